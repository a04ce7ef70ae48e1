"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each one.

This is the evidence that the pins are strong enough: a dropped term, a wrong sign or index, a
swapped operand or a wrong order anywhere in the oracle must make at least one check fail.
"""
import numpy as np
import pytest

import oracle.attention as A
import oracle.cache as C
import oracle.rope as R
import oracle_pins as pins


def _rope_sign_flip(x, pos, theta):
    return R.__dict__["_orig_rope"](x, -np.asarray(pos), theta)


def _rope_interleaved(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * R.inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty(np.broadcast_shapes(x.shape, c.shape[:-1] + (D,)))
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return out


def _inv_freq_half_exponent(head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -1.0 * i / head_dim)


def _view_others_descending(self, p, w):
    order = list(self.common[p]) + [self.live[p][u] for u in reversed(range(self.W)) if u != w] + \
        [self.live[p][w]]
    return _entries(self, order)


def _view_own_first(self, p, w):
    order = list(self.common[p]) + [self.live[p][w]] + \
        [self.live[p][u] for u in range(self.W) if u != w]
    return _entries(self, order)


def _entries(self, order, shift=0, iq_shift=0):
    entries, off = [], 0
    for sid in order:
        n = self.segments[sid].visible
        if n:
            entries.append((sid, off + shift, n))
            off += n
    return entries, off - 1 + iq_shift


def _view_offsets_shifted(self, p, w):
    order = list(self.common[p]) + [self.live[p][u] for u in range(self.W) if u != w] + \
        [self.live[p][w]]
    return _entries(self, order, shift=1)


def _view_iq_off_by_one(self, p, w):
    order = list(self.common[p]) + [self.live[p][u] for u in range(self.W) if u != w] + \
        [self.live[p][w]]
    return _entries(self, order, iq_shift=1)


def _partial_no_scale(stored_k, v, q_rot, scale):
    return A.__dict__["_orig_partial"](stored_k, v, q_rot, 1.0)


def _partial_transposed_value(stored_k, v, q_rot, scale):
    # uses the keys where the values belong
    return A.__dict__["_orig_partial"](stored_k, stored_k, q_rot, scale)


def _merge_drop_rescale(parts):
    M = np.max(np.stack([m for m, _, _ in parts]), axis=0)
    L = sum(l for m, l, _ in parts)                          # forgot exp(m - M)
    O = sum(o * np.exp(m - M)[:, None] for m, _, o in parts)
    return O / L[:, None], M + np.log(L)


def _allocate_lifo(self, n_new):
    self.free = type(self.free)(reversed(self.free))
    try:
        return C.HogwildCache.__dict__["_orig_allocate"](self, n_new)
    finally:
        self.free = type(self.free)(reversed(self.free))


def _step_end_commit_descending(self, finished):
    finished = np.asarray(finished, dtype=np.uint8).reshape(self.P, self.W)
    for seg in self.segments:
        seg.length += seg.pending
        seg.pending = 0
    self.step_pending = None
    self.appended_layers = set()
    for p in range(self.P):
        for w in reversed(range(self.W)):
            if finished[p, w] and self.segments[self.live[p][w]].length > 0:
                self.common[p].append(self.live[p][w])
                self.live[p][w] = self._new_segment(p, w)


def _view_layout_ignored(self, p, w):
    saved = self.layout
    self.layout = "combined"
    try:
        return _orig_view(self, p, w)
    finally:
        self.layout = saved


def _view_step_wise_shows_others(self, p, w):
    saved = self.layout
    if saved == "step_wise":
        self.layout = "combined"
    try:
        return _orig_view(self, p, w)
    finally:
        self.layout = saved


def _view_contiguous_own_first(self, p, w):
    entries, i_q = _orig_view(self, p, w)
    if self.layout != "contiguous" or len(entries) < 3:
        return entries, i_q
    own = [e for e in entries if self.segments[e[0]].origin == w]
    rest = [e for e in entries if self.segments[e[0]].origin != w]
    out, off = [], 0
    for sid, _, n in rest[:1] + own + rest[1:]:
        out.append((sid, off, n))
        off += n
    return out, i_q


_orig_view = C.HogwildCache.view


def _merged_positions_local(segments):
    return np.concatenate([np.arange(s.length) for s in segments] or [np.zeros(0, int)])


def _own_visible_one_more(n, back):
    return min(n, n - back + 1)


def _query_position_unshifted(i_q, back):
    return i_q

def _entry_spans_live_descending(cache, p):
    first, n = {}, 0
    for sid in list(cache.common[p]) + list(reversed(cache.live[p])):
        first[sid] = n
        n += cache.segments[sid].visible
    return first, n


def _selected_end_inclusive(first_entry, n, begin, end):
    a = min(max(begin - first_entry, 0), n)
    b = min(max(end + 1 - first_entry, 0), n)
    return a, max(a, b)


def _merge_parts_unweighted(outs, lses):
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    return outs.mean(axis=0), np.log(np.exp(lses).sum(axis=0))


def _method_range_rotated_from_range_start(cache, layer, q, ranges):
    """method_range with each segment's query rotated from the first selected token."""
    import math
    P, W, Hq, D = np.asarray(q).shape
    q = np.asarray(q, dtype=np.float64)
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((P, W, Hq, D))
    lse = np.full((P, W, Hq), -np.inf)
    for p in range(P):
        first, _ = A.entry_spans(cache, p)
        begin, end = ranges[p]
        for w in range(W):
            entries, i_q = cache.view(p, w)
            parts = {h: [] for h in range(cache.H_kv)}
            for sid, off, n in entries:
                a, b = A.selected(first[sid], n, begin, end)
                if a == b:
                    continue
                seg = cache.segments[sid]
                q_rot = A.rope(q[p, w], i_q - off - a, cache.theta)
                for kh in range(cache.H_kv):
                    parts[kh].append(A.segment_partial(seg.stored_k(layer)[a:b, kh, :],
                                                       seg.raw_v(layer)[a:b, kh, :],
                                                       q_rot[kh * G:(kh + 1) * G], scale))
            if not parts[0]:
                continue
            for kh in range(cache.H_kv):
                o, l = A.lse_merge(parts[kh])
                out[p, w, kh * G:(kh + 1) * G] = o
                lse[p, w, kh * G:(kh + 1) * G] = l
    return out, lse


MUTATIONS = {
    "entry_numbering_live_descending": [(A, "entry_spans", _entry_spans_live_descending)],
    "range_end_inclusive": [(A, "selected", _selected_end_inclusive)],
    "merge_parts_unweighted": [(A, "merge_parts", _merge_parts_unweighted)],
    "range_query_rotated_from_range_start": [(A, "method_range",
                                              _method_range_rotated_from_range_start)],
    "rope_rotates_backwards": [(R, "rope", _rope_sign_flip), (A, "rope", _rope_sign_flip),
                               (C, "rope", _rope_sign_flip)],
    "rope_interleaved_pairs": [(R, "rope", _rope_interleaved), (A, "rope", _rope_interleaved),
                               (C, "rope", _rope_interleaved)],
    "inv_freq_wrong_exponent": [(R, "inv_freq", _inv_freq_half_exponent)],
    "others_in_descending_id": [(C.HogwildCache, "view", _view_others_descending)],
    "own_block_not_last": [(C.HogwildCache, "view", _view_own_first)],
    "view_offset_off_by_one": [(C.HogwildCache, "view", _view_offsets_shifted)],
    "query_position_off_by_one": [(C.HogwildCache, "view", _view_iq_off_by_one)],
    "score_scale_dropped": [(A, "segment_partial", _partial_no_scale)],
    "keys_used_as_values": [(A, "segment_partial", _partial_transposed_value)],
    "merge_forgets_rescale": [(A, "lse_merge", _merge_drop_rescale)],
    "pages_popped_lifo": [(C.HogwildCache, "_allocate", _allocate_lifo)],
    "commits_in_descending_id": [(C.HogwildCache, "step_end", _step_end_commit_descending)],
    "layout_ignored": [(C.HogwildCache, "view", _view_layout_ignored)],
    "causal_cut_off_by_one": [(A, "own_visible", _own_visible_one_more)],
    "compaction_keeps_block_local_positions": [(C, "merged_positions", _merged_positions_local)],
    "chunk_queries_share_one_position": [(A, "query_position", _query_position_unshifted)],
    "step_wise_shows_others": [(C.HogwildCache, "view", _view_step_wise_shows_others)],
    "contiguous_own_output_first": [(C.HogwildCache, "view", _view_contiguous_own_first)],
}


def _failing_checks():
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check()
        except (AssertionError, C.CacheError, ValueError, IndexError, FloatingPointError):
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    R.__dict__.setdefault("_orig_rope", R.rope)
    A.__dict__.setdefault("_orig_partial", A.segment_partial)
    if "_orig_allocate" not in C.HogwildCache.__dict__:
        C.HogwildCache._orig_allocate = C.HogwildCache._allocate
    for obj, attr, repl in MUTATIONS[name]:
        monkeypatch.setattr(obj, attr, repl)
    with np.errstate(all="ignore"):
        failed = _failing_checks()
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_unmutated_oracle_passes_every_pin():
    assert _failing_checks() == []
