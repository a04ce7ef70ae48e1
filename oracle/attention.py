"""Concurrent attention in fp64, two independent ways (oracle; test infrastructure only).

Both compute, for every problem p, worker w and query head h, softmax attention of the worker's
query over every token of its view (Hogwild! Inference summary, gentlecold.top, sections 4-5
and 9), with score scale 1/sqrt(D), GQA head h -> KV head floor(h / G), no other mask:

* ``brute_force`` is the plain definition: lay the view's raw keys out at positions 0 .. n-1,
  rotate each key at its view position, rotate the query at i_q, and run an ordinary softmax.
  This is the "re-encode every token at its new position" formulation the summary calls too
  costly for real use (section 4) -- exactly what makes it a good check.
* ``method`` is the summary's section-5 identity: keys stay rotated at block-local positions,
  and for each block of the view the query is rotated once by (i_q - the block's view offset);
  per-block softmax partials (max, sum, weighted values) are then merged by log-sum-exp, the
  "aggregate in the softmax weighting" / "partial result reduction" of sections 5 and 9.

Returned ``lse`` is the natural-log log-sum-exp of the scaled scores (-inf for an empty view).

Several query tokens per worker (``*_mq``; the paragraph header a worker prefills after a
commit, section 8 step 4, or any chunk of tokens a worker appends in one step): the queries of
worker w are the last n_q[p][w] tokens of its own block, in order.  Query token t sits at view
position i_q - (n_q - 1 - t) and attends causally -- to every token of the view up to and
including its own position.  The own block is last in every view (section 6), so only its
newest tokens are ever masked, and the other workers' tokens of the same step stay visible
(the inference flow appends every worker's tokens before any attention).
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np

from .cache import HogwildCache
from .rope import rope


def _check_q(cache: HogwildCache, q: np.ndarray, num_q_heads: int) -> np.ndarray:
    q = np.asarray(q, dtype=np.float64)
    if q.shape != (cache.P, cache.W, num_q_heads, cache.D):
        raise ValueError("q must be [P][W][H_q][D]")
    if num_q_heads % cache.H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    return q


def brute_force(cache: HogwildCache, layer: int, q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Re-rotate every raw key at its full view position; plain softmax attention."""
    P, W, Hq, D = np.asarray(q).shape
    q = _check_q(cache, q, Hq)
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((P, W, Hq, D))
    lse = np.full((P, W, Hq), -np.inf)
    for p in range(P):
        for w in range(W):
            entries, i_q = cache.view(p, w)
            if not entries:
                continue
            kr = np.concatenate([cache.segments[s].raw_k(layer)[:n] for s, _, n in entries])
            vr = np.concatenate([cache.segments[s].raw_v(layer)[:n] for s, _, n in entries])
            pos = np.arange(kr.shape[0])
            k = rope(kr, pos[:, None], cache.theta)              # [n][H_kv][D]
            qr = rope(q[p, w], i_q, cache.theta)                  # [H_q][D]
            for h in range(Hq):
                s = (k[:, h // G, :] @ qr[h]) * scale
                m = s.max()
                e = np.exp(s - m)
                out[p, w, h] = (e @ vr[:, h // G, :]) / e.sum()
                lse[p, w, h] = m + math.log(e.sum())
    return out, lse


def segment_partial(stored_k: np.ndarray, v: np.ndarray, q_rot: np.ndarray, scale: float):
    """Softmax partial of one block for a group of query rows sharing one KV head.

    stored_k, v: [n][D]; q_rot: [rows][D].  Returns (m [rows], l [rows], o [rows][D]) with
    m = max score, l = sum exp(score - m), o = sum exp(score - m) v (unnormalised).
    """
    s = (q_rot @ stored_k.T) * scale                 # [rows][n]
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    return m, e.sum(axis=1), e @ v


def lse_merge(parts):
    """Merge softmax partials [(m, l, o)] into (out, lse) by log-sum-exp."""
    M = np.max(np.stack([m for m, _, _ in parts]), axis=0)
    L = sum(l * np.exp(m - M) for m, l, _ in parts)
    O = sum(o * np.exp(m - M)[:, None] for m, _, o in parts)
    return O / L[:, None], M + np.log(L)


def method(cache: HogwildCache, layer: int, q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Keys at block-local positions, one query rotation per (worker, block), LSE merge."""
    P, W, Hq, D = np.asarray(q).shape
    q = _check_q(cache, q, Hq)
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((P, W, Hq, D))
    lse = np.full((P, W, Hq), -np.inf)
    for p in range(P):
        for w in range(W):
            entries, i_q = cache.view(p, w)
            if not entries:
                continue
            parts = {h: [] for h in range(cache.H_kv)}
            for sid, off, n in entries:
                seg = cache.segments[sid]
                ks = seg.stored_k(layer)[:n]
                vs = seg.raw_v(layer)[:n]
                q_rot = rope(q[p, w], i_q - off, cache.theta)      # rotate by (i_q - offset)
                for kh in range(cache.H_kv):
                    parts[kh].append(segment_partial(ks[:, kh, :], vs[:, kh, :],
                                                     q_rot[kh * G:(kh + 1) * G], scale))
            for kh in range(cache.H_kv):
                o, l = lse_merge(parts[kh])
                out[p, w, kh * G:(kh + 1) * G] = o
                lse[p, w, kh * G:(kh + 1) * G] = l
    return out, lse


# ------------------------------------------------------------------ several queries per worker


def _mq_rows(cache: HogwildCache, n_q):
    """(p, w, t, back) of every query row in order (problem, worker, token); back = n_q-1-t."""
    n_q = np.asarray(n_q, dtype=np.int64).reshape(cache.P, cache.W)
    rows = []
    for p in range(cache.P):
        for w in range(cache.W):
            nq = int(n_q[p, w])
            if nq < 0:
                raise ValueError("negative query count")
            if nq == 0:
                continue
            entries, _ = cache.view(p, w)
            own = cache.live[p][w]
            if not entries or entries[-1][0] != own or entries[-1][2] < nq:
                raise ValueError("a worker's queries must be tokens of its own block")
            rows += [(p, w, t, nq - 1 - t) for t in range(nq)]
    return rows


def _check_q_mq(cache, q, rows):
    q = np.asarray(q, dtype=np.float64)
    if q.ndim != 3 or q.shape[0] != len(rows) or q.shape[2] != cache.D or q.shape[1] % cache.H_kv:
        raise ValueError("q must be [sum n_q][H_q][D]")
    return q


def brute_force_mq(cache: HogwildCache, layer: int, q: np.ndarray, n_q):
    """Causal textbook attention: view keys re-rotated at positions 0 .. n-1, each query token
    rotated at its own position and masked to the positions up to it."""
    rows = _mq_rows(cache, n_q)
    q = _check_q_mq(cache, q, rows)
    Hq, D = q.shape[1], q.shape[2]
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros(q.shape)
    lse = np.full(q.shape[:2], -np.inf)
    for i, (p, w, t, back) in enumerate(rows):
        entries, i_q = cache.view(p, w)
        pos = i_q - back
        kr = np.concatenate([cache.segments[s].raw_k(layer)[:n] for s, _, n in entries])[:pos + 1]
        vr = np.concatenate([cache.segments[s].raw_v(layer)[:n] for s, _, n in entries])[:pos + 1]
        k = rope(kr, np.arange(pos + 1)[:, None], cache.theta)
        qr = rope(q[i], pos, cache.theta)
        for h in range(Hq):
            sc = (k[:, h // G, :] @ qr[h]) * scale
            m = sc.max()
            e = np.exp(sc - m)
            out[i, h] = (e @ vr[:, h // G, :]) / e.sum()
            lse[i, h] = m + math.log(e.sum())
    return out, lse


def query_position(i_q: int, back: int) -> int:
    """View position of a query token that has ``back`` newer query tokens after it."""
    return i_q - back


def own_visible(n: int, back: int) -> int:
    """Tokens of the own block (n visible) that a query with ``back`` newer tokens may see."""
    return n - back


def method_mq(cache: HogwildCache, layer: int, q: np.ndarray, n_q):
    """The method with several causal query tokens per worker: token t is rotated once per
    block by (its position - the block's view offset); the own block contributes only its
    tokens up to the query's own; partials merged by log-sum-exp."""
    rows = _mq_rows(cache, n_q)
    q = _check_q_mq(cache, q, rows)
    Hq, D = q.shape[1], q.shape[2]
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros(q.shape)
    lse = np.full(q.shape[:2], -np.inf)
    for i, (p, w, t, back) in enumerate(rows):
        entries, i_q = cache.view(p, w)
        own = cache.live[p][w]
        pos = query_position(i_q, back)
        parts = {h: [] for h in range(cache.H_kv)}
        for sid, off, n in entries:
            nv = own_visible(n, back) if sid == own else n      # causal cut in the own block
            seg = cache.segments[sid]
            q_rot = rope(q[i], pos - off, cache.theta)
            for kh in range(cache.H_kv):
                parts[kh].append(segment_partial(seg.stored_k(layer)[:nv, kh, :],
                                                 seg.raw_v(layer)[:nv, kh, :],
                                                 q_rot[kh * G:(kh + 1) * G], scale))
        for kh in range(cache.H_kv):
            o, l = lse_merge(parts[kh])
            out[i, kh * G:(kh + 1) * G] = o
            lse[i, kh * G:(kh + 1) * G] = l
    return out, lse


# ------------------------------------------------------------------ split over KV entries
#
# The work of one decode step can be split over KV entries and the partial results reduced
# afterwards (summary section 9: the kernel is balanced by KV entries, then the partial results
# are reduced) -- also across GPUs, each taking a range of the entries.  The entries of a
# problem are numbered in segment order: the common segments in commit order, then the
# workers' current blocks in ascending id.  Every view holds whole segments of that list in its
# own order, so an entry's number does not depend on the worker; a worker attends to the
# selected entries of its view, each still at its position in the worker's view.


def entry_spans(cache: HogwildCache, p: int):
    """Problem p's entry numbering: {segment id: number of its first token} and the total."""
    first, n = {}, 0
    for sid in list(cache.common[p]) + list(cache.live[p]):
        first[sid] = n
        n += cache.segments[sid].visible
    return first, n


def selected(first_entry: int, n: int, begin: int, end: int):
    """Block-local tokens [a, b) of a segment holding entries [first_entry, first_entry + n)
    that lie in the entry range [begin, end) (a == b when none do)."""
    a = min(max(begin - first_entry, 0), n)
    b = min(max(end - first_entry, 0), n)
    return a, max(a, b)


def brute_force_range(cache: HogwildCache, layer: int, q: np.ndarray, ranges):
    """Plain definition of the attention over selected entries: worker w's view laid out with
    every raw key rotated at its view position, and softmax attention of rho(q, i_q) over the
    keys whose entry number lies in ranges[p] = (begin, end) only.  Returns (out, lse); a worker
    that selects no key gets out = 0 and lse = -inf."""
    P, W, Hq, D = np.asarray(q).shape
    q = _check_q(cache, q, Hq)
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((P, W, Hq, D))
    lse = np.full((P, W, Hq), -np.inf)
    for p in range(P):
        first, _ = entry_spans(cache, p)
        begin, end = (int(x) for x in ranges[p])
        for w in range(W):
            entries, i_q = cache.view(p, w)
            if not entries:
                continue
            kr = np.concatenate([cache.segments[s].raw_k(layer)[:n] for s, _, n in entries])
            vr = np.concatenate([cache.segments[s].raw_v(layer)[:n] for s, _, n in entries])
            number = np.concatenate([first[s] + np.arange(n) for s, _, n in entries])
            keep = (number >= begin) & (number < end)
            if not keep.any():
                continue
            pos = np.arange(kr.shape[0])
            k = rope(kr, pos[:, None], cache.theta)[keep]
            v = vr[keep]
            qr = rope(q[p, w], i_q, cache.theta)
            for h in range(Hq):
                s = (k[:, h // G, :] @ qr[h]) * scale
                m = s.max()
                e = np.exp(s - m)
                out[p, w, h] = (e @ v[:, h // G, :]) / e.sum()
                lse[p, w, h] = m + math.log(e.sum())
    return out, lse


def method_range(cache: HogwildCache, layer: int, q: np.ndarray, ranges):
    """The method over selected entries: for each segment of worker w's view, its tokens in the
    range, stored at block-local positions, attended with the query rotated once by
    (i_q - the segment's view offset); the per-segment partials merged by log-sum-exp."""
    P, W, Hq, D = np.asarray(q).shape
    q = _check_q(cache, q, Hq)
    G = Hq // cache.H_kv
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((P, W, Hq, D))
    lse = np.full((P, W, Hq), -np.inf)
    for p in range(P):
        first, _ = entry_spans(cache, p)
        begin, end = (int(x) for x in ranges[p])
        for w in range(W):
            entries, i_q = cache.view(p, w)
            parts = {h: [] for h in range(cache.H_kv)}
            for sid, off, n in entries:
                a, b = selected(first[sid], n, begin, end)
                if a == b:
                    continue
                seg = cache.segments[sid]
                q_rot = rope(q[p, w], i_q - off, cache.theta)
                for kh in range(cache.H_kv):
                    parts[kh].append(segment_partial(seg.stored_k(layer)[a:b, kh, :],
                                                     seg.raw_v(layer)[a:b, kh, :],
                                                     q_rot[kh * G:(kh + 1) * G], scale))
            if not parts[0]:
                continue
            for kh in range(cache.H_kv):
                o, l = lse_merge(parts[kh])
                out[p, w, kh * G:(kh + 1) * G] = o
                lse[p, w, kh * G:(kh + 1) * G] = l
    return out, lse


def merge_parts(outs, lses):
    """Merge normalised partial results of the same queries over disjoint sets of keys:
    LSE = log sum_i exp(lse_i), out = sum_i exp(lse_i - LSE) out_i (out = 0, LSE = -inf when
    every part is empty).  outs: [n][...][D], lses: [n][...] (natural log)."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    M = lses.max(axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    wts = np.where(np.isfinite(lses), np.exp(lses - Ms), 0.0)
    L = wts.sum(axis=0)
    out = np.where(finite[..., None], (wts[..., None] * outs).sum(axis=0) /
                   np.where(finite, L, 1.0)[..., None], 0.0)
    return out, np.where(finite, Ms + np.log(np.where(finite, L, 1.0)), -np.inf)
