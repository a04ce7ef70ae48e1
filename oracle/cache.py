"""The shared Hogwild! cache as a plain state machine (oracle; test infrastructure only).

What it models (Hogwild! Inference summary, gentlecold.top):

* section 9: the cache is a set of blocks -- one common block and one current block per
  worker -- each holding K/V of every layer at block-local positions 0 .. len-1;
* section 8 (inference flow): every worker appends its new token's K/V to its own block before
  any worker attends; when a worker finishes a reasoning step its block is moved to the end of
  the common history, the worker's current block is cleared and it starts a new one;
* sections 4 and 6: worker w sees the common history, then the other workers' current blocks,
  then its own current block last.

Readings where the pages are silent (each is also listed in the design notes):

* A "segment" is a block piece with one RoPE frame: the prompt, each committed paragraph, and
  each worker's current block.  A commit moves the worker's segment, unchanged, to the end of
  the common list; its positions stay block-local and the query rotation absorbs the new
  offset (the "RoPE offset correction" of section 8 done on the query side).  A commit of an
  empty block does nothing.
* Other workers' blocks appear in ascending worker id (the ocdem.com article, section 2.1);
  with two workers this gives the C+B+A / C+A+B views of section 4.
* ``n_new[p][0]`` tokens are appended to the last common segment, ``n_new[p][1 + w]`` to
  worker w's current block.  All layers of a step append the same counts; the lengths advance
  at ``step_end``; attention in the step sees the appended tokens.
* Pages are handed out FIFO from a free list initialised from ``page_order``, visiting problems
  in order, then the common block, then workers in ascending id, each in position order, one
  new page whenever a block-local position is a multiple of the page size (for a contiguous
  cache: one page, of the block's capacity, at position 0).  Pages are never freed.
* Segment ids count up in creation order: per problem the prompt segment then workers
  0 .. W-1 at creation; then each fresh block started by a commit, in commit order.

Cache layouts (section 6 compares three; section 10 adds the no-sync baseline of its
collaboration scores).  The blocks, commits and pages are the same in all of them; only the
order and the membership of a worker's view change:

* ``combined`` (token-wise, the main method): common history, then the other workers' current
  blocks, then the own current block -- as above.
* ``step_wise`` (interleaved): only finished steps are shared -- the common history, then the
  own current block; other workers' unfinished blocks are not visible.
* ``contiguous``: each worker's output is one contiguous run -- the prompt, then every other
  worker's whole output (its committed paragraphs in commit order, then its current block),
  in ascending id, then the worker's own whole output.
* ``no_sync``: workers generate independently -- the prompt, the worker's own committed
  paragraphs in commit order, then its own current block.
In ``contiguous`` and ``no_sync`` a committed paragraph belongs to the worker that wrote it
(its segment's origin); tokens appended to the last common segment belong to that segment.

The stored keys are the raw keys rotated to their block-local positions in fp64
(``rope(k, j)``); the brute-force attention uses the raw keys instead.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from .rope import rope


class CacheError(Exception):
    """Base class; ``kind`` names the library status the same misuse must produce."""

    kind = "invalid_arg"


class InvalidArg(CacheError):
    kind = "invalid_arg"


class OutOfPages(CacheError):
    kind = "out_of_pages"


class Capacity(CacheError):
    kind = "capacity"


class Segment:
    def __init__(self, sid: int, problem: int, origin: int, num_layers: int):
        self.id = sid
        self.problem = problem
        self.origin = origin          # -1 for the prompt segment, else the worker that wrote it
        self.length = 0               # committed tokens
        self.pending = 0              # tokens appended in the current step
        self.pages: List[int] = []
        self._raw_k = [[] for _ in range(num_layers)]
        self._raw_v = [[] for _ in range(num_layers)]
        self._stored_k = [[] for _ in range(num_layers)]
        self._cat: Dict[Tuple[str, int], np.ndarray] = {}

    @property
    def visible(self) -> int:
        return self.length + self.pending

    def _get(self, which: str, layer: int) -> np.ndarray:
        key = (which, layer)
        lst = {"k": self._raw_k, "v": self._raw_v, "ks": self._stored_k}[which][layer]
        n = sum(a.shape[0] for a in lst)
        c = self._cat.get(key)
        if c is None or c.shape[0] != n:
            c = np.concatenate(lst) if lst else None
            if len(lst) > 1:
                lst[:] = [c]
            self._cat[key] = c
        return c

    def raw_k(self, layer):
        return self._get("k", layer)

    def raw_v(self, layer):
        return self._get("v", layer)

    def stored_k(self, layer):
        return self._get("ks", layer)


LAYOUTS = ("combined", "step_wise", "contiguous", "no_sync")


def merged_positions(segments) -> np.ndarray:
    """Position of every token of ``segments`` (in order) in the segment they merge into."""
    return np.arange(sum(s.length for s in segments))


class HogwildCache:
    def __init__(self, num_problems: int, num_workers: int, num_layers: int, num_kv_heads: int,
                 head_dim: int, rope_theta: float, page_size: int, num_pages: int,
                 contiguous: bool = False, page_order: Optional[Sequence[int]] = None,
                 layout: str = "combined"):
        if layout not in LAYOUTS:
            raise InvalidArg("unknown cache layout")
        self.layout = layout
        self.P, self.W, self.L = num_problems, num_workers, num_layers
        self.H_kv, self.D, self.theta = num_kv_heads, head_dim, float(rope_theta)
        self.S, self.contiguous = page_size, bool(contiguous)
        order = list(range(num_pages)) if page_order is None else [int(x) for x in page_order]
        self.free = deque(order)
        self.segments: List[Segment] = []
        self.common: List[List[int]] = []
        self.live: List[List[int]] = []
        for p in range(self.P):
            self.common.append([self._new_segment(p, -1)])
            self.live.append([self._new_segment(p, w) for w in range(self.W)])
        self.step_pending: Optional[np.ndarray] = None
        self.appended_layers = set()

    # -- structure -----------------------------------------------------------------------

    def _new_segment(self, problem: int, origin: int) -> int:
        seg = Segment(len(self.segments), problem, origin, self.L)
        self.segments.append(seg)
        return seg.id

    def block_segment(self, p: int, b: int) -> Segment:
        """Block b of problem p: 0 = last common segment, 1 + w = worker w's current block."""
        return self.segments[self.common[p][-1] if b == 0 else self.live[p][b - 1]]

    def view(self, p: int, w: int) -> Tuple[List[Tuple[int, int, int]], int]:
        """Worker w's view: [(segment id, view offset, visible length)], and i_q.

        Order (combined layout): common segments in commit order, other workers' current
        blocks in ascending id, own block last; the other layouts are listed in the module
        docstring.  Empty segments are skipped.  i_q = view length - 1 (the query is the last
        token of the worker's own block once this step's token is appended).
        """
        common, live = self.common[p], self.live[p]
        others = [u for u in range(self.W) if u != w]
        if self.layout == "combined":
            order = list(common) + [live[u] for u in others] + [live[w]]
        elif self.layout == "step_wise":
            order = list(common) + [live[w]]
        else:
            def output(u):          # worker u's committed paragraphs, then its current block
                return [s for s in common if self.segments[s].origin == u] + [live[u]]
            order = [s for s in common if self.segments[s].origin == -1]
            if self.layout == "contiguous":
                for u in others:
                    order += output(u)
            order += output(w)
        entries, off = [], 0
        for sid in order:
            n = self.segments[sid].visible
            if n == 0:
                continue
            entries.append((sid, off, n))
            off += n
        return entries, off - 1

    # -- the step protocol ---------------------------------------------------------------

    def append(self, layer: int, n_new, k_raw, v_raw) -> None:
        """Append raw K/V of ``layer``; tokens ordered problem-major, then block 0 .. W."""
        if not (0 <= layer < self.L):
            raise InvalidArg("layer out of range")
        n_new = np.asarray(n_new, dtype=np.int64).reshape(self.P, self.W + 1)
        if (n_new < 0).any():
            raise InvalidArg("negative token count")
        total = int(n_new.sum())
        k_raw = np.asarray(k_raw)
        v_raw = np.asarray(v_raw)
        if k_raw.shape != (total, self.H_kv, self.D) or v_raw.shape != k_raw.shape:
            raise InvalidArg("k/v shape does not match n_new")
        if self.step_pending is None:
            self._allocate(n_new)
            self.step_pending = n_new.copy()
        else:
            if not np.array_equal(self.step_pending, n_new):
                raise InvalidArg("every layer of a step must append the same token counts")
            if layer in self.appended_layers:
                raise InvalidArg("layer already appended in this step")
        self.appended_layers.add(layer)
        i = 0
        for p in range(self.P):
            for b in range(self.W + 1):
                n = int(n_new[p, b])
                if n == 0:
                    continue
                seg = self.block_segment(p, b)
                j0 = self._layer_len(seg, layer)      # equals seg.length: one append per step
                kr = np.asarray(k_raw[i:i + n], dtype=np.float64)
                vr = np.asarray(v_raw[i:i + n], dtype=np.float64)
                seg._raw_k[layer].append(kr)
                seg._raw_v[layer].append(vr)
                pos = np.arange(j0, j0 + n, dtype=np.int64)[:, None]
                seg._stored_k[layer].append(rope(kr, pos, self.theta))
                i += n

    @staticmethod
    def _layer_len(seg: Segment, layer: int) -> int:
        return sum(a.shape[0] for a in seg._raw_k[layer])

    def _allocate(self, n_new: np.ndarray) -> None:
        need: List[Tuple[Segment, int]] = []
        for p in range(self.P):
            for b in range(self.W + 1):
                n = int(n_new[p, b])
                if n == 0:
                    continue
                seg = self.block_segment(p, b)
                j0 = seg.length
                if self.contiguous:
                    if j0 + n > self.S:
                        raise Capacity("block capacity exceeded")
                    if j0 == 0:
                        need.append((seg, 1))
                else:
                    first = -(-j0 // self.S)               # first page index starting at or after j0
                    last = (j0 + n - 1) // self.S          # page index of the last new token
                    cnt = max(0, last - first + 1)
                    if cnt:
                        need.append((seg, cnt))
        if sum(c for _, c in need) > len(self.free):
            raise OutOfPages("page pool exhausted")
        for seg, c in need:
            for _ in range(c):
                seg.pages.append(self.free.popleft())
        for p in range(self.P):
            for b in range(self.W + 1):
                n = int(n_new[p, b])
                if n:
                    self.block_segment(p, b).pending = n

    def step_end(self, finished) -> None:
        """Advance lengths, then commit finished workers' blocks in ascending worker id."""
        finished = np.asarray(finished, dtype=np.uint8).reshape(self.P, self.W)
        if self.step_pending is not None and len(self.appended_layers) != self.L:
            raise InvalidArg("step_end before every layer was appended")
        for seg in self.segments:
            seg.length += seg.pending
            seg.pending = 0
        self.step_pending = None
        self.appended_layers = set()
        for p in range(self.P):
            for w in range(self.W):
                if finished[p, w] and self.segments[self.live[p][w]].length > 0:
                    self.common[p].append(self.live[p][w])
                    self.live[p][w] = self._new_segment(p, w)

    def compact(self, p: int, first: int, count: int) -> int:
        """Merge common segments first .. first+count-1 of problem p into one segment with one
        RoPE frame (reading 1 of section 8's "correct by RoPE offset": the moved block's keys are
        re-rotated to their positions in the common history, here relative to the merged
        segment's start).  Returns the new segment id.

        Readings (the pages name the correction, not its bookkeeping):
        * only between steps, on committed (common) segments, in commit order; count >= 2;
        * the merged segment is written into fresh pages taken FIFO from the free list (one per
          S positions; a contiguous cache takes one page and the merge must fit its capacity);
          the old segments' pages then go back to the end of the free list, segment by segment
          in commit order, each in its page order; the old segments stay in the table, empty;
        * the merged segment's writer is the segments' common origin, or -1 (shared history)
          when they differ -- which the contiguous and no-sync layouts, whose views depend on
          the writer, refuse;
        * keys: the token at merged position j is stored rotated at j (the fp64 oracle re-rotates
          from the raw key); values unchanged.  Views are unchanged: the merged segment takes the
          span the old ones had, so every attention output stays the same.
        """
        if self.step_pending is not None:
            raise InvalidArg("compaction between steps only")
        common = self.common[p]
        if count < 2 or first < 0 or first + count > len(common):
            raise InvalidArg("bad segment range")
        olds = [self.segments[sid] for sid in common[first:first + count]]
        origins = {s.origin for s in olds}
        origin = next(iter(origins)) if len(origins) == 1 else -1
        if len(origins) > 1 and self.layout in ("contiguous", "no_sync"):
            raise InvalidArg("the layout's views depend on the writer")
        total = sum(s.length for s in olds)
        if self.contiguous:
            if total > self.S:
                raise Capacity("block capacity exceeded")
            need = 1 if total else 0
        else:
            need = -(-total // self.S)
        if need > len(self.free):
            raise OutOfPages("page pool exhausted")
        new = Segment(len(self.segments), p, origin, self.L)
        self.segments.append(new)
        new.pages = [self.free.popleft() for _ in range(need)]
        new.length = total
        for layer in range(self.L):
            kr = [s.raw_k(layer) for s in olds if s.length]
            vr = [s.raw_v(layer) for s in olds if s.length]
            if kr:
                k = np.concatenate(kr)
                new._raw_k[layer] = [k]
                new._raw_v[layer] = [np.concatenate(vr)]
                new._stored_k[layer] = [rope(k, merged_positions(olds)[:, None], self.theta)]
        for s in olds:
            self.free.extend(s.pages)
            s.pages = []
            s.length = 0
            for lst in (s._raw_k, s._raw_v, s._stored_k):
                for layer in range(self.L):
                    lst[layer] = []
            s._cat.clear()
        common[first:first + count] = [new.id]
        return new.id

    # -- exports for bit-exact comparison ------------------------------------------------

    def tables(self) -> dict:
        return {
            "segments": [(s.problem, s.origin, s.length, s.pending, list(s.pages))
                         for s in self.segments],
            "common": [list(c) for c in self.common],
            "live": [list(l) for l in self.live],
            "free_count": len(self.free),
        }

    def slot_of(self, sid: int, j: int) -> Tuple[int, int]:
        """(physical page, slot) of block-local position j of segment sid."""
        seg = self.segments[sid]
        if self.contiguous:
            return seg.pages[0], j
        return seg.pages[j // self.S], j % self.S
