// K2 (CUDA-core form) -- concurrent attention with per-(worker, block) query rotation for fewer
// than 16 query rows per KV head; the per-unit partial results are merged by K3 (merge.cu).
//
// Method (Hogwild! Inference summary, gentlecold.top): keys are stored rotated at block-local
// positions; for a block at offset o in worker w's view the query is rotated by (i_q - o)
// (section 5), so one KV tile serves every worker and every query head of its GQA group, each
// with its own rotated query.  Work is split over KV entries, not over blocks, and the partial
// results are reduced afterwards (section 9, Flash-Decoding style kernel).
//
// One CTA per unit (a run of pieces of one (problem, KV head)), 8 warps.  Each piece's K and V
// tiles (128 rows x D bf16 from the pool, the same 128-byte-swizzled TMA boxes the tensor-core
// kernel loads) are staged once into a ring of one or two slots in shared memory, completion
// on an mbarrier, and kept in bf16; the rotated, pre-scaled queries (log2(e)/sqrt(D)) and the
// running output O of every row stay in shared memory in fp32.  Per tile and per chunk of 16
// query rows, warp w takes rows 2w and 2w + 1 in both passes: S = Q~ K^T and the online softmax
// (running max and sum, rescale factor) with a lane per (half of the dims, 8 tokens) of both
// rows, the halves swapping partial sums and a row's 16 lanes reducing by shuffles; then
// O = alpha O + P V with a lane per (half of the tokens, 8 columns) of both rows, the halves
// again swapping partial sums (D = 64: a lane per 4 columns of both rows over all the tokens).
// So every K or V chunk read from shared memory feeds two rows.
// In a decode step the CTA first writes its unit's appended
// tokens itself (fused append).  Every wait is bounded (about a second): one that runs out records
// ERR_TIMEOUT, and the CTA waits (bounded by the clock) for its copies in flight, then writes
// empty partials.  The kernel is launched as a programmatic dependent: it waits for the grid
// it follows (which may write the queries or this step's tokens) before it reads anything.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hw_device.cuh"
#include "tc_ptx.cuh"

#include <algorithm>

namespace hw {
namespace {

using tc::fence_mbar_init;
using tc::fence_proxy_async_global;
using tc::fence_proxy_async_smem;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mbar_wait_drain;
using tc::smem_u32;
using tc::tma_load_2d;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 128;            // tokens per tile (one TMA box of rows)
constexpr int kChunkRows = 16;        // query rows per pass over a tile, at most
constexpr int kSStride = kTile + 4;   // floats per row of P (padded: two rows' stores share no bank)
constexpr uint64_t kWaitNs = 1000000000ull;

template <int D>
struct FmaCfg {
  static constexpr int kHalves = D / 64;                       // 128-byte swizzle atoms per row
  static constexpr uint32_t kHalfBytes = kTile * 128;          // one {64, 128} TMA box
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes; // K or V tile
  static constexpr uint32_t kSlotBytes = 2 * kTileBytes;       // K then V
};

// Shared-memory layout for R query rows and `slots` ring slots (offsets from a 1024-byte
// aligned base): ring, Q~ [R][D] f32, O [R][D] f32, P [16][132] f32, M/L/alpha [R] f32, row
// cut [R] i32, barriers, flags.
template <int D>
struct FmaLayout {
  uint32_t q, o, s, m, l, al, cut, bars, flags, total;
  __host__ __device__ FmaLayout(int R, int slots) {
    uint32_t off = (uint32_t)slots * FmaCfg<D>::kSlotBytes;
    q = off;    off += (uint32_t)R * D * 4;
    o = off;    off += (uint32_t)R * D * 4;
    s = off;    off += kChunkRows * kSStride * 4;
    m = off;    off += (uint32_t)R * 4;
    l = off;    off += (uint32_t)R * 4;
    al = off;   off += (uint32_t)R * 4;
    cut = off;  off += (uint32_t)R * 4;
    off = (off + 7) / 8 * 8;
    bars = off; off += 8 * 2;
    flags = off; off += 16;
    total = off + 1024;                  // + alignment slack
  }
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// c + a * b on two fp32 lanes at once (packed FMA, each lane rounded as fma.rn.f32).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long ar, br, cr;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ar) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(br) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(cr) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(cr) : "l"(ar), "l"(br));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(cr));
  return r;
}

// Byte offset, inside a {64, 128} swizzled box pair, of the 16-byte chunk holding elements
// 8c .. 8c + 7 (c = d / 8) of tile row j.
template <int D>
__device__ __forceinline__ uint32_t swz(int j, int c) {
  return (uint32_t)(c >> 3) * FmaCfg<D>::kHalfBytes + (uint32_t)j * 128 +
         ((uint32_t)((c & 7) ^ (j & 7)) << 4);
}

__device__ __forceinline__ bool piece_ok(const AttnArgs& a, const Piece& pc) {
  return pc.page >= 0 && pc.page < a.num_pages && pc.slot0 >= 0 && pc.ntok >= 1 &&
         pc.ntok <= kTile && pc.slot0 + pc.ntok <= a.S && pc.seg_slot >= 0 &&
         pc.seg_slot < a.num_seg_slots;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fma_kernel(const AttnArgs a, const __grid_constant__ TcMaps maps, const int32_t layer,
                    const int32_t slots) {
  using C = FmaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int R = a.rows;
  const FmaLayout<D> L(R, slots);
  float* Qs = reinterpret_cast<float*>(smem + L.q);
  float* Os = reinterpret_cast<float*>(smem + L.o);
  float* Ss = reinterpret_cast<float*>(smem + L.s);
  float* Ms = reinterpret_cast<float*>(smem + L.m);
  float* Ls = reinterpret_cast<float*>(smem + L.l);
  float* As = reinterpret_cast<float*>(smem + L.al);
  int* cut = reinterpret_cast<int*>(smem + L.cut);     // tokens of the segment a row sees (-1: none)
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);   // [0] plan ok, [1] abort
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L.bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int PS = part_stride(D);

  // Set-up that touches no global memory: barriers, running output and row statistics.
  if (tid == 0) {
    for (int k = 0; k < slots; ++k) mbar_init(bars + 8u * k, 1);
    fence_mbar_init();
    flags[1] = 0;
  }
  for (int i = tid; i < R * D; i += kThreads) Os[i] = 0.f;
  for (int r = tid; r < R; r += kThreads) {
    Ms[r] = -CUDART_INF_F;
    Ls[r] = 0.f;
  }
  // Before the programmatic wait this kernel reads only what belongs to its plan (delivered on
  // the library's copy stream and checked through its sequence word, or copied before the
  // launch), the constant rotation table, and K/V tiles that the plan marks as written before
  // the grids this one may overlap; it writes nothing global but the error word.
  // The unit record is read while thread 0 checks that the plan has arrived: each of its three
  // 16-byte vectors carries the low 32 bits of the plan's sequence number, and a vector read
  // before the plan landed (its copy differs) is read again once the plan is confirmed.
  const int4* urec = reinterpret_cast<const int4*>(a.units + blockIdx.x);
  int4 uv[3] = {__ldcg(urec), __ldcg(urec + 1), __ldcg(urec + 2)};
  if (tid == 0) flags[0] = plan_arrived(a.gate, plan_seq_now(a.gate), a.err, KID_ATTN_FMA) ? 1 : 0;
  __syncthreads();
  const bool plan_ok = flags[0] != 0;
  Unit u{};
  Group g{};
  bool unit_ok = false;
  if (plan_ok) {
    static_assert(sizeof(Unit) == 48, "unit record: three 16-byte vectors");
    const uint32_t want = (uint32_t)a.gate.plan_expect;
    if ((uint32_t)uv[0].z != want) uv[0] = __ldcg(urec);
    if ((uint32_t)uv[1].w != want) uv[1] = __ldcg(urec + 1);
    if ((uint32_t)uv[2].z != want) uv[2] = __ldcg(urec + 2);
    int4* ud = reinterpret_cast<int4*>(&u);
    ud[0] = uv[0];
    ud[1] = uv[1];
    ud[2] = uv[2];
    // (problem, KV head) from the group index (groups are numbered p * H_kv + h): no dependent
    // load of the group record
    if (u.group >= 0 && u.group < a.num_groups) {
      g.p = u.group / a.H_kv;
      g.h = u.group % a.H_kv;
      unit_ok = g.p < a.P && u.piece_begin >= 0 && u.piece_begin <= u.piece_end;
    }
    if (!unit_ok && tid == 0) record_error(a.err, ERR_PLAN, KID_ATTN_FMA, blockIdx.x, 0);
  }
  const int pb = unit_ok ? u.piece_begin : 0, pe = unit_ok ? u.piece_end : 0;
  const int64_t page_base = (int64_t)layer * a.num_pages;   // first page of this layer's pool
  // This CTA writes the unit's appended tokens of its KV head itself (fused append).
  const bool fresh_here = unit_ok && a.k_raw != nullptr && u.fresh_end > u.fresh_begin;

  // Producer (thread 0): the first valid piece at or after `from`, its K and V tiles into ring
  // slot `slot` (pool rows ((page_base + page) * H_kv + h) * S + slot0 ..).  Returns the index
  // of the piece it loaded, -1 when none is left, or -2 - index for a piece with tokens of this
  // step while those may not be loaded yet (fresh_ok false: the fused append has not run).
  auto issue = [&](int from, int slot, bool fresh_ok) -> int {
    for (int pi = from; pi < pe; ++pi) {
      const Piece pc = a.pieces[pi];
      if (!piece_ok(a, pc)) continue;
      if (pc.fresh && !fresh_ok) return -2 - pi;
      const uint32_t dst = sbase + (uint32_t)slot * C::kSlotBytes;
      const int32_t y = (int32_t)(((page_base + pc.page) * a.H_kv + g.h) * a.S + pc.slot0);
      mbar_arrive_expect_tx(bars + 8u * slot, C::kSlotBytes);
#pragma unroll
      for (int hh = 0; hh < C::kHalves; ++hh) {
        tma_load_2d(dst + hh * C::kHalfBytes, &maps.k, 64 * hh, y, bars + 8u * slot,
                    tc::l2_policy_evict_first());
        tma_load_2d(dst + C::kTileBytes + hh * C::kHalfBytes, &maps.v, 64 * hh, y,
                    bars + 8u * slot, tc::l2_policy_evict_first());
      }
      return pi;
    }
    return -1;
  };
  int next_issue = pb;            // (thread 0) first piece not yet looked at
  uint32_t issued = 0;            // (thread 0) tiles issued
  auto fill_ring = [&](bool fresh_ok) {
    while (issued < (uint32_t)slots && next_issue < pe) {
      const int got = issue(next_issue, (int)issued, fresh_ok);
      if (got <= -2) {            // resumes there once the fused append is written
        next_issue = -2 - got;
        return;
      }
      next_issue = got < 0 ? pe : got + 1;
      if (got >= 0) ++issued;
    }
  };
  // The unit record names its first tile's pool position when that tile holds no token of
  // this step or of the step before (first_tok): it goes out now, before the programmatic wait,
  // without waiting for the piece record, which is checked against it afterwards.  The other
  // tiles go out after the wait (those with tokens this CTA appends, after the append).
  if (tid == 0 && pb < pe) {
    tc::tma_prefetch(&maps.k);
    tc::tma_prefetch(&maps.v);
    if (u.first_tok >= 0 && u.first_tok < a.num_pages * a.S) {
      const int32_t pg = u.first_tok / a.S, sl = u.first_tok % a.S;
      const int32_t y = (int32_t)(((page_base + pg) * a.H_kv + g.h) * a.S + sl);
      const uint32_t dst = sbase;                     // slot 0
      mbar_arrive_expect_tx(bars, C::kSlotBytes);
#pragma unroll
      for (int hh = 0; hh < C::kHalves; ++hh) {
        tma_load_2d(dst + hh * C::kHalfBytes, &maps.k, 64 * hh, y, bars,
                    tc::l2_policy_evict_first());
        tma_load_2d(dst + C::kTileBytes + hh * C::kHalfBytes, &maps.v, 64 * hh, y, bars,
                    tc::l2_policy_evict_first());
      }
      issued = 1;
      next_issue = pb + 1;
      const Piece pc0 = a.pieces[pb];
      if (!piece_ok(a, pc0) || pc0.fresh || pc0.page != pg || pc0.slot0 != sl)
        record_error(a.err, ERR_PLAN, KID_ATTN_FMA, blockIdx.x, 7);
    }
  }

  // Rotation of every row's query for segment slot `seg` by (i_q - the segment's view offset),
  // pre-scaled; rows of workers that do not see it are zero and cut = -1.  Threads t0 .. t0 + nt
  // of the CTA share the work (t = tid - t0), in two passes with the same items per thread:
  // rot_factors puts each item's (cos, sin) where its rotated pair goes (plan and table data
  // only: it may run before the programmatic wait), rot_apply reads the query pair and
  // replaces them (zero factors: a row that does not see the segment).
  constexpr int half = D / 2;
  auto rot_factors = [&](int seg, int t, int nt) {
    const int* dl = a.delta + (size_t)seg * a.W;
    for (int idx = t; idx < R * half; idx += nt) {
      const int r = idx / half, i = idx % half;
      const int w = r / a.G;
      const int delta = dl[w];
      const bool vis = delta >= 0 && delta < a.max_position;
      float c = 0.f, sn = 0.f;
      if (vis) {
        c = a.rope_cos[(size_t)delta * half + i];
        sn = a.rope_sin[(size_t)delta * half + i];
      } else if (delta >= a.max_position && i == 0) {
        record_error(a.err, ERR_POS_RANGE, KID_ATTN_FMA, blockIdx.x, delta);
      }
      Qs[r * D + i] = c;
      Qs[r * D + i + half] = sn;
      // causal cut (several query tokens per worker): tokens of the segment it may see
      if (i == 0) cut[r] = !vis ? -1 : (a.vlen ? a.vlen[(size_t)seg * a.W + w] : 0x7fffffff);
    }
  };
  auto rot_apply = [&](int t, int nt) {
    for (int idx = t; idx < R * half; idx += nt) {
      const int r = idx / half, i = idx % half;
      const int w = r / a.G, hq = g.h * a.G + r % a.G;
      const float c = Qs[r * D + i], sn = Qs[r * D + i + half];
      float y1 = 0.f, y2 = 0.f;
      const int qr = query_row(a, g.p, w);
      if ((c != 0.f || sn != 0.f) && qr >= 0) {      // (cos and sin of an angle are never both 0)
        const size_t qo = ((size_t)qr * a.H_q + hq) * D;
        const float q1 = __bfloat162float(a.q[qo + i]);
        const float q2 = __bfloat162float(a.q[qo + i + half]);
        y1 = (q1 * c - q2 * sn) * a.scale_log2;
        y2 = (q2 * c + q1 * sn) * a.scale_log2;
      }
      Qs[r * D + i] = y1;
      Qs[r * D + i + half] = y2;
    }
  };
  // The unit's first segment (named by its record): its rotation factors before the wait.  The
  // fused append, if the unit has appended tokens, runs after it on two warps while the other
  // six finish the rotation; the async-proxy fence orders the pool writes before the CTA's TMA
  // reads of them; every (token, KV head) belongs to exactly one unit.
  const bool pre_rot = unit_ok && u.seg0 >= 0 && u.seg0 < a.num_seg_slots;
  const int rot_t = fresh_here ? tid - 64 : tid, rot_nt = fresh_here ? kThreads - 64 : kThreads;
  if (pre_rot && rot_t >= 0) rot_factors(u.seg0, rot_t, rot_nt);
  // Wait for the grid this one follows (it may write the queries, this step's tokens, or read
  // the partials this grid overwrites).
  tc::pdl_wait();
  if (tid == 0 && pb < pe) fill_ring(!fresh_here);
  if (fresh_here && tid < 64) {
    append_fresh<D, 64>(a, g.h, u.fresh_begin, u.fresh_end, tid, KID_ATTN_FMA);
    fence_proxy_async_global();
  } else if (pre_rot) {
    rot_apply(rot_t, rot_nt);
  }
  __syncthreads();
  if (fresh_here && tid == 0) fill_ring(true);

  int cur_seg = pre_rot ? u.seg0 : -1;
  uint32_t tile = 0;              // tiles consumed
  for (int pi = pb; pi < pe; ++pi) {
    const Piece pc = a.pieces[pi];
    if (!piece_ok(a, pc)) continue;                 // every thread skips it the same way
    if (pc.seg_slot != cur_seg) {                   // a new segment: its query rotation
      cur_seg = pc.seg_slot;
      rot_factors(cur_seg, tid, kThreads);
      rot_apply(tid, kThreads);
    }
    const int slot = (int)(tile % (uint32_t)slots);
    const uint32_t parity = (tile / (uint32_t)slots) & 1u;
    // every thread waits for the tile (bounded); an expiry anywhere ends the loop for all
    if (!mbar_wait(bars + 8u * slot, parity, flags + 1, kWaitNs)) flags[1] = 1;
    __syncthreads();                                // also: the rotated queries are written
    if (flags[1]) break;
    const uint8_t* kt = smem + (uint32_t)slot * C::kSlotBytes;
    const uint8_t* vt = kt + C::kTileBytes;
    const int nv = pc.ntok;
    for (int r0 = 0; r0 < R; r0 += kChunkRows) {
      const int CR = min(kChunkRows, R - r0);
      {
        // S = Q~ K^T and the online softmax of the tile, fused.  Warp w takes chunk rows
        // ra = 2w and rb = 2w + 1; lane = (half dh, token group tg): tokens tg + 16 k (k < 8) of
        // both rows over the dims of half dh, so every K chunk loaded feeds two rows (the bytes
        // shared memory delivers to registers, not the FMAs, set the pace of this loop).  The
        // 8-element query chunks stay in registers across the eight tokens; the 16 lanes of a
        // half read 16 consecutive tokens' chunks (swizzled rows: no bank conflict).  The halves
        // then swap partial sums -- half 0 keeps row ra, half 1 row rb -- and the 16 lanes of a
        // half reduce their row's maximum and sum with shuffles.
        const int ra = 2 * warp, rb = ra + 1;
        if (ra < CR) {                                  // (uniform in the warp)
          const bool has_b = rb < CR;
          const int dh = lane >> 4, tg = lane & 15;
          constexpr int NCH = D / 16;                   // 8-element chunks per half of the dims
          float acc_a[kTile / 16], acc_b[kTile / 16];    // per token: this half's dot product
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) acc_a[k] = acc_b[k] = 0.f;
          const float* qa_row = Qs + (size_t)(r0 + ra) * D;
          const float* qb_row = Qs + (size_t)(r0 + (has_b ? rb : ra)) * D;
#pragma unroll 1
          for (int cc = 0; cc < NCH; ++cc) {
            const int c = dh * NCH + cc;
            const float4 a0 = *reinterpret_cast<const float4*>(qa_row + 8 * c);
            const float4 a1 = *reinterpret_cast<const float4*>(qa_row + 8 * c + 4);
            const float4 b0 = *reinterpret_cast<const float4*>(qb_row + 8 * c);
            const float4 b1 = *reinterpret_cast<const float4*>(qb_row + 8 * c + 4);
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k) {
              const uint4 kw = *reinterpret_cast<const uint4*>(kt + swz<D>(tg + 16 * k, c));
              const float k0 = bf_lo(kw.x), k1 = bf_hi(kw.x), k2 = bf_lo(kw.y), k3 = bf_hi(kw.y);
              const float k4 = bf_lo(kw.z), k5 = bf_hi(kw.z), k6 = bf_lo(kw.w), k7 = bf_hi(kw.w);
              float x = acc_a[k], y = acc_b[k];
              x = fmaf(a0.x, k0, x); y = fmaf(b0.x, k0, y);
              x = fmaf(a0.y, k1, x); y = fmaf(b0.y, k1, y);
              x = fmaf(a0.z, k2, x); y = fmaf(b0.z, k2, y);
              x = fmaf(a0.w, k3, x); y = fmaf(b0.w, k3, y);
              x = fmaf(a1.x, k4, x); y = fmaf(b1.x, k4, y);
              x = fmaf(a1.y, k5, x); y = fmaf(b1.y, k5, y);
              x = fmaf(a1.z, k6, x); y = fmaf(b1.z, k6, y);
              x = fmaf(a1.w, k7, x); y = fmaf(b1.w, k7, y);
              acc_a[k] = x;
              acc_b[k] = y;
            }
          }
          // swap the halves' partial sums: this lane keeps its own row's score
          float sv[kTile / 16];
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            const float mine = dh ? acc_b[k] : acc_a[k], other = dh ? acc_a[k] : acc_b[k];
            sv[k] = mine + __shfl_xor_sync(0xffffffffu, other, 16);
          }
          const int r = dh ? rb : ra;                   // this half's row (in the chunk)
          if (r < CR) {                                 // (uniform in the half)
            const unsigned hmask = dh ? 0xffff0000u : 0x0000ffffu;
            // Online softmax of the row over this tile: tokens past the piece or past the row's
            // causal cut (cut -1: the row does not see the segment) score -inf.
            const int rr = r0 + r;
            const int cap = cut[rr];
            const int lim = cap < 0 ? 0 : min(nv, cap - pc.pos0);
            const float m_old = Ms[rr];
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k) {
              if (tg + 16 * k >= lim) sv[k] = -CUDART_INF_F;
              mx = fmaxf(mx, sv[k]);
            }
#pragma unroll
            for (int off = 8; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(hmask, mx, off));
            const float m_new = fmaxf(m_old, mx);
            float alpha = 1.f, ps = 0.f;
            float* prow = Ss + r * kSStride;
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k) {
              const float pk = (sv[k] == -CUDART_INF_F) ? 0.f : exp2f(sv[k] - m_new);
              ps += pk;
              prow[tg + 16 * k] = pk;
            }
            if (m_new != -CUDART_INF_F) alpha = (m_old == -CUDART_INF_F) ? 0.f : exp2f(m_old - m_new);
#pragma unroll
            for (int off = 8; off; off >>= 1) ps += __shfl_xor_sync(hmask, ps, off);
            if (tg == 0) {             // (every lane of the row has read Ms above)
              Ms[rr] = m_new;
              Ls[rr] = Ls[rr] * alpha + ps;
              As[rr] = alpha;
            }
          }
        }
      }
      // Warp w computed P and the statistics of chunk rows 2w and 2w + 1 -- the rows it takes in
      // O = alpha O + P V below: no other warp reads or writes them.
      __syncwarp();
      if constexpr (D == 128) {
        // O = alpha O + P V.  Warp w, rows ra = 2w and rb = 2w + 1; lane = (token half th, column
        // group cg): tokens [64 th, 64 th + 64) and columns 8 cg .. 8 cg + 7 of both rows, so
        // every V chunk loaded feeds two rows.  The halves then swap partial sums (half 0 keeps
        // row ra, half 1 row rb) and each writes its row's columns.  P is zero past the piece's
        // tokens, so a group of four that runs past them adds nothing.
        const int ra = 2 * warp, rb = ra + 1;
        if (ra < CR) {                                  // (uniform in the warp)
          const bool has_b = rb < CR;
          const int th = lane >> 4, cg = lane & 15;
          const float* pa = Ss + ra * kSStride;
          const float* pbr = Ss + (has_b ? rb : ra) * kSStride;
          float2 ya[4], yb[4];                          // 8 columns per row, as (even, odd)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            ya[i] = make_float2(0.f, 0.f);
            yb[i] = make_float2(0.f, 0.f);
          }
          const int nv4 = (nv + 3) & ~3;
          const int k_end = min(nv4, 64 * th + 64);
#pragma unroll 1
          for (int k = 64 * th; k < k_end; k += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pa + k);
            const float4 q4 = *reinterpret_cast<const float4*>(pbr + k);
            uint4 vw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) vw[e] = *reinterpret_cast<const uint4*>(vt + swz<D>(k + e, cg));
            const float pp[4] = {p4.x, p4.y, p4.z, p4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 pe = make_float2(pp[e], pp[e]), qe = make_float2(qq[e], qq[e]);
              const uint32_t wv[4] = {vw[e].x, vw[e].y, vw[e].z, vw[e].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 v = make_float2(bf_lo(wv[i]), bf_hi(wv[i]));
                ya[i] = fma2(pe, v, ya[i]);
                yb[i] = fma2(qe, v, yb[i]);
              }
            }
          }
          float fin[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 mine = th ? yb[i] : ya[i], other = th ? ya[i] : yb[i];
            fin[2 * i] = mine.x + __shfl_xor_sync(0xffffffffu, other.x, 16);
            fin[2 * i + 1] = mine.y + __shfl_xor_sync(0xffffffffu, other.y, 16);
          }
          const int r = th ? rb : ra;
          if (r < CR) {
            float4* o = reinterpret_cast<float4*>(Os + (size_t)(r0 + r) * D + 8 * cg);
            const float al = As[r0 + r];
            const float4 o0 = o[0], o1 = o[1];
            o[0] = make_float4(fmaf(al, o0.x, fin[0]), fmaf(al, o0.y, fin[1]), fmaf(al, o0.z, fin[2]),
                               fmaf(al, o0.w, fin[3]));
            o[1] = make_float4(fmaf(al, o1.x, fin[4]), fmaf(al, o1.y, fin[5]), fmaf(al, o1.z, fin[6]),
                               fmaf(al, o1.w, fin[7]));
          }
        }
      } else {
        // O = alpha O + P V: thread (row pair rp, columns 4 dg .. 4 dg + 3)
        const int rp = tid >> 5, dg = lane;
        const int ra = 2 * rp, rb = 2 * rp + 1;
        if (dg < D / 4 && ra < CR) {
          const bool has_b = rb < CR;
          float4* oa = reinterpret_cast<float4*>(Os + (size_t)(r0 + ra) * D) + dg;
          float4* ob = reinterpret_cast<float4*>(Os + (size_t)(r0 + (has_b ? rb : ra)) * D) + dg;
          float4 xa = *oa, xb = *ob;
          const float aa = As[r0 + ra], ab = has_b ? As[r0 + rb] : 1.f;
          xa = make_float4(xa.x * aa, xa.y * aa, xa.z * aa, xa.w * aa);
          xb = make_float4(xb.x * ab, xb.y * ab, xb.z * ab, xb.w * ab);
          const float* pa = Ss + ra * kSStride;
          const float* pbr = Ss + (has_b ? rb : ra) * kSStride;
          const int d = 4 * dg;
          const uint8_t* vcol = vt + (uint32_t)(d >> 6) * C::kHalfBytes + (uint32_t)((d & 7) * 2);
          const int vc = (d & 63) >> 3;
          // four tokens at a time: their P values (one float4 per row) and V words loaded first
          // (P is zero past the piece's tokens, so the tail of the last group adds nothing)
          const int nv4 = (nv + 3) & ~3;
          float2 xa01 = make_float2(xa.x, xa.y), xa23 = make_float2(xa.z, xa.w);
          float2 xb01 = make_float2(xb.x, xb.y), xb23 = make_float2(xb.z, xb.w);
#pragma unroll 1
          for (int k = 0; k < nv4; k += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pa + k);
            const float4 q4 = *reinterpret_cast<const float4*>(pbr + k);
            uint2 vw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              vw[e] = *reinterpret_cast<const uint2*>(
                  vcol + (uint32_t)(k + e) * 128 + ((uint32_t)(vc ^ ((k + e) & 7)) << 4));
            const float pp[4] = {p4.x, p4.y, p4.z, p4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 v01 = make_float2(bf_lo(vw[e].x), bf_hi(vw[e].x));
              const float2 v23 = make_float2(bf_lo(vw[e].y), bf_hi(vw[e].y));
              const float2 pe = make_float2(pp[e], pp[e]), qe = make_float2(qq[e], qq[e]);
              xa01 = fma2(pe, v01, xa01);
              xa23 = fma2(pe, v23, xa23);
              xb01 = fma2(qe, v01, xb01);
              xb23 = fma2(qe, v23, xb23);
            }
          }
          *oa = make_float4(xa01.x, xa01.y, xa23.x, xa23.y);
          if (has_b) *ob = make_float4(xb01.x, xb01.y, xb23.x, xb23.y);
        }
      }
      __syncwarp();                                 // (the next chunk rewrites this warp's P rows)
    }
    __syncthreads();                                // every warp is done with the slot and Q~
    ++tile;
    // the slot is free: its next piece goes out (the generic reads of the slot are ordered
    // before the copy's writes)
    if (tid == 0 && next_issue < pe) {
      fence_proxy_async_smem();
      const int got = issue(next_issue, slot, true);
      next_issue = got < 0 ? pe : got + 1;
      if (got >= 0) ++issued;
    }
  }
  if (tid == 0) tc::pdl_launch_dependents();       // the merge may start its prologue
  if (flags[1] || !plan_ok) {
    // A wait ran out (or the plan never arrived): the copies in flight land before the CTA
    // leaves, and the unit's partials are written empty.
    if (tid == 0) {
      if (flags[1]) record_error(a.err, ERR_TIMEOUT, KID_ATTN_FMA, blockIdx.x, 1);
      for (uint32_t k = tile; k < issued; ++k)
        mbar_wait_drain(bars + 8u * (k % (uint32_t)slots), (k / (uint32_t)slots) & 1u, kWaitNs);
    }
    float* part = a.partials + (size_t)blockIdx.x * R * PS;
    for (int e = tid; e < R * PS; e += kThreads) part[e] = (e % PS == D) ? -CUDART_INF_F : 0.f;
    return;
  }
  // Partial result of this unit: o (unnormalised), m, l in the log2 domain.
  float* part = a.partials + (size_t)blockIdx.x * R * PS;
  for (int r = warp; r < R; r += kWarps) {
    if (lane < D / 4)
      reinterpret_cast<float4*>(part + (size_t)r * PS)[lane] =
          reinterpret_cast<const float4*>(Os + (size_t)r * D)[lane];
    if (lane == 0)
      *reinterpret_cast<float4*>(part + (size_t)r * PS + D) = make_float4(Ms[r], Ls[r], 0.f, 0.f);
  }
}

// Ring slots for R query rows: one, so that two CTAs share an SM (each computes while the
// other's tile lands); the occupancy, not a second slot, hides the load latency.
template <int D>
int fma_slots(int rows) {
  (void)rows;
  return 1;
}

template <int D>
void launch_fma_d(const AttnArgs& a, const TcMaps& maps, int layer, cudaStream_t s) {
  const int slots = fma_slots<D>(a.rows);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = FmaLayout<D>(a.rows, slots).total;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, attn_fma_kernel<D>, a, maps, (int32_t)layer, (int32_t)slots);
}

}  // namespace

cudaError_t prepare_attention_fma(int D) {
  // Shared-memory limit: the largest layout any row count up to 128 uses.
  int most = 0;
  for (int r = 1; r <= 128; ++r)
    most = std::max(most, (int)(D == 64 ? FmaLayout<64>(r, fma_slots<64>(r)).total
                                        : FmaLayout<128>(r, fma_slots<128>(r)).total));
  if (D == 64)
    return cudaFuncSetAttribute(attn_fma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                most);
  return cudaFuncSetAttribute(attn_fma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              most);
}

void launch_attention_fma(const AttnArgs& a, const TcMaps& maps, int layer, cudaStream_t s) {
  if (a.num_units <= 0) return;
  if (a.D == 64)
    launch_fma_d<64>(a, maps, layer, s);
  else
    launch_fma_d<128>(a, maps, layer, s);
}

}  // namespace hw
