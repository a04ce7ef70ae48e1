// K2 (tensor-core form) -- concurrent attention on sm_103a with tcgen05, TMEM and TMA.
//
// Method (Hogwild! Inference summary, gentlecold.top): the keys of every block stay rotated at
// block-local positions; for the block at offset o in worker w's view the query is rotated by
// (i_q - o) (section 5), so one K/V tile serves every worker and every query head of the GQA
// group, each through its own rotated query.  The work is split over KV entries and the
// partial results reduced afterwards (section 9).
//
// One CTA = one unit: a run of pieces (<= 256 tokens of one segment inside one page) of one
// (problem, KV head).  Per 128-token tile:
//   S  = Q~ K^T      tcgen05.mma, M = 128 query rows (W*G real rows, the rest zero),
//                    N = 128 tokens, K = D; A = rotated queries (smem), B = K tile (smem, TMA)
//   P  = 2^(S - m)   softmax threads, one query row per thread (row = TMEM lane), max and sum
//                    thread-local; the running max only moves when it grows by > 2^8, and then
//                    the thread rescales its own row of O in TMEM; P goes back to TMEM as bf16
//   O += P V         tcgen05.mma with A = P from TMEM, B = V tile (smem, MN-major), D = TMEM
// Warp roles: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-3 query rotation per segment,
// 4-7 softmax / correction / epilogue.  Every K/V element is loaded from HBM once per unit and
// used by all W*G rows; S is double-buffered so the softmax of tile i overlaps MMA2(i-1) and
// MMA1(i+1).  All waits are bounded: a wait that runs out raises a CTA abort flag, records
// ERR_TIMEOUT in the error word, drains the copies and MMAs already issued and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hw_device.cuh"
#include "tc_ptx.cuh"

namespace hw {

namespace {

using namespace tc;

constexpr int kTile = 128;                  // tokens per tile = N of the first MMA
constexpr int kRowsM = 128;                 // M of both MMAs (query rows, zero padded)
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                       // 128-byte swizzle atoms per row
  static constexpr uint32_t kHalfBytes = kTile * 128;          // one {64, 128} TMA box
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes; // K or V tile
  static constexpr uint32_t kQBytes = kRowsM * D * 2;
  static constexpr int kSlots = D == 128 ? 5 : 8;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kRingOff = 2 * kQBytes;
  static constexpr uint32_t kBarOff = kRingOff + kSlots * kTileBytes;
  // barriers: full[S], empty[S], q_full[2], q_empty[2], s_full[2], p_full[2], o_done, fin
  static constexpr int kNumBars = 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 1;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
};

struct TileInfo {
  int32_t seg_slot, page, slot0, nvalid;
};

// Walk the tiles of a unit in order; every role runs the same walk.
struct TileWalker {
  const Piece* pieces;
  int32_t pi, pe, k, ntiles_piece;
  Piece pc;
  int32_t num_pages, S, num_seg_slots;
  int32_t last_slot;
  __device__ bool valid(const Piece& p) const {
    return p.page >= 0 && p.page < num_pages && p.slot0 >= 0 && p.ntok >= 1 &&
           p.slot0 + p.ntok <= S && (p.slot0 % kTile) == 0 && p.seg_slot >= 0 &&
           p.seg_slot < num_seg_slots;
  }
  __device__ void init(const AttnArgs& a, const Unit& u) {
    pieces = a.pieces;
    pi = u.piece_begin - 1;
    pe = u.piece_end;
    k = 0;
    ntiles_piece = 0;
    num_pages = a.num_pages;
    S = a.S;
    num_seg_slots = a.num_seg_slots;
    last_slot = -1;
  }
  // Next tile; new_seg is set when the tile starts a new segment (a new query rotation).
  __device__ bool next(TileInfo* t, bool* new_seg) {
    while (k >= ntiles_piece) {
      if (++pi >= pe) return false;
      pc = pieces[pi];
      k = 0;
      ntiles_piece = valid(pc) ? (pc.ntok + kTile - 1) / kTile : 0;
    }
    t->seg_slot = pc.seg_slot;
    t->page = pc.page;
    t->slot0 = pc.slot0 + k * kTile;
    t->nvalid = min(kTile, pc.ntok - k * kTile);
    *new_seg = pc.seg_slot != last_slot;
    last_slot = pc.seg_slot;
    ++k;
    return true;
  }
  // Whether the tile just returned is the last one of its segment in this unit.
  __device__ bool last_of_segment() const {
    if (k < ntiles_piece) return false;
    for (int32_t j = pi + 1; j < pe; ++j) {
      const Piece n = pieces[j];
      if (!valid(n)) continue;
      return n.seg_slot != pc.seg_slot;
    }
    return true;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ TcMaps maps, const int32_t layer) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_base = sbase + C::kQOff;
  const uint32_t ring = sbase + C::kRingOff;
  const uint32_t bars = sbase + C::kBarOff;
  auto bar_full = [&](int s) { return bars + 8u * s; };
  auto bar_empty = [&](int s) { return bars + 8u * (C::kSlots + s); };
  auto bar_qfull = [&](int b) { return bars + 8u * (2 * C::kSlots + b); };
  auto bar_qempty = [&](int b) { return bars + 8u * (2 * C::kSlots + 2 + b); };
  auto bar_sfull = [&](int b) { return bars + 8u * (2 * C::kSlots + 4 + b); };
  auto bar_pfull = [&](int b) { return bars + 8u * (2 * C::kSlots + 6 + b); };
  const uint32_t bar_odone = bars + 8u * (2 * C::kSlots + 8);
  const uint32_t bar_fin = bars + 8u * (2 * C::kSlots + 9);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Unit u = a.units[blockIdx.x];
  const Group g = a.groups[u.group];
  const int R = a.rows;
  const int active_softmax_warps = (R + 31) / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_qfull(b), 64);
      mbar_init(bar_qempty(b), 1);
      mbar_init(bar_sfull(b), 1);
      mbar_init(bar_pfull(b), 32 * active_softmax_warps);
    }
    mbar_init(bar_odone, 1);
    mbar_init(bar_fin, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&maps.k);
    tma_prefetch(&maps.v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t page_base = (int64_t)layer * a.num_pages;   // first page of this layer's pool

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      TileWalker tw;
      tw.init(a, u);
      TileInfo t;
      bool ns;
      uint32_t j = 0;
      bool ok = true;
      while (ok && tw.next(&t, &ns)) {
        const int32_t y = (int32_t)(((page_base + t.page) * a.H_kv + g.h) * a.S + t.slot0);
        for (int part = 0; part < 2 && ok; ++part, ++j) {
          const int s = j % C::kSlots;
          if (j >= (uint32_t)C::kSlots)
            ok = mbar_wait(bar_empty(s), ((j / C::kSlots) - 1) & 1, abort, kWaitLimitNs);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_full(s), C::kTileBytes);
          const CUtensorMap* m = part == 0 ? &maps.k : &maps.v;
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(ring + s * C::kTileBytes + h * C::kHalfBytes, m, 64 * h, y, bar_full(s),
                        policy);
        }
      }
      // Drain: every load issued must have landed before the CTA can exit.
      for (uint32_t s = 0; s < (uint32_t)C::kSlots && s < j; ++s) {
        const uint32_t last = s + ((j - 1 - s) / C::kSlots) * C::kSlots;
        mbar_wait(bar_full(s), (last / C::kSlots) & 1, abort, kWaitLimitNs);
      }
      if (!ok && (*abort)) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc1 = idesc_bf16(kRowsM, kTile, 0, 0);
      constexpr uint32_t idesc2 = idesc_bf16(kRowsM, D, 0, 1);
      TileWalker tw;
      tw.init(a, u);
      TileInfo t;
      bool new_seg;
      uint32_t i = 0, seg = 0;
      int qbuf = 0;
      bool ok = true;
      bool issued_any = false;
      auto issue_mma2 = [&](uint32_t jt) -> bool {
        const int b = jt & 1;
        if (!mbar_wait(bar_pfull(b), (jt >> 1) & 1, abort, kWaitLimitNs)) return false;
        const uint32_t jv = 2 * jt + 1;
        const int s = jv % C::kSlots;
        if (!mbar_wait(bar_full(s), (jv / C::kSlots) & 1, abort, kWaitLimitNs)) return false;
        tc_fence_after();
        const uint32_t vb = ring + s * C::kTileBytes;
        const uint32_t p_tmem = tmem + (b ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bdesc = smem_desc(vb + kk * 2048, C::kHalfBytes, 1024, kSwizzle128);
          mma_ts(tmem + kColO, p_tmem + kk * 8, bdesc, idesc2, (jt > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_empty(s));
        mma_commit(bar_odone);
        return true;
      };
      while (ok && tw.next(&t, &new_seg)) {
        if (new_seg) {
          qbuf = seg & 1;
          ok = mbar_wait(bar_qfull(qbuf), (seg >> 1) & 1, abort, kWaitLimitNs);
          ++seg;
          if (!ok) break;
        }
        const uint32_t jk = 2 * i;
        const int s = jk % C::kSlots;
        ok = mbar_wait(bar_full(s), (jk / C::kSlots) & 1, abort, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        const int b = i & 1;
        const uint32_t qb = q_base + qbuf * C::kQBytes;
        const uint32_t kb = ring + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          const uint64_t adesc = smem_desc(qb + off, 16, 1024, kSwizzle128);
          const uint64_t bdesc = smem_desc(kb + off, 16, 1024, kSwizzle128);
          mma_ss(tmem + (b ? kColS1 : kColS0), adesc, bdesc, idesc1, kk > 0 ? 1u : 0u);
        }
        issued_any = true;
        mma_commit(bar_empty(s));
        mma_commit(bar_sfull(b));
        if (tw.last_of_segment()) mma_commit(bar_qempty(qbuf));
        if (i > 0) ok = issue_mma2(i - 1);
        ++i;
      }
      if (ok && i > 0) ok = issue_mma2(i - 1);
      if (issued_any) {
        mma_commit(bar_fin);
        mbar_wait(bar_fin, 0, abort, kWaitLimitNs);
      }
      if (!ok && (*abort)) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 1);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- query rotation
    const int tq = threadIdx.x - 64;          // 0..63, rows tq and tq + 64
    TileWalker tw;
    tw.init(a, u);
    TileInfo t;
    bool new_seg;
    uint32_t seg = 0;
    const int half = D / 2;
    while (tw.next(&t, &new_seg)) {
      if (!new_seg) continue;
      const int qb = seg & 1;
      if (seg >= 2 && !mbar_wait(bar_qempty(qb), ((seg >> 1) - 1) & 1, abort, kWaitLimitNs)) break;
      uint8_t* qs = smem + C::kQOff + qb * C::kQBytes;
      const int32_t* dl = a.delta + (size_t)t.seg_slot * a.W;
      for (int rr = 0; rr < 2; ++rr) {
        const int r = tq + 64 * rr;
        int delta = -1;
        size_t qo = 0;
        if (r < R) {
          const int w = r / a.G, hq = g.h * a.G + r % a.G;
          delta = dl[w];
          qo = (((size_t)g.p * a.W + w) * a.H_q + hq) * D;
          if (delta >= a.max_position) {
            record_error(a.err, ERR_POS_RANGE, KID_ATTN_TC, blockIdx.x, delta);
            delta = -1;
          }
        }
        // 8-element chunks: chunk c of the first half pairs with chunk c of the second half.
#pragma unroll 1
        for (int c = 0; c < half / 8; ++c) {
          uint32_t lo[4] = {0, 0, 0, 0}, hi[4] = {0, 0, 0, 0};
          if (delta >= 0) {
            const uint4 q1v = *reinterpret_cast<const uint4*>(a.q + qo + 8 * c);
            const uint4 q2v = *reinterpret_cast<const uint4*>(a.q + qo + half + 8 * c);
            const __nv_bfloat162* q1 = reinterpret_cast<const __nv_bfloat162*>(&q1v);
            const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&q2v);
            const float* cs = a.rope_cos + (size_t)delta * half + 8 * c;
            const float* sn = a.rope_sin + (size_t)delta * half + 8 * c;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 x1 = __bfloat1622float2(q1[e]);
              const float2 x2 = __bfloat1622float2(q2[e]);
              const float c0 = cs[2 * e], c1 = cs[2 * e + 1];
              const float s0 = sn[2 * e], s1 = sn[2 * e + 1];
              const __nv_bfloat162 y1 = __floats2bfloat162_rn((x1.x * c0 - x2.x * s0) * a.scale_log2,
                                                              (x1.y * c1 - x2.y * s1) * a.scale_log2);
              const __nv_bfloat162 y2 = __floats2bfloat162_rn((x2.x * c0 + x1.x * s0) * a.scale_log2,
                                                              (x2.y * c1 + x1.y * s1) * a.scale_log2);
              lo[e] = *reinterpret_cast<const uint32_t*>(&y1);
              hi[e] = *reinterpret_cast<const uint32_t*>(&y2);
            }
          }
          // element d of row r: atom d / 64, 16-byte chunk ((d % 64) / 8) ^ (r % 8)
          const int d_lo = 8 * c, d_hi = half + 8 * c;
          uint8_t* p_lo = qs + (d_lo >> 6) * C::kHalfBytes + r * 128 + ((((d_lo & 63) >> 3) ^ (r & 7)) << 4);
          uint8_t* p_hi = qs + (d_hi >> 6) * C::kHalfBytes + r * 128 + ((((d_hi & 63) >> 3) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(p_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(p_hi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar_qfull(qb));
      ++seg;
    }
  } else {
    // ---------------------------------------------------------------- softmax / epilogue
    const int wq = warp - 4;                  // TMEM lane quarter of this warp
    const int r = 32 * wq + lane;
    if (wq < active_softmax_warps) {
      const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
      float m_run = -CUDART_INF_F, l_sum = 0.f;
      TileWalker tw;
      tw.init(a, u);
      TileInfo t;
      bool new_seg;
      uint32_t i = 0;
      bool ok = true;
      bool row_visible = false;
      while (tw.next(&t, &new_seg)) {
        if (new_seg) {
          row_visible = r < R && a.delta[(size_t)t.seg_slot * a.W + r / a.G] >= 0;
        }
        const int b = i & 1;
        if (!mbar_wait(bar_sfull(b), (i >> 1) & 1, abort, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_tmem = tmem + lane_off + (b ? kColS1 : kColS0);
        float s[kTile];
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(s_tmem + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) s[32 * c + e] = __uint_as_float(v[e]);
        }
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          if (c >= t.nvalid || !row_visible) s[c] = -CUDART_INF_F;
          mx = fmaxf(mx, s[c]);
        }
        const bool need = mx > m_run + kRescaleThreshold || (m_run == -CUDART_INF_F && mx > m_run);
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? fmaxf(m_run, mx) : m_run;
          const float alpha = (m_run == -CUDART_INF_F) ? 0.f : exp2f(m_run - m_new);
          l_sum *= need ? alpha : 1.f;
          if (i > 0) {
            // O holds MMA2 results up to tile i-1: wait for the last of them, rescale this row.
            if (!mbar_wait(bar_odone, (i - 1) & 1, abort, kWaitLimitNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float sc = need ? alpha : 1.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(tmem + lane_off + kColO + 32 * c, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * sc);
              tmem_st32(tmem + lane_off + kColO + 32 * c, v);
            }
            tmem_wait_st();
          }
          m_run = m_new;
        }
        const float m_use = (m_run == -CUDART_INF_F) ? 0.f : m_run;
#pragma unroll
        for (int c = 0; c < kTile / 64; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float p0 = exp2f(s[64 * c + 2 * e] - m_use);
            const float p1 = exp2f(s[64 * c + 2 * e + 1] - m_use);
            l_sum += p0 + p1;
            const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
            pk[e] = *reinterpret_cast<const uint32_t*>(&pp);
          }
          tmem_st32(s_tmem + 32 * c, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_pfull(b));
        ++i;
      }
      // Epilogue: unnormalised o, running max and sum of this row (log2 domain).
      float* part = a.partials + ((size_t)blockIdx.x * R + r) * (D + 2);
      bool have = ok && i > 0;
      if (have) {
        have = mbar_wait(bar_odone, (i - 1) & 1, abort, kWaitLimitNs);
        tc_fence_after();
      }
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(tmem + lane_off + kColO + 32 * c, v);
          tmem_wait_ld();
        }
        if (r < R) {
#pragma unroll
          for (int e = 0; e < 32; ++e) part[32 * c + e] = have ? __uint_as_float(v[e]) : 0.f;
        }
      }
      if (r < R) {
        part[D] = have ? m_run : -CUDART_INF_F;
        part[D + 1] = have ? l_sum : 0.f;
      }
      if (!ok && (*abort) && lane == 0) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

template <int D>
static void launch_tc_d(const AttnArgs& a, const TcMaps& maps, int layer, cudaStream_t s) {
  using C = Cfg<D>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)C::kSmemBytes);
  attn_tc_kernel<D><<<a.num_units, kThreads, C::kSmemBytes, s>>>(a, maps, layer);
}

void launch_attention_tc(const AttnArgs& a, const TcMaps& maps, int layer, cudaStream_t s) {
  if (a.num_units <= 0) return;
  if (a.D == 64)
    launch_tc_d<64>(a, maps, layer, s);
  else
    launch_tc_d<128>(a, maps, layer, s);
}

// ---- tensor maps (host) ------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_tc_maps(const hw_config& cfg, void* k_pool, void* v_pool, TcMaps* out) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t rows = (cuuint64_t)cfg.num_layers * cfg.num_pages * cfg.num_kv_heads * cfg.page_size;
  const cuuint64_t dims[2] = {(cuuint64_t)cfg.head_dim, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cfg.head_dim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  const cuuint32_t estr[2] = {1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = enc(i == 0 ? &out->k : &out->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     i == 0 ? k_pool : v_pool, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

}  // namespace hw
