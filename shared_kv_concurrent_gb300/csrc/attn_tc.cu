// K2 (tensor-core form) -- concurrent attention on sm_103a with tcgen05, TMEM and TMA.
//
// Method (Hogwild! Inference summary, gentlecold.top): the keys of every block stay rotated at
// block-local positions; for the block at offset o in worker w's view the query is rotated by
// (i_q - o) (section 5), so one K/V tile serves every worker and every query head of the GQA
// group, each through its own rotated query.  The work is split over KV entries and the
// partial results reduced afterwards (section 9).
//
// One CTA = one unit: a run of pieces (<= 128 tokens of one segment inside one page) of one
// (problem, KV head).  Per segment of the unit, the query-rotation warps build the rotated,
// pre-scaled (log2(e)/sqrt(D)) 128-row bf16 A tile in shared memory, in the swizzled layout the
// MMA reads.  Per 128-token tile:
//     S  = Q~ K^T     tcgen05.mma, M = 128 TMEM lanes, N = 128 tokens, K = D; A = rotated
//                     queries (smem), B = K tile (smem, TMA, 128-byte swizzle)
//     P  = 2^(S - m)  softmax threads, one TMEM lane each.  Every real query row is repeated T
//                     times in A, once per softmax warp group, and warp group j takes tokens
//                     [j*128/T, (j+1)*128/T) of every tile: each lane keeps its own running max
//                     (moved only when it grows by more than 2^8, then the lane rescales its
//                     own O row in TMEM), sum and O row over its tokens.  P goes to dedicated
//                     TMEM columns as bf16, zero outside the warp's token range.
//     O += P V        tcgen05.mma with A = P from TMEM, B = V tile (smem, MN-major), D = TMEM;
//                     the epilogue merges the T partial rows of each query row by log-sum-exp
// T = 4, 2, 1 for up to 32, 64, 128 real rows, so that every SM sub-partition runs softmax.
// Warp roles: 0 TMA producer (K and V tiles), 1 MMA issuer and TMEM owner, 2-3 query rotation,
// 4-7 softmax / correction / epilogue.  Every K/V element is loaded from HBM once per unit and
// used by all W*G rows; S is double-buffered so the softmax of tile i overlaps MMA2(i-1) and
// MMA1(i+1), and the query tile is double-buffered so the next segment's rotation overlaps
// the current segment's tiles.  All waits are bounded: one that runs out raises a CTA abort
// flag, records ERR_TIMEOUT in the error word, and the CTA drains the copies and MMAs it
// issued and frees its TMEM.  Launch chaining (programmatic dependent launch): the kernel may
// start while the preceding kernel of the stream (the previous call's merge, or the append
// kernel) still runs; meanwhile it sets up and loads its first tile, when that tile holds only
// tokens no launch still in flight can have written, and it waits for that kernel before it
// reads the queries or any other tile; it lets the merge kernel launch before its partial
// results are stored.  What a CTA of the first wave needs before the plan is read (its first
// tile's row, the first query tile's group, segment and rotation) comes with the launch as a
// kernel parameter, so that nothing at the start waits on a dependent load.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hw_device.cuh"
#include "tc_ptx.cuh"

namespace hw {

namespace {

using namespace tc;

constexpr int kTile = 128;                  // tokens per tile = N of the first MMA
constexpr int kRowsM = 128;                 // M of both MMAs (TMEM lanes)
constexpr int kThreads = 256;
constexpr int kRotThreads = 64;             // warps 2-3: query rotation
constexpr uint32_t kTmemCols = 512;
// TMEM columns: two S buffers, O, and two P buffers of their own.  P must not alias S: the
// MMA that writes S(i+2) is issued right after the one that reads P(i), and the tensor core
// may overlap the two.
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kChunkRing = 16;              // published tile ranges in flight (see TileWalker)

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                       // 128-byte swizzle atoms per row
  static constexpr uint32_t kHalfBytes = kTile * 128;          // one {64, 128} TMA box
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes; // K or V tile
  static constexpr uint32_t kQBytes = kRowsM * D * 2;          // rotated query tile
  // K/V ring slots: at D = 128 two tiles in flight; a fifth slot measured 1 % slower per
  // chained step (the early fills compete with the previous step's last tiles), a third fewer
  // starves the MMA.
  static constexpr int kSlots = D == 128 ? 4 : 8;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kRingOff = 2 * kQBytes;
  static constexpr uint32_t kBarOff = kRingOff + kSlots * kTileBytes;
  // barriers: full[S], empty[S], q_full[2], q_empty[2], s_full[2], p_full[2], o_done, fin,
  // fresh, chunk_full[kChunkRing], chunk_empty[kChunkRing]
  static constexpr int kNumBars = 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 1 + 1 + 2 * kChunkRing;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kUnitOff = (kMiscOff + 8 + 15) / 16 * 16;   // the CTA's Unit
  static constexpr uint32_t kChunkOff = kUnitOff + sizeof(Unit);   // int2[kChunkRing]
  static constexpr uint32_t kSmemBytes = kChunkOff + 8 * kChunkRing + 1024;  // + alignment slack
};

// Timeline tracing, compiled in only with -DHW_TRACE (a separate debug build of the library):
// %globaltimer stamps per CTA -- 0 start, 1 set-up done, 2 first query tile issued,
// 3 producer done, 4 MMA issuer done, 5 epilogue start, 6 epilogue end, 7 end; then per tile
// i < 60: 8+4i K(i) issued, 9+4i MMA1(i) issued, 10+4i S(i) seen by softmax, 11+4i P(i) written.
#ifdef HW_TRACE
constexpr int kTraceCtas = 160, kTraceEvents = 256;
__device__ unsigned long long g_trace[kTraceCtas][kTraceEvents];
#define HW_TRACE_EV(idx)                                                   \
  do {                                                                     \
    const int ev_ = (idx);                                                 \
    if (blockIdx.x < kTraceCtas && ev_ < kTraceEvents)                     \
      g_trace[blockIdx.x][ev_] = globaltimer_ns();                         \
  } while (0)
#else
#define HW_TRACE_EV(idx) \
  do {                   \
  } while (0)
#endif

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct TileInfo {
  int32_t seg_slot, page, slot0, nvalid, fresh, pos0;
};

// The CTA's sequence of tiles: the producer publishes ranges of pieces, {begin, end}, in a
// shared-memory ring of kChunkRing entries (end < 0 closes the sequence); every other role
// reads the ring through a TileWalker, so all of them see the same tiles in the same order.
// A piece is one tile.

struct TileWalker {
  const Piece* pieces;
  const int2* ring;
  uint32_t full_bars, empty_bars;             // kChunkRing mbarriers each
  volatile int* abort;
  uint32_t ci;                                // ring entries consumed
  int32_t pi, pe;
  int32_t num_pages, S, num_seg_slots, last_slot;
  bool done;
  __device__ bool valid(const Piece& p) const {
    return p.page >= 0 && p.page < num_pages && p.slot0 >= 0 && p.ntok >= 1 && p.ntok <= kTile &&
           p.slot0 + p.ntok <= S && p.seg_slot >= 0 &&
           p.seg_slot < num_seg_slots;
  }
  __device__ void init(const AttnArgs& a, const int2* ring_, uint32_t full_, uint32_t empty_,
                       volatile int* abort_) {
    pieces = a.pieces;
    ring = ring_;
    full_bars = full_;
    empty_bars = empty_;
    abort = abort_;
    ci = 0;
    pi = pe = 0;
    num_pages = a.num_pages;
    S = a.S;
    num_seg_slots = a.num_seg_slots;
    last_slot = -1;
    done = false;
  }
  // Next tile; new_seg is set when the tile starts a new segment (a new query rotation).
  // False at the end of the sequence, or when a wait gave up (the abort flag is then set).
  __device__ bool next(TileInfo* t, bool* new_seg) {
    Piece pc;
    for (;;) {
      while (pi >= pe) {
        if (done) return false;
        const uint32_t e = ci % kChunkRing;
        if (!mbar_wait(full_bars + 8u * e, (ci / kChunkRing) & 1, abort, kWaitLimitNs)) {
          done = true;
          return false;
        }
        const int2 r = ring[e];
        mbar_arrive(empty_bars + 8u * e);
        ++ci;
        if (r.y < 0) {
          done = true;
          return false;
        }
        pi = r.x;
        pe = r.y;
      }
      pc = pieces[pi++];
      if (valid(pc)) break;
    }
    t->seg_slot = pc.seg_slot;
    t->page = pc.page;
    t->slot0 = pc.slot0;
    t->nvalid = pc.ntok;
    t->fresh = pc.fresh;
    t->pos0 = pc.pos0;
    *new_seg = pc.seg_slot != last_slot;
    last_slot = pc.seg_slot;
    return true;
  }
};

// ---------------------------------------------------------------------------- rotation

// Rotated query tile of segment slot `slot` for the unit's group (p, h): 128 M-rows x D bf16 in
// the MMA's shared-memory layout (D / 64 atoms of 128-byte rows, 128-byte swizzle: the 16-byte
// chunk c of M-row m sits at chunk c ^ (m % 8)).  Query row r of the group (worker r / G, head
// h*G + r % G) is rotated by its worker's delta for the segment and pre-scaled by
// log2(e)/sqrt(D), and stored at the T M-rows r + j * 128/T (softmax warp group j reads copy
// j); rows past W*G and rows whose worker does not see the segment are zero.  uniform_delta
// >= 0 is the rotation of every row (no delta-table load), -1 = look it up per row.  Run by NT
// threads; each takes (row, 8-pair chunk) items and issues the loads of up to four items
// before using any.
template <int D, int T, int NT>
__device__ __forceinline__ void rotate_tile(const AttnArgs& a, const Group& g, int slot,
                                            int uniform_delta, uint8_t* tile, int tid) {
  constexpr int half = D / 2;
  constexpr int CH = half / 8;                 // 8-pair chunks per row
  constexpr int RR = kRowsM / T;               // M-rows per copy
  constexpr int ITEMS = RR * CH;
  constexpr int PER = (ITEMS + NT - 1) / NT;   // items per thread
  constexpr int B = PER < 4 ? PER : (PER % 4 == 0 ? 4 : 3);  // loads in flight together
  constexpr uint32_t kHalfBytes = kTile * 128;
  static_assert(PER % B == 0, "rotation work split");
#pragma unroll 1
  for (int b0 = 0; b0 < PER; b0 += B) {
    uint4 q1[B], q2[B];
    float4 cs[B][2], sn[B][2];
    int dl[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int item = tid + NT * (b0 + k);
      const int r = item / CH, c = item % CH;
      int delta = -1;
      size_t qo = 0;
      if (item < ITEMS && r < a.rows) {
        const int w = r / a.G, hq = g.h * a.G + r % a.G;
        delta = uniform_delta >= 0 ? uniform_delta : a.delta[(size_t)slot * a.W + w];
        qo = ((size_t)query_row(a, g.p, w) * a.H_q + hq) * D;
        if (delta >= a.max_position) {
          record_error(a.err, ERR_POS_RANGE, KID_ATTN_TC, blockIdx.x, delta);
          delta = -1;
        }
      }
      dl[k] = delta;
      if (delta >= 0) {
        q1[k] = *reinterpret_cast<const uint4*>(a.q + qo + 8 * c);
        q2[k] = *reinterpret_cast<const uint4*>(a.q + qo + half + 8 * c);
        const float4* cp = reinterpret_cast<const float4*>(a.rope_cos + (size_t)delta * half + 8 * c);
        const float4* sp = reinterpret_cast<const float4*>(a.rope_sin + (size_t)delta * half + 8 * c);
        cs[k][0] = cp[0];
        cs[k][1] = cp[1];
        sn[k][0] = sp[0];
        sn[k][1] = sp[1];
      }
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int item = tid + NT * (b0 + k);
      if (item >= ITEMS) break;
      const int r = item / CH, c = item % CH;
      uint32_t lo[4] = {0, 0, 0, 0}, hi[4] = {0, 0, 0, 0};
      if (dl[k] >= 0) {
        const __nv_bfloat162* x1p = reinterpret_cast<const __nv_bfloat162*>(&q1[k]);
        const __nv_bfloat162* x2p = reinterpret_cast<const __nv_bfloat162*>(&q2[k]);
        const float cv[8] = {cs[k][0].x, cs[k][0].y, cs[k][0].z, cs[k][0].w,
                             cs[k][1].x, cs[k][1].y, cs[k][1].z, cs[k][1].w};
        const float sv[8] = {sn[k][0].x, sn[k][0].y, sn[k][0].z, sn[k][0].w,
                             sn[k][1].x, sn[k][1].y, sn[k][1].z, sn[k][1].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x1 = __bfloat1622float2(x1p[e]);
          const float2 x2 = __bfloat1622float2(x2p[e]);
          const float ca = cv[2 * e], cb = cv[2 * e + 1];
          const float sa = sv[2 * e], sb = sv[2 * e + 1];
          const __nv_bfloat162 y1 = __floats2bfloat162_rn((x1.x * ca - x2.x * sa) * a.scale_log2,
                                                          (x1.y * cb - x2.y * sb) * a.scale_log2);
          const __nv_bfloat162 y2 = __floats2bfloat162_rn((x2.x * ca + x1.x * sa) * a.scale_log2,
                                                          (x2.y * cb + x1.y * sb) * a.scale_log2);
          lo[e] = *reinterpret_cast<const uint32_t*>(&y1);
          hi[e] = *reinterpret_cast<const uint32_t*>(&y2);
        }
      }
      const int d_lo = 8 * c, d_hi = half + 8 * c;
#pragma unroll
      for (int j = 0; j < T; ++j) {
        const int m = r + j * RR;
        uint8_t* p_lo = tile + (d_lo >> 6) * kHalfBytes + m * 128 + ((((d_lo & 63) >> 3) ^ (m & 7)) << 4);
        uint8_t* p_hi = tile + (d_hi >> 6) * kHalfBytes + m * 128 + ((((d_hi & 63) >> 3) ^ (m & 7)) << 4);
        *reinterpret_cast<uint4*>(p_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(p_hi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------- attention

template <int D, int T>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ TcMaps maps, const int32_t layer,
                   const __grid_constant__ LaunchUnits lu) {
  using C = Cfg<D>;
  static_assert(T == 1 || T == 2 || T == 4, "T copies of each query row, one per column chunk");
  constexpr int WPC = 4 / T;                  // softmax warps per column chunk
  constexpr int CPT = kTile / T;              // token columns per lane
  constexpr int PCPT = CPT / 2;               // packed bf16 P columns per lane
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
  const uint32_t bar_fresh = bars + 8u * (2 * C::kSlots + 10);   // fused append written
  const uint32_t bar_cfull0 = bars + 8u * (2 * C::kSlots + 11);   // chunk ring: published
  const uint32_t bar_cempty0 = bar_cfull0 + 8u * kChunkRing;      // chunk ring: read by all
  int2* cring = reinterpret_cast<int2*>(smem + C::kChunkOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Unit* u_smem = reinterpret_cast<Unit*>(smem + C::kUnitOff);
  const int R = a.rows;
  const int64_t page_base0 = (int64_t)layer * a.num_pages;  // first page of this layer's pool
  int active_softmax_warps = 0;               // softmax warps that own at least one real row
  for (int q = 0; q < 4; ++q) active_softmax_warps += (32 * (q % WPC) < R) ? 1 : 0;
  if (threadIdx.x == 0) HW_TRACE_EV(0);

  // The launch parameters describe this CTA's unit before any of the plan is read (first wave).
  const bool in_lu = blockIdx.x < (unsigned)kLaunchUnits;
  const int32_t lu_row0 = in_lu ? lu.row0[blockIdx.x] : -1;
  const int32_t lu_group = in_lu ? lu.group[blockIdx.x] : -1;
  const int32_t lu_seg0 = in_lu ? lu.seg0[blockIdx.x] : -1;
  const int32_t lu_delta0 = in_lu ? lu.delta0[blockIdx.x] : -1;

  // Warps 2-7 rotate the first query tile before set-up is done when it needs nothing of the
  // plan: one rotation for every row (no delta table) and one query per worker (no row map).
  // Otherwise they do after set-up, once the plan has arrived.
  bool pre_q = false;
  if (warp >= 2) {
    pdl_wait();                       // the queries may come from the kernel this grid follows
    if (lu_delta0 >= 0 && a.qrow == nullptr && lu_group >= 0 && lu_group < a.P * a.H_kv &&
        lu_seg0 >= 0 && lu_seg0 < a.num_seg_slots) {
      const Group g0{lu_group / a.H_kv, lu_group % a.H_kv, 0, 0};
      rotate_tile<D, T, kThreads - 64>(a, g0, lu_seg0, lu_delta0, smem + C::kQOff,
                                       threadIdx.x - 64);
      pre_q = true;
    }
  }

  if (threadIdx.x == 0) {
    // The unit record (three vectors) and the plan's sequence word are read first and used
    // once the plan's arrival is confirmed.
    const int4* urec = reinterpret_cast<const int4*>(a.units + blockIdx.x);
    int4 uv[3];                                     // (L2, not a stale L1 line)
#pragma unroll
    for (int k = 0; k < 3; ++k) uv[k] = __ldcg(urec + k);
    const unsigned long long seq0 = plan_seq_now(a.gate);   // in flight with the record
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_qfull(b), 1);
      mbar_init(bar_qempty(b), 1);
      mbar_init(bar_sfull(b), 1);
      mbar_init(bar_pfull(b), 32 * active_softmax_warps);
    }
    mbar_init(bar_odone, 1);
    mbar_init(bar_fin, 1);
    mbar_init(bar_fresh, 1);
    // every tile-walking thread reads each ring entry: MMA issuer, rotation warps, softmax
    for (int e = 0; e < kChunkRing; ++e) {
      mbar_init(bar_cfull0 + 8u * e, 1);
      mbar_init(bar_cempty0 + 8u * e, 1 + kRotThreads + 32 * active_softmax_warps);
    }
    fence_mbar_init();
    // Meanwhile the first query tile's inputs and the unit's first K/V tile go out from the
    // launch parameters, which need no load.
    const uint32_t want = a.gate.plan_seq ? (uint32_t)a.gate.plan_expect : 0u;
    int early = 0;
    if (lu_group >= 0 && lu_group < a.P * a.H_kv && a.qrow == nullptr) {
      // The first query tile's inputs into L2 before the K/V loads start: the rotation warps
      // read them right after the wait, and would otherwise queue behind every CTA's tiles.
      const int p = lu_group / a.H_kv, h = lu_group % a.H_kv;
      for (int w = 0; w < a.W; ++w)       // query row w's G heads of this KV head
        bulk_prefetch_l2(a.q + ((size_t)(p * a.W + w) * a.H_q + (size_t)h * a.G) * D,
                         (uint32_t)(a.G * D * 2));
      if (lu_delta0 >= 0 && lu_delta0 < a.max_position) {
        bulk_prefetch_l2(a.rope_cos + (size_t)lu_delta0 * (D / 2), D / 2 * 4);
        bulk_prefetch_l2(a.rope_sin + (size_t)lu_delta0 * (D / 2), D / 2 * 4);
      }
    }
    if (lu_row0 >= 0 && lu_row0 < a.num_pages * a.H_kv * a.S) {
      tma_prefetch(&maps.k);
      tma_prefetch(&maps.v);
      const int32_t y = (int32_t)(page_base0 * a.H_kv * a.S + lu_row0);
      mbar_arrive_expect_tx(bar_full(0), C::kTileBytes);
      mbar_arrive_expect_tx(bar_full(1), C::kTileBytes);
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h) {
        tma_load_2d(sbase + C::kRingOff + h * C::kHalfBytes, &maps.k, 64 * h, y, bar_full(0),
                    l2_policy_evict_first());
        tma_load_2d(sbase + C::kRingOff + C::kTileBytes + h * C::kHalfBytes, &maps.v, 64 * h, y,
                    bar_full(1), l2_policy_evict_first());
      }
      HW_TRACE_EV(8);
      early = 1;
    }
    *abort = plan_arrived(a.gate, seq0, a.err, KID_ATTN_TC) ? 0 : 1;
    // a vector read before the plan had landed is read again (the plan is complete now)
    if ((uint32_t)uv[0].z != want) uv[0] = __ldcg(urec);
    if ((uint32_t)uv[1].w != want) uv[1] = __ldcg(urec + 1);
    if ((uint32_t)uv[2].z != want) uv[2] = __ldcg(urec + 2);
    Unit uu;
    static_assert(sizeof(Unit) == 48, "unit record: three 16-byte vectors");
    int4* ud = reinterpret_cast<int4*>(&uu);
    ud[0] = uv[0];
    ud[1] = uv[1];
    ud[2] = uv[2];
    uu.flags = early;                   // tells the producer that tile 0 is on its way
    if (*abort) {                       // no plan: an empty unit (the error word says why)
      uu.piece_begin = uu.piece_end = 0;
      uu.seg0 = uu.first_tok = -1;
      uu.fresh_end = uu.fresh_begin;
    } else if (early) {                 // the launch parameters must name the record's tile
      const int32_t rec_row = uu.first_tok < 0 ? -1
          : ((uu.first_tok / a.S) * a.H_kv + uu.group % a.H_kv) * a.S + uu.first_tok % a.S;
      if (rec_row != lu_row0) record_error(a.err, ERR_PLAN, KID_ATTN_TC, blockIdx.x, 6);
    }
    *u_smem = uu;
  }

  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Unit u = *u_smem;
  // (problem, KV head) of the unit, from its group index (no dependent load)
  const Group g{u.group / a.H_kv, u.group % a.H_kv, 0, 0};
  if (threadIdx.x == 0) HW_TRACE_EV(1);

  const int64_t page_base = page_base0;

  // The first query tile (segment slot u.seg0, known from the unit record without a dependent
  // load), finished by warps 2-7 together (the softmax warps have nothing to do before the
  // first S).
  const bool first_q = u.seg0 >= 0 && u.seg0 < a.num_seg_slots;
  const bool fused = a.k_raw != nullptr;      // this kernel writes the step's appended tokens
  if (warp >= 2) {
    if (first_q) {
      if (!pre_q)
        rotate_tile<D, T, kThreads - 64>(a, g, u.seg0, u.delta0, smem + C::kQOff, threadIdx.x - 64);
      fence_proxy_async_smem();           // generic-proxy writes -> operands of the MMA
      asm volatile("bar.sync 3, %0;" ::"r"(kThreads - 64) : "memory");
      if (threadIdx.x == 64) {
        mbar_arrive(bar_qfull(0));
        HW_TRACE_EV(2);
      }
    }
  }

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      uint32_t j = 0;          // K/V ring loads issued
      uint32_t pub = 0;        // chunk-ring entries published
      bool ok = true;
      // Tiles holding tokens of the current step are written by this CTA's rotation warps
      // (fused append) or by the append kernel, which may still run (this grid is its
      // programmatic dependent): wait for those writes before the first such tile.  Tiles of
      // older tokens are streamed right away.
      bool waited = false;
      auto publish = [&](int32_t b, int32_t e) -> bool {
        const uint32_t slot = pub % kChunkRing;
        if (pub >= (uint32_t)kChunkRing &&
            !mbar_wait(bar_cempty0 + 8u * slot, ((pub / kChunkRing) - 1) & 1, abort, kWaitLimitNs))
          return false;
        cring[slot] = make_int2(b, e);
        mbar_arrive(bar_cfull0 + 8u * slot);          // release: the entry is visible to readers
        ++pub;
        return true;
      };
      // Issue the K and V loads of tile j (two ring slots) at pool row y.
      auto issue_tile = [&](int32_t y) -> bool {
        for (int part = 0; part < 2; ++part, ++j) {
          const int s = j % C::kSlots;
          if (j >= (uint32_t)C::kSlots &&
              !mbar_wait(bar_empty(s), ((j / C::kSlots) - 1) & 1, abort, kWaitLimitNs))
            return false;
          if (part == 0) HW_TRACE_EV(8 + 4 * (j >> 1));
          mbar_arrive_expect_tx(bar_full(s), C::kTileBytes);
          const CUtensorMap* m = part == 0 ? &maps.k : &maps.v;
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(ring + s * C::kTileBytes + h * C::kHalfBytes, m, 64 * h, y, bar_full(s),
                        policy);
        }
        return true;
      };
      // The unit's first tile may have gone out during set-up (see above): its two ring slots
      // are then taken.
      const bool early = u.flags != 0;
      if (early) j = 2;
      auto load_range = [&](int32_t b, int32_t e) -> bool {
        for (int32_t pi = b; pi < e; ++pi) {
          if (early && pi == u.piece_begin) continue;  // issued above
          const Piece pc = a.pieces[pi];
          const bool valid = pc.page >= 0 && pc.page < a.num_pages && pc.slot0 >= 0 &&
                             pc.ntok >= 1 && pc.ntok <= kTile && pc.slot0 + pc.ntok <= a.S &&
                             pc.seg_slot >= 0 &&
                             pc.seg_slot < a.num_seg_slots;
          if (!valid) continue;                        // every role skips it the same way
          if (pc.fresh && !waited) {
            if (fused) {
              if (!mbar_wait(bar_fresh, 0, abort, kWaitLimitNs)) return false;
            } else {
              pdl_wait();
            }
            waited = true;
            HW_TRACE_EV(248);
          }
          if (!issue_tile((int32_t)(((page_base + pc.page) * a.H_kv + g.h) * a.S + pc.slot0)))
            return false;
        }
        return true;
      };
      // The unit's pieces in plan order, then the end of the sequence.
      if (ok && u.piece_end > u.piece_begin)
        ok = publish(u.piece_begin, u.piece_end) && load_range(u.piece_begin, u.piece_end);
      publish(0, -1);                                  // end of the sequence (also on abort)
      HW_TRACE_EV(3);
      // Drain: every copy issued must have landed before the CTA can exit, abort or not.
      bool drained = true;
      for (uint32_t s = 0; s < (uint32_t)C::kSlots && s < j; ++s) {
        const uint32_t last = s + ((j - 1 - s) / C::kSlots) * C::kSlots;
        drained = mbar_wait_drain(bar_full(s), (last / C::kSlots) & 1, kWaitLimitNs) && drained;
      }
      if ((!ok && (*abort)) || !drained) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc1 = idesc_bf16(kRowsM, kTile, 0, 0);
      constexpr uint32_t idesc2 = idesc_bf16(kRowsM, D, 0, 1);
      TileWalker tw;
      tw.init(a, cring, bar_cfull0, bar_cempty0, abort);
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
        const uint32_t p_tmem = tmem + (b ? kColP1 : kColP0);
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
          // the previous segment's query buffer is free once every MMA issued so far is done
          if (seg > 0) mma_commit(bar_qempty(qbuf));
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
        HW_TRACE_EV(9 + 4 * i);
        mma_commit(bar_empty(s));
        mma_commit(bar_sfull(b));
        if (i > 0) ok = issue_mma2(i - 1);
        ++i;
      }
      if (ok && i > 0) ok = issue_mma2(i - 1);
      HW_TRACE_EV(4);
      // Every MMA issued must have completed before TMEM is freed, abort or not.
      bool drained = true;
      if (issued_any) {
        mma_commit(bar_fin);
        drained = mbar_wait_drain(bar_fin, 0, kWaitLimitNs);
      }
      if ((!ok && (*abort)) || !drained) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 1);
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------------------------------------------------------- query rotation
    // Fused append first (the producer holds this unit's tiles of new tokens until it is
    // written), then the query tiles of the unit's later segments, into the two query buffers
    // in turn.
    const int tid = threadIdx.x - 64;
    if (fused) {
      append_fresh<D, kRotThreads>(a, g.h, u.fresh_begin, u.fresh_end, tid, KID_ATTN_TC);
      fence_proxy_async_global();         // generic-proxy pool writes -> this CTA's TMA loads
      asm volatile("bar.sync 4, %0;" ::"r"(kRotThreads) : "memory");
      if (tid == 0) mbar_arrive(bar_fresh);
    }
    TileWalker tw;
    tw.init(a, cring, bar_cfull0, bar_cempty0, abort);
    TileInfo t;
    bool new_seg;
    uint32_t seg = 0;
    bool ok = true;
    while (ok && tw.next(&t, &new_seg)) {
      if (!new_seg) continue;
      if (seg == 0 && first_q) {
        // built above; the plan names the unit's first segment in u.seg0
        if (t.seg_slot != u.seg0 && tid == 0) record_error(a.err, ERR_PLAN, KID_ATTN_TC, blockIdx.x, 4);
        ++seg;
        continue;
      }
      const int qb = seg & 1;
      if (seg >= 2) ok = mbar_wait(bar_qempty(qb), ((seg >> 1) - 1) & 1, abort, kWaitLimitNs);
      if (!ok) break;
      rotate_tile<D, T, kRotThreads>(a, g, t.seg_slot, -1, smem + C::kQOff + qb * C::kQBytes, tid);
      fence_proxy_async_smem();           // generic-proxy writes -> operands of the MMA
      asm volatile("bar.sync 4, %0;" ::"r"(kRotThreads) : "memory");
      if (tid == 0) {
        mbar_arrive(bar_qfull(qb));
        HW_TRACE_EV(249);
      }
      ++seg;
    }
#ifdef HW_TRACE
    if (tid == 0 && blockIdx.x < kTraceCtas) g_trace[blockIdx.x][254] = seg;
#endif
    if (!ok && (*abort) && tid == 0) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 3);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax / epilogue
    // Softmax warp q takes the token columns [cq * 128/T, (cq + 1) * 128/T) of every tile,
    // cq = q / (4/T), for query rows 32 * (q % (4/T)) + lane.  The column range is the same for
    // the whole warp, so S and P move with warp-uniform TMEM addresses, and every lane keeps
    // its own running max, sum and O row over its columns; the epilogue merges the T lanes of
    // a row by log-sum-exp.
    const int wq = warp - 4;                  // TMEM lane quarter of this warp
    const int cq = wq / WPC;                  // column chunk of this warp
    const int r = 32 * (wq % WPC) + lane;     // query row of this lane
    if (32 * (wq % WPC) < R) {
      const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
      {
        // This warp only ever writes its own P columns: zero both P buffers once.
        uint32_t z[kTile / 2];
#pragma unroll
        for (int e = 0; e < kTile / 2; ++e) z[e] = 0u;
        tmem_st64_sync(tmem + lane_off + kColP0, z);
        tmem_st64_sync(tmem + lane_off + kColP1, z);
      }
      float m_run = -CUDART_INF_F, l_sum = 0.f;
      TileWalker tw;
      tw.init(a, cring, bar_cfull0, bar_cempty0, abort);
      TileInfo t;
      bool new_seg;
      uint32_t i = 0;
      bool ok = true;
      bool row_visible = false;
      int row_cap = 0x7fffffff;
      while (tw.next(&t, &new_seg)) {
        if (new_seg) {
          row_visible = r < R && a.delta[(size_t)t.seg_slot * a.W + r / a.G] >= 0;
          // causal cut (several query tokens per worker): tokens of the segment it may see
          row_cap = (row_visible && a.vlen) ? a.vlen[(size_t)t.seg_slot * a.W + r / a.G]
                                            : 0x7fffffff;
        }
        const int b = i & 1;
        // (warp-uniform outcome: the TMEM accesses below need every lane)
        if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(b), (i >> 1) & 1, abort, kWaitLimitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (threadIdx.x == 128) HW_TRACE_EV(10 + 4 * i);
        float s[CPT];
        {
          uint32_t v[CPT];
          tmem_ld_sync<CPT>(tmem + lane_off + (b ? kColS1 : kColS0) + cq * CPT, v);
#pragma unroll
          for (int k = 0; k < CPT; ++k) s[k] = __uint_as_float(v[k]);
        }
        const int nv = min(t.nvalid, row_cap - t.pos0);   // (nvalid unless cut)
        const int limit = row_visible ? max(0, min(CPT, nv - cq * CPT)) : 0;
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
          if (k >= limit) s[k] = -CUDART_INF_F;
          mx = fmaxf(mx, s[k]);
        }
        const bool need = mx > m_run + kRescaleThreshold || (m_run == -CUDART_INF_F && mx > m_run);
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? fmaxf(m_run, mx) : m_run;
          const float alpha = (m_run == -CUDART_INF_F) ? 0.f : fast_exp2(m_run - m_new);
          const float sc = need ? alpha : 1.f;
          l_sum *= sc;
          if (i > 0) {
            // O holds MMA2 results up to tile i-1: wait for the last of them, rescale the row.
            if (!__all_sync(0xffffffffu, mbar_wait(bar_odone, (i - 1) & 1, abort, kWaitLimitNs))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32_sync(tmem + lane_off + kColO + 32 * c, v);
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * sc);
              tmem_st32_sync(tmem + lane_off + kColO + 32 * c, v);
            }
          }
          m_run = m_new;
        }
        const float m_use = (m_run == -CUDART_INF_F) ? 0.f : m_run;
        uint32_t own[PCPT];
#pragma unroll
        for (int e = 0; e < PCPT; ++e) {
          const float p0 = fast_exp2(s[2 * e] - m_use);
          const float p1 = fast_exp2(s[2 * e + 1] - m_use);
          l_sum += p0 + p1;
          const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
          own[e] = *reinterpret_cast<const uint32_t*>(&pp);
        }
        tmem_st_sync<PCPT>(tmem + lane_off + (b ? kColP1 : kColP0) + cq * PCPT, own);
        tc_fence_before();
        mbar_arrive(bar_pfull(b));
        if (threadIdx.x == 128) HW_TRACE_EV(11 + 4 * i);
        ++i;
      }
      if (threadIdx.x == 128) HW_TRACE_EV(5);
      // Epilogue.  Each lane's (O row, max, sum) over its columns goes to shared memory (the
      // K/V ring is idle once the last MMA has completed) as stage[chunk][row][PS], with the
      // log-sum-exp weights of the T chunks of every row; after the role branches all warps
      // merge the chunks and store the unit's partials.
      // Wait for every MMA through the single-use `fin` barrier, not o_done: here o_done may be
      // two phases behind (the last two P.V products can both be in flight), and a parity
      // wait cannot tell that apart from "done".
      constexpr int PS = part_stride(D);
      bool have = ok && i > 0;
      if (have) {
        have = mbar_wait(bar_fin, 0, abort, kWaitLimitNs);
        tc_fence_after();
      }
      have = __all_sync(0xffffffffu, have);
      if (threadIdx.x == 128) HW_TRACE_EV(250);
      float* stage = reinterpret_cast<float*>(smem + C::kRingOff);
      const bool writer = r < R;
      float4* srow = reinterpret_cast<float4*>(stage + ((size_t)cq * R + r) * PS);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        if (have) tmem_ld32_sync(tmem + lane_off + kColO + 32 * c, v);
        if (writer) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            srow[8 * c + e] = have ? make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                 __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (writer)
        srow[D / 4] = make_float4(have ? m_run : -CUDART_INF_F, have ? l_sum : 0.f, 0.f, 0.f);
      const int nthr = 32 * active_softmax_warps;
      asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
      if (threadIdx.x == 128) HW_TRACE_EV(251);
      // Per row: M = max over the T chunks, each chunk's weight 2^(m_j - M), and the merged
      // sum L = sum_j l_j 2^(m_j - M); the merged rows are written after the role branches by
      // all warps.
      float* rowM = stage + (size_t)T * R * PS;
      float* rowW = rowM + R;                                  // [T][R]
      float* rowL = rowW + T * R;
      for (int rr = threadIdx.x - 128; rr < R; rr += nthr) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < T; ++j) M = fmaxf(M, stage[((size_t)j * R + rr) * PS + D]);
        rowM[rr] = M;
        float Ls = 0.f;
#pragma unroll
        for (int j = 0; j < T; ++j) {
          const float wj =
              (M == -CUDART_INF_F) ? 0.f : fast_exp2(stage[((size_t)j * R + rr) * PS + D] - M);
          rowW[j * R + rr] = wj;
          Ls = fmaf(stage[((size_t)j * R + rr) * PS + D + 1], wj, Ls);
        }
        rowL[rr] = Ls;
      }
      if (threadIdx.x == 128) HW_TRACE_EV(252);
      if (!ok && (*abort) && lane == 0) record_error(a.err, ERR_TIMEOUT, KID_ATTN_TC, blockIdx.x, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  // The merge kernel may launch once every CTA is here (it waits for this grid before reading
  // the partials).  Triggering right after the softmax loop instead measured 1 % slower per
  // chained step: the merge's CTAs then take the SMs that free up first.
  if (threadIdx.x == 0) pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  {
    // The unit's partials, [R][PS] fp32 -- unnormalised o, then (M, L, 0, 0) in the log2
    // domain -- from the T staged chunks of every row: all eight warps, a warp per row and a
    // float4 column per lane (coalesced 16-byte stores).
    constexpr int PS = part_stride(D);
    constexpr int Q4 = PS / 4, DQ = D / 4;
    const float* stage = reinterpret_cast<const float*>(smem + C::kRingOff);
    const float4* st4 = reinterpret_cast<const float4*>(stage);
    const float* rowM = stage + (size_t)T * R * PS;
    const float* rowW = rowM + R;
    const float* rowL = rowW + T * R;
    float4* part = reinterpret_cast<float4*>(a.partials + (size_t)blockIdx.x * R * PS);
#pragma unroll 2
    for (int rr = warp; rr < R; rr += kThreads / 32) {
      if (lane < DQ) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < T; ++j) {
          const float wj = rowW[j * R + rr];
          const float4 x = st4[((size_t)j * R + rr) * Q4 + lane];
          acc.x = fmaf(x.x, wj, acc.x);
          acc.y = fmaf(x.y, wj, acc.y);
          acc.z = fmaf(x.z, wj, acc.z);
          acc.w = fmaf(x.w, wj, acc.w);
        }
        part[(size_t)rr * Q4 + lane] = acc;
      }
      if (lane == (DQ < 32 ? DQ : 0))                         // a spare lane, else lane 0
        part[(size_t)rr * Q4 + DQ] = make_float4(rowM[rr], rowL[rr], 0.f, 0.f);
    }
    if (threadIdx.x == 128) HW_TRACE_EV(6);
  }
  if (threadIdx.x == 0) HW_TRACE_EV(7);
}

}  // namespace

#ifdef HW_TRACE
// Debug builds only: copy out / clear the timeline stamps (uint64 [160][256], ns).
extern "C" int hw_trace_read(void* dst, size_t bytes) {
  const size_t n = bytes < sizeof(g_trace) ? bytes : sizeof(g_trace);
  return (int)cudaMemcpyFromSymbol(dst, g_trace, n);
}
extern "C" int hw_trace_clear(void) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_trace);
  if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(g_trace));
  return (int)e;
}
#endif

template <int D, int T>
static void launch_tc_dt(const AttnArgs& a, const TcMaps& maps, const LaunchUnits& lu, int layer,
                         cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  using C = Cfg<D>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = e0 ? 0 : 1;        // a timing event in between ends the programmatic chain
  if (e0) cudaEventRecord(e0, s);
  cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, T>, a, maps, (int32_t)layer, lu);
  if (e1) cudaEventRecord(e1, s);
}

template <int D>
static void launch_tc_d(const AttnArgs& a, const TcMaps& maps, const LaunchUnits& lu, int layer,
                        cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
  if (a.rows <= 32)
    launch_tc_dt<D, 4>(a, maps, lu, layer, s, e0, e1);
  else if (a.rows <= 64)
    launch_tc_dt<D, 2>(a, maps, lu, layer, s, e0, e1);
  else
    launch_tc_dt<D, 1>(a, maps, lu, layer, s, e0, e1);
}

template <int D>
static cudaError_t prepare_tc_d() {
  constexpr int smem = (int)Cfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

cudaError_t prepare_attention_tc(int D) { return D == 64 ? prepare_tc_d<64>() : prepare_tc_d<128>(); }

void launch_attention_tc(const AttnArgs& a, const TcMaps& maps, const LaunchUnits& lu, int layer,
                         cudaStream_t s, cudaEvent_t ev_before, cudaEvent_t ev_after) {
  if (a.num_units <= 0) return;
  if (a.D == 64)
    launch_tc_d<64>(a, maps, lu, layer, s, ev_before, ev_after);
  else
    launch_tc_d<128>(a, maps, lu, layer, s, ev_before, ev_after);
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
