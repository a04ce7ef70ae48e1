// Internal declarations of libhogwild: the per-call plans the host uploads, the kernel
// argument blocks, and the launchers.  Host planning lives in hw_api.cpp, kernels in the .cu
// files.  Nothing here is part of the public ABI (include/hogwild.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hogwild.h"

namespace hw {

// Device error word layout (uint32[4] at the start of the workspace):
//   [0] OR of error bits, [1] id of the first kernel that failed, [2], [3] its details.
enum : uint32_t {
  ERR_PAGE_RANGE = 1u << 0,    // a physical page index outside [0, num_pages)
  ERR_SLOT_RANGE = 1u << 1,    // a slot range outside the page
  ERR_POS_RANGE = 1u << 2,     // a RoPE position outside [0, max_position)
  ERR_TIMEOUT = 1u << 3,       // a bounded wait gave up
  ERR_PLAN = 1u << 4,          // an inconsistent plan entry
};
enum : uint32_t { KID_APPEND = 1, KID_ATTN_FMA = 2, KID_MERGE = 3, KID_ATTN_TC = 4, KID_COMPACT = 5 };

// One run of appended tokens: ntok consecutive tokens of one block that land in one page.
struct AppendRun {
  int32_t src_tok;   // first token in k_raw / v_raw
  int32_t ntok;
  int32_t page;      // physical page
  int32_t slot0;     // slot of the first token in the page
  int32_t pos0;      // block-local position of the first token (RoPE angle)
  int32_t pad;
};

// Compaction: n tokens copied from (src_page, src_slot ..) to (dst_page, dst_slot ..) of every
// layer, keys turned by rot positions on the way (the run never crosses a page on either side).
struct CompactRun {
  int32_t src_page, src_slot, dst_page, dst_slot, n, rot;
};

struct CompactArgs {
  const CompactRun* runs;
  int32_t num_runs, num_layers;
  __nv_bfloat16* k_pool;      // pool bases: [L][num_pages][H_kv][S][D]
  __nv_bfloat16* v_pool;
  size_t layer_elems;
  const float* rope_cos;
  const float* rope_sin;
  uint32_t* err;
  int32_t H_kv, D, S, num_pages, max_position;
};

// A piece: <= 128 consecutive tokens (one kernel tile) of one segment, inside one page.
struct Piece {
  int32_t seg_slot;  // row of the delta table (problem, segment) -> per-worker rotation
  int32_t page;
  int32_t slot0;
  int32_t ntok;
  int32_t fresh;     // 1 if the piece holds tokens appended in the current step
  int32_t pos0;      // block-local position of its first token
};

// A token appended in the current step whose K/V the tensor-core attention kernel writes
// itself (fused append): pool (page, slot), block-local position, row of k_raw / v_raw.
struct FreshTok {
  int32_t page;
  int32_t slot;
  int32_t pos;
  int32_t src;
};

// Row stride (floats) of a partial result: o[D], m, l, 2 pad -- 16-byte aligned rows.
__host__ __device__ constexpr int part_stride(int D) { return D + 4; }

// A unit: consecutive pieces of one (problem, KV head) group, one CTA, one partial result.
// Read as three 16-byte vectors, possibly before the plan's arrival is confirmed: each vector
// carries the low 32 bits of the plan's sequence number (seq, seq_b, seq_c; 0 when the plan is
// not gated), and a vector whose copy matches belongs to the current plan.
struct __align__(16) Unit {
  int32_t first_tok;  // page * S + slot of the first piece if the kernel may load it before
                      // it waits for the kernel it follows, else -1: a piece with no token of
                      // this step (the kernel writes or waits for those) and none written by
                      // the previous step or a compaction since (a launch that may still be in
                      // flight could have written them)
  int32_t group;      // p * H_kv + h
  uint32_t seq;
  int32_t seg0;       // seg_slot of the first piece, -1 if the unit has none
  int32_t piece_begin;
  int32_t piece_end;
  int32_t delta0;     // the rotation of seg0 if it is the same for every worker, else -1
  uint32_t seq_b;
  int32_t fresh_begin, fresh_end;  // appended tokens it writes, in the FreshTok table
  uint32_t seq_c;
  int32_t flags;      // kernel-side use
};

// What the tensor-core kernel needs of its unit before it has read any of the plan, for the
// first kLaunchUnits CTAs of a launch, passed as a kernel parameter (no load, always current):
// the layer-relative pool row of the unit's first K/V tile if it may be loaded before the
// kernel waits for the one it follows (Unit::first_tok), and the group, first segment slot and
// shared rotation of the unit's first query tile (Unit::group, seg0, delta0).  -1 = none.
constexpr int kLaunchUnits = 160;
struct LaunchUnits {
  int32_t row0[kLaunchUnits];     // ((page * H_kv + h) * S + slot), layer offset not included
  int32_t group[kLaunchUnits];
  int32_t seg0[kLaunchUnits];
  int32_t delta0[kLaunchUnits];
};

// A group: one (problem, KV head); its units are [unit_begin, unit_end).
struct Group {
  int32_t p;
  int32_t h;
  int32_t unit_begin;
  int32_t unit_end;
};

// A plan goes up on the library's copy stream, followed by an 8-byte sequence number; a kernel
// that reads the plan first checks that *plan_seq == plan_expect (spinning, bounded, while the
// copy is still in flight), so the compute stream needs no wait on the copy stream.  plan_seq
// is null when the plan was copied in stream order.
struct PlanGate {
  const unsigned long long* plan_seq;
  unsigned long long plan_expect;
};

struct AppendArgs {
  PlanGate gate;
  const AppendRun* runs;
  int32_t num_runs;
  int32_t max_run;
  const __nv_bfloat16* k_raw;
  const __nv_bfloat16* v_raw;
  __nv_bfloat16* k_layer;     // pool base of this layer: [num_pages][H_kv][S][D]
  __nv_bfloat16* v_layer;
  const float* rope_cos;      // [max_position][D/2]
  const float* rope_sin;
  uint32_t* err;
  int32_t H_kv, D, S, num_pages, max_position;
};

struct AttnArgs {
  PlanGate gate;
  const Piece* pieces;
  const Unit* units;
  const Group* groups;
  const int32_t* delta;       // [seg_slots][W]: i_q(w) - view offset, or -1 (not visible)
  // Several query tokens per worker: W counts query rows per problem ("virtual workers"
  // v = (worker, token)), and the two tables below are set; both are null for one query per
  // worker (then v = w and q row = p * W + w).
  const int32_t* qrow;        // [P][W]: row of q / out / lse of (problem, v), or -1 (padding)
  const int32_t* vlen;        // [seg_slots][W]: tokens of the segment v may see (causal cut)
  const FreshTok* fresh;      // appended tokens, per problem in piece order (fused append)
  const __nv_bfloat16* k_raw; // fused append: this layer's new keys / values [n][H_kv][D],
  const __nv_bfloat16* v_raw; //   or null when the append kernel has written them already
  int32_t num_units, num_groups, num_seg_slots;
  __nv_bfloat16* k_layer;     // pool base of this layer: [num_pages][H_kv][S][D]
  __nv_bfloat16* v_layer;
  const __nv_bfloat16* q;     // [P][W][H_q][D]
  void* out;                  // [P][W][H_q][D] bf16 or fp32
  int32_t out_f32;
  float* lse;                 // [P][W][H_q] or null
  float* partials;            // [units][rows][part_stride(D)]: o[D], m, l (log2 domain), pad
  const float* rope_cos;
  const float* rope_sin;
  uint32_t* err;
  int32_t P, W, H_q, H_kv, G, D, S, num_pages, max_position, rows;
  float scale_log2;           // log2(e) / sqrt(D)
};

// TMA descriptors of the two pools, each viewed as a 2-D tensor [L*pages*H_kv*S rows][D] bf16
// with {64 elements, 128 rows} boxes and 128-byte swizzle.
struct TcMaps {
  CUtensorMap k;
  CUtensorMap v;
};

// Per-device kernel attributes (shared-memory limits), set once when a context is created.
cudaError_t prepare_attention_fma(int D);
cudaError_t prepare_attention_tc(int D);

void launch_append(const AppendArgs& a, cudaStream_t s);
void launch_compact(const CompactArgs& a, cudaStream_t s);
// The CUDA-core attention kernel (fewer than 16 query rows), K/V tiles staged through the same
// tensor maps as the tensor-core kernel; a programmatic dependent of whatever precedes it.
void launch_attention_fma(const AttnArgs& a, const TcMaps& maps, int layer, cudaStream_t s);
// Launches the attention kernel; ev_before / ev_after (optional) are recorded directly around
// it (and it is then launched without programmatic chaining).
void launch_attention_tc(const AttnArgs& a, const TcMaps& maps, const LaunchUnits& lu, int layer,
                         cudaStream_t s, cudaEvent_t ev_before = nullptr,
                         cudaEvent_t ev_after = nullptr);
// The merge of the units' partials.  pdl: launch as a programmatic dependent of the preceding
// kernel (it waits for its writes).  max_group_units (the most units of any group) sets how many
// warps share a query row.
void launch_merge(const AttnArgs& a, cudaStream_t s, bool pdl, int max_group_units);
bool make_tc_maps(const hw_config& cfg, void* k_pool, void* v_pool, TcMaps* out);

// HW_OK for cudaSuccess; otherwise records the error for hw_last_cuda_error and returns
// HW_ERR_CUDA.
hw_status cuda_status(cudaError_t e);

// hw_concurrent_attention with the plan and the partial results in `scratch` (device).
hw_status attention_into_scratch(hw_ctx* c, int32_t layer, const void* q, void* out,
                                 int32_t out_dtype, float* lse, void* stream, char* scratch,
                                 size_t scratch_bytes);

}  // namespace hw
