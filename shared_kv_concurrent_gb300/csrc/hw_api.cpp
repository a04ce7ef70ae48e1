// Host side of libhogwild: argument checking, the cache's host tables (segments, page
// allocator, commits), per-call plans and kernel launches.  See include/hogwild.h for the
// contract of every entry point.
//
// The cache model is Hogwild! Inference's (summary at gentlecold.top): a common block plus one
// current block per worker, K/V at block-local positions (section 9); views common ++ other
// workers ascending ++ own (sections 4 and 6); append before attention and paragraph commits
// at step end (section 8).  The host is the single owner of the tables: it knows how many
// tokens every call appends, so no call ever reads state back from the GPU.
#include "hogwild.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "hw_internal.h"

namespace {

constexpr int kMaxSlots = 32;          // pinned staging / device plan slots in flight, at most
constexpr size_t kSlotBudget = 64u << 20;  // ... and at most this many bytes of them (>= 4 slots)
constexpr size_t kAlign = 256;
constexpr int kPieceMax = 128;         // tokens per piece = one kernel tile (never crosses a page)
constexpr int kProfPairs = 4096;       // timed launches kept per hw_profile_read
// A step whose blocks each append at most this many tokens has them written by the attention
// kernel itself (fused append, either kernel); larger appends use the append kernel.
constexpr int kFuseTok = 16;
constexpr int kMaxRows = 128;          // query rows of one (problem, KV head): one MMA tile
// Tensor-core plans: about this many tiles per SM per wave of units, at most kMaxWaves waves.
constexpr int64_t kWaveTiles = 24;
constexpr int64_t kMaxWaves = 4;

thread_local int g_cuda_err = 0;
// Plan sequence numbers, unique in the process: a slot word left by an earlier context in
// recycled memory never equals a number this context waits for.
std::atomic<uint64_t> g_upload_seq{0};
std::mutex g_msg_mu;
std::string g_cuda_msg;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

hw_status cuda_fail(cudaError_t e) {
  g_cuda_err = (int)e;
  std::lock_guard<std::mutex> lk(g_msg_mu);
  g_cuda_msg = cudaGetErrorString(e);
  return HW_ERR_CUDA;
}

#define HW_CUDA(call)                              \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_);   \
  } while (0)

struct Layout {
  size_t err, cos, sin, slots, partials, total;
  size_t slot_bytes, slot_seq_off;   // a slot ends with the plan's 8-byte sequence number
  int32_t max_segments, max_append, max_pieces, max_units, max_seg_slots, rows;
  int32_t num_slots, max_fresh;
};

bool valid_config(const hw_config* c) {
  if (!c) return false;
  if (c->num_problems < 1 || c->num_workers < 1 || c->num_layers < 1) return false;
  if (c->num_kv_heads < 1 || c->num_q_heads < c->num_kv_heads) return false;
  if (c->num_q_heads % c->num_kv_heads) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->page_size < 128 || c->page_size % 128) return false;
  if (c->contiguous != 0 && c->contiguous != 1) return false;
  if (c->num_pages < 1 || c->max_position < 1) return false;
  if (c->max_segments < 0 || c->max_append_tokens < 0) return false;
  if (!(c->rope_theta > 1.0) || !std::isfinite(c->rope_theta)) return false;
  if (c->layout < HW_LAYOUT_COMBINED || c->layout > HW_LAYOUT_NO_SYNC || c->reserved != 0)
    return false;
  const int64_t rows = (int64_t)c->num_workers * (c->num_q_heads / c->num_kv_heads);
  if (rows > 128) return false;
  const int64_t pool_tokens = (int64_t)c->num_pages * c->page_size;
  if (pool_tokens > (1ll << 30) || c->max_position > (1 << 26)) return false;
  return true;
}

Layout make_layout(const hw_config* c) {
  Layout L{};
  const int64_t P = c->num_problems, W = c->num_workers, H = c->num_kv_heads;
  L.rows = (int32_t)(W * (c->num_q_heads / c->num_kv_heads));
  L.max_segments = c->max_segments ? c->max_segments : (int32_t)(P * (1 + 4 * W));
  const int64_t pool_tokens = (int64_t)c->num_pages * c->page_size;
  L.max_append = c->max_append_tokens ? c->max_append_tokens : (int32_t)pool_tokens;
  // Pieces are listed once per problem (shared by its KV heads); a piece never leaves its
  // page and pieces start every kPieceMax slots of it, so a page holds at most
  // ceil(S / kPieceMax) of them.
  L.max_pieces = (int32_t)((int64_t)c->num_pages * ((c->page_size + kPieceMax - 1) / kPieceMax) + 1);
  L.max_units = (int32_t)(P * H + 2048);
  L.max_seg_slots = L.max_segments;
  L.max_fresh = (int32_t)(P * (W + 1) * kFuseTok);
  const size_t runs = (size_t)P * (W + 1) + (size_t)L.max_append / 128 + 2;
  const size_t append_bytes = runs * sizeof(hw::AppendRun);
  // Rotation tables are [segment slot][query rows per problem / G]: W wide for one query per
  // worker, up to 128 / G wide for several (hw_concurrent_attention_mq), which adds the causal
  // length table of the same shape and the query-row map.
  const int64_t Wt = std::max<int64_t>(W, kMaxRows / (c->num_q_heads / c->num_kv_heads));
  const size_t attn_bytes = align_up((size_t)L.max_pieces * sizeof(hw::Piece), 16) +
                            align_up((size_t)L.max_units * sizeof(hw::Unit), 16) +
                            align_up((size_t)P * H * sizeof(hw::Group), 16) +
                            2 * align_up((size_t)L.max_seg_slots * Wt * sizeof(int32_t), 16) +
                            align_up((size_t)P * Wt * sizeof(int32_t), 16) +
                            align_up((size_t)L.max_fresh * sizeof(hw::FreshTok), 16);
  // A slot holds a step's append runs followed by its attention plan (uploaded together), and
  // last the plan's sequence number.
  L.slot_seq_off = align_up(append_bytes, kAlign) + align_up(attn_bytes, kAlign);
  L.slot_bytes = L.slot_seq_off + kAlign;
  // Staging slots let the host run that many calls ahead of the device.
  L.num_slots = (int32_t)std::max<size_t>(4, std::min<size_t>(kMaxSlots, kSlotBudget / L.slot_bytes));
  size_t off = 0;
  L.err = off;
  off += kAlign;
  const size_t tab = align_up((size_t)c->max_position * (c->head_dim / 2) * sizeof(float), kAlign);
  L.cos = off;
  off += tab;
  L.sin = off;
  off += tab;
  L.slots = off;
  off += (size_t)L.num_slots * L.slot_bytes;
  L.partials = off;
  off += align_up((size_t)L.max_units * L.rows * hw::part_stride(c->head_dim) * sizeof(float), kAlign);
  L.total = off;
  return L;
}

// Offsets of the arrays of an attention plan inside its buffer, and their sizes.
struct PlanOffsets {
  size_t pieces, units, groups, delta, vlen, qrow, fresh, bytes;
  int32_t num_pieces, num_units, num_groups, num_seg_slots, num_fresh;
  int32_t width;                       // columns of the rotation table (query rows / G)
  int32_t max_group_units;             // the most units of any (problem, KV head) group
};

// An append-only array that keeps its storage across plans: `grow(k)` hands out k slots to be
// written by index (no per-element capacity check, no zero-fill of slots that are written).
template <class T>
struct Buf {
  std::vector<T> v;
  size_t n = 0;
  void clear() { n = 0; }
  T* grow(size_t k) {
    if (n + k > v.size()) v.resize(std::max<size_t>(2 * v.size(), n + k + 64));
    T* p = v.data() + n;
    n += k;
    return p;
  }
  void push_back(const T& x) { *grow(1) = x; }
  size_t size() const { return n; }
  bool empty() const { return n == 0; }
  T* data() { return v.data(); }
  const T* data() const { return v.data(); }
  T& operator[](size_t i) { return v[i]; }
  const T& operator[](size_t i) const { return v[i]; }
  T* begin() { return v.data(); }
  T* end() { return v.data() + n; }
};

// Reused host buffers of the plan builder (no allocation per call once they have grown).
struct PlanScratch {
  struct Part {
    int32_t unit, ref, t0, t1;        // tiles [t0, t1) of segment reference `ref` go to `unit`
  };
  // The plan's arrays are built here (memory the planner keeps warm) and copied into the
  // staging slot in one pass at the end: a slot comes back only after the others have been
  // used, and stores scattered over its cold lines cost more than the copy.
  Buf<hw::Piece> pieces;
  Buf<hw::Unit> units;
  Buf<hw::Group> groups;
  Buf<hw::FreshTok> fresh;
  std::vector<int32_t> delta, refs, src_base, ref_of, view_ref, vlen, qrow;
  Buf<uint8_t> piece_early;             // the piece may be loaded before the programmatic wait
  int32_t qrow_next = 0;
  std::vector<int64_t> view_off;
  // per segment reference: its tokens [ref_lo, ref_hi) are attended (the whole segment, or its
  // part inside an entry range), in ref_tiles tiles starting at tile ref_lo / kPieceMax
  std::vector<int32_t> ref_lo, ref_hi;
  std::vector<int32_t> ref_sid, ref_slot, ref_tiles, prob_ref_begin, prob_common_refs, unit_rem,
      order, prob_units;
  std::vector<int64_t> prob_tiles;
  std::vector<Part> parts;
};

// The pieces of a segment as the planner last emitted them, with what they depend on: a plan
// reuses them while all of it is unchanged (common segments between decode steps).
struct PieceCache {
  int32_t seg_slot = -1, lo = -1, hi = -1, len = -1, recent = -1, npages = -1;
  std::vector<hw::Piece> pieces;
  std::vector<uint8_t> early;
};

struct Seg {
  int32_t problem, origin, length, pending;
  std::vector<int32_t> pages;
  PieceCache cache;
  // Positions >= recent_from were written in the last completed step or by a compaction
  // since: the next attention launch may not load them before its programmatic wait.
  int32_t recent_from = INT32_MAX;
  int32_t visible() const { return length + pending; }
};

}  // namespace

struct hw_ctx {
  hw_config cfg{};
  Layout lay{};
  int32_t G = 0, rows = 0, num_sms = 0;
  __nv_bfloat16* k_pool = nullptr;
  __nv_bfloat16* v_pool = nullptr;
  char* ws = nullptr;
  size_t layer_elems = 0;
  char* h_slots = nullptr;                 // pinned staging, lay.num_slots * slot_bytes
  cudaEvent_t slot_ev[kMaxSlots] = {};     // compute stream: last kernel reading the slot
  bool slot_used[kMaxSlots] = {};
  // Plans go up on a stream of their own, each followed by its sequence number, which the
  // kernels check before reading the plan: the compute stream never waits on the copy stream,
  // so its kernels stay back to back (programmatic launch chaining across calls).
  cudaStream_t copy_stream = nullptr;
  int next_slot = 0;
  int32_t expire_plans = 0;                // fault injection: plans announced with a dead number
  hw::TcMaps maps{};
  bool use_tc = false;                     // tensor-core attention (W*G >= 16 rows)
  // CTAs of one wave of units: the tensor-core kernel holds an SM alone (its shared memory and
  // TMEM); the CUDA-core kernel runs two CTAs per SM, one computing while the other's tile lands.
  int64_t wave_ctas() const { return use_tc ? num_sms : 2 * (int64_t)num_sms; }
  std::deque<int32_t> free_pages;
  std::vector<Seg> segs;
  std::vector<std::vector<int32_t>> common, live;
  bool step_active = false;
  std::vector<int32_t> step_n;
  std::vector<uint8_t> appended;
  // The step's append runs and attention plan, uploaded together by its first append and
  // reused by every layer while the tables stay unchanged (epoch counts table changes).
  uint64_t epoch = 0, step_epoch = ~0ull;
  int step_slot = -1;
  int32_t step_runs = 0, step_max_run = 0;
  size_t step_plan_off = 0;
  bool step_plan_ok = false;
  PlanOffsets step_po{};
  hw::PlanGate step_gate{};
  // Set by hw_decode_step_host while it records the step's appends: the step's plan is then
  // copied on the call's stream, in order with the step's kernels, and needs no sequence word.
  bool plan_in_order = false;
  PlanScratch ps;
  // Fused append: when the step's plan lists its appended tokens (step_fused), hw_append_kv
  // only records the layer's k_raw / v_raw here and the layer's attention kernel writes them;
  // whatever else needs the pool first launches the append kernel (flush_append).
  bool step_fused = false;
  std::vector<const void*> pend_k, pend_v;
  // measurement
  bool prof_on = false;
  int64_t n_launch = 0, n_attn = 0, n_append = 0;
  std::vector<cudaEvent_t> prof_ev;       // 2 * kProfPairs, created on first enable
  std::vector<int8_t> prof_kind;          // 0 = attention, 1 = append, 2 = merge, per pair
  int prof_next = 0;

  // Reserve an event pair for a timed launch (the caller records it); -1 when not timing.
  int prof_reserve(int8_t kind) {
    if (!prof_on || prof_next >= kProfPairs) return -1;
    const int i = prof_next++;
    prof_kind[i] = kind;
    return i;
  }
  // Record the opening event of a timed launch; returns the pair index or -1.
  int prof_begin(cudaStream_t s, int8_t kind) {
    const int i = prof_reserve(kind);
    if (i >= 0) cudaEventRecord(prof_ev[2 * i], s);
    return i;
  }
  void prof_end(int i, cudaStream_t s) {
    if (i >= 0) cudaEventRecord(prof_ev[2 * i + 1], s);
  }

  uint32_t* d_err() const { return reinterpret_cast<uint32_t*>(ws + lay.err); }
  float* d_cos() const { return reinterpret_cast<float*>(ws + lay.cos); }
  float* d_sin() const { return reinterpret_cast<float*>(ws + lay.sin); }
  float* d_partials() const { return reinterpret_cast<float*>(ws + lay.partials); }
  char* d_slot(int i) const { return ws + lay.slots + (size_t)i * lay.slot_bytes; }
  char* h_slot(int i) const { return h_slots + (size_t)i * lay.slot_bytes; }

  int32_t new_segment(int32_t p, int32_t origin) {
    segs.push_back(Seg{p, origin, 0, 0, {}});
    return (int32_t)segs.size() - 1;
  }
  Seg& block(int32_t p, int32_t b) {
    return segs[b == 0 ? common[p].back() : live[p][b - 1]];
  }
  // Worker w's view: (segment, offset, visible length); returns i_q.
  // Worker w's view in the context's layout (summary section 6; section 10 for no-sync): calls
  // f(segment, view offset, visible length) for each non-empty segment in view order and
  // returns the view length (i_q + 1).  A committed paragraph's writer is its segment origin.
  template <class F>
  int64_t for_each_view(int32_t p, int32_t w, F&& f) const {
    int64_t off = 0;
    auto add = [&](int32_t sid) {
      const int32_t n = segs[sid].visible();
      if (n == 0) return;
      f(sid, off, n);
      off += n;
    };
    auto output = [&](int32_t u) {        // worker u's paragraphs, then its current block
      for (int32_t sid : common[p])
        if (segs[sid].origin == u) add(sid);
      add(live[p][u]);
    };
    switch (cfg.layout) {
      case HW_LAYOUT_STEP_WISE:
        for (int32_t sid : common[p]) add(sid);
        add(live[p][w]);
        break;
      case HW_LAYOUT_CONTIGUOUS:
      case HW_LAYOUT_NO_SYNC:
        for (int32_t sid : common[p])
          if (segs[sid].origin < 0) add(sid);
        if (cfg.layout == HW_LAYOUT_CONTIGUOUS)
          for (int32_t u = 0; u < cfg.num_workers; ++u)
            if (u != w) output(u);
        output(w);
        break;
      default:                            // HW_LAYOUT_COMBINED
        for (int32_t sid : common[p]) add(sid);
        for (int32_t u = 0; u < cfg.num_workers; ++u)
          if (u != w) add(live[p][u]);
        add(live[p][w]);
    }
    return off;
  }
  int32_t view(int32_t p, int32_t w, std::vector<int32_t>* ids, std::vector<int32_t>* offs,
               std::vector<int32_t>* lens) const {
    const int64_t total = for_each_view(p, w, [&](int32_t sid, int64_t off, int32_t n) {
      ids->push_back(sid);
      offs->push_back((int32_t)off);
      lens->push_back(n);
    });
    return (int32_t)(total - 1);
  }
  // Launch the append kernel of `layer` for the step's runs (uploaded with the step's plan).
  hw_status launch_append(int32_t layer, const void* k_raw, const void* v_raw, cudaStream_t s) {
    const int slot = step_slot;
    hw::AppendArgs a{};
    a.gate = step_gate;
    a.runs = reinterpret_cast<const hw::AppendRun*>(d_slot(slot));
    a.num_runs = step_runs;
    a.max_run = step_max_run;
    a.k_raw = (const __nv_bfloat16*)k_raw;
    a.v_raw = (const __nv_bfloat16*)v_raw;
    a.k_layer = k_pool + (size_t)layer * layer_elems;
    a.v_layer = v_pool + (size_t)layer * layer_elems;
    a.rope_cos = d_cos();
    a.rope_sin = d_sin();
    a.err = d_err();
    a.H_kv = cfg.num_kv_heads;
    a.D = cfg.head_dim;
    a.S = cfg.page_size;
    a.num_pages = cfg.num_pages;
    a.max_position = cfg.max_position;
    const int pi = prof_begin(s, 1);
    hw::launch_append(a, s);
    prof_end(pi, s);
    HW_CUDA(cudaGetLastError());
    n_launch += (step_runs + 65534) / 65535;
    n_append += 1;
    HW_CUDA(cudaEventRecord(slot_ev[slot], s));
    slot_used[slot] = true;
    return HW_OK;
  }
  // Write a recorded (fused) append of `layer` with the append kernel, if one is pending.
  hw_status flush_append(int32_t layer, cudaStream_t s) {
    if (layer < 0 || layer >= (int32_t)pend_k.size() || !pend_k[layer]) return HW_OK;
    const void* k = pend_k[layer];
    const void* v = pend_v[layer];
    pend_k[layer] = pend_v[layer] = nullptr;
    return launch_append(layer, k, v, s);
  }
  // Copy `bytes` of staging slot `slot` to its device copy on the copy stream, then the plan's
  // sequence number `seq` (from next_seq(); *gate is set to check for it).  The slot's previous readers have
  // completed (acquire_slot), and the next ones check the number before reading.
  hw_status upload_slot(int slot, size_t bytes, uint64_t seq, hw::PlanGate* gate) {
    std::memcpy(h_slot(slot) + lay.slot_seq_off, &seq, sizeof(seq));
    HW_CUDA(cudaMemcpyAsync(d_slot(slot), h_slot(slot), bytes, cudaMemcpyHostToDevice, copy_stream));
    HW_CUDA(cudaMemcpyAsync(d_slot(slot) + lay.slot_seq_off, h_slot(slot) + lay.slot_seq_off,
                            sizeof(seq), cudaMemcpyHostToDevice, copy_stream));
    gate->plan_seq = reinterpret_cast<const unsigned long long*>(d_slot(slot) + lay.slot_seq_off);
    gate->plan_expect = seq;
    if (expire_plans > 0) {
      // ~seq: never a sequence number (those count up from 1), and every 32-bit part of it
      // differs from seq's, so no unit record looks current either
      gate->plan_expect = ~seq;
      --expire_plans;
    }
    return HW_OK;
  }
  // The same, copied on `s` in stream order, in one copy: whatever `s` runs afterwards reads
  // the plan without checking for it (a null gate; the plan carries sequence number 0).
  hw_status upload_slot_in_order(int slot, size_t bytes, cudaStream_t s, hw::PlanGate* gate) {
    HW_CUDA(cudaMemcpyAsync(d_slot(slot), h_slot(slot), bytes, cudaMemcpyHostToDevice, s));
    *gate = hw::PlanGate{nullptr, 0};
    return HW_OK;
  }
  static uint64_t next_seq() { return ++g_upload_seq; }
  // Pick the next staging slot; waits only if the slot's previous use is still in flight.  The
  // current step's plan slot is passed over: every later append flush and attention call of the
  // step reads it, however many other plans (several-query calls) go up in between.
  hw_status acquire_slot(int* slot) {
    int i = next_slot;
    if (i == step_slot) i = (i + 1) % lay.num_slots;      // num_slots >= 4
    next_slot = (i + 1) % lay.num_slots;
    if (slot_used[i]) HW_CUDA(cudaEventSynchronize(slot_ev[i]));
    *slot = i;
    return HW_OK;
  }
};

extern "C" {

const char* hw_status_string(hw_status s) {
  switch (s) {
    case HW_OK: return "HW_OK";
    case HW_ERR_INVALID_ARG: return "HW_ERR_INVALID_ARG";
    case HW_ERR_OUT_OF_PAGES: return "HW_ERR_OUT_OF_PAGES";
    case HW_ERR_CAPACITY: return "HW_ERR_CAPACITY";
    case HW_ERR_CUDA: return "HW_ERR_CUDA";
    case HW_ERR_DEVICE_CHECK: return "HW_ERR_DEVICE_CHECK";
    case HW_ERR_DEVICE_TIMEOUT: return "HW_ERR_DEVICE_TIMEOUT";
    case HW_ERR_UNSUPPORTED: return "HW_ERR_UNSUPPORTED";
  }
  return "HW_ERR_UNKNOWN";
}

int32_t hw_last_cuda_error(const char** message) {
  if (message) {
    std::lock_guard<std::mutex> lk(g_msg_mu);
    *message = g_cuda_msg.c_str();
  }
  return g_cuda_err;
}

hw_status hw_pool_size(const hw_config* cfg, size_t* bytes) {
  if (!valid_config(cfg) || !bytes) return HW_ERR_INVALID_ARG;
  *bytes = (size_t)cfg->num_layers * cfg->num_pages * cfg->num_kv_heads * cfg->page_size *
           cfg->head_dim * sizeof(__nv_bfloat16);
  return HW_OK;
}

hw_status hw_workspace_size(const hw_config* cfg, size_t* bytes) {
  if (!valid_config(cfg) || !bytes) return HW_ERR_INVALID_ARG;
  *bytes = make_layout(cfg).total;
  return HW_OK;
}

void hw_destroy(hw_ctx* ctx) {
  if (!ctx) return;
  for (cudaEvent_t e : ctx->prof_ev)
    if (e) cudaEventDestroy(e);
  for (int i = 0; i < kMaxSlots; ++i)
    if (ctx->slot_ev[i]) {
      cudaEventSynchronize(ctx->slot_ev[i]);
      cudaEventDestroy(ctx->slot_ev[i]);
    }
  if (ctx->copy_stream) {
    cudaStreamSynchronize(ctx->copy_stream);
    cudaStreamDestroy(ctx->copy_stream);
  }
  if (ctx->h_slots) cudaFreeHost(ctx->h_slots);
  delete ctx;
}

hw_status hw_create(const hw_config* cfg, void* k_pool, void* v_pool, void* workspace,
                    size_t workspace_bytes, const int32_t* page_order, void* stream,
                    hw_ctx** out) {
  if (!out) return HW_ERR_INVALID_ARG;
  *out = nullptr;
  if (!valid_config(cfg) || !k_pool || !v_pool || !workspace) return HW_ERR_INVALID_ARG;
  if (((uintptr_t)k_pool | (uintptr_t)v_pool | (uintptr_t)workspace) % kAlign)
    return HW_ERR_INVALID_ARG;
  const Layout lay = make_layout(cfg);
  if (workspace_bytes < lay.total) return HW_ERR_CAPACITY;
  const int32_t P = cfg->num_problems, W = cfg->num_workers;
  if ((int64_t)P * (1 + W) > lay.max_segments) return HW_ERR_CAPACITY;
  std::vector<int32_t> order(cfg->num_pages);
  if (page_order) {
    std::vector<uint8_t> seen(cfg->num_pages, 0);
    for (int32_t i = 0; i < cfg->num_pages; ++i) {
      const int32_t pg = page_order[i];
      if (pg < 0 || pg >= cfg->num_pages || seen[pg]) return HW_ERR_INVALID_ARG;
      seen[pg] = 1;
      order[i] = pg;
    }
  } else {
    for (int32_t i = 0; i < cfg->num_pages; ++i) order[i] = i;
  }
  cudaStream_t s = (cudaStream_t)stream;
  hw_ctx* c = new (std::nothrow) hw_ctx();
  if (!c) return HW_ERR_CAPACITY;
  c->cfg = *cfg;
  c->lay = lay;
  c->G = cfg->num_q_heads / cfg->num_kv_heads;
  c->rows = lay.rows;
  c->k_pool = (__nv_bfloat16*)k_pool;
  c->v_pool = (__nv_bfloat16*)v_pool;
  c->ws = (char*)workspace;
  c->layer_elems = (size_t)cfg->num_pages * cfg->num_kv_heads * cfg->page_size * cfg->head_dim;
  c->free_pages.assign(order.begin(), order.end());
  for (int32_t p = 0; p < P; ++p) {
    c->common.push_back({c->new_segment(p, -1)});
    std::vector<int32_t> lv;
    for (int32_t w = 0; w < W; ++w) lv.push_back(c->new_segment(p, w));
    c->live.push_back(lv);
  }
  auto fail = [&](hw_status st) {
    hw_destroy(c);
    return st;
  };
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  // Tensor cores take the contraction once a dense 16-row tile of query rows exists; the TMA
  // row coordinate of the pools must fit in int32.
  const int64_t pool_rows = (int64_t)cfg->num_layers * cfg->num_pages * cfg->num_kv_heads *
                            cfg->page_size;
  // Both attention kernels stage K/V tiles through TMA tensor maps of the pools, whose row
  // coordinate must fit in int32.
  if (pool_rows >= (1ll << 31)) return fail(HW_ERR_UNSUPPORTED);
  c->use_tc = c->rows >= 16;
  if (!hw::make_tc_maps(*cfg, k_pool, v_pool, &c->maps)) return fail(HW_ERR_UNSUPPORTED);
  e = hw::prepare_attention_fma(cfg->head_dim);
  if (e == cudaSuccess && c->use_tc) e = hw::prepare_attention_tc(cfg->head_dim);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  e = cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  e = cudaHostAlloc((void**)&c->h_slots, (size_t)lay.num_slots * lay.slot_bytes,
                    cudaHostAllocDefault);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  for (int i = 0; i < kMaxSlots; ++i) {
    e = cudaEventCreateWithFlags(&c->slot_ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(cuda_fail(e));
  }
  // RoPE table: cos/sin of p * theta^(-2i/D) in fp64 on the host, stored as fp32.
  const int32_t half = cfg->head_dim / 2;
  std::vector<float> tc((size_t)cfg->max_position * half), ts(tc.size());
  for (int32_t i = 0; i < half; ++i) {
    const double f = std::pow(cfg->rope_theta, -2.0 * i / cfg->head_dim);
    for (int32_t p = 0; p < cfg->max_position; ++p) {
      const double a = (double)p * f;
      tc[(size_t)p * half + i] = (float)std::cos(a);
      ts[(size_t)p * half + i] = (float)std::sin(a);
    }
  }
  size_t pool_bytes = 0;
  hw_pool_size(cfg, &pool_bytes);
  e = cudaMemsetAsync(k_pool, 0, pool_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(v_pool, 0, pool_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->ws + lay.err, 0, kAlign, s);
  if (e == cudaSuccess)                      // plan slots, with their sequence words
    e = cudaMemsetAsync(c->ws + lay.slots, 0, (size_t)lay.num_slots * lay.slot_bytes, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->d_cos(), tc.data(), tc.size() * sizeof(float), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->d_sin(), ts.data(), ts.size() * sizeof(float), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  *out = c;
  return HW_OK;
}

}  // extern "C"

namespace {
bool build_attention_plan(hw_ctx* c, char* buf, size_t cap, PlanOffsets* po, int64_t unit_cap,
                          int64_t target_override, bool fuse, uint64_t seq,
                          const int32_t* n_q = nullptr, const int64_t* ranges = nullptr,
                          const int32_t* q_row0 = nullptr, const int32_t* q_tail = nullptr);
}  // namespace

extern "C" {

hw_status hw_append_kv(hw_ctx* c, int32_t layer, const int32_t* n_new, const void* k_raw,
                       const void* v_raw, void* stream) {
  if (!c || !n_new || layer < 0 || layer >= c->cfg.num_layers) return HW_ERR_INVALID_ARG;
  const int32_t P = c->cfg.num_problems, W = c->cfg.num_workers, S = c->cfg.page_size;
  const int32_t B = W + 1;
  int64_t total = 0;
  for (int32_t i = 0; i < P * B; ++i) {
    if (n_new[i] < 0) return HW_ERR_INVALID_ARG;
    total += n_new[i];
  }
  if (total > 0 && (!k_raw || !v_raw)) return HW_ERR_INVALID_ARG;
  if (total > 0 && (((uintptr_t)k_raw | (uintptr_t)v_raw) % 16)) return HW_ERR_INVALID_ARG;
  if (total > c->lay.max_append) return HW_ERR_CAPACITY;
  if (!c->step_active) {
    // First append of the step: check, then allocate pages (all-or-nothing).
    int64_t need = 0;
    for (int32_t p = 0; p < P; ++p) {
      // Every view of problem p spans all its tokens: RoPE angles reach the view length - 1.
      int64_t view_len = 0;
      for (int32_t sid : c->common[p]) view_len += c->segs[sid].length;
      for (int32_t sid : c->live[p]) view_len += c->segs[sid].length;
      for (int32_t b = 0; b < B; ++b) view_len += n_new[p * B + b];
      if (view_len > c->cfg.max_position) return HW_ERR_CAPACITY;
      for (int32_t b = 0; b < B; ++b) {
        const int32_t n = n_new[p * B + b];
        if (!n) continue;
        const Seg& sg = c->block(p, b);
        const int64_t j0 = sg.length;
        if (c->cfg.contiguous) {
          if (j0 + n > S) return HW_ERR_CAPACITY;
          if (j0 == 0) need += 1;
        } else {
          const int64_t first = (j0 + S - 1) / S, last = (j0 + n - 1) / S;
          need += std::max<int64_t>(0, last - first + 1);
        }
      }
    }
    if (need > (int64_t)c->free_pages.size()) return HW_ERR_OUT_OF_PAGES;
    for (int32_t p = 0; p < P; ++p)
      for (int32_t b = 0; b < B; ++b) {
        const int32_t n = n_new[p * B + b];
        if (!n) continue;
        Seg& sg = c->block(p, b);
        const int64_t j0 = sg.length;
        int64_t cnt;
        if (c->cfg.contiguous) {
          cnt = (j0 == 0) ? 1 : 0;
        } else {
          const int64_t first = (j0 + S - 1) / S, last = (j0 + n - 1) / S;
          cnt = std::max<int64_t>(0, last - first + 1);
        }
        for (int64_t k = 0; k < cnt; ++k) {
          sg.pages.push_back(c->free_pages.front());
          c->free_pages.pop_front();
        }
        sg.pending = n;
      }
    c->step_active = true;
    ++c->epoch;                            // tables changed: any uploaded plan is stale
    c->step_n.assign(n_new, n_new + P * B);
    c->appended.assign(c->cfg.num_layers, 0);
    c->pend_k.assign(c->cfg.num_layers, nullptr);
    c->pend_v.assign(c->cfg.num_layers, nullptr);
  } else {
    if (!std::equal(c->step_n.begin(), c->step_n.end(), n_new)) return HW_ERR_INVALID_ARG;
    if (c->appended[layer]) return HW_ERR_INVALID_ARG;
  }
  if (total == 0) {
    c->appended[layer] = 1;
    return HW_OK;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (c->step_slot < 0 || c->step_epoch != c->epoch) {
    // First append since the tables changed: the runs (identical for every layer of the step)
    // and the attention plan of the post-append state go up in one copy.
    int slot = 0;
    hw_status st = c->acquire_slot(&slot);
    if (st != HW_OK) return st;
    hw::AppendRun* runs = reinterpret_cast<hw::AppendRun*>(c->h_slot(slot));
    const size_t max_runs = c->lay.slot_seq_off / sizeof(hw::AppendRun);
    int32_t nr = 0, src = 0, max_run = 0;
    for (int32_t p = 0; p < P; ++p)
      for (int32_t b = 0; b < B; ++b) {
        const int32_t n = n_new[p * B + b];
        if (!n) continue;
        const Seg& sg = c->block(p, b);
        int32_t j = sg.length;
        const int32_t end = sg.length + n;
        while (j < end) {
          const int32_t pg_idx = c->cfg.contiguous ? 0 : j / S;
          const int32_t slot0 = c->cfg.contiguous ? j : j % S;
          const int32_t len = std::min(end - j, S - slot0);
          if ((size_t)nr >= max_runs) return HW_ERR_CAPACITY;
          runs[nr++] = hw::AppendRun{src, len, sg.pages[pg_idx], slot0, j, 0};
          max_run = std::max(max_run, len);
          src += len;
          j += len;
        }
      }
    const size_t plan_off = align_up((size_t)nr * sizeof(hw::AppendRun), kAlign);
    PlanOffsets po{};
    // Small appends (decode) are written by the attention kernel itself.
    bool fuse = true;
    for (int32_t i = 0; i < P * B && fuse; ++i) fuse = n_new[i] <= kFuseTok;
    const uint64_t seq = c->plan_in_order ? 0 : c->next_seq();
    bool plan_ok = plan_off < c->lay.slot_seq_off &&
                   build_attention_plan(c, c->h_slot(slot) + plan_off, c->lay.slot_seq_off - plan_off,
                                        &po, 0, c->wave_ctas(), fuse, seq);
    if (!plan_ok && fuse) {
      fuse = false;
      plan_ok = plan_off < c->lay.slot_seq_off &&
                build_attention_plan(c, c->h_slot(slot) + plan_off, c->lay.slot_seq_off - plan_off,
                                     &po, 0, c->wave_ctas(), false, seq);
    }
    const size_t up = plan_off + (plan_ok ? po.bytes : 0);
    st = c->plan_in_order ? c->upload_slot_in_order(slot, up, s, &c->step_gate)
                          : c->upload_slot(slot, up, seq, &c->step_gate);
    if (st != HW_OK) return st;
    c->step_slot = slot;
    c->step_runs = nr;
    c->step_max_run = max_run;
    c->step_plan_off = plan_off;
    c->step_plan_ok = plan_ok;
    c->step_fused = plan_ok && fuse;
    c->step_po = po;
    c->step_epoch = c->epoch;
  }
  if (c->step_fused) {
    c->pend_k[layer] = k_raw;
    c->pend_v[layer] = v_raw;
    c->appended[layer] = 1;
    return HW_OK;
  }
  const hw_status st = c->launch_append(layer, k_raw, v_raw, s);
  if (st != HW_OK) return st;
  c->appended[layer] = 1;
  return HW_OK;
}


}  // extern "C"

namespace {

// Build the attention plan of the current state into host buffer `buf` (`cap` bytes long).
// Returns false if a table would overflow (the buffer's contents are then undefined).  Offsets
// of each array are written to `po`.
//
// The pieces of a problem are listed once and shared by its KV heads: the units of group
// (p, h) index the problem's piece list, and the head comes from the group.  A segment's
// delta for worker w is i_q(w) minus the segment's offset in w's view (in the context's
// layout), or -1 when w's view does not hold it; in the combined layout every view holds every
// segment and i_q is the problem's visible length - 1.
// unit_cap > 0 bounds the number of units (one partial result each); 0 = the default split.
// n_q (host [P][W], or null for one query per worker): several causal query tokens per worker;
// the rotation table then has one column per query row of a problem (its width WT is the
// largest count of any problem), with the causal length table and the query-row map.  q_row0
// (host [P][W], or null): the q / out / lse row of each worker's first query token, for a call
// that covers only some workers' tokens (null: the tokens present, numbered in order); q_tail
// (host [P][W], or null for none): the worker's query tokens after this call's, for a call that
// takes a worker's first tokens only (the causal offsets count from its last token).
bool build_attention_plan(hw_ctx* c, char* buf, size_t cap, PlanOffsets* po, int64_t unit_cap = 0,
                          int64_t target_override = 0, bool fuse = false, uint64_t seq = 0,
                          const int32_t* n_q, const int64_t* ranges, const int32_t* q_row0,
                          const int32_t* q_tail) {
  const int32_t P = c->cfg.num_problems, W = c->cfg.num_workers, H = c->cfg.num_kv_heads;
  int32_t WT = W;                       // rotation-table width: query rows per problem / G
  if (n_q) {
    WT = 1;
    for (int32_t p = 0; p < P; ++p) {
      int32_t v = 0;
      for (int32_t w = 0; w < W; ++w) v += n_q[(size_t)p * W + w];
      WT = std::max(WT, v);
    }
  }
  const int32_t S = c->cfg.page_size;
  const Layout& L = c->lay;
  PlanScratch& ps = c->ps;
  ps.delta.clear();
  ps.ref_sid.clear();
  ps.ref_slot.clear();
  ps.ref_tiles.clear();
  ps.ref_lo.clear();
  ps.ref_hi.clear();
  ps.prob_ref_begin.assign(P + 1, 0);
  ps.prob_common_refs.assign(P, 0);
  ps.prob_tiles.assign(P, 0);
  ps.vlen.clear();
  ps.qrow.assign(n_q ? (size_t)P * WT : 0, -1);
  ps.qrow_next = 0;
  // fuse: list the step's appended tokens (k_raw rows in append order: problems, then block 0 =
  // common, 1 + w = worker w, each in position order) for the attention kernel to write.
  if (fuse) {
    if (!c->step_active || c->step_n.size() != (size_t)P * (W + 1)) return false;
    ps.src_base.assign(c->segs.size(), -1);
    int32_t run = 0;
    for (int32_t p = 0; p < P; ++p)
      for (int32_t b = 0; b <= W; ++b) {
        const int32_t n = c->step_n[(size_t)p * (W + 1) + b];
        const int32_t sid = b == 0 ? c->common[p].back() : c->live[p][b - 1];
        if (n > 0) ps.src_base[sid] = run;
        run += n;
      }
  }
  // Pass 1, per problem: the non-empty segments (common part in commit order, then the live
  // blocks by worker), their rotation table and their tile counts.  A segment is streamed once
  // for every row of its problem; the table says which rows see it, and at what rotation.
  if (ps.ref_of.size() < c->segs.size()) ps.ref_of.resize(c->segs.size(), -1);
  for (int32_t p = 0; p < P; ++p) {
    ps.prob_ref_begin[p] = (int32_t)ps.ref_sid.size();
    ps.refs.clear();
    for (int32_t sid : c->common[p])
      if (c->segs[sid].visible() > 0) ps.refs.push_back(sid);
    const int32_t n_common_refs = (int32_t)ps.refs.size();
    for (int32_t w = 0; w < W; ++w) {
      const int32_t sid = c->live[p][w];
      if (c->segs[sid].visible() > 0) ps.refs.push_back(sid);
    }
    const int32_t slot_base = (int32_t)(ps.delta.size() / (size_t)WT);
    if (slot_base + (int64_t)ps.refs.size() > L.max_seg_slots) return false;
    ps.delta.resize(ps.delta.size() + ps.refs.size() * (size_t)WT, -1);
    int32_t* delta = ps.delta.data() + (size_t)slot_base * WT;
    int32_t* vlen = nullptr;
    if (n_q) {
      ps.vlen.resize(ps.delta.size(), 0);
      vlen = ps.vlen.data() + (size_t)slot_base * WT;
    }
    // Rotation of reference r for worker w: i_q(w) minus r's offset in w's view, or -1 when the
    // layout keeps r out of that view.  With several query tokens, worker w's token t (back =
    // n_q - 1 - t newer tokens after it) is query row v: its rotation is back less, and in the
    // own block (last in every view) it sees back tokens fewer -- the causal cut.
    for (size_t r = 0; r < ps.refs.size(); ++r) ps.ref_of[ps.refs[r]] = (int32_t)r;
    int32_t v0 = 0;                        // first query row of worker w
    for (int32_t w = 0; w < W; ++w) {
      const int32_t nq = n_q ? n_q[(size_t)p * W + w] : 1;
      if (nq == 0) continue;
      ps.view_ref.clear();
      ps.view_off.clear();
      const int64_t total = c->for_each_view(p, w, [&](int32_t sid, int64_t off, int32_t) {
        ps.view_ref.push_back(ps.ref_of[sid]);
        ps.view_off.push_back(off);
      });
      const int32_t vb = n_q ? v0 : w;
      for (int32_t t = 0; t < nq; ++t) {
        const int32_t back = nq - 1 - t + (q_tail ? q_tail[(size_t)p * W + w] : 0), v = vb + t;
        for (size_t k = 0; k < ps.view_ref.size(); ++k) {
          const int32_t r = ps.view_ref[k];
          delta[(size_t)r * WT + v] = (int32_t)(total - 1 - back - ps.view_off[k]);
          if (vlen) {
            const int32_t n = c->segs[ps.refs[r]].visible();
            vlen[(size_t)r * WT + v] = k + 1 == ps.view_ref.size() ? n - back : n;
          }
        }
        if (n_q) ps.qrow[(size_t)p * WT + v] = q_row0 ? q_row0[(size_t)p * W + w] + t : ps.qrow_next++;
      }
      v0 += nq;
    }
    // Tokens attended of each reference: all of them, or, with an entry range, those whose
    // entry number (segment order: the common segments in commit order, then the workers'
    // blocks by id -- the order of the references) lies in [begin, end).
    int64_t tiles = 0, entry = 0;
    for (size_t r = 0; r < ps.refs.size(); ++r) {
      const int32_t vis = c->segs[ps.refs[r]].visible();
      int32_t lo = 0, hi = vis;
      if (ranges) {
        const int64_t b = ranges[2 * (size_t)p], e = ranges[2 * (size_t)p + 1];
        lo = (int32_t)std::min<int64_t>(std::max<int64_t>(b - entry, 0), vis);
        hi = (int32_t)std::max<int64_t>(lo, std::min<int64_t>(std::max<int64_t>(e - entry, 0), vis));
      }
      entry += vis;
      const int32_t nt = hi > lo ? (hi + kPieceMax - 1) / kPieceMax - lo / kPieceMax : 0;
      ps.ref_sid.push_back(ps.refs[r]);
      ps.ref_slot.push_back(slot_base + (int32_t)r);
      ps.ref_tiles.push_back(nt);
      ps.ref_lo.push_back(lo);
      ps.ref_hi.push_back(hi);
      tiles += nt;
    }
    ps.prob_common_refs[p] = n_common_refs;
    ps.prob_tiles[p] = tiles;
  }
  ps.prob_ref_begin[P] = (int32_t)ps.ref_sid.size();
  // Units per problem: KV-entry balanced (summary section 9: the kernel balances by KV
  // entries, not by blocks, then reduces the partial results); every 128-token tile costs the
  // kernels the same, so the balance is in tiles.
  int64_t total_tiles = 0;
  for (int64_t t : ps.prob_tiles) total_tiles += t * H;
  // target_override: the tensor-core kernel's CTA count per wave (one CTA per SM).  A unit never
  // spans two groups, so when groups differ in size one wave of units leaves some SMs with far
  // more tiles than others; a step with many tiles per SM and such an imbalance gets several
  // waves of smaller units instead, and the block scheduler hands the next unit to whichever
  // SM is free.  (With units of about equal size, more waves only add per-unit set-up.)
  int64_t waves = 1;
  if (target_override > 0 && total_tiles > 0) {
    const int64_t per_sm = total_tiles / target_override;
    int64_t largest = 0, units1 = 0;                // the one-wave plan, as computed below
    for (int32_t p = 0; p < P; ++p) {
      const int64_t Tt = ps.prob_tiles[p];
      if (Tt == 0) continue;
      const int64_t n1 = std::max<int64_t>(
          1, std::min<int64_t>(Tt, (target_override * Tt * H + total_tiles / 2) / (total_tiles * H)));
      largest = std::max(largest, (Tt + n1 - 1) / n1);
      units1 += n1 * H;
    }
    const bool unbalanced = units1 > 0 && largest * units1 * 4 > total_tiles * 5;  // > 1.25 x mean
    if (unbalanced)
      waves = std::max<int64_t>(1, std::min<int64_t>(kMaxWaves, (per_sm + kWaveTiles / 2) / kWaveTiles));
  }
  int64_t target_units = std::max<int64_t>((int64_t)P * H,
                                           target_override > 0 ? target_override * waves
                                                               : 4ll * c->num_sms);
  if (unit_cap > 0) {
    if (unit_cap < (int64_t)P * H) return false;
    // per-group counts are floored and then raised to >= 1: keep room for that raise
    target_units = std::max<int64_t>(0, std::min<int64_t>(target_units, unit_cap - (int64_t)P * H));
  }
  // Sizes, known before anything is built: every tile of a problem is one piece, and a
  // problem's units (the same for every KV head) follow from its share of the tiles.
  ps.prob_units.resize((size_t)P);
  int64_t n_pieces = 0, n_units_all = 0;
  for (int32_t p = 0; p < P; ++p) {
    const int64_t Tt = ps.prob_tiles[p];
    int64_t nu = total_tiles ? (target_units * Tt * H + (unit_cap > 0 ? 0 : total_tiles / 2)) /
                                   (total_tiles * H)
                             : 1;
    nu = std::max<int64_t>(1, std::min<int64_t>(nu, Tt));
    ps.prob_units[p] = (int32_t)nu;
    n_pieces += Tt;
    n_units_all += nu * H;
  }
  if (n_pieces > L.max_pieces || n_units_all > L.max_units) return false;
  if (unit_cap > 0 && n_units_all > unit_cap) return false;
  size_t off = 0;
  po->pieces = off;
  off = align_up(off + (size_t)n_pieces * sizeof(hw::Piece), 16);
  po->units = off;
  off = align_up(off + (size_t)n_units_all * sizeof(hw::Unit), 16);
  po->groups = off;
  off = align_up(off + (size_t)P * H * sizeof(hw::Group), 16);
  po->delta = off;
  off = align_up(off + ps.delta.size() * sizeof(int32_t), 16);
  po->vlen = off;
  off = align_up(off + ps.vlen.size() * sizeof(int32_t), 16);
  po->qrow = off;
  off = align_up(off + ps.qrow.size() * sizeof(int32_t), 16);
  po->fresh = off;
  if (off > cap) return false;
  const int64_t max_fresh =
      std::min<int64_t>(L.max_fresh, (int64_t)((cap - off) / sizeof(hw::FreshTok)));
  ps.pieces.clear();
  ps.units.clear();
  ps.groups.clear();
  ps.fresh.clear();
  ps.piece_early.clear();
  hw::Piece* const pieces = ps.pieces.grow((size_t)n_pieces);
  hw::Unit* const units = ps.units.grow((size_t)n_units_all);
  hw::Group* const groups = ps.groups.grow((size_t)P * H);
  hw::FreshTok* const fresh = ps.fresh.grow((size_t)max_fresh);
  uint8_t* const early_all = ps.piece_early.grow((size_t)n_pieces);
  int32_t np = 0, nf = 0, nu_done = 0;                 // pieces, fresh tokens, units written
  // The pieces of segment reference r at its tiles [t0, t1) (counted from the reference's
  // first tile): the reference's tokens inside one kPieceMax-aligned tile each -- so inside one
  // page -- with the step's appended tokens in it listed for the fused append.  Only the first
  // piece of a reference can start inside its tile (an entry range that cuts the segment).
  // (Segment data is read once per run; the page index advances with the tile.)
  const bool contiguous = c->cfg.contiguous != 0;
  const int32_t tiles_per_page = S / kPieceMax;
  auto emit = [&](int32_t r, int32_t t0, int32_t t1) -> bool {
    if (t1 <= t0) return true;
    if ((int64_t)np + (t1 - t0) > n_pieces) return false;
    const int32_t sid = ps.ref_sid[r];
    Seg& sg = c->segs[sid];
    if (sg.pending == 0) {
      // No token of this step in it: its pieces are those of the last plan while the segment,
      // its slot in the rotation table and the attended range are unchanged.
      PieceCache& pc = sg.cache;
      if (pc.seg_slot != ps.ref_slot[r] || pc.lo != ps.ref_lo[r] || pc.hi != ps.ref_hi[r] ||
          pc.len != sg.length || pc.recent != sg.recent_from ||
          pc.npages != (int32_t)sg.pages.size()) {
        const int32_t nt = ps.ref_tiles[r];
        const int32_t lo = ps.ref_lo[r], hi = ps.ref_hi[r];
        pc.pieces.resize((size_t)nt);
        pc.early.resize((size_t)nt);
        const int32_t Tb = lo / kPieceMax;
        int32_t pi = contiguous ? 0 : Tb / tiles_per_page;
        int32_t sub = contiguous ? 0 : Tb - pi * tiles_per_page;
        for (int32_t T = Tb; T < Tb + nt; ++T) {
          const int32_t j = std::max(lo, T * kPieceMax);
          const int32_t end = std::min(hi, (T + 1) * kPieceMax);
          const int32_t slot0 = contiguous ? j : sub * kPieceMax + (j - T * kPieceMax);
          pc.pieces[T - Tb] = hw::Piece{ps.ref_slot[r], sg.pages[pi], slot0, end - j, 0, j};
          pc.early[T - Tb] = end <= sg.recent_from ? 1 : 0;
          if (!contiguous && ++sub == tiles_per_page) {
            sub = 0;
            ++pi;
          }
        }
        pc.seg_slot = ps.ref_slot[r];
        pc.lo = lo;
        pc.hi = hi;
        pc.len = sg.length;
        pc.recent = sg.recent_from;
        pc.npages = (int32_t)sg.pages.size();
      }
      const size_t n = (size_t)(t1 - t0);
      std::memcpy(pieces + np, pc.pieces.data() + t0, n * sizeof(hw::Piece));
      std::memcpy(early_all + np, pc.early.data() + t0, n);
      np += (int32_t)n;
      return true;
    }
    const int32_t* pages = sg.pages.data();
    const int32_t seg_slot = ps.ref_slot[r], len = sg.length;
    const int32_t lo = ps.ref_lo[r], hi = ps.ref_hi[r];
    const int32_t recent = sg.recent_from;
    const int32_t T0 = lo / kPieceMax + t0, T1 = lo / kPieceMax + t1;   // tiles of the segment
    int32_t pi = contiguous ? 0 : T0 / tiles_per_page;     // page of tile T
    int32_t sub = contiguous ? 0 : T0 - pi * tiles_per_page;  // tile T's place in it
    for (int32_t T = T0; T < T1; ++T) {
      const int32_t j = std::max(lo, T * kPieceMax);              // first token of the piece
      const int32_t end = std::min(hi, (T + 1) * kPieceMax);      // one past its last
      const int32_t pg = pages[pi];
      const int32_t slot0 = contiguous ? j : sub * kPieceMax + (j - T * kPieceMax);
      const int32_t cnt = end - j;
      // fresh: holds tokens appended in this step (the kernels read it only after the append)
      const int32_t is_fresh = end > len ? 1 : 0;
      early_all[np] = !is_fresh && end <= recent ? 1 : 0;
      pieces[np++] = hw::Piece{seg_slot, pg, slot0, cnt, is_fresh, j};
      if (fuse && is_fresh) {
        if (ps.src_base[sid] < 0) return false;
        for (int32_t k = std::max<int32_t>(0, len - j); k < cnt; ++k) {
          if (nf >= max_fresh) return false;
          fresh[nf++] = hw::FreshTok{pg, slot0 + k, j + k, ps.src_base[sid] + (j + k - len)};
        }
      }
      if (!contiguous && ++sub == tiles_per_page) {
        sub = 0;
        ++pi;
      }
    }
    return true;
  };
  for (int32_t p = 0; p < P; ++p) {
    const int32_t rb = ps.prob_ref_begin[p], re = ps.prob_ref_begin[p + 1];
    const int32_t rc = rb + ps.prob_common_refs[p];      // first live-block reference
    const int64_t Tt = ps.prob_tiles[p];
    const int32_t n = ps.prob_units[p];
    // Layout of the problem's units (the same for every KV head): unit k holds cap_k tiles;
    // each live block (largest first) goes to the unit with the most room left, split over
    // units only when it does not fit; the rest of every unit is filled with common-part tiles,
    // which come first in the unit.  So a unit crosses at most a few segments, its first
    // segment is usually common (one rotation for every worker), and a block's query tile is
    // built while the unit's common tiles stream.
    ps.unit_rem.assign(n, 0);
    for (int32_t k = 0; k < n; ++k) ps.unit_rem[k] = (int32_t)(Tt / n + (k < Tt % n ? 1 : 0));
    ps.parts.clear();                                    // (unit, ref, tile begin, tile end)
    ps.order.clear();
    // live blocks by tile count, largest first, ties in worker order (a stable insertion sort:
    // W is small)
    for (int32_t r = rc; r < re; ++r) {
      size_t i = ps.order.size();
      ps.order.push_back(r);
      while (i > 0 && ps.ref_tiles[ps.order[i - 1]] < ps.ref_tiles[r]) {
        ps.order[i] = ps.order[i - 1];
        --i;
      }
      ps.order[i] = r;
    }
    for (int32_t r : ps.order) {
      int32_t t = 0;
      const int32_t nt = ps.ref_tiles[r];
      while (t < nt) {
        int32_t best = 0;
        for (int32_t k = 1; k < n; ++k)
          if (ps.unit_rem[k] > ps.unit_rem[best]) best = k;
        if (ps.unit_rem[best] <= 0) return false;
        const int32_t take = std::min(nt - t, ps.unit_rem[best]);
        ps.parts.push_back({best, r, t, t + take});
        ps.unit_rem[best] -= take;
        t += take;
      }
    }
    // Pieces, unit by unit (common-part tiles in order, then the unit's live-block parts), and
    // the units of KV head 0 over them; every other head's units are copies (but the group).
    hw::Unit* const us = units + nu_done;
    int32_t cr = rb, ct = 0;                             // common-part cursor
    for (int32_t k = 0; k < n; ++k) {
      const int32_t ub = np, fb = nf;
      for (int32_t left = ps.unit_rem[k]; left > 0;) {
        while (cr < rc && ct >= ps.ref_tiles[cr]) {
          ++cr;
          ct = 0;
        }
        if (cr >= rc) return false;
        const int32_t take = std::min(left, ps.ref_tiles[cr] - ct);
        if (!emit(cr, ct, ct + take)) return false;
        ct += take;
        left -= take;
      }
      for (const auto& pt : ps.parts) {
        if (pt.unit != k) continue;
        if (!emit(pt.ref, pt.t0, pt.t1)) return false;
      }
      hw::Unit& u = us[k];
      u = hw::Unit{};
      u.piece_begin = ub;
      u.piece_end = np;
      u.group = p * H;
      u.seg0 = np > ub ? pieces[ub].seg_slot : -1;
      u.seq = u.seq_b = u.seq_c = (uint32_t)seq;
      u.first_tok = np > ub && early_all[ub] ? pieces[ub].page * S + pieces[ub].slot0 : -1;
      // a unit's appended tokens are those of its pieces
      u.fresh_begin = fb;
      u.fresh_end = nf;
      // A segment seen by every worker at the same view offset (every common segment) has one
      // rotation for all query rows: the kernels then need no delta-table load for it.
      u.delta0 = -1;
      if (u.seg0 >= 0 && !n_q) {           // (with a causal cut the rows differ anyway)
        const int32_t* row = ps.delta.data() + (size_t)u.seg0 * WT;
        bool same = row[0] >= 0;
        for (int32_t w = 1; w < WT && same; ++w) same = row[w] == row[0];
        if (same) u.delta0 = row[0];
      }
    }
    for (int32_t h = 0; h < H; ++h) {
      hw::Unit* const uh = us + (size_t)h * n;
      if (h > 0) {
        std::memcpy(uh, us, (size_t)n * sizeof(hw::Unit));
        for (int32_t k = 0; k < n; ++k) uh[k].group = p * H + h;
      }
      groups[p * H + h] = hw::Group{p, h, nu_done + h * n, nu_done + (h + 1) * n};
    }
    nu_done += n * H;
  }
  if (np != n_pieces || nu_done != n_units_all) return false;
  std::memcpy(buf + po->pieces, pieces, (size_t)np * sizeof(hw::Piece));
  std::memcpy(buf + po->units, units, (size_t)nu_done * sizeof(hw::Unit));
  std::memcpy(buf + po->groups, groups, (size_t)P * H * sizeof(hw::Group));
  if (nf) std::memcpy(buf + po->fresh, fresh, (size_t)nf * sizeof(hw::FreshTok));
  std::memcpy(buf + po->delta, ps.delta.data(), ps.delta.size() * sizeof(int32_t));
  if (!ps.vlen.empty())
    std::memcpy(buf + po->vlen, ps.vlen.data(), ps.vlen.size() * sizeof(int32_t));
  if (!ps.qrow.empty())
    std::memcpy(buf + po->qrow, ps.qrow.data(), ps.qrow.size() * sizeof(int32_t));
  po->bytes = align_up(off + (size_t)nf * sizeof(hw::FreshTok), 16);
  po->num_pieces = np;
  po->num_units = nu_done;
  po->num_groups = P * H;
  po->max_group_units = 0;
  for (int32_t p = 0; p < P; ++p) po->max_group_units = std::max(po->max_group_units, ps.prob_units[p]);
  po->num_seg_slots = (int32_t)(ps.delta.size() / (size_t)WT);
  po->width = WT;
  po->num_fresh = nf;
  return true;
}

// One attention call: one query per worker (n_q null), or n_q[p][w] causal query tokens per
// worker (the last tokens of its own block).
static hw_status attend(hw_ctx* c, int32_t layer, const void* q, const int32_t* n_q, void* out,
                        int32_t out_dtype, float* lse, void* stream,
                        const int64_t* ranges = nullptr, const int32_t* q_row0 = nullptr,
                        const int32_t* q_tail = nullptr) {
  if (!c || layer < 0 || layer >= c->cfg.num_layers) return HW_ERR_INVALID_ARG;
  if (out_dtype != HW_OUT_BF16 && out_dtype != HW_OUT_F32) return HW_ERR_INVALID_ARG;
  if (c->step_active && !c->appended[layer]) return HW_ERR_INVALID_ARG;
  int64_t width = c->cfg.num_workers;       // query rows per problem / G
  if (n_q) {
    const int32_t P = c->cfg.num_problems, W = c->cfg.num_workers;
    int64_t total = 0;
    width = 0;
    for (int32_t p = 0; p < P; ++p) {
      int64_t rows = 0;
      for (int32_t w = 0; w < W; ++w) {
        const int32_t n = n_q[(size_t)p * W + w];
        const int32_t tail = q_tail ? q_tail[(size_t)p * W + w] : 0;
        if (n < 0 || tail < 0 || (int64_t)n + tail > c->segs[c->live[p][w]].visible())
          return HW_ERR_INVALID_ARG;
        rows += n;
      }
      total += rows;
      width = std::max(width, rows);
    }
    if (width * c->G > kMaxRows) return HW_ERR_CAPACITY;
    if (total == 0) return HW_OK;                 // no query: nothing to compute
  }
  if (!q || !out) return HW_ERR_INVALID_ARG;
  if (((uintptr_t)q | (uintptr_t)out) % 16) return HW_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int slot = 0;
  PlanOffsets po{};
  char* dbase = nullptr;
  // (the step's plan has one query per worker and lists the step's tokens for the kernel)
  const bool step_plan =
      !n_q && !ranges && c->step_slot >= 0 && c->step_epoch == c->epoch && c->step_plan_ok;
  // The layer's recorded append is written by the attention kernel when the step's plan lists
  // the appended tokens; otherwise by the append kernel, now.
  const bool fused = step_plan && c->step_fused && layer < (int32_t)c->pend_k.size() &&
                     c->pend_k[layer] != nullptr;
  if (!fused) {
    const hw_status st = c->flush_append(layer, s);
    if (st != HW_OK) return st;
  }
  hw::PlanGate gate{};
  const char* hbase = nullptr;               // host copy of the plan (the staging slot)
  if (step_plan) {
    // The plan of this step went up with its first append.
    slot = c->step_slot;
    po = c->step_po;
    dbase = c->d_slot(slot) + c->step_plan_off;
    hbase = c->h_slot(slot) + c->step_plan_off;
    gate = c->step_gate;
  } else {
    hw_status st = c->acquire_slot(&slot);
    if (st != HW_OK) return st;
    // One CTA per SM holds all of its shared memory (and, tensor-core kernel, TMEM), so one
    // unit per SM, balanced by KV entries.
    const uint64_t seq = c->next_seq();
    // partials fit the workspace: units * rows stays within its max_units * (W * G) rows
    const int64_t cap = n_q ? (int64_t)c->lay.max_units * c->rows / (width * c->G) : 0;
    if (!build_attention_plan(c, c->h_slot(slot), c->lay.slot_seq_off, &po, cap, c->wave_ctas(),
                              false, seq, n_q, ranges, q_row0, q_tail))
      return HW_ERR_CAPACITY;
    dbase = c->d_slot(slot);
    hbase = c->h_slot(slot);
    st = c->upload_slot(slot, po.bytes, seq, &gate);
    if (st != HW_OK) return st;
  }
  hw::AttnArgs a{};
  a.gate = gate;
  a.pieces = reinterpret_cast<const hw::Piece*>(dbase + po.pieces);
  a.units = reinterpret_cast<const hw::Unit*>(dbase + po.units);
  a.groups = reinterpret_cast<const hw::Group*>(dbase + po.groups);
  a.delta = reinterpret_cast<const int32_t*>(dbase + po.delta);
  if (n_q) {
    a.vlen = reinterpret_cast<const int32_t*>(dbase + po.vlen);
    a.qrow = reinterpret_cast<const int32_t*>(dbase + po.qrow);
  }
  a.fresh = reinterpret_cast<const hw::FreshTok*>(dbase + po.fresh);
  a.k_raw = fused ? (const __nv_bfloat16*)c->pend_k[layer] : nullptr;
  a.v_raw = fused ? (const __nv_bfloat16*)c->pend_v[layer] : nullptr;
  a.num_units = po.num_units;
  a.num_groups = po.num_groups;
  a.num_seg_slots = po.num_seg_slots;
  a.k_layer = c->k_pool + (size_t)layer * c->layer_elems;
  a.v_layer = c->v_pool + (size_t)layer * c->layer_elems;
  a.q = (const __nv_bfloat16*)q;
  a.out = out;
  a.out_f32 = out_dtype == HW_OUT_F32;
  a.lse = lse;
  a.partials = c->d_partials();
  a.rope_cos = c->d_cos();
  a.rope_sin = c->d_sin();
  a.err = c->d_err();
  a.P = c->cfg.num_problems;
  a.W = po.width;                      // query rows per problem / G (= W for decode)
  a.H_q = c->cfg.num_q_heads;
  a.H_kv = c->cfg.num_kv_heads;
  a.G = c->G;
  a.D = c->cfg.head_dim;
  a.S = c->cfg.page_size;
  a.num_pages = c->cfg.num_pages;
  a.max_position = c->cfg.max_position;
  a.rows = po.width * c->G;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  // Timing events (when enabled) go directly around the attention kernel only.
  const int pi = c->prof_reserve(0);
  cudaEvent_t e0 = pi >= 0 ? c->prof_ev[2 * pi] : nullptr;
  cudaEvent_t e1 = pi >= 0 ? c->prof_ev[2 * pi + 1] : nullptr;
  if (c->use_tc) {
    // What the first CTAs need of their units before reading the plan, as launch parameters.
    hw::LaunchUnits lu;
    const hw::Unit* hu = reinterpret_cast<const hw::Unit*>(hbase + po.units);
    const int32_t S = c->cfg.page_size, H = c->cfg.num_kv_heads;
    for (int32_t i = 0; i < hw::kLaunchUnits; ++i) {
      lu.row0[i] = lu.group[i] = lu.seg0[i] = lu.delta0[i] = -1;
      if (i >= po.num_units) continue;
      const hw::Unit& u = hu[i];
      if (u.first_tok >= 0)
        lu.row0[i] = ((u.first_tok / S) * H + u.group % H) * S + u.first_tok % S;
      lu.group[i] = u.group;
      lu.seg0[i] = u.seg0;
      lu.delta0[i] = u.delta0;
    }
    // the attention kernel and the merge, both as programmatic dependents
    hw::launch_attention_tc(a, c->maps, lu, layer, s, e0, e1);
  } else {
    if (e0) cudaEventRecord(e0, s);
    hw::launch_attention_fma(a, c->maps, layer, s);
    if (e1) cudaEventRecord(e1, s);
  }
  HW_CUDA(cudaGetLastError());
  if (fused) c->pend_k[layer] = c->pend_v[layer] = nullptr;
  const int pm = c->prof_begin(s, 2);      // (a timed merge is not chained to the attention)
  hw::launch_merge(a, s, pm < 0, po.max_group_units);
  c->prof_end(pm, s);
  HW_CUDA(cudaGetLastError());
  c->n_launch += 2;
  c->n_attn += 1;
  HW_CUDA(cudaEventRecord(c->slot_ev[slot], s));
  c->slot_used[slot] = true;
  return HW_OK;
}

}  // namespace

extern "C" {

hw_status hw_concurrent_attention(hw_ctx* c, int32_t layer, const void* q, void* out,
                                  int32_t out_dtype, float* lse, void* stream) {
  return attend(c, layer, q, nullptr, out, out_dtype, lse, stream);
}

hw_status hw_concurrent_attention_mq(hw_ctx* c, int32_t layer, const void* q, const int32_t* n_q,
                                     void* out, int32_t out_dtype, float* lse, void* stream) {
  if (!c || !n_q) return HW_ERR_INVALID_ARG;
  const int32_t P = c->cfg.num_problems, W = c->cfg.num_workers;
  const int64_t cap = kMaxRows / c->G;          // query tokens of a problem per attention call
  int64_t width = 0;
  for (int32_t p = 0; p < P; ++p) {
    int64_t rows = 0;
    for (int32_t w = 0; w < W; ++w) {
      const int32_t n = n_q[(size_t)p * W + w];
      if (n < 0 || n > c->segs[c->live[p][w]].visible()) return HW_ERR_INVALID_ARG;
      rows += n;
    }
    width = std::max(width, rows);
  }
  if (width <= cap) return attend(c, layer, q, n_q, out, out_dtype, lse, stream);
  // Row split: each problem's query tokens, worker by worker in order, are cut into parts of
  // at most `cap` tokens (a worker's tokens may straddle parts); part k of every problem is
  // attended in launch k.  A worker's piece of a part is a run of its tokens: their q / out /
  // lse rows (row0) and the worker's tokens after them (tail, which keeps the causal offsets)
  // go with it.  The K/V are streamed once per launch.
  std::vector<int32_t> first_row((size_t)P * W);
  int32_t next_row = 0, parts = 0;
  for (size_t i = 0; i < first_row.size(); ++i) {
    first_row[i] = next_row;
    next_row += n_q[i];
  }
  for (int32_t p = 0; p < P; ++p) {
    int64_t rows = 0;
    for (int32_t w = 0; w < W; ++w) rows += n_q[(size_t)p * W + w];
    parts = std::max<int32_t>(parts, (int32_t)((rows + cap - 1) / cap));
  }
  std::vector<int32_t> nq_k((size_t)P * W), row0_k((size_t)P * W), tail_k((size_t)P * W);
  for (int32_t k = 0; k < parts; ++k) {
    for (int32_t p = 0; p < P; ++p) {
      // tokens [k cap, (k + 1) cap) of the problem's token sequence
      const int64_t lo = (int64_t)k * cap, hi = lo + cap;
      int64_t start = 0;                        // the worker's first token in that sequence
      for (int32_t w = 0; w < W; ++w) {
        const size_t i = (size_t)p * W + w;
        const int64_t n = n_q[i];
        const int64_t a = std::max(lo, start), b = std::min(hi, start + n);
        nq_k[i] = b > a ? (int32_t)(b - a) : 0;
        row0_k[i] = first_row[i] + (int32_t)(b > a ? a - start : 0);
        tail_k[i] = b > a ? (int32_t)(start + n - b) : 0;
        start += n;
      }
    }
    const hw_status st = attend(c, layer, q, nq_k.data(), out, out_dtype, lse, stream, nullptr,
                                row0_k.data(), tail_k.data());
    if (st != HW_OK) return st;
  }
  return HW_OK;
}

hw_status hw_concurrent_attention_range(hw_ctx* c, int32_t layer, const void* q,
                                        const int64_t* ranges, float* out, float* lse,
                                        void* stream) {
  if (!c || !ranges || !lse) return HW_ERR_INVALID_ARG;
  for (int32_t p = 0; p < c->cfg.num_problems; ++p)
    if (ranges[2 * p] < 0 || ranges[2 * p + 1] < ranges[2 * p]) return HW_ERR_INVALID_ARG;
  if ((uintptr_t)lse % 4) return HW_ERR_INVALID_ARG;
  return attend(c, layer, q, nullptr, out, HW_OUT_F32, lse, stream, ranges);
}

}  // extern "C"

hw_status hw::cuda_status(cudaError_t e) { return e == cudaSuccess ? HW_OK : cuda_fail(e); }

// Same computation as hw_concurrent_attention, with the call's plan and the split-K partials
// placed in caller-given device scratch instead of the workspace (used by the allocation-free
// entry point).  The number of units is capped so that both fit.
hw_status hw::attention_into_scratch(hw_ctx* c, int32_t layer, const void* q, void* out,
                                     int32_t out_dtype, float* lse, void* stream, char* scratch,
                                     size_t scratch_bytes) {
  if (!c || !q || !out || !scratch || layer < 0 || layer >= c->cfg.num_layers)
    return HW_ERR_INVALID_ARG;
  if (out_dtype != HW_OUT_BF16 && out_dtype != HW_OUT_F32) return HW_ERR_INVALID_ARG;
  if (((uintptr_t)q | (uintptr_t)out) % 16) return HW_ERR_INVALID_ARG;
  if (c->step_active && !c->appended[layer]) return HW_ERR_INVALID_ARG;
  const size_t per_unit = (size_t)c->rows * hw::part_stride(c->cfg.head_dim) * sizeof(float);
  const size_t plan_region = align_up(std::min(c->lay.slot_bytes, scratch_bytes / 4), kAlign);
  if (plan_region >= scratch_bytes) return HW_ERR_CAPACITY;
  const int64_t unit_cap = (int64_t)((scratch_bytes - plan_region) / per_unit);
  if (unit_cap < (int64_t)c->cfg.num_problems * c->cfg.num_kv_heads) return HW_ERR_CAPACITY;
  int slot = 0;
  hw_status st = c->acquire_slot(&slot);
  if (st != HW_OK) return st;
  // The plan is built and checked before anything is enqueued: a refusal leaves the stream and
  // the layer's recorded append untouched.
  PlanOffsets po{};
  if (!build_attention_plan(c, c->h_slot(slot), std::min(plan_region, c->lay.slot_seq_off), &po,
                            unit_cap))
    return HW_ERR_CAPACITY;
  cudaStream_t s = (cudaStream_t)stream;
  st = c->flush_append(layer, s);
  if (st != HW_OK) return st;
  HW_CUDA(cudaMemcpyAsync(scratch, c->h_slot(slot), po.bytes, cudaMemcpyHostToDevice, s));
  hw::AttnArgs a{};
  a.pieces = reinterpret_cast<const hw::Piece*>(scratch + po.pieces);
  a.units = reinterpret_cast<const hw::Unit*>(scratch + po.units);
  a.groups = reinterpret_cast<const hw::Group*>(scratch + po.groups);
  a.delta = reinterpret_cast<const int32_t*>(scratch + po.delta);
  a.fresh = reinterpret_cast<const hw::FreshTok*>(scratch + po.fresh);
  a.num_units = po.num_units;
  a.num_groups = po.num_groups;
  a.num_seg_slots = po.num_seg_slots;
  a.k_layer = c->k_pool + (size_t)layer * c->layer_elems;
  a.v_layer = c->v_pool + (size_t)layer * c->layer_elems;
  a.q = (const __nv_bfloat16*)q;
  a.out = out;
  a.out_f32 = out_dtype == HW_OUT_F32;
  a.lse = lse;
  a.partials = reinterpret_cast<float*>(scratch + plan_region);
  a.rope_cos = c->d_cos();
  a.rope_sin = c->d_sin();
  a.err = c->d_err();
  a.P = c->cfg.num_problems;
  a.W = po.width;                      // query rows per problem / G (= W for decode)
  a.H_q = c->cfg.num_q_heads;
  a.H_kv = c->cfg.num_kv_heads;
  a.G = c->G;
  a.D = c->cfg.head_dim;
  a.S = c->cfg.page_size;
  a.num_pages = c->cfg.num_pages;
  a.max_position = c->cfg.max_position;
  a.rows = po.width * c->G;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  hw::launch_attention_fma(a, c->maps, layer, s);
  HW_CUDA(cudaGetLastError());
  hw::launch_merge(a, s, false, po.max_group_units);
  HW_CUDA(cudaGetLastError());
  HW_CUDA(cudaEventRecord(c->slot_ev[slot], s));
  c->slot_used[slot] = true;
  c->n_launch += 2;
  c->n_attn += 1;
  return HW_OK;
}

extern "C" {

hw_status hw_step_end(hw_ctx* c, const uint8_t* finished, void* stream) {
  if (!c) return HW_ERR_INVALID_ARG;
  const int32_t P = c->cfg.num_problems, W = c->cfg.num_workers;
  if (c->step_active)
    for (uint8_t a : c->appended)
      if (!a) return HW_ERR_INVALID_ARG;
  int64_t commits = 0;
  if (finished)
    for (int32_t p = 0; p < P; ++p)
      for (int32_t w = 0; w < W; ++w)
        if (finished[p * W + w] && c->segs[c->live[p][w]].visible() > 0) ++commits;
  if ((int64_t)c->segs.size() + commits > c->lay.max_segments) return HW_ERR_CAPACITY;
  // Appends no attention call has written yet go to the pool now.
  for (int32_t l = 0; l < (int32_t)c->pend_k.size(); ++l) {
    const hw_status st = c->flush_append(l, (cudaStream_t)stream);
    if (st != HW_OK) return st;
  }
  c->pend_k.clear();
  c->pend_v.clear();
  for (Seg& sg : c->segs) {
    sg.recent_from = sg.pending > 0 ? sg.length : INT32_MAX;
    sg.length += sg.pending;
    sg.pending = 0;
  }
  c->step_active = false;
  ++c->epoch;
  c->step_slot = -1;
  c->appended.clear();
  c->step_n.clear();
  if (finished)
    for (int32_t p = 0; p < P; ++p)
      for (int32_t w = 0; w < W; ++w)
        if (finished[p * W + w] && c->segs[c->live[p][w]].length > 0) {
          c->common[p].push_back(c->live[p][w]);
          c->live[p][w] = c->new_segment(p, w);
        }
  return HW_OK;
}

hw_status hw_compact_segments(hw_ctx* c, int32_t problem, int32_t first, int32_t count,
                              void* stream) {
  if (!c || problem < 0 || problem >= c->cfg.num_problems) return HW_ERR_INVALID_ARG;
  if (c->step_active) return HW_ERR_INVALID_ARG;          // between steps only
  std::vector<int32_t>& com = c->common[problem];
  if (count < 2 || first < 0 || (int64_t)first + count > (int64_t)com.size())
    return HW_ERR_INVALID_ARG;
  const int32_t S = c->cfg.page_size;
  int64_t total = 0;
  bool mixed = false;
  const int32_t origin0 = c->segs[com[first]].origin;
  for (int32_t i = first; i < first + count; ++i) {
    total += c->segs[com[i]].length;
    mixed |= c->segs[com[i]].origin != origin0;
  }
  if (mixed && (c->cfg.layout == HW_LAYOUT_CONTIGUOUS || c->cfg.layout == HW_LAYOUT_NO_SYNC))
    return HW_ERR_INVALID_ARG;                            // these views depend on the writer
  if ((int64_t)c->segs.size() + 1 > c->lay.max_segments) return HW_ERR_CAPACITY;
  if (c->cfg.contiguous && total > S) return HW_ERR_CAPACITY;
  const int64_t need = c->cfg.contiguous ? (total > 0 ? 1 : 0) : (total + S - 1) / S;
  if (need > (int64_t)c->free_pages.size()) return HW_ERR_OUT_OF_PAGES;
  std::vector<int32_t> dst_pages(c->free_pages.begin(), c->free_pages.begin() + need);
  // Runs of tokens that stay inside one page on both sides, at most 128 each.
  std::vector<hw::CompactRun> runs;
  int64_t pos = 0;                                        // position in the merged segment
  for (int32_t i = first; i < first + count; ++i) {
    const Seg& sg = c->segs[com[i]];
    const int64_t rot = pos;
    for (int32_t j = 0; j < sg.length;) {
      const int32_t sp = c->cfg.contiguous ? 0 : j / S, ss = c->cfg.contiguous ? j : j % S;
      const int64_t d = pos;
      const int32_t dp = c->cfg.contiguous ? 0 : (int32_t)(d / S);
      const int32_t ds = c->cfg.contiguous ? (int32_t)d : (int32_t)(d % S);
      const int32_t n = (int32_t)std::min<int64_t>({(int64_t)S - ss, (int64_t)S - ds,
                                                    (int64_t)sg.length - j, 128});
      runs.push_back(hw::CompactRun{sg.pages[sp], ss, dst_pages[dp], ds, n, (int32_t)rot});
      j += n;
      pos += n;
    }
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (!runs.empty()) {
    const size_t bytes = runs.size() * sizeof(hw::CompactRun);
    if (bytes > c->lay.slot_seq_off) return HW_ERR_CAPACITY;
    int slot = 0;
    hw_status st = c->acquire_slot(&slot);
    if (st != HW_OK) return st;
    std::memcpy(c->h_slot(slot), runs.data(), bytes);
    // in stream order: after every earlier call's reads of the old pages, before any later use
    HW_CUDA(cudaMemcpyAsync(c->d_slot(slot), c->h_slot(slot), bytes, cudaMemcpyHostToDevice, s));
    hw::CompactArgs a{};
    a.runs = reinterpret_cast<const hw::CompactRun*>(c->d_slot(slot));
    a.num_runs = (int32_t)runs.size();
    a.num_layers = c->cfg.num_layers;
    a.k_pool = c->k_pool;
    a.v_pool = c->v_pool;
    a.layer_elems = c->layer_elems;
    a.rope_cos = c->d_cos();
    a.rope_sin = c->d_sin();
    a.err = c->d_err();
    a.H_kv = c->cfg.num_kv_heads;
    a.D = c->cfg.head_dim;
    a.S = S;
    a.num_pages = c->cfg.num_pages;
    a.max_position = c->cfg.max_position;
    hw::launch_compact(a, s);
    HW_CUDA(cudaGetLastError());
    HW_CUDA(cudaEventRecord(c->slot_ev[slot], s));
    c->slot_used[slot] = true;
    c->n_launch += 1;
  }
  // Tables: the merged segment takes the range's place; the old pages go back to the free list.
  for (int64_t k = 0; k < need; ++k) c->free_pages.pop_front();
  int32_t origin = mixed ? -1 : origin0;
  const int32_t sid = c->new_segment(problem, origin);
  c->segs[sid].pages = dst_pages;
  c->segs[sid].length = (int32_t)total;
  c->segs[sid].recent_from = 0;           // written by the compaction kernel
  for (int32_t i = first; i < first + count; ++i) {
    Seg& sg = c->segs[com[i]];
    for (int32_t pg : sg.pages) c->free_pages.push_back(pg);
    sg.pages.clear();
    sg.length = 0;
  }
  com.erase(com.begin() + first, com.begin() + first + count);
  com.insert(com.begin() + first, sid);
  ++c->epoch;                     // tables changed: no plan of the old state is reused
  return HW_OK;
}

hw_status hw_compact_auto(hw_ctx* c, int32_t max_paragraphs, void* stream, int32_t* merged) {
  if (!c || max_paragraphs < 1) return HW_ERR_INVALID_ARG;
  if (merged) *merged = 0;
  if (c->step_active) return HW_ERR_INVALID_ARG;          // between steps only
  const bool by_writer =
      c->cfg.layout == HW_LAYOUT_CONTIGUOUS || c->cfg.layout == HW_LAYOUT_NO_SYNC;
  for (int32_t p = 0; p < c->cfg.num_problems; ++p) {
    const std::vector<int32_t>& com = c->common[p];
    if ((int64_t)com.size() - 1 <= max_paragraphs) continue;
    if (!by_writer) {
      // every committed paragraph (all but the prompt) into one RoPE frame
      const hw_status st = hw_compact_segments(c, p, 1, (int32_t)com.size() - 1, stream);
      if (st != HW_OK) return st;
      if (merged) ++*merged;
      continue;
    }
    // views that depend on the writer: each run of consecutive paragraphs of one writer
    for (int32_t i = 1; i < (int32_t)c->common[p].size(); ++i) {   // (a merged run: one entry)
      const std::vector<int32_t>& cm = c->common[p];
      const int32_t origin = c->segs[cm[i]].origin;
      int32_t j = i + 1;
      while (j < (int32_t)cm.size() && c->segs[cm[j]].origin == origin) ++j;
      if (j - i >= 2) {
        const hw_status st = hw_compact_segments(c, p, i, j - i, stream);
        if (st != HW_OK) return st;
        if (merged) ++*merged;
      }
    }
  }
  return HW_OK;
}

hw_status hw_check_device_errors(hw_ctx* c, void* stream, uint32_t* info) {
  if (!c) return HW_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t w[4] = {0, 0, 0, 0};
  HW_CUDA(cudaStreamSynchronize(s));
  HW_CUDA(cudaMemcpy(w, c->d_err(), sizeof(w), cudaMemcpyDeviceToHost));
  if (info) std::memcpy(info, w, sizeof(w));
  if (!w[0]) return HW_OK;
  HW_CUDA(cudaMemset(c->d_err(), 0, sizeof(w)));
  return (w[0] & hw::ERR_TIMEOUT) ? HW_ERR_DEVICE_TIMEOUT : HW_ERR_DEVICE_CHECK;
}

hw_status hw_debug_expire_plans(hw_ctx* c, int32_t count) {
  if (!c || count < 0) return HW_ERR_INVALID_ARG;
  c->expire_plans = count;
  return HW_OK;
}

hw_status hw_profile_enable(hw_ctx* c, int32_t enable) {
  if (!c) return HW_ERR_INVALID_ARG;
  if (enable && c->prof_ev.empty()) {
    c->prof_ev.assign(2 * kProfPairs, nullptr);
    c->prof_kind.assign(kProfPairs, 0);
    for (auto& e : c->prof_ev) HW_CUDA(cudaEventCreate(&e));
  }
  c->prof_on = enable != 0;
  return HW_OK;
}

hw_status hw_profile_read(hw_ctx* c, hw_profile* out) {
  if (!c || !out) return HW_ERR_INVALID_ARG;
  hw_profile r{};
  r.launches = c->n_launch;
  r.attention_launches = c->n_attn;
  r.append_launches = c->n_append;
  for (int i = 0; i < c->prof_next; ++i) {
    HW_CUDA(cudaEventSynchronize(c->prof_ev[2 * i + 1]));
    float ms = 0.f;
    HW_CUDA(cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]));
    if (c->prof_kind[i] == 0) {
      r.attention_ms += ms;
      r.timed_attention += 1;
    } else if (c->prof_kind[i] == 2) {
      r.merge_ms += ms;
      r.timed_merge += 1;
    } else {
      r.append_ms += ms;
      r.timed_append += 1;
    }
  }
  c->prof_next = 0;
  c->n_launch = c->n_attn = c->n_append = 0;
  *out = r;
  return HW_OK;
}

hw_status hw_get_counts(const hw_ctx* c, int32_t* num_segments, int32_t* free_pages) {
  if (!c || !num_segments || !free_pages) return HW_ERR_INVALID_ARG;
  *num_segments = (int32_t)c->segs.size();
  *free_pages = (int32_t)c->free_pages.size();
  return HW_OK;
}

hw_status hw_get_segment(const hw_ctx* c, int32_t seg, int32_t* problem, int32_t* origin,
                         int32_t* length, int32_t* pending, int32_t* num_pages,
                         int32_t* pages_out, int32_t pages_cap) {
  if (!c || seg < 0 || seg >= (int32_t)c->segs.size()) return HW_ERR_INVALID_ARG;
  if (!problem || !origin || !length || !pending || !num_pages) return HW_ERR_INVALID_ARG;
  const Seg& sg = c->segs[seg];
  *problem = sg.problem;
  *origin = sg.origin;
  *length = sg.length;
  *pending = sg.pending;
  *num_pages = (int32_t)sg.pages.size();
  if ((int32_t)sg.pages.size() > pages_cap || (!pages_out && !sg.pages.empty()))
    return HW_ERR_CAPACITY;
  std::copy(sg.pages.begin(), sg.pages.end(), pages_out);
  return HW_OK;
}

hw_status hw_get_blocks(const hw_ctx* c, int32_t problem, int32_t* common_ids, int32_t cap,
                        int32_t* num_common, int32_t* live_ids) {
  if (!c || problem < 0 || problem >= c->cfg.num_problems || !num_common || !live_ids)
    return HW_ERR_INVALID_ARG;
  const auto& cm = c->common[problem];
  *num_common = (int32_t)cm.size();
  std::copy(c->live[problem].begin(), c->live[problem].end(), live_ids);
  if ((int32_t)cm.size() > cap || !common_ids) return HW_ERR_CAPACITY;
  std::copy(cm.begin(), cm.end(), common_ids);
  return HW_OK;
}

hw_status hw_get_view(const hw_ctx* c, int32_t problem, int32_t worker, int32_t* seg_ids,
                      int32_t* view_offsets, int32_t* lengths, int32_t cap, int32_t* n,
                      int32_t* i_q) {
  if (!c || problem < 0 || problem >= c->cfg.num_problems || worker < 0 ||
      worker >= c->cfg.num_workers || !n || !i_q)
    return HW_ERR_INVALID_ARG;
  std::vector<int32_t> ids, offs, lens;
  *i_q = c->view(problem, worker, &ids, &offs, &lens);
  *n = (int32_t)ids.size();
  if ((int32_t)ids.size() > cap || !seg_ids || !view_offsets || !lengths) return HW_ERR_CAPACITY;
  std::copy(ids.begin(), ids.end(), seg_ids);
  std::copy(offs.begin(), offs.end(), view_offsets);
  std::copy(lens.begin(), lens.end(), lengths);
  return HW_OK;
}

}  // extern "C"

// ------------------------------------------------------------------- decode step from host

namespace {
// Device scratch of hw_decode_step_host: [K][V][Q][out], each 256-byte aligned.
struct StepScratch {
  size_t k, v, q, out, bytes;
};
StepScratch step_scratch_layout(const hw_config& cfg, int64_t total_new, int32_t out_elem) {
  const size_t L = (size_t)cfg.num_layers, D = (size_t)cfg.head_dim;
  const size_t kv = L * (size_t)total_new * cfg.num_kv_heads * D * sizeof(__nv_bfloat16);
  const size_t rows = (size_t)cfg.num_problems * cfg.num_workers * cfg.num_q_heads;
  StepScratch s{};
  s.k = 0;
  s.v = align_up(kv, kAlign);
  s.q = s.v + align_up(kv, kAlign);
  s.out = s.q + align_up(L * rows * D * sizeof(__nv_bfloat16), kAlign);
  s.bytes = s.out + align_up(L * rows * D * out_elem, kAlign);
  return s;
}
}  // namespace

extern "C" {

hw_status hw_step_scratch_size(const hw_ctx* c, const int32_t* n_new, int32_t out_dtype,
                               size_t* bytes) {
  if (!c || !n_new || !bytes) return HW_ERR_INVALID_ARG;
  if (out_dtype != HW_OUT_BF16 && out_dtype != HW_OUT_F32) return HW_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int32_t i = 0; i < c->cfg.num_problems * (c->cfg.num_workers + 1); ++i) {
    if (n_new[i] < 0) return HW_ERR_INVALID_ARG;
    total += n_new[i];
  }
  *bytes = step_scratch_layout(c->cfg, total, out_dtype == HW_OUT_F32 ? 4 : 2).bytes;
  return HW_OK;
}

hw_status hw_decode_step_host(hw_ctx* c, const int32_t* n_new, const void* in_host,
                              size_t in_bytes, void* out_host, int32_t out_dtype,
                              const uint8_t* finished, void* scratch, size_t scratch_bytes,
                              int32_t sync, void* stream) {
  if (!c || !n_new || !in_host || !out_host || !scratch) return HW_ERR_INVALID_ARG;
  if (out_dtype != HW_OUT_BF16 && out_dtype != HW_OUT_F32) return HW_ERR_INVALID_ARG;
  if (c->step_active || (uintptr_t)scratch % kAlign) return HW_ERR_INVALID_ARG;
  const hw_config& cfg = c->cfg;
  int64_t total = 0;
  for (int32_t i = 0; i < cfg.num_problems * (cfg.num_workers + 1); ++i) {
    if (n_new[i] < 0) return HW_ERR_INVALID_ARG;
    total += n_new[i];
  }
  const int32_t out_elem = out_dtype == HW_OUT_F32 ? 4 : 2;
  const StepScratch sl = step_scratch_layout(cfg, total, out_elem);
  if (scratch_bytes < sl.bytes) return HW_ERR_CAPACITY;
  const size_t L = (size_t)cfg.num_layers, D = (size_t)cfg.head_dim;
  const size_t kv_layer = (size_t)total * cfg.num_kv_heads * D * sizeof(__nv_bfloat16);
  const size_t q_layer = (size_t)cfg.num_problems * cfg.num_workers * cfg.num_q_heads * D *
                         sizeof(__nv_bfloat16);
  const size_t out_layer = q_layer / sizeof(__nv_bfloat16) * out_elem;
  if (in_bytes != L * (2 * kv_layer + q_layer)) return HW_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* dev = (char*)scratch;
  const char* in = (const char*)in_host;
  // Inputs up: one copy when the scratch holds K, V and Q back to back (no alignment gaps),
  // else one copy per part.
  if (sl.v == L * kv_layer && sl.q == 2 * L * kv_layer) {
    HW_CUDA(cudaMemcpyAsync(dev, in, in_bytes, cudaMemcpyHostToDevice, s));
  } else {
    if (kv_layer) {
      HW_CUDA(cudaMemcpyAsync(dev + sl.k, in, L * kv_layer, cudaMemcpyHostToDevice, s));
      HW_CUDA(cudaMemcpyAsync(dev + sl.v, in + L * kv_layer, L * kv_layer,
                              cudaMemcpyHostToDevice, s));
    }
    HW_CUDA(cudaMemcpyAsync(dev + sl.q, in + 2 * L * kv_layer, L * q_layer,
                            cudaMemcpyHostToDevice, s));
  }
  // Every layer's append, then every layer's attention: an error from an attention call leaves
  // a step that hw_step_end can close.  (An append after the first one fails only on the
  // arguments checked above.)  The step's plan goes up with the first append on this stream,
  // in order with the kernels that read it (one copy, no sequence word).
  struct InOrder {
    hw_ctx* c;
    ~InOrder() { c->plan_in_order = false; }
  } in_order{c};
  c->plan_in_order = true;
  for (int32_t l = 0; l < cfg.num_layers; ++l) {
    const hw_status st = hw_append_kv(c, l, n_new, total ? dev + sl.k + l * kv_layer : nullptr,
                                      total ? dev + sl.v + l * kv_layer : nullptr, stream);
    if (st != HW_OK) return st;
  }
  c->plan_in_order = false;
  for (int32_t l = 0; l < cfg.num_layers; ++l) {
    const hw_status st = attend(c, l, dev + sl.q + l * q_layer, nullptr,
                                dev + sl.out + l * out_layer, out_dtype, nullptr, stream);
    if (st != HW_OK) return st;
  }
  HW_CUDA(cudaMemcpyAsync(out_host, dev + sl.out, L * out_layer, cudaMemcpyDeviceToHost, s));
  const hw_status st = hw_step_end(c, finished, stream);
  if (st != HW_OK) return st;
  if (sync) HW_CUDA(cudaStreamSynchronize(s));
  return HW_OK;
}

}  // extern "C"
