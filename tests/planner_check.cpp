// Host-only check of the attention planner (build_attention_plan in hw_api.cpp, compiled here
// with the kernel launchers stubbed out): random cache states -- segment lengths, this step's
// appended tokens, commits, page orders, every view layout -- and every kind of plan the
// library builds (a decode step's plan with the fused append, a plain call, several query
// tokens per worker, a capped unit count, entry ranges).  Each plan is checked against facts
// computed here from the tables alone, token by token:
//   - every visible token (or every token in the entry range) of every segment of a problem is
//     covered exactly once by the pieces of each (problem, KV head) group's units;
//   - pieces stay inside one page and one 128-token tile, and name the segment's page;
//   - groups tile the unit array in (problem, KV head) order, a problem's units have the same
//     pieces for every KV head, and a problem's units share its tiles exactly (sizes differ by
//     at most one tile when uncapped);
//   - the rotation table holds i_q(w) minus the segment's offset in w's view, or -1 where the
//     layout hides it (views rebuilt here from the layout's definition);
//   - several query tokens: each token has its own output row and its causal cut;
//   - fused append: every token appended in the step is listed once, with its source row, page,
//     slot and position, inside the unit that holds its piece;
//   - a unit's first_tok names its first piece only when that piece holds no token of this
//     step or of the last one.
// Exit status 0 and "planner ok" on success; the first failed fact otherwise.
#include "hw_api.cpp"

#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <set>

namespace hw {
void launch_append(const AppendArgs&, cudaStream_t) {}
void launch_compact(const CompactArgs&, cudaStream_t) {}
void launch_attention_fma(const AttnArgs&, const TcMaps&, int, cudaStream_t) {}
void launch_attention_tc(const AttnArgs&, const TcMaps&, const LaunchUnits&, int, cudaStream_t,
                         cudaEvent_t, cudaEvent_t) {}
void launch_merge(const AttnArgs&, cudaStream_t, bool, int) {}
bool make_tc_maps(const hw_config&, void*, void*, TcMaps*) { return true; }
cudaError_t prepare_attention_fma(int) { return cudaSuccess; }
cudaError_t prepare_attention_tc(int) { return cudaSuccess; }
}  // namespace hw

static int g_case = 0;
#define CHECK(cond, ...)                                                   \
  do {                                                                     \
    if (!(cond)) {                                                         \
      std::printf("case %d: failed: %s -- ", g_case, #cond);               \
      std::printf(__VA_ARGS__);                                            \
      std::printf("\n");                                                   \
      std::exit(1);                                                        \
    }                                                                      \
  } while (0)

// Worker w's view of problem p from the layout's definition: (segment, offset) in order.
static std::vector<std::pair<int32_t, int64_t>> view_of(const hw_ctx* c, int p, int w,
                                                        int64_t* len) {
  std::vector<int32_t> order;
  const auto& com = c->common[p];
  const int W = c->cfg.num_workers;
  auto paragraphs_then_block = [&](int u) {
    for (int32_t sid : com)
      if (c->segs[sid].origin == u) order.push_back(sid);
    order.push_back(c->live[p][u]);
  };
  switch (c->cfg.layout) {
    case HW_LAYOUT_STEP_WISE:
      order = com;
      order.push_back(c->live[p][w]);
      break;
    case HW_LAYOUT_CONTIGUOUS:
    case HW_LAYOUT_NO_SYNC:
      for (int32_t sid : com)
        if (c->segs[sid].origin < 0) order.push_back(sid);
      if (c->cfg.layout == HW_LAYOUT_CONTIGUOUS)
        for (int u = 0; u < W; ++u)
          if (u != w) paragraphs_then_block(u);
      paragraphs_then_block(w);
      break;
    default:
      order = com;
      for (int u = 0; u < W; ++u)
        if (u != w) order.push_back(c->live[p][u]);
      order.push_back(c->live[p][w]);
  }
  std::vector<std::pair<int32_t, int64_t>> v;
  int64_t off = 0;
  for (int32_t sid : order) {
    const int32_t n = c->segs[sid].visible();
    if (n == 0) continue;
    v.push_back({sid, off});
    off += n;
  }
  *len = off;
  return v;
}

// One plan, checked.  nq: [P][W] query tokens per worker or empty; ranges: [P][2] or empty.
static void check_plan(hw_ctx* c, const char* buf, const PlanOffsets& po, bool fuse,
                       const std::vector<int32_t>& nq, const std::vector<int64_t>& ranges,
                       int64_t unit_cap, uint64_t seq) {
  const int P = c->cfg.num_problems, W = c->cfg.num_workers, H = c->cfg.num_kv_heads;
  const int S = c->cfg.page_size;
  const bool contiguous = c->cfg.contiguous != 0;
  const auto* pieces = reinterpret_cast<const hw::Piece*>(buf + po.pieces);
  const auto* units = reinterpret_cast<const hw::Unit*>(buf + po.units);
  const auto* groups = reinterpret_cast<const hw::Group*>(buf + po.groups);
  const auto* delta = reinterpret_cast<const int32_t*>(buf + po.delta);
  const auto* vlen = reinterpret_cast<const int32_t*>(buf + po.vlen);
  const auto* qrow = reinterpret_cast<const int32_t*>(buf + po.qrow);
  const auto* fresh = reinterpret_cast<const hw::FreshTok*>(buf + po.fresh);
  for (size_t o : {po.pieces, po.units, po.groups, po.delta, po.vlen, po.qrow, po.fresh})
    CHECK(o % 16 == 0, "offset %zu", o);
  const int WT = po.width;
  // segment slots: per problem, the non-empty common segments in commit order, then the
  // non-empty worker blocks by id
  std::vector<int32_t> slot_sid;
  std::vector<int> slot_problem;
  std::vector<int64_t> slot_entry0;                    // entry number of the segment's token 0
  for (int p = 0; p < P; ++p) {
    int64_t entry = 0;
    std::vector<int32_t> refs;
    for (int32_t sid : c->common[p])
      if (c->segs[sid].visible() > 0) refs.push_back(sid);
    for (int w = 0; w < W; ++w)
      if (c->segs[c->live[p][w]].visible() > 0) refs.push_back(c->live[p][w]);
    for (int32_t sid : refs) {
      slot_sid.push_back(sid);
      slot_problem.push_back(p);
      slot_entry0.push_back(entry);
      entry += c->segs[sid].visible();
    }
  }
  CHECK(po.num_seg_slots == (int)slot_sid.size(), "slots %d vs %zu", po.num_seg_slots,
        slot_sid.size());
  // groups and units
  CHECK(po.num_groups == P * H, "groups %d", po.num_groups);
  int32_t next_unit = 0;
  for (int gi = 0; gi < P * H; ++gi) {
    const hw::Group& g = groups[gi];
    CHECK(g.p == gi / H && g.h == gi % H, "group %d is (%d, %d)", gi, g.p, g.h);
    CHECK(g.unit_begin == next_unit && g.unit_end > g.unit_begin, "group %d units [%d, %d)", gi,
          g.unit_begin, g.unit_end);
    next_unit = g.unit_end;
    for (int k = g.unit_begin; k < g.unit_end; ++k) {
      const hw::Unit& u = units[k];
      CHECK(u.group == gi, "unit %d group %d", k, u.group);
      CHECK(u.seq == (uint32_t)seq && u.seq_b == (uint32_t)seq && u.seq_c == (uint32_t)seq,
            "unit %d sequence", k);
      CHECK(0 <= u.piece_begin && u.piece_begin <= u.piece_end && u.piece_end <= po.num_pieces,
            "unit %d pieces [%d, %d)", k, u.piece_begin, u.piece_end);
      // the same pieces for every KV head of the problem
      const hw::Group& g0 = groups[g.p * H];
      const hw::Unit& u0 = units[g0.unit_begin + (k - g.unit_begin)];
      CHECK(g.unit_end - g.unit_begin == g0.unit_end - g0.unit_begin &&
                u.piece_begin == u0.piece_begin && u.piece_end == u0.piece_end,
            "unit %d differs from head 0", k);
      CHECK(u.seg0 == (u.piece_end > u.piece_begin ? pieces[u.piece_begin].seg_slot : -1),
            "unit %d seg0", k);
    }
  }
  CHECK(next_unit == po.num_units, "units %d vs %d", next_unit, po.num_units);
  if (unit_cap > 0) CHECK(po.num_units <= unit_cap, "units %d over the cap %ld", po.num_units,
                          (long)unit_cap);
  // coverage, token by token, per group; pieces inside one page and one tile
  for (int gi = 0; gi < P * H; ++gi) {
    const hw::Group& g = groups[gi];
    std::map<int32_t, std::vector<int>> seen;              // slot -> count per token
    int64_t min_tiles = INT64_MAX, max_tiles = 0;
    for (int k = g.unit_begin; k < g.unit_end; ++k) {
      const hw::Unit& u = units[k];
      min_tiles = std::min<int64_t>(min_tiles, u.piece_end - u.piece_begin);
      max_tiles = std::max<int64_t>(max_tiles, u.piece_end - u.piece_begin);
      for (int i = u.piece_begin; i < u.piece_end; ++i) {
        const hw::Piece& pc = pieces[i];
        CHECK(pc.seg_slot >= 0 && pc.seg_slot < po.num_seg_slots, "piece %d slot", i);
        CHECK(slot_problem[pc.seg_slot] == g.p, "piece %d of another problem", i);
        const Seg& sg = c->segs[slot_sid[pc.seg_slot]];
        CHECK(pc.ntok >= 1 && pc.ntok <= 128 && pc.pos0 >= 0 && pc.pos0 + pc.ntok <= sg.visible(),
              "piece %d tokens [%d, +%d) of %d", i, pc.pos0, pc.ntok, sg.visible());
        CHECK(pc.pos0 / 128 == (pc.pos0 + pc.ntok - 1) / 128, "piece %d crosses a tile", i);
        const int pg_idx = contiguous ? 0 : pc.pos0 / S;
        CHECK(pg_idx < (int)sg.pages.size() && pc.page == sg.pages[pg_idx], "piece %d page", i);
        CHECK(pc.slot0 == (contiguous ? pc.pos0 : pc.pos0 % S) && pc.slot0 + pc.ntok <= S,
              "piece %d slot %d", i, pc.slot0);
        CHECK(pc.fresh == (pc.pos0 + pc.ntok > sg.length ? 1 : 0), "piece %d fresh flag", i);
        auto& cnt = seen[pc.seg_slot];
        cnt.resize(sg.visible(), 0);
        for (int t = pc.pos0; t < pc.pos0 + pc.ntok; ++t) ++cnt[t];
      }
    }
    if (unit_cap == 0 && ranges.empty())
      CHECK(max_tiles - min_tiles <= 1, "group %d unit sizes %ld..%ld", gi, (long)min_tiles,
            (long)max_tiles);
    for (size_t sl = 0; sl < slot_sid.size(); ++sl) {
      if (slot_problem[sl] != g.p) continue;
      const Seg& sg = c->segs[slot_sid[sl]];
      auto it = seen.find((int32_t)sl);
      for (int t = 0; t < sg.visible(); ++t) {
        int want = 1;
        if (!ranges.empty()) {
          const int64_t e = slot_entry0[sl] + t;
          want = (e >= ranges[2 * g.p] && e < ranges[2 * g.p + 1]) ? 1 : 0;
        }
        const int got = it == seen.end() ? 0 : it->second[t];
        CHECK(got == want, "group %d slot %zu token %d covered %d times, want %d", gi, sl, t, got,
              want);
      }
    }
  }
  // rotation table (and, with several query tokens, the causal cut and the row map)
  std::set<int32_t> rows_seen;
  int32_t rows_total = 0;
  for (int p = 0; p < P; ++p) {
    int v0 = 0;
    for (int w = 0; w < W; ++w) {
      const int n = nq.empty() ? 1 : nq[p * W + w];
      int64_t len = 0;
      const auto view = view_of(c, p, w, &len);
      for (int t = 0; t < n; ++t) {
        const int back = n - 1 - t, v = nq.empty() ? w : v0 + t;
        for (size_t sl = 0; sl < slot_sid.size(); ++sl) {
          if (slot_problem[sl] != p) continue;
          int64_t want = -1;
          int own_cut = -1;
          for (size_t k = 0; k < view.size(); ++k)
            if (view[k].first == slot_sid[sl]) {
              want = len - 1 - back - view[k].second;
              const int vis = c->segs[slot_sid[sl]].visible();
              own_cut = k + 1 == view.size() ? vis - back : vis;
            }
          CHECK(delta[sl * WT + v] == want, "problem %d worker %d token %d slot %zu delta %d want %ld",
                p, w, t, sl, delta[sl * WT + v], (long)want);
          if (!nq.empty() && want >= 0)
            CHECK(vlen[sl * WT + v] == own_cut, "causal cut %d want %d", vlen[sl * WT + v], own_cut);
        }
        if (!nq.empty()) {
          const int32_t r = qrow[p * WT + v];
          CHECK(r == rows_total, "query row %d want %d", r, rows_total);
          CHECK(rows_seen.insert(r).second, "row %d twice", r);
          ++rows_total;
        }
      }
      v0 += n;
    }
  }
  // fused append: every appended token once, in the unit that holds its piece
  if (fuse) {
    std::map<std::tuple<int32_t, int32_t>, int> listed;    // (page, slot) -> count
    int32_t src = 0;
    for (int p = 0; p < P; ++p)
      for (int b = 0; b <= W; ++b) {
        const int n = c->step_n[(size_t)p * (W + 1) + b];
        const int32_t sid = b == 0 ? c->common[p].back() : c->live[p][b - 1];
        const Seg& sg = c->segs[sid];
        for (int k = 0; k < n; ++k) {
          const int j = sg.length + k;
          const int pg = sg.pages[contiguous ? 0 : j / S];
          const int sl = contiguous ? j : j % S;
          bool found = false;
          for (int f = 0; f < po.num_fresh; ++f)
            if (fresh[f].page == pg && fresh[f].slot == sl) {
              CHECK(!found, "token (%d, %d) listed twice", pg, sl);
              found = true;
              CHECK(fresh[f].pos == j && fresh[f].src == src + k, "token (%d, %d) pos %d src %d",
                    pg, sl, fresh[f].pos, fresh[f].src);
            }
          CHECK(found, "appended token (%d, %d) not listed", pg, sl);
        }
        src += n;
      }
    int64_t appended = 0;
    for (int32_t n : c->step_n) appended += n;
    CHECK(po.num_fresh == appended, "fresh %d appended %ld", po.num_fresh, (long)appended);
    for (int k = 0; k < po.num_units; ++k) {
      const hw::Unit& u = units[k];
      for (int f = u.fresh_begin; f < u.fresh_end; ++f) {
        bool inside = false;
        for (int i = u.piece_begin; i < u.piece_end && !inside; ++i)
          inside = pieces[i].page == fresh[f].page && fresh[f].slot >= pieces[i].slot0 &&
                   fresh[f].slot < pieces[i].slot0 + pieces[i].ntok;
        CHECK(inside, "unit %d lists a token outside its pieces", k);
      }
    }
  }
  // first_tok: only a first piece with no token of this step or of the last one
  for (int k = 0; k < po.num_units; ++k) {
    const hw::Unit& u = units[k];
    if (u.first_tok < 0) continue;
    const hw::Piece& pc = pieces[u.piece_begin];
    const Seg& sg = c->segs[slot_sid[pc.seg_slot]];
    CHECK(u.first_tok == pc.page * S + pc.slot0, "unit %d first_tok", k);
    CHECK(!pc.fresh && pc.pos0 + pc.ntok <= sg.recent_from, "unit %d early tile is recent", k);
  }
}

int main() {
  std::mt19937 g(20261202);
  auto R = [&](int lo, int hi) { return std::uniform_int_distribution<int>(lo, hi)(g); };
  int plans = 0;
  for (int it = 0; it < 600; ++it) {
    hw_config cfg{};
    cfg.num_problems = R(1, 3);
    cfg.num_workers = R(1, 8);
    cfg.num_layers = 1;
    cfg.num_kv_heads = R(1, 3);
    int G = R(1, 8);
    while (cfg.num_workers * G > 128) --G;
    cfg.num_q_heads = cfg.num_kv_heads * G;
    cfg.head_dim = R(0, 1) ? 128 : 64;
    cfg.page_size = 128 * R(1, 3);
    cfg.contiguous = R(0, 4) == 0;
    cfg.layout = R(0, 3);
    cfg.rope_theta = 1e4;
    const int P = cfg.num_problems, W = cfg.num_workers, S = cfg.page_size;
    const int ncommit = R(0, 4);
    cfg.max_segments = P * (1 + W) + P * ncommit + 8;
    const int cap = cfg.contiguous ? S : 4096;
    cfg.num_pages = P * (1 + W + ncommit) * (cfg.contiguous ? 1 : (cap + S - 1) / S + 2) + 8;
    cfg.max_position = P * (1 + W + ncommit) * cap + 16;
    hw_ctx* c = new hw_ctx();
    c->cfg = cfg;
    c->lay = make_layout(&cfg);
    c->G = G;
    c->rows = c->lay.rows;
    c->num_sms = R(0, 1) ? 152 : R(4, 40);
    c->use_tc = c->rows >= 16;
    std::vector<int32_t> order(cfg.num_pages);
    for (int i = 0; i < cfg.num_pages; ++i) order[i] = i;
    std::shuffle(order.begin(), order.end(), g);
    c->free_pages.assign(order.begin(), order.end());
    const bool step = R(0, 2) > 0;
    auto fill = [&](int sid, int len, int pend) {
      Seg& s = c->segs[sid];
      s.length = len;
      s.pending = pend;
      const int vis = len + pend;
      if (cfg.contiguous) {
        if (vis > 0) {
          s.pages.push_back(c->free_pages.front());
          c->free_pages.pop_front();
        }
      } else {
        for (int j = 0; j < vis; j += S) {
          s.pages.push_back(c->free_pages.front());
          c->free_pages.pop_front();
        }
      }
      s.recent_from = R(0, 3) == 0 ? R(0, std::max(0, len)) : INT32_MAX;
    };
    const int maxlen = cfg.contiguous ? S - 20 : R(0, 1) ? 700 : 2000;
    for (int p = 0; p < P; ++p) {
      c->common.push_back({c->new_segment(p, -1)});
      for (int k = 0; k < ncommit; ++k) c->common[p].push_back(c->new_segment(p, R(0, W - 1)));
      std::vector<int32_t> lv;
      for (int k = 0; k < W; ++k) lv.push_back(c->new_segment(p, k));
      c->live.push_back(lv);
    }
    c->step_n.assign((size_t)P * (W + 1), 0);
    for (int p = 0; p < P; ++p) {
      for (size_t k = 0; k < c->common[p].size(); ++k) {
        const bool last = k + 1 == c->common[p].size();
        const int pend = (step && last) ? R(0, 3) : 0;
        fill(c->common[p][k], R(0, 1) ? R(0, maxlen) : R(0, 3), pend);
        if (last) c->step_n[(size_t)p * (W + 1)] = pend;
      }
      for (int k = 0; k < W; ++k) {
        const int pend = step ? R(0, 2) : 0;
        fill(c->live[p][k], R(0, 3) == 0 ? 0 : R(0, maxlen), pend);
        c->step_n[(size_t)p * (W + 1) + 1 + k] = pend;
      }
    }
    c->step_active = step;
    std::vector<char> buf(c->lay.slot_bytes);
    for (int call = 0; call < 5; ++call) {
      g_case = it * 5 + call;
      PlanOffsets po{};
      const int64_t target = c->use_tc ? c->num_sms : 2 * c->num_sms;
      const bool fuse = step && call == 0;
      std::vector<int32_t> nq;
      std::vector<int64_t> ranges;
      int64_t ucap = 0;
      if (call == 2) {                      // several query tokens per worker
        nq.assign((size_t)P * W, 0);
        int64_t width = 1;
        for (int p = 0; p < P; ++p) {
          int64_t v = 0;
          for (int k = 0; k < W; ++k) {
            nq[(size_t)p * W + k] = std::min(R(0, 3), c->segs[c->live[p][k]].visible());
            v += nq[(size_t)p * W + k];
          }
          width = std::max(width, v);
        }
        if (width * G > 128) nq.clear();
        else ucap = (int64_t)c->lay.max_units * c->rows / (width * G);
      }
      if (call == 3) ucap = P * cfg.num_kv_heads + R(0, 50);
      if (call == 4) {                      // entry ranges
        for (int p = 0; p < P; ++p) {
          int64_t total = 0;
          for (int32_t sid : c->common[p]) total += c->segs[sid].visible();
          for (int k = 0; k < W; ++k) total += c->segs[c->live[p][k]].visible();
          const int64_t a = R(0, (int)total), b = R((int)a, (int)total);
          ranges.push_back(a);
          ranges.push_back(b);
        }
      }
      const uint64_t seq = 1000 + g_case;
      const bool ok = build_attention_plan(c, buf.data(), c->lay.slot_seq_off, &po, ucap, target,
                                           fuse, seq, nq.empty() ? nullptr : nq.data(),
                                           ranges.empty() ? nullptr : ranges.data());
      if (!ok) {
        CHECK(call == 3, "an uncapped plan was refused");     // only a tight unit cap may refuse
        continue;
      }
      check_plan(c, buf.data(), po, fuse, nq, ranges, ucap, seq);
      ++plans;
    }
    delete c;
  }
  std::printf("planner ok: %d plans\n", plans);
  return 0;
}
