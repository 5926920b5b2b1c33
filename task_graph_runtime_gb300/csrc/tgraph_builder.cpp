// Host tGraph builder.  See tgraph_builder.h for the passes and sources.
#include "tgraph_builder.h"

#include "device_abi.h"

#include <algorithm>
#include <deque>
#include <unordered_map>

namespace mpk {
namespace {

// Activation tensors of one step, each written once (single assignment), so
// the only hazards are read-after-write and the only events are overlaps of
// an output region with an input region.
enum TensorKind {
  T_H = 0,     // residual stream entering layer l (h_l), [B, hidden]
  T_QKV,       // [B, (Hq + 2Hkv) d]
  T_OPART,     // attention partials [B Hkv, chunks]
  T_ATTN,      // attention output [B, Hq d]
  T_O,         // o-projection output [B, hidden]
  T_HMID,      // h_l + o
  T_ACT,       // SwiGLU (or SiLU) activation [B, ffn]
  T_DOUT,      // down-projection output [B, hidden]
  T_Z,         // chained mode: W2 output
  T_LOGITS,
  T_AMAX,      // per-tile (max, argmax) [B, lm_head tiles]
  T_NEXT,
  T_NKINDS
};

constexpr int kWhole = 1 << 30;   // "to the end" of a tensor axis

struct Decomposer {
  const BuildConfig& cfg;
  std::vector<BOp>& ops;
  std::vector<BTask>& tasks;
  int nl1;  // layers + 1 (tensor interning stride)
  bool bad_rows = false;   // an explicit tile size above a tile cap

  int tid(int kind, int layer) const { return kind * nl1 + layer; }

  void begin_op(int kind, int layer) {
    ops.push_back(BOp{kind, layer, (int)tasks.size(), 0});
  }
  BTask& add_task() {
    BOp& op = ops.back();
    tasks.emplace_back();
    BTask& t = tasks.back();
    t.kind = op.kind;
    t.op = (int)ops.size() - 1;
    t.layer = op.layer;
    t.tile = op.n++;
    return t;
  }
  // A read of a whole tensor (or, with coarse events, every read).
  void read(BTask& t, int tensor, int r0, int r1, int c0, int c1) {
    if (cfg.coarse_events)
      t.reads.push_back({tensor, 0, kWhole, 0, kWhole});
    else
      t.reads.push_back({tensor, r0, r1, c0, c1});
  }
  // MatMul tiles: each reads its whole input rows (the sources of its
  // prologue); tile 0 also writes `resid` when the prologue forms one.
  void gemv(int kind, int layer, int n_rows, bool dual,
            std::initializer_list<int> srcs, int k_cols, int dst, int resid,
            int extra_dst) {
    const int B = cfg.batch;
    begin_op(kind, layer);
    const int rpt =
        B >= 8 ? cfg.mma_rows_per_task : cfg.gemv_rows_per_task;
    const int cap = tile_row_cap(B, dual, k_cols);
    if (rpt > cap) bad_rows = true;
    auto tl = row_tiles(n_rows, rpt, cfg.num_workers, cap, B == 1 ? 1 : 8);
    for (size_t i = 0; i < tl.size(); ++i) {
      BTask& t = add_task();
      t.row0 = tl[i].first;
      t.row1 = tl[i].second;
      for (int src : srcs) read(t, src, 0, B, 0, k_cols);
      t.writes.push_back({dst, 0, B, t.row0, t.row1});
      if (i == 0 && resid >= 0) t.writes.push_back({resid, 0, B, 0, k_cols});
      if (extra_dst >= 0)
        t.writes.push_back({extra_dst, 0, B, (int)i, (int)i + 1});
    }
  }

  void run() {
    const mpk_model_shape& s = cfg.shape;
    const int B = cfg.batch, h = s.hidden, d = s.head_dim;
    const int Hq = s.n_q_heads, Hkv = s.n_kv_heads;
    const int L = s.n_layers;
    if (s.chain_ffn > 0) {
      // x = RMSNorm(embed[token]) is the prologue of every W1 tile
      gemv(MPK_TASK_CHAIN_UP, 0, s.chain_ffn, false, {}, h, tid(T_ACT, 0), -1,
           -1);
      gemv(MPK_TASK_CHAIN_DOWN, 0, h, false, {tid(T_ACT, 0)}, s.chain_ffn,
           tid(T_Z, 0), -1, -1);
      gemv(MPK_TASK_LM_HEAD, 0, s.vocab, false, {tid(T_Z, 0)}, h,
           tid(T_LOGITS, 0), -1, tid(T_AMAX, 0));
    } else {
      const int grp = Hq / Hkv, C = cfg.attn_chunks;
      for (int l = 0; l < L; ++l) {
        // prologue: h_l = hmid_{l-1} + dout_{l-1} (layer 0: embedding), then
        // RMSNorm; tile 0 stores h_l
        if (l == 0)
          gemv(MPK_TASK_QKV, l, (Hq + 2 * Hkv) * d, false, {}, h,
               tid(T_QKV, l), tid(T_H, l), -1);
        else
          gemv(MPK_TASK_QKV, l, (Hq + 2 * Hkv) * d, false,
               {tid(T_HMID, l - 1), tid(T_DOUT, l - 1)}, h, tid(T_QKV, l),
               tid(T_H, l), -1);
        begin_op(MPK_TASK_ATTN, l);
        for (int b = 0; b < B; ++b)
          for (int g = 0; g < Hkv; ++g)
            for (int c = 0; c < C; ++c) {
              BTask& t = add_task();
              t.b = b;
              t.g = g;
              t.c = c;
              const int q0 = g * grp * d, q1 = (g + 1) * grp * d;
              const int k0 = Hq * d + g * d, v0 = (Hq + Hkv) * d + g * d;
              read(t, tid(T_QKV, l), b, b + 1, q0, q1);
              read(t, tid(T_QKV, l), b, b + 1, k0, k0 + d);
              read(t, tid(T_QKV, l), b, b + 1, v0, v0 + d);
              t.writes.push_back(
                  {tid(T_OPART, l), b * Hkv + g, b * Hkv + g + 1, c, c + 1});
              // the last chunk to finish merges (b, g): every chunk may
              // write the group's attention output
              t.writes.push_back({tid(T_ATTN, l), b, b + 1, q0, q1});
            }
        gemv(MPK_TASK_O, l, h, false, {tid(T_ATTN, l)}, Hq * d, tid(T_O, l),
             -1, -1);
        // prologue: hmid_l = h_l + o_l, RMSNorm; tile 0 stores hmid_l
        gemv(MPK_TASK_GATEUP, l, s.ffn, true, {tid(T_H, l), tid(T_O, l)}, h,
             tid(T_ACT, l), tid(T_HMID, l), -1);
        gemv(MPK_TASK_DOWN, l, h, false, {tid(T_ACT, l)}, s.ffn,
             tid(T_DOUT, l), -1, -1);
      }
      // prologue: the final residual sum + RMSNorm; tile 0 stores h_L
      gemv(MPK_TASK_LM_HEAD, L, s.vocab, false,
           {tid(T_HMID, L - 1), tid(T_DOUT, L - 1)}, h, tid(T_LOGITS, 0),
           tid(T_H, L), tid(T_AMAX, 0));
    }
    const int n_lm = ops.back().n;
    begin_op(MPK_TASK_ARGMAX, L);
    BTask& t = add_task();
    read(t, tid(T_AMAX, 0), 0, B, 0, n_lm);
    t.writes.push_back({tid(T_NEXT, 0), 0, B, 0, 1});
  }
};

inline bool overlaps(const Region& a, const Region& b) {
  return a.r0 < b.r1 && b.r0 < a.r1 && a.c0 < b.c1 && b.c0 < a.c1;
}

// Raw events: all (producer, consumer) pairs whose regions overlap, sorted
// by (producer, consumer).  Per tensor, writers are sorted by c0 so each
// reader scans only writers starting left of its right edge.
std::vector<std::pair<int, int>> raw_events(const std::vector<BTask>& tasks,
                                            int n_tensors) {
  struct Ref {
    int task;
    Region r;
  };
  std::vector<std::vector<Ref>> writers(n_tensors), readers(n_tensors);
  for (int i = 0; i < (int)tasks.size(); ++i) {
    for (const Region& w : tasks[i].writes) writers[w.tensor].push_back({i, w});
    for (const Region& r : tasks[i].reads) readers[r.tensor].push_back({i, r});
  }
  std::vector<std::pair<int, int>> pairs;
  for (int tsr = 0; tsr < n_tensors; ++tsr) {
    auto& ws = writers[tsr];
    if (ws.empty() || readers[tsr].empty()) continue;
    std::sort(ws.begin(), ws.end(),
              [](const Ref& a, const Ref& b) { return a.r.c0 < b.r.c0; });
    for (const Ref& rd : readers[tsr]) {
      for (const Ref& w : ws) {
        if (w.r.c0 >= rd.r.c1) break;
        if (w.task != rd.task && overlaps(w.r, rd.r))
          pairs.emplace_back(w.task, rd.task);
      }
    }
  }
  std::sort(pairs.begin(), pairs.end());
  pairs.erase(std::unique(pairs.begin(), pairs.end()), pairs.end());
  return pairs;
}

struct VecHash {
  size_t operator()(const std::vector<int>& v) const {
    uint64_t h = 1469598103934665603ull ^ v.size();
    for (int x : v) {
      h ^= (uint64_t)(uint32_t)x + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    }
    return (size_t)h;
  }
};

struct Ev {
  std::vector<int> in, out;  // sorted task ids
  bool alive = true;
};

void sort_unique(std::vector<int>& v) {
  std::sort(v.begin(), v.end());
  v.erase(std::unique(v.begin(), v.end()), v.end());
}

// Def 4.1 (equal OutTasks: union the InTasks) then Def 4.2 (equal InTasks:
// union the OutTasks), repeated until a full round merges nothing.  The
// merged event keeps the smallest id of its group.
void fuse(std::vector<Ev>& ev) {
  bool changed = true;
  while (changed) {
    changed = false;
    for (int pass = 0; pass < 2; ++pass) {
      const bool by_out = (pass == 0);
      std::unordered_map<std::vector<int>, int, VecHash> keeper;
      keeper.reserve(ev.size() * 2);
      std::vector<int> touched;
      for (int i = 0; i < (int)ev.size(); ++i) {
        if (!ev[i].alive) continue;
        const std::vector<int>& key = by_out ? ev[i].out : ev[i].in;
        auto it = keeper.find(key);
        if (it == keeper.end()) {
          keeper.emplace(key, i);
          continue;
        }
        Ev& k = ev[it->second];
        std::vector<int>& dst = by_out ? k.in : k.out;
        const std::vector<int>& src = by_out ? ev[i].in : ev[i].out;
        dst.insert(dst.end(), src.begin(), src.end());
        touched.push_back(it->second);
        ev[i].alive = false;
        ev[i].in.clear();
        ev[i].out.clear();
        changed = true;
      }
      for (int k : touched) sort_unique(by_out ? ev[k].in : ev[k].out);
    }
  }
}

}  // namespace

int tile_row_cap(int batch, bool dual, int K) {
  int rows;
  if (batch == 1)
    rows = kB1Partials / b1_warps_per_row(K);
  else
    rows = batch < 8 ? 64 : 128;
  if (dual) rows /= 2;
  return std::max(8, rows / 8 * 8);
}

std::vector<std::pair<int, int>> row_tiles(int n_rows, int rows_per_task,
                                           int num_workers, int cap_rows,
                                           int unit) {
  std::vector<std::pair<int, int>> out;
  if (rows_per_task > 0) {
    for (int s = 0; s < n_rows; s += rows_per_task)
      out.emplace_back(s, std::min(n_rows, s + rows_per_task));
    return out;
  }
  const int64_t U = (n_rows + unit - 1) / unit;
  const int64_t cap_u = std::max(1, cap_rows / unit);
  const int64_t T0 = (U + cap_u - 1) / cap_u;
  const int64_t W = std::max(1, num_workers);
  const int64_t T = std::max<int64_t>(1, std::min(U, W * ((T0 + W - 1) / W)));
  for (int64_t i = 0; i < T; ++i) {
    const int64_t u0 = (i * U) / T, u1 = ((i + 1) * U) / T;
    out.emplace_back((int)(unit * u0),
                     (int)std::min<int64_t>(n_rows, unit * u1));
  }
  return out;
}

bool attn_is_aot(int batch, int max_ctx, int chunks) {
  return batch == 1 && chunks > 0 && (max_ctx + chunks - 1) / chunks <= 128;
}

int default_attn_chunks(int batch, int n_kv_heads, int max_ctx,
                        int num_workers) {
  const int by_len = (max_ctx + 127) / 128;
  const int denom = batch * n_kv_heads;
  const int by_workers = (4 * num_workers + denom - 1) / denom;
  return std::max(1, std::min(by_len, by_workers));
}

mpk_status build_tgraph(const BuildConfig& cfg_in, BuiltGraph* out,
                        std::string* err) {
  BuildConfig cfg = cfg_in;
  const mpk_model_shape& s = cfg.shape;
  auto fail = [&](mpk_status st, const char* m) {
    if (err) *err = m;
    return st;
  };
  if (cfg.batch < 1 || cfg.num_workers < 1) return fail(MPK_ERR_INVALID_ARG, "batch and workers must be >= 1");
  if (s.hidden < 8 || s.vocab < 1) return fail(MPK_ERR_INVALID_ARG, "bad hidden/vocab");
  if (s.hidden % 8) return fail(MPK_ERR_UNSUPPORTED, "hidden must be a multiple of 8");
  if (s.hidden > 8192) return fail(MPK_ERR_UNSUPPORTED, "hidden must be <= 8192 (RMSNorm prologue)");
  const bool chain = s.chain_ffn > 0;
  int max_ctx = 0;
  if (chain) {
    if (s.n_layers != 0) return fail(MPK_ERR_INVALID_ARG, "chained mode needs n_layers == 0");
    if (s.chain_ffn % 8) return fail(MPK_ERR_UNSUPPORTED, "chain_ffn must be a multiple of 8");
  } else {
    if (s.n_layers < 1 || s.n_q_heads < 1 || s.n_kv_heads < 1 || s.ffn < 8 ||
        s.page_size < 1 || s.max_pages_per_seq < 1)
      return fail(MPK_ERR_INVALID_ARG, "bad decoder shape");
    if (s.n_q_heads % s.n_kv_heads) return fail(MPK_ERR_INVALID_ARG, "n_q_heads % n_kv_heads != 0");
    if (s.head_dim != 32 && s.head_dim != 64 && s.head_dim != 128)
      return fail(MPK_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 128");
    const int grp = s.n_q_heads / s.n_kv_heads;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8)
      return fail(MPK_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8");
    if (s.ffn % 8) return fail(MPK_ERR_UNSUPPORTED, "ffn must be a multiple of 8");
    max_ctx = s.max_pages_per_seq * s.page_size;
    if (cfg.attn_chunks <= 0)
      cfg.attn_chunks = default_attn_chunks(cfg.batch, s.n_kv_heads, max_ctx,
                                            cfg.num_workers);
  }
  if (cfg.batch > 16) return fail(MPK_ERR_UNSUPPORTED, "batch > 16");
  if (cfg.gemv_rows_per_task < 0 || cfg.gemv_rows_per_task % 8 ||
      cfg.mma_rows_per_task < 0 || cfg.mma_rows_per_task % 8)
    return fail(MPK_ERR_INVALID_ARG, "rows per task must be a multiple of 8");
  {
    const int kmax = chain ? std::max(s.hidden, s.chain_ffn)
                           : std::max({s.hidden, s.n_q_heads * s.head_dim, s.ffn});
    if (kmax > 16384)
      return fail(MPK_ERR_UNSUPPORTED, "MatMul reduction length above 16384");
  }
  if (chain) cfg.attn_chunks = 0;
  const bool attn_aot = !chain && attn_is_aot(cfg.batch, max_ctx, cfg.attn_chunks);

  BuiltGraph g;
  g.cfg = cfg;
  Decomposer dec{cfg, g.ops, g.tasks, s.n_layers + 1};
  dec.run();
  if (dec.bad_rows)
    return fail(MPK_ERR_UNSUPPORTED, "rows per task above the tile cap");
  g.n_real = (int)g.tasks.size();
  const int n_tensors = T_NKINDS * (s.n_layers + 1);

  // 1. raw events by overlap; 2. fusion
  auto raw = raw_events(g.tasks, n_tensors);
  g.n_raw = (int64_t)raw.size();
  std::vector<Ev> ev(raw.size());
  for (size_t i = 0; i < raw.size(); ++i) {
    ev[i].in = {raw[i].first};
    ev[i].out = {raw[i].second};
  }
  std::vector<std::pair<int, int>>().swap(raw);
  fuse(ev);
  int64_t n_fused = 0;
  for (auto& e : ev) n_fused += e.alive;
  g.n_fused = n_fused;

  // 3. normalisation: fan-outs (tasks ascending), then fan-ins
  std::vector<std::vector<int>> trig_of(g.tasks.size()), dep_of(g.tasks.size());
  for (int i = 0; i < (int)ev.size(); ++i) {
    if (!ev[i].alive) continue;
    for (int t : ev[i].in) trig_of[t].push_back(i);
    for (int t : ev[i].out) dep_of[t].push_back(i);
  }
  auto new_empty = [&]() {
    g.tasks.emplace_back();
    trig_of.emplace_back();
    dep_of.emplace_back();
    return (int)g.tasks.size() - 1;
  };
  auto erase_val = [](std::vector<int>& v, int x) {
    v.erase(std::find(v.begin(), v.end(), x));
  };
  for (int t = 0; t < g.n_real; ++t) {
    if (trig_of[t].size() < 2) continue;
    std::vector<int> old = trig_of[t];
    std::sort(old.begin(), old.end());
    const int e1 = (int)ev.size();
    ev.emplace_back();
    ev[e1].in = {t};
    trig_of[t] = {e1};
    for (int ei : old) {
      const int Ti = new_empty();
      erase_val(ev[ei].in, t);
      ev[ei].in.push_back(Ti);
      ev[e1].out.push_back(Ti);
      trig_of[Ti] = {ei};
      dep_of[Ti] = {e1};
    }
  }
  for (int t = 0; t < (int)g.tasks.size(); ++t) {
    if (dep_of[t].size() < 2) continue;
    std::vector<int> old = dep_of[t];
    std::sort(old.begin(), old.end());
    const int e2 = (int)ev.size();
    ev.emplace_back();
    ev[e2].out = {t};
    dep_of[t] = {e2};
    for (int ei : old) {
      const int Ti = new_empty();
      erase_val(ev[ei].out, t);
      ev[ei].out.push_back(Ti);
      ev[e2].in.push_back(Ti);
      dep_of[Ti] = {ei};
      trig_of[Ti] = {e2};
    }
  }
  const int nT = (int)g.tasks.size();
  const int root = (int)ev.size();
  ev.emplace_back();
  const int end = (int)ev.size();
  ev.emplace_back();
  for (int t = 0; t < nT; ++t) {
    if (dep_of[t].empty()) {
      ev[root].out.push_back(t);
      dep_of[t] = {root};
    }
    if (trig_of[t].empty()) {
      ev[end].in.push_back(t);
      trig_of[t] = {end};
    }
  }
  for (auto& e : ev) {
    std::sort(e.in.begin(), e.in.end());
    std::sort(e.out.begin(), e.out.end());
  }

  // 4. Kahn-style BFS linearisation from the root
  const int nE = (int)ev.size();
  std::vector<int> remaining(nE), ev_pos(nE, -1), task_pos(nT, -1);
  for (int i = 0; i < nE; ++i) remaining[i] = (int)ev[i].in.size();
  std::deque<int> q{root};
  std::vector<int> ev_order;
  g.order.reserve(nT);
  std::vector<int32_t> first_of, last_of;
  while (!q.empty()) {
    const int e = q.front();
    q.pop_front();
    ev_pos[e] = (int)ev_order.size();
    ev_order.push_back(e);
    first_of.push_back((int32_t)g.order.size());
    for (int t : ev[e].out) {
      task_pos[t] = (int)g.order.size();
      g.order.push_back(t);
    }
    last_of.push_back((int32_t)g.order.size() - 1);
    for (int t : ev[e].out) {
      const int te = trig_of[t][0];
      if (--remaining[te] == 0) q.push_back(te);
    }
  }
  int n_alive = 0;
  for (int i = 0; i < nE; ++i) n_alive += (ev[i].alive ? 1 : 0);
  if ((int)g.order.size() != nT || (int)ev_order.size() != n_alive)
    return fail(MPK_ERR_GRAPH_INVALID, "linearisation did not reach every task/event");

  // 5. encode in linear order; AOT round-robin over workers
  g.dep.resize(nT);
  g.trig.resize(nT);
  g.launch.resize(nT);
  g.worker.resize(nT);
  int k = 0;
  for (int p = 0; p < nT; ++p) {
    const int t = g.order[p];
    g.dep[p] = ev_pos[dep_of[t][0]];
    g.trig[p] = ev_pos[trig_of[t][0]];
    const int kind = g.tasks[t].kind;
    if (kind == MPK_TASK_EMPTY) {
      g.launch[p] = MPK_LAUNCH_INLINE;
      g.worker[p] = -1;
    } else if (kind == MPK_TASK_ATTN && !attn_aot) {
      g.launch[p] = MPK_LAUNCH_JIT;
      g.worker[p] = -1;
    } else {
      g.launch[p] = MPK_LAUNCH_AOT;
      g.worker[p] = k++ % cfg.num_workers;
    }
  }
  g.ev_count.resize(ev_order.size());
  for (size_t i = 0; i < ev_order.size(); ++i)
    g.ev_count[i] = (int32_t)ev[ev_order[i]].in.size();
  g.ev_first = std::move(first_of);
  g.ev_last = std::move(last_of);
  g.root_lin = ev_pos[root];
  g.end_lin = ev_pos[end];
  if (!validate(g, err)) return MPK_ERR_GRAPH_INVALID;
  *out = std::move(g);
  return MPK_OK;
}

bool validate(const BuiltGraph& g, std::string* err) {
  const int nT = (int)g.order.size(), nE = (int)g.ev_count.size();
  std::vector<int> n_prod(nE, 0), max_prod(nE, -1);
  for (int p = 0; p < nT; ++p) {
    if (g.dep[p] < 0 || g.dep[p] >= nE || g.trig[p] < 0 || g.trig[p] >= nE) {
      if (err) *err = "event index out of range";
      return false;
    }
    n_prod[g.trig[p]]++;
    max_prod[g.trig[p]] = std::max(max_prod[g.trig[p]], p);
    const int e = g.dep[p];
    if (p < g.ev_first[e] || p > g.ev_last[e]) {
      if (err) *err = "task outside its event's [first,last]";
      return false;
    }
  }
  int covered = 0;
  for (int e = 0; e < nE; ++e) {
    if (n_prod[e] != g.ev_count[e]) {
      if (err) *err = "event count != number of triggering tasks";
      return false;
    }
    const int n = g.ev_last[e] - g.ev_first[e] + 1;
    if (n < 0) {
      if (err) *err = "negative fan-out range";
      return false;
    }
    covered += n;
    if (n > 0 && max_prod[e] >= g.ev_first[e]) {
      if (err) *err = "producer after consumer (not topological)";
      return false;
    }
  }
  if (covered != nT) {
    if (err) *err = "fan-out ranges do not partition the tasks";
    return false;
  }
  return true;
}

}  // namespace mpk
