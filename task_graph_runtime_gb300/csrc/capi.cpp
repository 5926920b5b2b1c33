// C ABI (include/mpk.h): graph construction, device encoding, weight
// binding and step launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include "device_abi.h"
#include "graph_state.h"
#include "launch.h"
#include "layout.h"
#include "mpk.h"
#include "tgraph_builder.h"

using namespace mpk;

using namespace mpk_detail;

namespace {

mpk_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MPK_OK;
  if (e == cudaErrorMemoryAllocation) return MPK_ERR_OOM;
  if (e == cudaErrorCooperativeLaunchTooLarge) return MPK_ERR_NOT_CORESIDENT;
  return MPK_ERR_CUDA;
}

#define CK(expr)                                   \
  do {                                             \
    cudaError_t e__ = (expr);                      \
    if (e__ != cudaSuccess) return cuda_status(e__); \
  } while (0)

void fill_export(mpk_graph* g) {
  const BuiltGraph& bg = g->bg;
  const int nT = (int)bg.order.size();
  auto rs = [nT](std::vector<int32_t>& v) { v.assign(nT, 0); };
  rs(g->x_kind); rs(g->x_op); rs(g->x_layer); rs(g->x_tile); rs(g->x_row0);
  rs(g->x_row1); rs(g->x_b); rs(g->x_g); rs(g->x_c); rs(g->x_pre);
  for (int p = 0; p < nT; ++p) {
    const BTask& t = bg.tasks[bg.order[p]];
    g->x_kind[p] = t.kind;
    g->x_op[p] = t.op;
    g->x_layer[p] = t.layer;
    g->x_tile[p] = t.tile;
    g->x_row0[p] = t.row0;
    g->x_row1[p] = t.row1;
    g->x_b[p] = t.b;
    g->x_g[p] = t.g;
    g->x_c[p] = t.c;
    g->x_pre[p] = bg.order[p];
  }
  g->op_kind.clear();
  g->op_layer.clear();
  g->op_n.clear();
  for (const BOp& o : bg.ops) {
    g->op_kind.push_back(o.kind);
    g->op_layer.push_back(o.layer);
    g->op_n.push_back(o.n);
  }
}

// Fixed-size descriptors in linear order; per-worker AOT lists; per-op task
// lists for the kernel-per-operator mode.
bool encode(mpk_graph* g) {
  const BuiltGraph& bg = g->bg;
  const int nT = (int)bg.order.size(), nE = (int)bg.ev_count.size();
  const int W = bg.cfg.num_workers;
  g->h_tasks.assign(nT, TaskDesc{});
  std::vector<int> pos_of(bg.tasks.size(), -1);
  for (int p = 0; p < nT; ++p) {
    const BTask& t = bg.tasks[bg.order[p]];
    pos_of[bg.order[p]] = p;
    TaskDesc& d = g->h_tasks[p];
    d.kind = (int16_t)t.kind;
    d.launch = (uint8_t)bg.launch[p];
    d.flags = task_flags(bg, t.kind, t.tile);
    d.layer = (int16_t)t.layer;
    d.b = (int16_t)t.b;
    d.g = (int16_t)t.g;
    d.c = (int16_t)t.c;
    d.dep = bg.dep[p];
    d.trig = bg.trig[p];
    d.row0 = t.row0;
    d.row1 = t.row1;
    d.tile = t.tile;
  }
  g->h_events.assign(nE, EventDesc{});
  for (int e = 0; e < nE; ++e) {
    EventDesc& d = g->h_events[e];
    d.count = (uint32_t)bg.ev_count[e];
    d.first = bg.ev_first[e];
    d.last = bg.ev_last[e];
    d.flags = 0;
    uint32_t n_inline = 0;
    for (int p = d.first; p <= d.last; ++p) {
      if (bg.launch[p] == MPK_LAUNCH_JIT) d.flags |= EV_HAS_JIT;
      if (bg.launch[p] == MPK_LAUNCH_INLINE) {
        d.flags |= EV_HAS_INLINE;
        ++n_inline;
      }
    }
    d.flags |= n_inline << kEvInlineShift;
  }
  std::vector<std::vector<int32_t>> lists(W);
  for (int p = 0; p < nT; ++p)
    if (bg.launch[p] == MPK_LAUNCH_AOT) lists[bg.worker[p]].push_back(p);
  g->h_aot.clear();
  g->h_aot_off.assign(W + 1, 0);
  for (int w = 0; w < W; ++w) {
    g->h_aot_off[w] = (int32_t)g->h_aot.size();
    g->h_aot.insert(g->h_aot.end(), lists[w].begin(), lists[w].end());
  }
  g->h_aot_off[W] = (int32_t)g->h_aot.size();
  g->h_aot_rec.assign(g->h_aot.size(), AotRec{});
  for (size_t i = 0; i < g->h_aot.size(); ++i) {
    AotRec& r = g->h_aot_rec[i];
    r.desc = g->h_tasks[g->h_aot[i]];
    r.id = g->h_aot[i];
    r.dep_count = g->h_events[r.desc.dep].count;
    r.trig_ev = g->h_events[r.desc.trig];
    r.fan[0] = r.fan[1] = -1;
    const EventDesc& e = r.trig_ev;
    const int n_in = (int)(e.flags >> kEvInlineShift);
    bool cached = !(e.flags & EV_HAS_JIT) && (e.flags & EV_HAS_INLINE) &&
                  n_in == e.last - e.first + 1 && n_in <= 2;
    for (int k = 0; cached && k < n_in; ++k) {
      const int f = g->h_tasks[e.first + k].trig;
      if (g->h_events[f].flags != 0) cached = false;
      r.fan[k] = f;
    }
    if (cached) r.trig_ev.flags |= EV_FAN_CACHED;
    else r.fan[0] = r.fan[1] = -1;
  }
  g->h_op_tasks.clear();
  g->h_op_first.clear();
  for (const BOp& o : bg.ops) {
    g->h_op_first.push_back((int32_t)g->h_op_tasks.size());
    for (int i = 0; i < o.n; ++i) g->h_op_tasks.push_back(pos_of[o.first + i]);
  }
  // inline tasks must be the suffix of each event's range (see
  // kEvInlineShift); the builder's numbering guarantees it
  for (int e = 0; e < nE; ++e) {
    const EventDesc& d = g->h_events[e];
    const int n_in = (int)(d.flags >> kEvInlineShift);
    for (int p = d.last - n_in + 1; p <= d.last; ++p)
      if (bg.launch[p] != MPK_LAUNCH_INLINE) return false;
  }
  g->encoded = true;
  return true;
}

}  // namespace

extern "C" {

const char* mpk_status_string(mpk_status s) {
  switch (s) {
    case MPK_OK: return "ok";
    case MPK_ERR_INVALID_ARG: return "invalid argument";
    case MPK_ERR_UNSUPPORTED: return "unsupported shape";
    case MPK_ERR_CUDA: return "CUDA error";
    case MPK_ERR_OOM: return "out of memory";
    case MPK_ERR_NOT_CORESIDENT: return "persistent grid cannot be co-resident";
    case MPK_ERR_TIMEOUT: return "device wait timed out";
    case MPK_ERR_KV_PAGE: return "unmapped KV page";
    case MPK_ERR_QUEUE_OVERFLOW: return "device queue overflow";
    case MPK_ERR_GRAPH_INVALID: return "graph failed its invariants";
    case MPK_ERR_NOT_BOUND: return "weights not bound";
  }
  return "unknown status";
}

static bool has_jit_tasks(const BuiltGraph& bg) {
  for (int32_t l : bg.launch)
    if (l == MPK_LAUNCH_JIT) return true;
  return false;
}

mpk_status mpk_build_tgraph(const mpk_model_shape* shape,
                            const mpk_tile_sizes* tiles, int batch,
                            mpk_graph** out) {
  if (!shape || !out) return MPK_ERR_INVALID_ARG;
  *out = nullptr;
  mpk_tile_sizes t{};
  if (tiles) t = *tiles;
  // Scheduler SMs: as given, else (0) 4 (Table 1) when the graph has JIT
  // tasks and none when every task is AOT -- such a graph never dispatches,
  // so every SM becomes a worker.
  const bool auto_sched = t.num_sched_sms <= 0;
  int sched_sms = auto_sched ? 0 : t.num_sched_sms;
  int sched_warps = t.sched_warps_per_sm > 0 ? t.sched_warps_per_sm : 4;
  if (sched_warps > 9) return MPK_ERR_INVALID_ARG;
  int W = t.num_workers;
  if (W < 0) return MPK_ERR_INVALID_ARG;
  int sms = 0;
  if (W == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess)
      return MPK_ERR_CUDA;
    W = sms - sched_sms;
    if (W < 1) return MPK_ERR_NOT_CORESIDENT;
  }
  BuildConfig cfg;
  cfg.shape = *shape;
  cfg.batch = batch;
  cfg.num_workers = W;
  cfg.gemv_rows_per_task = t.gemv_rows_per_task;
  cfg.mma_rows_per_task = t.mma_rows_per_task;
  cfg.attn_chunks = t.attn_chunks;
  cfg.coarse_events = t.coarse_events ? 1 : 0;
  std::unique_ptr<mpk_graph> g(new (std::nothrow) mpk_graph());
  if (!g) return MPK_ERR_OOM;
  std::string err;
  mpk_status st = build_tgraph(cfg, &g->bg, &err);
  if (st != MPK_OK) return st;
  if (auto_sched && has_jit_tasks(g->bg)) {
    sched_sms = 4;
    if (sms > 0) {   // workers from the device: make room and rebuild
      cfg.num_workers = W = sms - sched_sms;
      if (W < 1) return MPK_ERR_NOT_CORESIDENT;
      g->bg = BuiltGraph{};
      st = build_tgraph(cfg, &g->bg, &err);
      if (st != MPK_OK) return st;
    }
  }
  static std::atomic<uint64_t> next_uid{1};
  g->uid = next_uid.fetch_add(1);
  g->num_sched_sms = sched_sms;
  g->sched_warps_per_sm = sched_warps;
  if (t.smem_pages < 0 || t.smem_pages > 8) return MPK_ERR_INVALID_ARG;
  g->pages_req = t.smem_pages;
  if (const char* env = std::getenv("MPK_WAIT_TIMEOUT_MS")) {
    const long ms = std::strtol(env, nullptr, 10);
    if (ms > 0) g->timeout_ns = (uint64_t)ms * 1000000ull;
  }
  fill_export(g.get());
  if (!encode(g.get())) return MPK_ERR_GRAPH_INVALID;
  *out = g.release();
  return MPK_OK;
}

mpk_status mpk_export_tgraph(const mpk_graph* g, mpk_graph_export* out) {
  if (!g || !out) return MPK_ERR_INVALID_ARG;
  const BuiltGraph& bg = g->bg;
  out->n_tasks = (int)bg.order.size();
  out->n_events = (int)bg.ev_count.size();
  out->n_ops = (int)bg.ops.size();
  out->n_empty = (int)bg.tasks.size() - bg.n_real;
  out->n_workers = bg.cfg.num_workers;
  out->attn_chunks = bg.cfg.attn_chunks;
  out->task_kind = g->x_kind.data();
  out->task_op = g->x_op.data();
  out->task_layer = g->x_layer.data();
  out->task_tile = g->x_tile.data();
  out->task_row0 = g->x_row0.data();
  out->task_row1 = g->x_row1.data();
  out->task_b = g->x_b.data();
  out->task_g = g->x_g.data();
  out->task_c = g->x_c.data();
  out->task_dep = bg.dep.data();
  out->task_trig = bg.trig.data();
  out->task_launch = bg.launch.data();
  out->task_worker = bg.worker.data();
  out->task_pre_id = g->x_pre.data();
  out->event_count = bg.ev_count.data();
  out->event_first = bg.ev_first.data();
  out->event_last = bg.ev_last.data();
  out->op_kind = g->op_kind.data();
  out->op_layer = g->op_layer.data();
  out->op_n_tasks = g->op_n.data();
  out->n_raw_events = bg.n_raw;
  out->n_fused_events = bg.n_fused;
  out->n_sched_sms = g->num_sched_sms;
  out->sched_warps_per_sm = g->sched_warps_per_sm;
  return MPK_OK;
}

mpk_status mpk_bind_weights(mpk_graph* g, const mpk_weights* w) {
  if (!g || !w || !w->embed || !w->final_norm || !w->lm_head)
    return MPK_ERR_INVALID_ARG;
  const BuildConfig& cfg = g->bg.cfg;
  const mpk_model_shape& s = cfg.shape;
  const bool chain = s.chain_ffn > 0;
  if (chain ? (!w->chain_w1 || !w->chain_w2) : !w->layers)
    return MPK_ERR_INVALID_ARG;
  auto aligned = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (!aligned(w->embed) || !aligned(w->final_norm) || !aligned(w->lm_head))
    return MPK_ERR_INVALID_ARG;
  if (chain && (!aligned(w->chain_w1) || !aligned(w->chain_w2)))
    return MPK_ERR_INVALID_ARG;
  if (!chain) {
    for (int l = 0; l < s.n_layers; ++l)
      for (int k = 0; k < MPK_LAYER_NTENSORS; ++k) {
        const bool need = s.qk_norm || (k != MPK_W_QNORM && k != MPK_W_KNORM);
        const void* p = w->layers[l * MPK_LAYER_NTENSORS + k];
        if (need && (!p || !aligned(p))) return MPK_ERR_INVALID_ARG;
      }
  }
  int dev = 0, sms = 0, optin = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  CK(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                            dev));
  const int W = cfg.num_workers;
  if (W + g->num_sched_sms > sms) return MPK_ERR_NOT_CORESIDENT;
  const int B = cfg.batch;
  SmemLayout sm{};
  if (!smem_layout(g->bg, g->pages_req, std::min(optin, kSmemLimit), &sm))
    return MPK_ERR_UNSUPPORTED;
  g->smem = sm.total;
  CK(configure_kernels(g->smem));
  if (megakernel_max_blocks_per_sm(g->smem) < 1) return MPK_ERR_NOT_CORESIDENT;
  g->device = dev;

  // graph encoding
  CK(g->d_tasks.upload(g->h_tasks));
  CK(g->d_events.upload(g->h_events));
  CK(g->d_aot.upload(g->h_aot.empty() ? std::vector<int32_t>{0} : g->h_aot));
  CK(g->d_aot_off.upload(g->h_aot_off));
  CK(g->d_aot_rec.upload(g->h_aot_rec.empty() ? std::vector<AotRec>(1)
                                              : g->h_aot_rec));
  CK(g->d_op_tasks.upload(g->h_op_tasks));
  const int nE = (int)g->h_events.size();
  const int S = g->num_sched_sms * g->sched_warps_per_sm;
  CK(g->d_counters.alloc(nE));
  CK(g->d_status.alloc(2));
  CK(g->d_merge_cnt.alloc((size_t)merge_counters(g->bg)));
  CK(g->d_jit_hdr.alloc(W));
  CK(g->d_jit_cost.alloc(1));
  CK(g->d_sched_hdr.alloc(S));
  CK(g->d_jit_slots.alloc((size_t)W * kJitCap));
  CK(g->d_sched_slots.alloc((size_t)S * kSchedCap));

  // activation workspace
  ActLayout A{};
  const int64_t act_bytes = act_layout(g->bg, &A);
  CK(g->d_act.alloc((size_t)act_bytes));
  CK(cudaMemset(g->d_act.p, 0, (size_t)act_bytes));
  A.base = g->d_act.p;

  // RoPE table
  if (!chain) {
    std::vector<float> cs((size_t)rope_table_floats(s));
    rope_table(s, cs.data());
    CK(g->d_rope.upload(cs));
  }

  // per-layer weight pointers
  const int L = s.n_layers;
  std::vector<const uint16_t*> ptrs((size_t)std::max(L, 1) * MPK_LAYER_NTENSORS,
                                    nullptr);
  for (int l = 0; l < L; ++l)
    for (int k = 0; k < MPK_LAYER_NTENSORS; ++k)
      ptrs[(size_t)l * MPK_LAYER_NTENSORS + k] = static_cast<const uint16_t*>(
          w->layers[(size_t)l * MPK_LAYER_NTENSORS + k]);
  CK(g->d_layer_ptrs.upload(ptrs));

  KernelParams& P = g->params;
  P = KernelParams{};
  P.dims = make_dims(g->bg);
  P.sm = sm;
  DevGraph& G = P.graph;
  G.tasks = g->d_tasks.p;
  G.events = g->d_events.p;
  G.n_tasks = (int)g->h_tasks.size();
  G.n_events = nE;
  G.root = g->bg.root_lin;
  G.end = g->bg.end_lin;
  G.aot_list = g->d_aot.p;
  G.aot_off = g->d_aot_off.p;
  G.aot_rec = g->d_aot_rec.p;
  G.op_tasks = g->d_op_tasks.p;
  G.counters = g->d_counters.p;
  G.merge_cnt = g->d_merge_cnt.p;
  G.jit_hdr = g->d_jit_hdr.p;
  G.jit_cost = g->d_jit_cost.p;
  G.jit_slots = g->d_jit_slots.p;
  G.sched_hdr = g->d_sched_hdr.p;
  G.sched_slots = g->d_sched_slots.p;
  G.jit_cap = kJitCap;
  G.sched_cap = kSchedCap;
  G.status = g->d_status.p;
  G.abort_flag = g->d_status.p + 1;
  G.W = W;
  G.S = S;
  G.has_jit = 0;
  for (const TaskDesc& t : g->h_tasks)
    if (t.launch == MPK_LAUNCH_JIT) G.has_jit = 1;
  G.sched_warps_per_sm = g->sched_warps_per_sm;
  P.w.embed = static_cast<const uint16_t*>(w->embed);
  P.w.final_norm = static_cast<const uint16_t*>(w->final_norm);
  P.w.lm_head = static_cast<const uint16_t*>(w->lm_head);
  P.w.chain_w1 = static_cast<const uint16_t*>(w->chain_w1);
  P.w.chain_w2 = static_cast<const uint16_t*>(w->chain_w2);
  P.w.layers = g->d_layer_ptrs.p;
  P.w.rope_cs = g->d_rope.p;
  P.act = A;
  (void)B;
  g->bound = true;
  return mpk_reset(g);
}

mpk_status mpk_reset(mpk_graph* g) {
  if (!g) return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  CK(cudaDeviceSynchronize());
  CK(cudaMemset(g->d_counters.p, 0, g->d_counters.n * sizeof(uint32_t)));
  CK(cudaMemset(g->d_status.p, 0, g->d_status.n * sizeof(uint32_t)));
  CK(cudaMemset(g->d_merge_cnt.p, 0, g->d_merge_cnt.n * sizeof(uint32_t)));
  CK(cudaMemset(g->d_jit_hdr.p, 0, g->d_jit_hdr.n * sizeof(RingHdr)));
  CK(cudaMemset(g->d_jit_cost.p, 0, sizeof(unsigned long long)));
  CK(cudaMemset(g->d_sched_hdr.p, 0, g->d_sched_hdr.n * sizeof(RingHdr)));
  CK(cudaMemset(g->d_jit_slots.p, 0, g->d_jit_slots.n * sizeof(uint64_t)));
  CK(cudaMemset(g->d_sched_slots.p, 0, g->d_sched_slots.n * sizeof(uint64_t)));
  CK(cudaDeviceSynchronize());
  g->epoch = 0;
  return MPK_OK;
}

mpk_status mpk_set_mode(mpk_graph* g, int mode) {
  if (!g || mode < MPK_MODE_MEGAKERNEL || mode > MPK_MODE_KPO_GRAPH)
    return MPK_ERR_INVALID_ARG;
  g->mode = mode;
  return MPK_OK;
}

static mpk_status enqueue_kpo(mpk_graph* g, cudaStream_t stream) {
  const KernelParams& P = g->params;
  for (size_t o = 0; o < g->bg.ops.size(); ++o) {
    CK(launch_kpo_op(P, g->h_op_first[o], g->bg.ops[o].n, g->smem, stream));
  }
  return MPK_OK;
}

mpk_status mpk_decode_step(mpk_graph* g, const int32_t* d_tokens,
                           const mpk_kv_cache* kv, float* d_logits,
                           int32_t* d_next_tokens, void* cuda_stream) {
  return mpk_decode_steps(g, d_tokens, kv, d_logits, d_next_tokens, 1,
                          cuda_stream);
}

mpk_status mpk_decode_steps(mpk_graph* g, const int32_t* d_tokens,
                            const mpk_kv_cache* kv, float* d_logits,
                            int32_t* d_next_tokens, int n_steps,
                            void* cuda_stream) {
  if (!g || !d_tokens || !d_logits || !d_next_tokens || n_steps < 1)
    return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  const mpk_model_shape& s = g->bg.cfg.shape;
  const bool chain = s.chain_ffn > 0;
  StepArgs a{};
  a.tokens = d_tokens;
  a.logits = d_logits;
  a.next_tokens = d_next_tokens;
  a.timeout_ns = g->timeout_ns;
  a.n_steps = 1;
  if (!chain) {
    if (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table ||
        !kv->seq_lens || kv->num_pages < 1 ||
        (((uintptr_t)kv->k_pool | (uintptr_t)kv->v_pool) & 15u))
      return MPK_ERR_INVALID_ARG;
    a.k_pool = static_cast<uint16_t*>(kv->k_pool);
    a.v_pool = static_cast<uint16_t*>(kv->v_pool);
    a.page_table = kv->page_table;
    a.seq_lens = kv->seq_lens;
    a.num_pages = kv->num_pages;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  CK(cudaSetDevice(g->device));
  if (g->mode == MPK_MODE_MEGAKERNEL) {
    // one launch runs all n_steps steps (the loop lives in the kernel)
    a.epoch = g->epoch + 1;
    a.n_steps = n_steps;
    g->params.step = a;
    const int grid = g->bg.cfg.num_workers + g->num_sched_sms;
    cudaError_t e = launch_megakernel(g->params, grid, g->smem, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cuda_status(e);
    }
    g->epoch += (uint32_t)n_steps;
    return MPK_OK;
  }
  if (n_steps > 1) {
    // kernel-per-operator: one step after another from the host
    const int B = g->bg.cfg.batch;
    for (int i = 0; i < n_steps; ++i) {
      mpk_status st = mpk_decode_steps(
          g, i == 0 ? d_tokens : d_next_tokens + (size_t)(i - 1) * B, kv,
          d_logits, d_next_tokens + (size_t)i * B, 1, cuda_stream);
      if (st != MPK_OK) return st;
    }
    return MPK_OK;
  }
  a.epoch = g->epoch;
  if (g->mode == MPK_MODE_KPO) {
    g->params.step = a;
    return enqueue_kpo(g, stream);
  }
  // MPK_MODE_KPO_GRAPH: capture once per distinct argument set and stream
  const bool same = g->kpo_exec && g->kpo_stream == stream &&
                    std::memcmp(&g->kpo_args, &a, sizeof(a)) == 0;
  if (!same) {
    if (g->kpo_exec) {
      cudaGraphExecDestroy(g->kpo_exec);
      g->kpo_exec = nullptr;
    }
    g->params.step = a;
    cudaStream_t cap = nullptr;
    CK(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    mpk_status st = MPK_OK;
    if (e == cudaSuccess) st = enqueue_kpo(g, cap);
    cudaError_t e2 = cudaStreamEndCapture(cap, &graph);
    cudaStreamDestroy(cap);
    if (e != cudaSuccess || e2 != cudaSuccess || st != MPK_OK) {
      if (graph) cudaGraphDestroy(graph);
      return st != MPK_OK ? st : MPK_ERR_CUDA;
    }
    e = cudaGraphInstantiate(&g->kpo_exec, graph, 0);
    cudaGraphDestroy(graph);
    CK(e);
    g->kpo_args = a;
    g->kpo_stream = stream;
  }
  CK(cudaGraphLaunch(g->kpo_exec, stream));
  return MPK_OK;
}

mpk_status mpk_get_status(mpk_graph* g) {
  if (!g) return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  CK(cudaDeviceSynchronize());
  uint32_t st = 0;
  CK(cudaMemcpy(&st, g->d_status.p, sizeof(st), cudaMemcpyDeviceToHost));
  return (mpk_status)st;
}

void mpk_destroy_tgraph(mpk_graph* g) {
  if (!g) return;
  if (g->bound) cudaDeviceSynchronize();
  delete g;
}

mpk_status mpk_debug_set_wait_timeout_ms(mpk_graph* g, int ms) {
  if (!g || ms <= 0) return MPK_ERR_INVALID_ARG;
  g->timeout_ns = (uint64_t)ms * 1000000ull;
  return MPK_OK;
}

mpk_status mpk_debug_add_event_count(mpk_graph* g, int event, int delta) {
  if (!g || event < 0 || event >= (int)g->h_events.size())
    return MPK_ERR_INVALID_ARG;
  g->h_events[event].count = (uint32_t)((int)g->h_events[event].count + delta);
  // the AOT records carry copies of their wait and trigger events' counts
  for (AotRec& r : g->h_aot_rec) {
    if (r.desc.dep == event) r.dep_count = g->h_events[event].count;
    if (r.desc.trig == event) r.trig_ev.count = g->h_events[event].count;
  }
  if (g->bound) {
    CK(cudaMemcpy(g->d_events.p + event, &g->h_events[event],
                  sizeof(EventDesc), cudaMemcpyHostToDevice));
    if (!g->h_aot_rec.empty())
      CK(cudaMemcpy(g->d_aot_rec.p, g->h_aot_rec.data(),
                    g->h_aot_rec.size() * sizeof(AotRec),
                    cudaMemcpyHostToDevice));
  }
  return MPK_OK;
}

mpk_status mpk_debug_set_trace(mpk_graph* g, int capacity) {
  if (!g || capacity < 0) return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  CK(cudaDeviceSynchronize());
  g->d_trace.reset();
  g->d_trace_count.reset();
  g->params.graph.trace = nullptr;
  g->params.graph.trace_count = nullptr;
  g->params.graph.trace_cap = 0;
  if (capacity == 0) return MPK_OK;
  CK(g->d_trace.alloc((size_t)capacity * 8));
  CK(g->d_trace_count.alloc(1));
  CK(cudaMemset(g->d_trace_count.p, 0, sizeof(uint32_t)));
  g->params.graph.trace = g->d_trace.p;
  g->params.graph.trace_count = g->d_trace_count.p;
  g->params.graph.trace_cap = (uint32_t)capacity;
  return MPK_OK;
}

mpk_status mpk_debug_read_trace(mpk_graph* g, uint64_t* host_records,
                                int capacity, int* n_records) {
  if (!g || !n_records || capacity < 0) return MPK_ERR_INVALID_ARG;
  if (!g->d_trace.p) return MPK_ERR_INVALID_ARG;
  CK(cudaDeviceSynchronize());
  uint32_t n = 0;
  CK(cudaMemcpy(&n, g->d_trace_count.p, sizeof(n), cudaMemcpyDeviceToHost));
  if (n > g->params.graph.trace_cap) n = g->params.graph.trace_cap;
  const int take = (int)n < capacity ? (int)n : capacity;
  if (take > 0 && host_records)
    CK(cudaMemcpy(host_records, g->d_trace.p, (size_t)take * 64,
                  cudaMemcpyDeviceToHost));
  CK(cudaMemset(g->d_trace_count.p, 0, sizeof(uint32_t)));
  *n_records = take;
  return MPK_OK;
}

mpk_status mpk_debug_read_hidden(mpk_graph* g, int layer, uint16_t* host_out) {
  if (!g || !host_out) return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  const mpk_model_shape& s = g->bg.cfg.shape;
  if (s.chain_ffn > 0 || layer < 0 || layer > s.n_layers)
    return MPK_ERR_INVALID_ARG;
  CK(cudaDeviceSynchronize());
  const KernelParams& P = g->params;
  const char* src = P.act.base + (int64_t)layer * P.act.layer_stride + P.act.o_h;
  CK(cudaMemcpy(host_out, src,
                (size_t)g->bg.cfg.batch * s.hidden * sizeof(uint16_t),
                cudaMemcpyDeviceToHost));
  return MPK_OK;
}

}  // extern "C"
