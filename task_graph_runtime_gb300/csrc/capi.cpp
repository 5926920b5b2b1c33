// C ABI (include/mpk.h): graph construction, device encoding, weight
// binding and step launches.
#include <cuda.h>
#include <cuda_runtime.h>

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
void encode(mpk_graph* g) {
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
    d.flags = 0;
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
    for (int p = d.first; p <= d.last; ++p) {
      if (bg.launch[p] == MPK_LAUNCH_JIT) d.flags |= EV_HAS_JIT;
      if (bg.launch[p] == MPK_LAUNCH_INLINE) d.flags |= EV_HAS_INLINE;
    }
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
  g->h_op_tasks.clear();
  g->h_op_first.clear();
  for (const BOp& o : bg.ops) {
    g->h_op_first.push_back((int32_t)g->h_op_tasks.size());
    for (int i = 0; i < o.n; ++i) g->h_op_tasks.push_back(pos_of[o.first + i]);
  }
  g->encoded = true;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                       cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  fn = reinterpret_cast<EncodeTiledFn>(p);
  return fn;
}

// bf16 matrix [rows][cols], boxes of 64 columns x 8 rows, 128-byte swizzle.
mpk_status make_tmap(uint8_t* dst, const void* base, int rows, int cols) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return MPK_ERR_CUDA;
  if (((uintptr_t)base) & 15u) return MPK_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 8};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MPK_ERR_INVALID_ARG;
  std::memcpy(dst, &m, 128);
  return MPK_OK;
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

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

mpk_status mpk_build_tgraph(const mpk_model_shape* shape,
                            const mpk_tile_sizes* tiles, int batch,
                            mpk_graph** out) {
  if (!shape || !out) return MPK_ERR_INVALID_ARG;
  *out = nullptr;
  mpk_tile_sizes t{};
  if (tiles) t = *tiles;
  int sched_sms = t.num_sched_sms > 0 ? t.num_sched_sms : 4;
  int sched_warps = t.sched_warps_per_sm > 0 ? t.sched_warps_per_sm : 4;
  if (sched_warps > 9) return MPK_ERR_INVALID_ARG;
  int W = t.num_workers;
  if (W < 0) return MPK_ERR_INVALID_ARG;
  if (W == 0) {
    int dev = 0, sms = 0;
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
  cfg.attn_chunks = t.attn_chunks;
  const mpk_model_shape& s = *shape;
  if (s.hidden > 8192) return MPK_ERR_UNSUPPORTED;
  if (s.chain_ffn == 0 && s.n_kv_heads > 0 && s.n_q_heads % s.n_kv_heads == 0) {
    const int grp = s.n_q_heads / s.n_kv_heads;
    if (s.head_dim % 32 || grp * (s.head_dim + 2) > 1024)
      return MPK_ERR_UNSUPPORTED;
  }
  std::unique_ptr<mpk_graph> g(new (std::nothrow) mpk_graph());
  if (!g) return MPK_ERR_OOM;
  std::string err;
  mpk_status st = build_tgraph(cfg, &g->bg, &err);
  if (st != MPK_OK) return st;
  g->num_sched_sms = sched_sms;
  g->sched_warps_per_sm = sched_warps;
  g->pages_req = t.smem_pages > 0 ? t.smem_pages : kDefaultPages;
  if (const char* env = std::getenv("MPK_WAIT_TIMEOUT_MS")) {
    const long ms = std::strtol(env, nullptr, 10);
    if (ms > 0) g->timeout_ns = (uint64_t)ms * 1000000ull;
  }
  fill_export(g.get());
  encode(g.get());
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
  if (!chain) {
    for (int l = 0; l < s.n_layers; ++l)
      for (int k = 0; k < MPK_LAYER_NTENSORS; ++k) {
        const bool need = s.qk_norm || (k != MPK_W_QNORM && k != MPK_W_KNORM);
        if (need && !w->layers[l * MPK_LAYER_NTENSORS + k])
          return MPK_ERR_INVALID_ARG;
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
  int pages = g->pages_req;
  const int limit = std::min(optin, kSmemLimit);
  while (pages > 2 && smem_bytes(pages, B) > limit) --pages;
  if (smem_bytes(pages, B) > limit || pages > 16) return MPK_ERR_UNSUPPORTED;
  g->n_pages = pages;
  g->smem = smem_bytes(pages, B);
  CK(configure_kernels(g->smem));
  g->device = dev;

  // graph encoding
  CK(g->d_tasks.upload(g->h_tasks));
  CK(g->d_events.upload(g->h_events));
  CK(g->d_aot.upload(g->h_aot.empty() ? std::vector<int32_t>{0} : g->h_aot));
  CK(g->d_aot_off.upload(g->h_aot_off));
  CK(g->d_op_tasks.upload(g->h_op_tasks));
  const int nE = (int)g->h_events.size();
  const int S = g->num_sched_sms * g->sched_warps_per_sm;
  CK(g->d_counters.alloc(nE));
  CK(g->d_status.alloc(2));
  CK(g->d_jit_hdr.alloc(W));
  CK(g->d_sched_hdr.alloc(S));
  CK(g->d_jit_slots.alloc((size_t)W * kJitCap));
  CK(g->d_sched_slots.alloc((size_t)S * kSchedCap));

  // activation workspace
  const int h = s.hidden, d = s.head_dim, Hq = s.n_q_heads, Hkv = s.n_kv_heads;
  const int grp = chain ? 1 : Hq / Hkv;
  const int C = chain ? 0 : cfg.attn_chunks;
  const int Nqkv = chain ? 0 : (Hq + 2 * Hkv) * d;
  const int Fa = std::max(s.ffn, s.chain_ffn);
  ActLayout A{};
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off += align_up(bytes, 256);
    return o;
  };
  A.o_h = take((int64_t)B * h * 2);
  A.o_n1 = take((int64_t)B * h * 2);
  A.o_qkv = take((int64_t)B * Nqkv * 2);
  A.o_q = take((int64_t)B * Hq * d * 2);
  A.o_opart = take((int64_t)B * Hkv * C * grp * (d + 2) * 4);
  A.o_attn = take((int64_t)B * Hq * d * 2);
  A.o_o = take((int64_t)B * h * 2);
  A.o_hmid = take((int64_t)B * h * 2);
  A.o_n2 = take((int64_t)B * h * 2);
  A.o_act = take((int64_t)B * Fa * 2);
  A.o_dout = take((int64_t)B * h * 2);
  A.layer_stride = off;
  const int nblocks = std::max(s.n_layers, 1) + 1;
  const int n_lm = g->op_n.empty() ? 0 : g->op_n[g->op_n.size() - 2];
  int64_t goff = 0;
  A.global_block = A.layer_stride * nblocks;
  A.g_nf = goff;
  goff += align_up((int64_t)B * h * 2, 256);
  A.g_z = goff;
  goff += align_up((int64_t)B * h * 2, 256);
  A.g_amax = goff;
  goff += align_up((int64_t)B * n_lm * 8, 256);
  CK(g->d_act.alloc((size_t)(A.global_block + goff)));
  CK(cudaMemset(g->d_act.p, 0, (size_t)(A.global_block + goff)));
  A.base = g->d_act.p;

  // RoPE table: cos/sin(pos * theta^(-2i/d)) evaluated in double
  const int max_ctx = chain ? 1 : s.max_pages_per_seq * s.page_size;
  if (!chain) {
    std::vector<float> cs((size_t)max_ctx * (d / 2) * 2);
    for (int p = 0; p < max_ctx; ++p)
      for (int i = 0; i < d / 2; ++i) {
        const double inv = std::pow((double)s.rope_theta, -2.0 * i / d);
        const double ang = (double)p * inv;
        cs[((size_t)p * (d / 2) + i) * 2] = (float)std::cos(ang);
        cs[((size_t)p * (d / 2) + i) * 2 + 1] = (float)std::sin(ang);
      }
    CK(g->d_rope.upload(cs));
  }

  // weights: pointer table and tensor maps
  const int L = s.n_layers;
  const int n_maps = 4 * L + 3;
  std::vector<uint8_t> maps((size_t)n_maps * 128, 0);
  std::vector<const uint16_t*> ptrs((size_t)std::max(L, 1) * MPK_LAYER_NTENSORS,
                                    nullptr);
  mpk_status st;
  for (int l = 0; l < L; ++l) {
    const void* const* lw = w->layers + (size_t)l * MPK_LAYER_NTENSORS;
    for (int k = 0; k < MPK_LAYER_NTENSORS; ++k)
      ptrs[(size_t)l * MPK_LAYER_NTENSORS + k] =
          static_cast<const uint16_t*>(lw[k]);
    if ((st = make_tmap(&maps[(4 * l + TM_QKV) * 128], lw[MPK_W_QKV], Nqkv, h)) != MPK_OK) return st;
    if ((st = make_tmap(&maps[(4 * l + TM_O) * 128], lw[MPK_W_O], h, Hq * d)) != MPK_OK) return st;
    if ((st = make_tmap(&maps[(4 * l + TM_GU) * 128], lw[MPK_W_GATEUP], 2 * s.ffn, h)) != MPK_OK) return st;
    if ((st = make_tmap(&maps[(4 * l + TM_DOWN) * 128], lw[MPK_W_DOWN], h, s.ffn)) != MPK_OK) return st;
  }
  if ((st = make_tmap(&maps[(4 * L) * 128], w->lm_head, s.vocab, h)) != MPK_OK) return st;
  if (chain) {
    if ((st = make_tmap(&maps[(4 * L + 1) * 128], w->chain_w1, s.chain_ffn, h)) != MPK_OK) return st;
    if ((st = make_tmap(&maps[(4 * L + 2) * 128], w->chain_w2, h, s.chain_ffn)) != MPK_OK) return st;
  }
  CK(g->d_tmaps.upload(maps));
  CK(g->d_layer_ptrs.upload(ptrs));

  KernelParams& P = g->params;
  P = KernelParams{};
  P.dims.L = L;
  P.dims.h = h;
  P.dims.Hq = Hq;
  P.dims.Hkv = Hkv;
  P.dims.d = d;
  P.dims.F = s.ffn;
  P.dims.V = s.vocab;
  P.dims.chain_ffn = s.chain_ffn;
  P.dims.qk_norm = s.qk_norm;
  P.dims.eps = s.rms_eps;
  P.dims.B = B;
  P.dims.C = C;
  P.dims.page_size = s.page_size;
  P.dims.max_pages = s.max_pages_per_seq;
  P.dims.n_lm_tiles = n_lm;
  P.dims.max_ctx = max_ctx;
  DevGraph& G = P.graph;
  G.tasks = g->d_tasks.p;
  G.events = g->d_events.p;
  G.n_tasks = (int)g->h_tasks.size();
  G.n_events = nE;
  G.root = g->bg.root_lin;
  G.end = g->bg.end_lin;
  G.aot_list = g->d_aot.p;
  G.aot_off = g->d_aot_off.p;
  G.op_tasks = g->d_op_tasks.p;
  G.counters = g->d_counters.p;
  G.jit_hdr = g->d_jit_hdr.p;
  G.jit_slots = g->d_jit_slots.p;
  G.sched_hdr = g->d_sched_hdr.p;
  G.sched_slots = g->d_sched_slots.p;
  G.jit_cap = kJitCap;
  G.sched_cap = kSchedCap;
  G.status = g->d_status.p;
  G.abort_flag = g->d_status.p + 1;
  G.W = W;
  G.S = S;
  G.sched_warps_per_sm = g->sched_warps_per_sm;
  G.n_pages = pages;
  P.w.embed = static_cast<const uint16_t*>(w->embed);
  P.w.final_norm = static_cast<const uint16_t*>(w->final_norm);
  P.w.lm_head = static_cast<const uint16_t*>(w->lm_head);
  P.w.layers = g->d_layer_ptrs.p;
  P.w.tmaps = g->d_tmaps.p;
  P.w.rope_cs = g->d_rope.p;
  P.act = A;
  g->bound = true;
  return mpk_reset(g);
}

mpk_status mpk_reset(mpk_graph* g) {
  if (!g) return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  CK(cudaDeviceSynchronize());
  CK(cudaMemset(g->d_counters.p, 0, g->d_counters.n * sizeof(uint32_t)));
  CK(cudaMemset(g->d_status.p, 0, g->d_status.n * sizeof(uint32_t)));
  CK(cudaMemset(g->d_jit_hdr.p, 0, g->d_jit_hdr.n * sizeof(RingHdr)));
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
  if (!g || !d_tokens || !d_logits || !d_next_tokens)
    return MPK_ERR_INVALID_ARG;
  if (!g->bound) return MPK_ERR_NOT_BOUND;
  const mpk_model_shape& s = g->bg.cfg.shape;
  const bool chain = s.chain_ffn > 0;
  StepArgs a{};
  a.tokens = d_tokens;
  a.logits = d_logits;
  a.next_tokens = d_next_tokens;
  a.timeout_ns = g->timeout_ns;
  if (!chain) {
    if (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table ||
        !kv->seq_lens || kv->num_pages < 1)
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
    a.epoch = g->epoch + 1;
    g->params.step = a;
    const int grid = g->bg.cfg.num_workers + g->num_sched_sms;
    cudaError_t e = launch_megakernel(g->params, grid, g->smem, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cuda_status(e);
    }
    g->epoch += 1;
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
  if (g->bound) {
    CK(cudaMemcpy(g->d_events.p + event, &g->h_events[event],
                  sizeof(EventDesc), cudaMemcpyHostToDevice));
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
  CK(g->d_trace.alloc((size_t)capacity * 4));
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
    CK(cudaMemcpy(host_records, g->d_trace.p, (size_t)take * 32,
                  cudaMemcpyDeviceToHost));
  CK(cudaMemset(g->d_trace_count.p, 0, sizeof(uint32_t)));
  *n_records = take;
  return MPK_OK;
}

}  // extern "C"
