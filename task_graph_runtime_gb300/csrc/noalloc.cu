// mpk_decode_step_noalloc: one decode step that allocates no device memory.
//
// Some callers cannot call cudaMalloc once they are running: a serving
// process whose device memory is entirely reserved up front by its own
// caching allocator, a latency-critical loop in which the implicit device
// synchronisation of cudaMalloc/cudaFree is not allowed, or a plugin whose
// host application owns all allocations.  For them this entry point runs the
// kernel-per-operator form of the step (the same task bodies as
// mpk_decode_step) with all of its scratch -- task descriptors, per-operator
// task lists, the layer pointer table, the RoPE table, the attention merge
// counters, the activation workspace and the status words -- placed in one
// file-scope __device__ array of MPK_NOALLOC_SCRATCH_BYTES.  Every GPU that
// loads the library holds that array until the process exits.  The caller
// still passes the weights, the KV cache and the outputs.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "device_abi.h"
#include "graph_state.h"
#include "launch.h"
#include "layout.h"
#include "mpk.h"

namespace {

using namespace mpk;

// Shared by every call on a device; contents persist between calls.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[MPK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};
// What the array of each device last received from the host: the graph
// (by its build number) and the layer pointer table it was uploaded with.
uint64_t g_uploaded_uid[kMaxDevices] = {};
std::vector<const void*> g_uploaded_ptrs[kMaxDevices];

// Device address of the scratch array on the current device.  Host code
// cannot use the array's name as a device address: it is a host-side
// stand-in.  Looked up once per device, with that device current.
cudaError_t scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return cudaSuccess;
}

// RoPE table (cos, sin of p * theta^(-2i/d), evaluated in double) written
// straight into the scratch array.
__global__ void rope_table_kernel(float* cs, int max_ctx, int half,
                                  double theta, int d) {
  const int64_t n = (int64_t)max_ctx * half;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(k / half), i = (int)(k % half);
    const double ang = (double)p * pow(theta, -2.0 * i / d);
    cs[2 * k] = (float)cos(ang);
    cs[2 * k + 1] = (float)sin(ang);
  }
}

__global__ void copy_status_kernel(const uint32_t* src, uint32_t* dst) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *dst = *src;
}

int64_t up256(int64_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" mpk_status mpk_decode_step_noalloc(
    const mpk_graph* g, const mpk_weights* w, const int32_t* d_tokens,
    const mpk_kv_cache* kv, float* d_logits, int32_t* d_next_tokens,
    uint32_t* d_status, void* cuda_stream) {
  if (!g || !w || !d_tokens || !d_logits || !d_next_tokens)
    return MPK_ERR_INVALID_ARG;
  const BuiltGraph& bg = g->bg;
  const mpk_model_shape& s = bg.cfg.shape;
  const bool chain = s.chain_ffn > 0;
  const int L = s.n_layers, d = s.head_dim;
  const int n_ptrs = (L > 0 ? L : 1) * MPK_LAYER_NTENSORS;

  // --- layout of the scratch array (bytes)
  ActLayout A{};
  const int64_t act_bytes = act_layout(bg, &A);
  const int64_t n_merge = merge_counters(bg);
  const int max_ctx = chain ? 1 : s.max_pages_per_seq * s.page_size;
  int64_t pos = 0;
  const int64_t o_status = pos;       pos += 256;
  const int64_t o_merge = pos;        pos += up256(n_merge * 4);
  const int64_t o_tasks = pos;        pos += up256((int64_t)g->h_tasks.size() * sizeof(TaskDesc));
  const int64_t o_optasks = pos;      pos += up256((int64_t)g->h_op_tasks.size() * 4);
  const int64_t o_ptrs = pos;         pos += up256((int64_t)n_ptrs * 8);
  const int64_t o_rope = pos;         pos += up256((int64_t)max_ctx * (d / 2) * 8);
  const int64_t o_act = pos;          pos += act_bytes;
  if (pos > (int64_t)MPK_NOALLOC_SCRATCH_BYTES) return MPK_ERR_UNSUPPORTED;

  if (chain ? (!w->embed || !w->final_norm || !w->lm_head || !w->chain_w1 ||
               !w->chain_w2)
            : (!w->embed || !w->final_norm || !w->lm_head || !w->layers))
    return MPK_ERR_INVALID_ARG;
  if (!chain && (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table ||
                 !kv->seq_lens || kv->num_pages < 1 ||
                 (((uintptr_t)kv->k_pool | (uintptr_t)kv->v_pool) & 15u)))
    return MPK_ERR_INVALID_ARG;

  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MPK_ERR_CUDA;
  unsigned char* base = nullptr;
  if (scratch_address(dev, &base) != cudaSuccess) return MPK_ERR_CUDA;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                             dev) != cudaSuccess)
    return MPK_ERR_CUDA;
  SmemLayout sm{};
  if (!smem_layout(bg, g->pages_req,
                   optin < mpk_detail::kSmemLimit ? optin
                                                  : mpk_detail::kSmemLimit,
                   &sm))
    return MPK_ERR_UNSUPPORTED;
  if (configure_kernels(sm.total) != cudaSuccess) return MPK_ERR_CUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  // --- fill the scratch array.  The status words and the merge counters
  // must start at zero on every call.
  if (cudaMemsetAsync(base + o_status, 0, 256, stream) != cudaSuccess ||
      cudaMemsetAsync(base + o_merge, 0, (size_t)n_merge * 4, stream) !=
          cudaSuccess)
    return MPK_ERR_CUDA;
  // The graph encoding, the layer pointers and the RoPE table are uploaded
  // again only when another graph or another set of layer pointers was the
  // last one uploaded to this device's array.
  std::vector<const void*> ptrs((size_t)n_ptrs, nullptr);
  if (!chain)
    std::memcpy(ptrs.data(), w->layers, (size_t)n_ptrs * sizeof(void*));
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    const bool fresh = g_uploaded_uid[dev] != g->uid ||
                       g_uploaded_ptrs[dev] != ptrs;
    if (fresh) {
      g_uploaded_uid[dev] = 0;   // until the uploads below are enqueued
      if (cudaMemcpyAsync(base + o_tasks, g->h_tasks.data(),
                          g->h_tasks.size() * sizeof(TaskDesc),
                          cudaMemcpyHostToDevice, stream) != cudaSuccess ||
          cudaMemcpyAsync(base + o_optasks, g->h_op_tasks.data(),
                          g->h_op_tasks.size() * 4, cudaMemcpyHostToDevice,
                          stream) != cudaSuccess)
        return MPK_ERR_CUDA;
      if (!chain) {
        if (cudaMemcpyAsync(base + o_ptrs, w->layers,
                            (size_t)n_ptrs * sizeof(void*),
                            cudaMemcpyHostToDevice, stream) != cudaSuccess)
          return MPK_ERR_CUDA;
        rope_table_kernel<<<64, 256, 0, stream>>>(
            reinterpret_cast<float*>(base + o_rope), max_ctx, d / 2,
            (double)s.rope_theta, d);
        if (cudaGetLastError() != cudaSuccess) return MPK_ERR_CUDA;
      }
      g_uploaded_uid[dev] = g->uid;
      g_uploaded_ptrs[dev] = ptrs;
    }
  }

  // --- launch parameters pointing into the scratch array
  KernelParams P{};
  P.dims = make_dims(bg);
  P.sm = sm;
  DevGraph& G = P.graph;
  G.tasks = reinterpret_cast<const TaskDesc*>(base + o_tasks);
  G.n_tasks = (int)g->h_tasks.size();
  G.op_tasks = reinterpret_cast<const int32_t*>(base + o_optasks);
  G.merge_cnt = reinterpret_cast<uint32_t*>(base + o_merge);
  G.status = reinterpret_cast<uint32_t*>(base + o_status);
  G.abort_flag = G.status + 1;
  G.W = bg.cfg.num_workers;
  P.w.embed = static_cast<const uint16_t*>(w->embed);
  P.w.final_norm = static_cast<const uint16_t*>(w->final_norm);
  P.w.lm_head = static_cast<const uint16_t*>(w->lm_head);
  P.w.chain_w1 = static_cast<const uint16_t*>(w->chain_w1);
  P.w.chain_w2 = static_cast<const uint16_t*>(w->chain_w2);
  P.w.layers = reinterpret_cast<const uint16_t* const*>(base + o_ptrs);
  P.w.rope_cs = reinterpret_cast<const float*>(base + o_rope);
  A.base = reinterpret_cast<char*>(base + o_act);
  P.act = A;
  StepArgs& a = P.step;
  a.tokens = d_tokens;
  a.logits = d_logits;
  a.next_tokens = d_next_tokens;
  a.timeout_ns = g->timeout_ns;
  a.n_steps = 1;
  if (!chain) {
    a.k_pool = static_cast<uint16_t*>(kv->k_pool);
    a.v_pool = static_cast<uint16_t*>(kv->v_pool);
    a.page_table = kv->page_table;
    a.seq_lens = kv->seq_lens;
    a.num_pages = kv->num_pages;
  }
  for (size_t o = 0; o < bg.ops.size(); ++o) {
    if (launch_kpo_op(P, g->h_op_first[o], bg.ops[o].n, sm.total, stream) !=
        cudaSuccess)
      return MPK_ERR_CUDA;
  }
  if (d_status) {
    copy_status_kernel<<<1, 32, 0, stream>>>(G.status, d_status);
    if (cudaGetLastError() != cudaSuccess) return MPK_ERR_CUDA;
  }
  return MPK_OK;
}
