// mpk_decode_step_noalloc: one decode step that allocates no device memory.
//
// Some callers cannot call cudaMalloc once they are running: a serving
// process whose device memory is entirely reserved up front by its own
// caching allocator, a latency-critical loop in which the implicit device
// synchronisation of cudaMalloc/cudaFree is not allowed, or a plugin whose
// host application owns all allocations.  For them this entry point runs the
// kernel-per-operator form of the step (the same task bodies as
// mpk_decode_step) with all of its scratch -- task descriptors, per-operator
// task lists, TMA descriptors, the layer pointer table, the RoPE table, the
// activation workspace and the status words -- placed in one file-scope
// __device__ array of MPK_NOALLOC_SCRATCH_BYTES.  Every GPU that loads the
// library holds that array until the process exits.  The caller still
// passes the weights, the KV cache and the outputs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "device_abi.h"
#include "graph_state.h"
#include "launch.h"
#include "mpk.h"

namespace {

using namespace mpk;

// Shared by every call on a device; contents persist between calls.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[MPK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

// Encode the TMA descriptor of a bf16 [rows][cols] matrix (64 x 8 boxes,
// 128-byte swizzle) and copy it into the scratch array.
mpk_status put_tmap(unsigned char* dst, const void* base, int rows, int cols,
                    cudaStream_t stream) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return MPK_ERR_CUDA;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  if (!base || (((uintptr_t)base) & 15u)) return MPK_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 8};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MPK_ERR_INVALID_ARG;
  // pageable source: the copy is staged before the call returns, so the
  // stack copy may go out of scope
  if (cudaMemcpyAsync(dst, &m, sizeof(m), cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return MPK_ERR_CUDA;
  return MPK_OK;
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
  const int B = bg.cfg.batch, L = s.n_layers, h = s.hidden, d = s.head_dim;
  const int Hq = s.n_q_heads, Hkv = s.n_kv_heads;
  const int grp = chain ? 1 : Hq / Hkv;
  const int C = chain ? 0 : bg.cfg.attn_chunks;
  const int Nqkv = chain ? 0 : (Hq + 2 * Hkv) * d;
  const int Fa = s.ffn > s.chain_ffn ? s.ffn : s.chain_ffn;
  const int n_lm = g->op_n.empty() ? 0 : g->op_n[g->op_n.size() - 2];
  const int max_ctx = chain ? 1 : s.max_pages_per_seq * s.page_size;
  const int n_maps = 4 * L + 3;
  const int n_ptrs = (L > 0 ? L : 1) * MPK_LAYER_NTENSORS;

  // --- layout of the scratch array (bytes)
  ActLayout A{};
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off += up256(bytes);
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
  const int nblocks = (L > 0 ? L : 1) + 1;
  A.global_block = A.layer_stride * nblocks;
  A.g_nf = 0;
  A.g_z = up256((int64_t)B * h * 2);
  A.g_amax = A.g_z + up256((int64_t)B * h * 2);
  const int64_t act_bytes = A.global_block + A.g_amax + up256((int64_t)B * n_lm * 8);
  int64_t pos = 0;
  const int64_t o_status = pos;       pos += 256;
  const int64_t o_tasks = pos;        pos += up256((int64_t)g->h_tasks.size() * sizeof(TaskDesc));
  const int64_t o_optasks = pos;      pos += up256((int64_t)g->h_op_tasks.size() * 4);
  const int64_t o_tmaps = pos;        pos += up256((int64_t)n_maps * 128);
  const int64_t o_ptrs = pos;         pos += up256((int64_t)n_ptrs * 8);
  const int64_t o_rope = pos;         pos += up256((int64_t)max_ctx * (d / 2) * 8);
  const int64_t o_act = pos;          pos += act_bytes;
  if (pos > (int64_t)MPK_NOALLOC_SCRATCH_BYTES) return MPK_ERR_UNSUPPORTED;

  if (chain ? (!w->embed || !w->final_norm || !w->lm_head || !w->chain_w1 ||
               !w->chain_w2)
            : (!w->embed || !w->final_norm || !w->lm_head || !w->layers))
    return MPK_ERR_INVALID_ARG;
  if (!chain && (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table ||
                 !kv->seq_lens || kv->num_pages < 1))
    return MPK_ERR_INVALID_ARG;

  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MPK_ERR_CUDA;
  unsigned char* base = nullptr;
  if (scratch_address(dev, &base) != cudaSuccess) return MPK_ERR_CUDA;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                             dev) != cudaSuccess)
    return MPK_ERR_CUDA;
  int pages = g->pages_req;
  const int limit = optin < mpk_detail::kSmemLimit ? optin : mpk_detail::kSmemLimit;
  while (pages > 2 && smem_bytes(pages, B) > limit) --pages;
  if (smem_bytes(pages, B) > limit || pages > 16) return MPK_ERR_UNSUPPORTED;
  const int smem = smem_bytes(pages, B);
  if (configure_kernels(smem) != cudaSuccess) return MPK_ERR_CUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  // --- fill the scratch array (status words must start at zero)
  if (cudaMemsetAsync(base + o_status, 0, 256, stream) != cudaSuccess)
    return MPK_ERR_CUDA;
  if (cudaMemcpyAsync(base + o_tasks, g->h_tasks.data(),
                      g->h_tasks.size() * sizeof(TaskDesc),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(base + o_optasks, g->h_op_tasks.data(),
                      g->h_op_tasks.size() * 4, cudaMemcpyHostToDevice,
                      stream) != cudaSuccess)
    return MPK_ERR_CUDA;
  mpk_status st;
  for (int l = 0; l < L; ++l) {
    const void* const* lw = w->layers + (size_t)l * MPK_LAYER_NTENSORS;
    unsigned char* m = base + o_tmaps + (int64_t)4 * l * 128;
    if ((st = put_tmap(m + TM_QKV * 128, lw[MPK_W_QKV], Nqkv, h, stream)) != MPK_OK) return st;
    if ((st = put_tmap(m + TM_O * 128, lw[MPK_W_O], h, Hq * d, stream)) != MPK_OK) return st;
    if ((st = put_tmap(m + TM_GU * 128, lw[MPK_W_GATEUP], 2 * s.ffn, h, stream)) != MPK_OK) return st;
    if ((st = put_tmap(m + TM_DOWN * 128, lw[MPK_W_DOWN], h, s.ffn, stream)) != MPK_OK) return st;
  }
  unsigned char* mt = base + o_tmaps + (int64_t)4 * L * 128;
  if ((st = put_tmap(mt, w->lm_head, s.vocab, h, stream)) != MPK_OK) return st;
  if (chain) {
    if ((st = put_tmap(mt + 128, w->chain_w1, s.chain_ffn, h, stream)) != MPK_OK) return st;
    if ((st = put_tmap(mt + 256, w->chain_w2, h, s.chain_ffn, stream)) != MPK_OK) return st;
  } else {
    if (cudaMemcpyAsync(base + o_ptrs, w->layers,
                        (size_t)L * MPK_LAYER_NTENSORS * sizeof(void*),
                        cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return MPK_ERR_CUDA;
    rope_table_kernel<<<64, 256, 0, stream>>>(
        reinterpret_cast<float*>(base + o_rope), max_ctx, d / 2,
        (double)s.rope_theta, d);
    if (cudaGetLastError() != cudaSuccess) return MPK_ERR_CUDA;
  }

  // --- launch parameters pointing into the scratch array
  KernelParams P{};
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
  G.tasks = reinterpret_cast<const TaskDesc*>(base + o_tasks);
  G.n_tasks = (int)g->h_tasks.size();
  G.op_tasks = reinterpret_cast<const int32_t*>(base + o_optasks);
  G.status = reinterpret_cast<uint32_t*>(base + o_status);
  G.abort_flag = G.status + 1;
  G.W = bg.cfg.num_workers;
  G.n_pages = pages;
  P.w.embed = static_cast<const uint16_t*>(w->embed);
  P.w.final_norm = static_cast<const uint16_t*>(w->final_norm);
  P.w.lm_head = static_cast<const uint16_t*>(w->lm_head);
  P.w.layers = reinterpret_cast<const uint16_t* const*>(base + o_ptrs);
  P.w.tmaps = base + o_tmaps;
  P.w.rope_cs = reinterpret_cast<const float*>(base + o_rope);
  A.base = reinterpret_cast<char*>(base + o_act);
  P.act = A;
  StepArgs& a = P.step;
  a.tokens = d_tokens;
  a.logits = d_logits;
  a.next_tokens = d_next_tokens;
  a.timeout_ns = g->timeout_ns;
  if (!chain) {
    a.k_pool = static_cast<uint16_t*>(kv->k_pool);
    a.v_pool = static_cast<uint16_t*>(kv->v_pool);
    a.page_table = kv->page_table;
    a.seq_lens = kv->seq_lens;
    a.num_pages = kv->num_pages;
  }
  for (size_t o = 0; o < bg.ops.size(); ++o) {
    if (launch_kpo_op(P, g->h_op_first[o], bg.ops[o].n, smem, stream) !=
        cudaSuccess)
      return MPK_ERR_CUDA;
  }
  if (d_status) {
    copy_status_kernel<<<1, 32, 0, stream>>>(G.status, d_status);
    if (cudaGetLastError() != cudaSuccess) return MPK_ERR_CUDA;
  }
  return MPK_OK;
}
