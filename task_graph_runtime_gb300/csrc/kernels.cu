// sm_103a task bodies and the persistent mega-kernel runtime.
//
// MPK: A Compiler and Runtime for Mega-Kernelizing Tensor Programs:
//   §2 Q2 -- workers run FIFO task queues, scheduler warps run event queues;
//   §2 Q2 / "Design space" -- hybrid launch: AOT tasks wait on their event
//     counter directly (one sync), JIT tasks are pushed by a scheduler warp
//     once their event fires (two syncs);
//   "Why this launch config (Table 1)" -- scheduler SMs x warps, 32 KB
//     shared-memory pages;
//   Figure 2 / "Optimization techniques inventory" -- cross-task software
//     pipelining: weight pages of the NEXT tasks stream in (TMA) while the
//     current task computes, and before the next task's event has fired,
//     because weights never depend on an event.
//
// GB300 layout of a worker CTA (one per SM, 288 threads):
//   warp 8      -- producer: walks this worker's AOT task list and issues
//                  2-D TMA loads (cp.async.bulk.tensor, 128-byte swizzle) of
//                  weight tiles into a ring of 32 KB pages;
//   warps 0..7  -- consumers: poll events and the JIT queue, run task bodies,
//                  release pages, trigger events.
// Every spin-wait is bounded by %globaltimer; on timeout the kernel latches
// MPK_ERR_TIMEOUT, raises an abort flag, drains its own copies in flight and
// returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_abi.h"
#include "mpk.h"

namespace mpk {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kPageBytes = 32768;
constexpr int kXsBytes = 32768;
constexpr int kPageCols = 256;   // 4 TMA boxes of 64 bf16 columns
constexpr int kMaxPageRows = 64;
constexpr int kBoxRows = 8;      // one TMA box = 8 rows x 128 bytes = 1 KB
constexpr int kCtrlBytes = 64;
constexpr int kScratchBytes = 1024;

__host__ __device__ inline int smem_bytes_for(int n_pages, int batch) {
  return n_pages * kPageBytes + kXsBytes + 4 * kMaxPageRows * batch * 4 +
         16 * n_pages + kCtrlBytes + kScratchBytes;
}

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap,
                                            uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];"
               : "=r"(v)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
               : "=r"(v)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_acquire64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];"
               : "=l"(v)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}
__device__ __forceinline__ void st_release64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v)
               : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// ------------------------------------------------------------ bf16 helpers
__device__ __forceinline__ float bf_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf_hi(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ float bf2f(uint16_t u) {
  return __uint_as_float(((uint32_t)u) << 16);
}
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float round_bf(float f) { return bf2f(f2bf(f)); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}
__device__ __forceinline__ float dot8(uint4 w, uint4 x, float acc) {
  acc = fmaf(bf_lo(w.x), bf_lo(x.x), acc);
  acc = fmaf(bf_hi(w.x), bf_hi(x.x), acc);
  acc = fmaf(bf_lo(w.y), bf_lo(x.y), acc);
  acc = fmaf(bf_hi(w.y), bf_hi(x.y), acc);
  acc = fmaf(bf_lo(w.z), bf_lo(x.z), acc);
  acc = fmaf(bf_hi(w.z), bf_hi(x.z), acc);
  acc = fmaf(bf_lo(w.w), bf_lo(x.w), acc);
  acc = fmaf(bf_hi(w.w), bf_hi(x.w), acc);
  return acc;
}
__device__ __forceinline__ float silu_f(float z) {
  return z / (1.0f + expf(-z));
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------ error latch
__device__ __forceinline__ void raise_error(const KernelParams& P,
                                            uint32_t code) {
  atomicCAS(P.graph.status, 0u, code);
  atomicExch(P.graph.abort_flag, 1u);
}
__device__ __forceinline__ bool aborted(const KernelParams& P) {
  return ld_relaxed(P.graph.abort_flag) != 0u;
}

// ------------------------------------------------------------ shared memory
struct Smem {
  uint8_t* pages;
  uint16_t* xs;
  float* red;
  uint64_t* full;
  uint64_t* empty;
  volatile int* ctrl;
  float* scratch;
};

__device__ __forceinline__ Smem carve(uint8_t* base, int n_pages, int B) {
  Smem s;
  size_t off = 0;
  s.pages = base;
  off += (size_t)n_pages * kPageBytes;
  s.xs = reinterpret_cast<uint16_t*>(base + off);
  off += kXsBytes;
  s.red = reinterpret_cast<float*>(base + off);
  off += (size_t)4 * kMaxPageRows * B * 4;
  s.full = reinterpret_cast<uint64_t*>(base + off);
  off += 8 * n_pages;
  s.empty = reinterpret_cast<uint64_t*>(base + off);
  off += 8 * n_pages;
  s.ctrl = reinterpret_cast<volatile int*>(base + off);
  off += kCtrlBytes;
  s.scratch = reinterpret_cast<float*>(base + off);
  return s;
}

// Position in the ring of weight pages, advanced identically by the
// producer and by every consumer thread.
struct Ring {
  uint32_t slot, phase;
  __device__ __forceinline__ void advance(int n) {
    if (++slot == (uint32_t)n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// ------------------------------------------------------------ tensors
__device__ __forceinline__ char* layer_base(const KernelParams& P, int l) {
  return P.act.base + (int64_t)l * P.act.layer_stride;
}
__device__ __forceinline__ char* global_base(const KernelParams& P) {
  return P.act.base + P.act.global_block;
}
__device__ __forceinline__ const uint16_t* layer_w(const KernelParams& P,
                                                   int l, int which) {
  return P.w.layers[l * MPK_LAYER_NTENSORS + which];
}
__device__ __forceinline__ const void* tmap_at(const KernelParams& P,
                                               int idx) {
  return P.w.tmaps + (size_t)idx * 128;
}

// Geometry of one MatMul task: which tensor map, rows, K, and paging.
struct Gemv {
  int kind, layer;
  int row0, rows;      // output rows [row0, row0 + rows)
  int K;               // reduction length
  int N;               // output width (ldo)
  int dual;            // gate/up pair: rows r of the gate and F + r
  int up_off;          // row offset of the up half (dual)
  int tmap;            // tensor-map slot
  const uint16_t* src; // activations [B][K]
  int rb_rows;         // output rows per row-block (64, or 32 when dual)
};

__device__ __forceinline__ bool is_gemv(int kind) {
  return kind == MPK_TASK_QKV || kind == MPK_TASK_O ||
         kind == MPK_TASK_GATEUP || kind == MPK_TASK_DOWN ||
         kind == MPK_TASK_LM_HEAD || kind == MPK_TASK_CHAIN_UP ||
         kind == MPK_TASK_CHAIN_DOWN;
}

__device__ Gemv gemv_geom(const KernelParams& P, const TaskDesc& t) {
  const Dims& D = P.dims;
  Gemv g;
  g.kind = t.kind;
  g.layer = t.layer;
  g.row0 = t.row0;
  g.rows = t.row1 - t.row0;
  g.dual = 0;
  g.up_off = 0;
  g.rb_rows = kMaxPageRows;
  const int l = t.layer;
  switch (t.kind) {
    case MPK_TASK_QKV:
      g.K = D.h;
      g.N = (D.Hq + 2 * D.Hkv) * D.d;
      g.tmap = 4 * l + TM_QKV;
      g.src = reinterpret_cast<const uint16_t*>(layer_base(P, l) + P.act.o_n1);
      break;
    case MPK_TASK_O:
      g.K = D.Hq * D.d;
      g.N = D.h;
      g.tmap = 4 * l + TM_O;
      g.src =
          reinterpret_cast<const uint16_t*>(layer_base(P, l) + P.act.o_attn);
      break;
    case MPK_TASK_GATEUP:
      g.K = D.h;
      g.N = D.F;
      g.dual = 1;
      g.up_off = D.F;
      g.rb_rows = kMaxPageRows / 2;
      g.tmap = 4 * l + TM_GU;
      g.src = reinterpret_cast<const uint16_t*>(layer_base(P, l) + P.act.o_n2);
      break;
    case MPK_TASK_DOWN:
      g.K = D.F;
      g.N = D.h;
      g.tmap = 4 * l + TM_DOWN;
      g.src = reinterpret_cast<const uint16_t*>(layer_base(P, l) + P.act.o_act);
      break;
    case MPK_TASK_LM_HEAD:
      g.K = D.h;
      g.N = D.V;
      g.tmap = 4 * D.L;
      g.src = reinterpret_cast<const uint16_t*>(
          global_base(P) + (D.chain_ffn > 0 ? P.act.g_z : P.act.g_nf));
      break;
    case MPK_TASK_CHAIN_UP:
      g.K = D.h;
      g.N = D.chain_ffn;
      g.tmap = 4 * D.L + 1;
      g.src = reinterpret_cast<const uint16_t*>(layer_base(P, 0) + P.act.o_n1);
      break;
    default:  // MPK_TASK_CHAIN_DOWN
      g.K = D.chain_ffn;
      g.N = D.h;
      g.tmap = 4 * D.L + 2;
      g.src = reinterpret_cast<const uint16_t*>(layer_base(P, 0) + P.act.o_act);
      break;
  }
  return g;
}

// Rows of row-block rb (output rows; a dual page holds them twice).
__device__ __forceinline__ int rb_count(const Gemv& g) {
  return (g.rows + g.rb_rows - 1) / g.rb_rows;
}
__device__ __forceinline__ int rb_len(const Gemv& g, int rb) {
  return min(g.rb_rows, g.rows - rb * g.rb_rows);
}
__device__ __forceinline__ int kpages(const Gemv& g) {
  return (g.K + kPageCols - 1) / kPageCols;
}

// ------------------------------------------------------------ producer
// Streams the weight pages of one MatMul task into the ring.  All 32 lanes
// of the producer warp take part; lane i issues box i of a page.
__device__ bool produce_gemv(const KernelParams& P, const Smem& S,
                             const Gemv& g, Ring& ring, uint32_t* issued,
                             uint64_t deadline, uint64_t policy) {
  const int lane = threadIdx.x & 31;
  const int n_pages = P.graph.n_pages;
  const void* tm = tmap_at(P, g.tmap);
  const int nrb = rb_count(g), nkp = kpages(g);
  for (int rb = 0; rb < nrb; ++rb) {
    const int len = rb_len(g, rb);
    const int r8 = (len + kBoxRows - 1) / kBoxRows;   // row boxes (per half)
    const int prow8 = g.dual ? 2 * r8 : r8;
    const int row_base = g.row0 + rb * g.rb_rows;
    for (int cb = 0; cb < nkp; ++cb) {
      const int c0 = cb * kPageCols;
      const int nbc = min(4, (g.K - c0 + 63) / 64);
      // wait until the consumers released this slot (lane 0 decides)
      int ok = 1;
      if (lane == 0) {
        uint32_t spins = 0;
        while (!mbar_try_wait(&S.empty[ring.slot], ring.phase ^ 1u)) {
          if ((++spins & 1023u) == 0u &&
              (aborted(P) || globaltimer() > deadline)) {
            if (!aborted(P)) raise_error(P, MPK_ERR_TIMEOUT);
            ok = 0;
            break;
          }
        }
        if (ok && aborted(P)) ok = 0;
        if (ok)
          mbar_arrive_expect_tx(&S.full[ring.slot],
                                (uint32_t)(nbc * prow8 * 1024));
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return false;
      uint8_t* page = S.pages + (size_t)ring.slot * kPageBytes;
      const int nbox = nbc * prow8;
      for (int i = lane; i < nbox; i += 32) {
        const int gb = i / prow8, rbi = i % prow8;
        int y;
        if (g.dual)
          y = (rbi < r8) ? row_base + rbi * kBoxRows
                         : g.up_off + row_base + (rbi - r8) * kBoxRows;
        else
          y = row_base + rbi * kBoxRows;
        tma_load_2d(page + (size_t)(gb * prow8 + rbi) * 1024, tm,
                    &S.full[ring.slot], c0 + gb * 64, y, policy);
      }
      issued[ring.slot] = 1u | (ring.phase << 1);
      ring.advance(n_pages);
      __syncwarp();
    }
  }
  return true;
}

// After an abort: wait (bounded) until every copy this producer issued has
// landed, so no TMA writes into shared memory after the CTA exits.
__device__ void drain_copies(const KernelParams& P, const Smem& S,
                             const uint32_t* issued) {
  if ((threadIdx.x & 31) != 0) return;
  const uint64_t limit = globaltimer() + 200000000ull;  // 200 ms
  for (int s = 0; s < P.graph.n_pages; ++s) {
    if (!(issued[s] & 1u)) continue;
    const uint32_t ph = (issued[s] >> 1) & 1u;
    while (!mbar_try_wait(&S.full[s], ph)) {
      if (globaltimer() > limit) return;
    }
  }
}

// ------------------------------------------------------------ task bodies
// RMSNorm family: x = a + c (bf16, rounded) or an embedding row; writes x
// (optional) and bf16((x * (mean(x^2) + eps)^-1/2) * w).
__device__ void task_norm(const KernelParams& P, const Smem& S,
                          const TaskDesc& t) {
  const Dims& D = P.dims;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = D.h, l = t.layer;
  const uint16_t *a = nullptr, *c = nullptr, *w;
  uint16_t *out_h = nullptr, *out_n;
  bool embed = false;
  switch (t.kind) {
    case MPK_TASK_NORM1:
      w = layer_w(P, l, MPK_W_LN1);
      out_h = reinterpret_cast<uint16_t*>(layer_base(P, l) + P.act.o_h);
      out_n = reinterpret_cast<uint16_t*>(layer_base(P, l) + P.act.o_n1);
      if (l == 0) {
        embed = true;
      } else {
        a = reinterpret_cast<const uint16_t*>(layer_base(P, l - 1) +
                                              P.act.o_hmid);
        c = reinterpret_cast<const uint16_t*>(layer_base(P, l - 1) +
                                              P.act.o_dout);
      }
      break;
    case MPK_TASK_NORM2:
      w = layer_w(P, l, MPK_W_LN2);
      a = reinterpret_cast<const uint16_t*>(layer_base(P, l) + P.act.o_h);
      c = reinterpret_cast<const uint16_t*>(layer_base(P, l) + P.act.o_o);
      out_h = reinterpret_cast<uint16_t*>(layer_base(P, l) + P.act.o_hmid);
      out_n = reinterpret_cast<uint16_t*>(layer_base(P, l) + P.act.o_n2);
      break;
    case MPK_TASK_FINAL_NORM:
      w = P.w.final_norm;
      a = reinterpret_cast<const uint16_t*>(layer_base(P, D.L - 1) +
                                            P.act.o_hmid);
      c = reinterpret_cast<const uint16_t*>(layer_base(P, D.L - 1) +
                                            P.act.o_dout);
      out_h = reinterpret_cast<uint16_t*>(layer_base(P, D.L) + P.act.o_h);
      out_n = reinterpret_cast<uint16_t*>(global_base(P) + P.act.g_nf);
      break;
    default:  // MPK_TASK_CHAIN_NORM
      w = P.w.final_norm;
      embed = true;
      out_n = reinterpret_cast<uint16_t*>(layer_base(P, 0) + P.act.o_n1);
      break;
  }
  constexpr int kMaxChunks = 4;  // h <= 4 * 8 * 256 = 8192
  const int nchunk = (h / 8 + kConsumers - 1) / kConsumers;
  for (int b = 0; b < D.B; ++b) {
    float x[kMaxChunks][8];
    float ss = 0.f;
    const uint16_t* erow = nullptr;
    if (embed) {
      int tok = __ldg(P.step.tokens + b);
      tok = min(max(tok, 0), D.V - 1);
      erow = P.w.embed + (int64_t)tok * h;
    }
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
      const int i = (tid + k * kConsumers) * 8;
      if (k < nchunk && i < h) {
        if (embed) {
          uint4 v = __ldg(reinterpret_cast<const uint4*>(erow + i));
          const uint32_t* pw = &v.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            x[k][2 * q] = bf_lo(pw[q]);
            x[k][2 * q + 1] = bf_hi(pw[q]);
          }
        } else {
          uint4 va = __ldcg(reinterpret_cast<const uint4*>(a + (int64_t)b * h + i));
          uint4 vc = __ldcg(reinterpret_cast<const uint4*>(c + (int64_t)b * h + i));
          const uint32_t* pa = &va.x;
          const uint32_t* pc = &vc.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            x[k][2 * q] = round_bf(__fadd_rn(bf_lo(pa[q]), bf_lo(pc[q])));
            x[k][2 * q + 1] = round_bf(__fadd_rn(bf_hi(pa[q]), bf_hi(pc[q])));
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) ss = fmaf(x[k][q], x[k][q], ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) S.scratch[warp] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int q = 0; q < kConsumerWarps; ++q) tot += S.scratch[q];
    const float r = 1.0f / sqrtf(tot / (float)h + D.eps);
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
      const int i = (tid + k * kConsumers) * 8;
      if (k < nchunk && i < h) {
        uint4 wv = __ldg(reinterpret_cast<const uint4*>(w + i));
        const uint32_t* pw = &wv.x;
        uint4 on, oh;
        uint32_t* pon = &on.x;
        uint32_t* poh = &oh.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float n0 = __fmul_rn(__fmul_rn(x[k][2 * q], r), bf_lo(pw[q]));
          const float n1 = __fmul_rn(__fmul_rn(x[k][2 * q + 1], r), bf_hi(pw[q]));
          pon[q] = pack_bf2(n0, n1);
          poh[q] = pack_bf2(x[k][2 * q], x[k][2 * q + 1]);
        }
        *reinterpret_cast<uint4*>(out_n + (int64_t)b * h + i) = on;
        if (out_h) *reinterpret_cast<uint4*>(out_h + (int64_t)b * h + i) = oh;
      }
    }
    consumer_sync();   // scratch reuse across rows
  }
}

// q/k RMSNorm (optional) + RoPE for the query heads of KV head g and for
// its key; appends k, v at position seq_lens[b] of the paged cache.
__device__ void task_rope(const KernelParams& P, const Smem& S,
                          const TaskDesc& t) {
  const Dims& D = P.dims;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = t.b, g = t.g, l = t.layer, d = D.d, half = d / 2;
  const int grp = D.Hq / D.Hkv;
  const int pos = __ldcg(P.step.seq_lens + b);
  const int pidx = pos / D.page_size;
  int page = -1;
  if (pos >= 0 && pidx < D.max_pages)
    page = __ldg(P.step.page_table + (int64_t)b * D.max_pages + pidx);
  if (page < 0 || page >= P.step.num_pages || pos >= D.max_ctx) {
    if (threadIdx.x == 0) raise_error(P, MPK_ERR_KV_PAGE);
    return;
  }
  const uint16_t* qkv = reinterpret_cast<const uint16_t*>(
      layer_base(P, l) + P.act.o_qkv) + (int64_t)b * (D.Hq + 2 * D.Hkv) * d;
  uint16_t* qout = reinterpret_cast<uint16_t*>(layer_base(P, l) + P.act.o_q) +
                   (int64_t)b * D.Hq * d;
  const int64_t slot = ((((int64_t)l * P.step.num_pages + page) * D.Hkv + g) *
                            D.page_size + pos % D.page_size) * d;
  const float* cs = P.w.rope_cs + (int64_t)pos * half * 2;
  for (int hh = warp; hh < grp + 2; hh += kConsumerWarps) {
    const uint16_t* src;
    uint16_t* dst;
    const uint16_t* nw = nullptr;
    bool rot = true;
    if (hh < grp) {
      src = qkv + (int64_t)(g * grp + hh) * d;
      dst = qout + (int64_t)(g * grp + hh) * d;
      if (D.qk_norm) nw = layer_w(P, l, MPK_W_QNORM);
    } else if (hh == grp) {
      src = qkv + (int64_t)(D.Hq + g) * d;
      dst = P.step.k_pool + slot;
      if (D.qk_norm) nw = layer_w(P, l, MPK_W_KNORM);
    } else {
      src = qkv + (int64_t)(D.Hq + D.Hkv + g) * d;
      dst = P.step.v_pool + slot;
      rot = false;
    }
    // pairs (i, i + d/2) for i = lane, lane + 32 (half <= 64)
    float x1[2], x2[2];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < half) {
        x1[k] = bf2f(__ldcg(src + i));
        x2[k] = bf2f(__ldcg(src + i + half));
        ss = fmaf(x1[k], x1[k], ss);
        ss = fmaf(x2[k], x2[k], ss);
      }
    }
    if (!rot) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = lane + 32 * k;
        if (i < half) {
          dst[i] = f2bf(x1[k]);
          dst[i + half] = f2bf(x2[k]);
        }
      }
      continue;
    }
    if (nw) {
      ss = warp_sum(ss);
      const float r = 1.0f / sqrtf(ss / (float)d + D.eps);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = lane + 32 * k;
        if (i < half) {
          x1[k] = round_bf(__fmul_rn(__fmul_rn(x1[k], r), bf2f(__ldg(nw + i))));
          x2[k] = round_bf(
              __fmul_rn(__fmul_rn(x2[k], r), bf2f(__ldg(nw + i + half))));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = lane + 32 * k;
      if (i < half) {
        const float c = __ldg(cs + 2 * i), s = __ldg(cs + 2 * i + 1);
        const float y1 = __fsub_rn(__fmul_rn(x1[k], c), __fmul_rn(x2[k], s));
        const float y2 = __fadd_rn(__fmul_rn(x2[k], c), __fmul_rn(x1[k], s));
        dst[i] = f2bf(y1);
        dst[i + half] = f2bf(y2);
      }
    }
  }
}

// Paged attention over KV chunk c of (sequence b, KV head g): tokens
// [c n / C, (c+1) n / C) of n = seq_lens[b] + 1.  Each warp runs an online
// softmax over a strided subset of the tokens for all query heads of the
// group; the warps are merged in shared memory into one partial
// (m, l, acc[d]) per query head.
template <int DL, int kMaxGrp>
__device__ void attn_body(const KernelParams& P, const Smem& S,
                          const TaskDesc& t) {
  const Dims& D = P.dims;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = t.b, g = t.g, l = t.layer, d = D.d;
  const int grp = D.Hq / D.Hkv;
  const int n = __ldcg(P.step.seq_lens + b) + 1;
  const int t0 = (int)(((int64_t)t.c * n) / D.C);
  const int t1 = (int)(((int64_t)(t.c + 1) * n) / D.C);
  const float scale = 1.0f / sqrtf((float)d);
  const uint16_t* q = reinterpret_cast<const uint16_t*>(
                          layer_base(P, l) + P.act.o_q) +
                      (int64_t)b * D.Hq * d + (int64_t)g * grp * d;
  float qr[kMaxGrp][DL];
  float m[kMaxGrp], lsum[kMaxGrp], acc[kMaxGrp][DL];
#pragma unroll
  for (int hh = 0; hh < kMaxGrp; ++hh) {
    m[hh] = -INFINITY;
    lsum[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) {
      acc[hh][e] = 0.f;
      qr[hh][e] = (hh < grp) ? bf2f(__ldcg(q + hh * d + lane * DL + e)) : 0.f;
    }
  }
  const int64_t head_stride = (int64_t)D.page_size * d;
  const int64_t page_stride = (int64_t)D.Hkv * head_stride;
  const int64_t layer_off = (int64_t)l * P.step.num_pages * page_stride +
                            (int64_t)g * head_stride;
  const int32_t* pt = P.step.page_table + (int64_t)b * D.max_pages;
  for (int tok = t0 + warp; tok < t1; tok += kConsumerWarps) {
    const int page = __ldg(pt + tok / D.page_size);
    if (page < 0 || page >= P.step.num_pages) {
      if (lane == 0) raise_error(P, MPK_ERR_KV_PAGE);
      break;
    }
    const int64_t off = layer_off + (int64_t)page * page_stride +
                        (int64_t)(tok % D.page_size) * d + lane * DL;
    float kf[DL], vf[DL];
    if (DL == 4) {
      uint2 kv = __ldcg(reinterpret_cast<const uint2*>(P.step.k_pool + off));
      uint2 vv = __ldcg(reinterpret_cast<const uint2*>(P.step.v_pool + off));
      kf[0] = bf_lo(kv.x); kf[1] = bf_hi(kv.x);
      kf[2 % DL] = bf_lo(kv.y); kf[3 % DL] = bf_hi(kv.y);
      vf[0] = bf_lo(vv.x); vf[1] = bf_hi(vv.x);
      vf[2 % DL] = bf_lo(vv.y); vf[3 % DL] = bf_hi(vv.y);
    } else if (DL == 2) {
      uint32_t kv = __ldcg(reinterpret_cast<const unsigned int*>(P.step.k_pool + off));
      uint32_t vv = __ldcg(reinterpret_cast<const unsigned int*>(P.step.v_pool + off));
      kf[0] = bf_lo(kv); kf[1 % DL] = bf_hi(kv);
      vf[0] = bf_lo(vv); vf[1 % DL] = bf_hi(vv);
    } else {
#pragma unroll
      for (int e = 0; e < DL; ++e) {
        kf[e] = bf2f(__ldcg(P.step.k_pool + off + e));
        vf[e] = bf2f(__ldcg(P.step.v_pool + off + e));
      }
    }
#pragma unroll
    for (int hh = 0; hh < kMaxGrp; ++hh) {
      if (hh < grp) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < DL; ++e) s = fmaf(qr[hh][e], kf[e], s);
        s = warp_sum(s) * scale;
        const float mn = fmaxf(m[hh], s);
        const float corr = expf(m[hh] - mn);
        const float p = expf(s - mn);
        lsum[hh] = lsum[hh] * corr + p;
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[hh][e] = fmaf(p, vf[e], acc[hh][e] * corr);
        m[hh] = mn;
      }
    }
  }
  // merge the 8 warps: layout [warp][grp][2 + d] floats in the x area
  float* wbuf = reinterpret_cast<float*>(S.xs);
  const int rec = 2 + d;
#pragma unroll
  for (int hh = 0; hh < kMaxGrp; ++hh) {
    if (hh < grp) {
      float* r = wbuf + ((int64_t)warp * grp + hh) * rec;
      if (lane == 0) {
        r[0] = m[hh];
        r[1] = lsum[hh];
      }
#pragma unroll
      for (int e = 0; e < DL; ++e) r[2 + lane * DL + e] = acc[hh][e];
    }
  }
  consumer_sync();
  float* out = reinterpret_cast<float*>(layer_base(P, l) + P.act.o_opart) +
               (((int64_t)(b * D.Hkv + g) * D.C + t.c) * grp) * rec;
  for (int o = threadIdx.x; o < grp * d; o += kConsumers) {
    const int hh = o / d, i = o % d;
    float M = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w)
      M = fmaxf(M, wbuf[((int64_t)w * grp + hh) * rec]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* r = wbuf + ((int64_t)w * grp + hh) * rec;
        const float sc = (r[0] == -INFINITY) ? 0.f : expf(r[0] - M);
        L = fmaf(r[1], sc, L);
        A = fmaf(r[2 + i], sc, A);
      }
    }
    out[(int64_t)hh * rec + 2 + i] = A;
    if (i == 0) {
      out[(int64_t)hh * rec] = M;
      out[(int64_t)hh * rec + 1] = L;
    }
  }
  consumer_sync();
}

__device__ void task_attn(const KernelParams& P, const Smem& S,
                          const TaskDesc& t) {
  const int grp = P.dims.Hq / P.dims.Hkv;
  const int dl = P.dims.d / 32;
  if (grp <= 4) {
    switch (dl) {
      case 1: attn_body<1, 4>(P, S, t); break;
      case 2: attn_body<2, 4>(P, S, t); break;
      case 3: attn_body<3, 4>(P, S, t); break;
      default: attn_body<4, 4>(P, S, t); break;
    }
  } else if (grp <= 8) {
    switch (dl) {
      case 1: attn_body<1, 8>(P, S, t); break;
      case 2: attn_body<2, 8>(P, S, t); break;
      case 3: attn_body<3, 8>(P, S, t); break;
      default: attn_body<4, 8>(P, S, t); break;
    }
  } else {
    switch (dl) {
      case 1: attn_body<1, 16>(P, S, t); break;
      default: attn_body<2, 16>(P, S, t); break;
    }
  }
}

// Log-sum-exp merge of the C chunk partials of (b, g) -> bf16 attention
// output of the group's query heads.
__device__ void task_merge(const KernelParams& P, const Smem& S,
                           const TaskDesc& t) {
  const Dims& D = P.dims;
  const int b = t.b, g = t.g, l = t.layer, d = D.d;
  const int grp = D.Hq / D.Hkv, rec = 2 + d;
  const float* part = reinterpret_cast<const float*>(layer_base(P, l) +
                                                     P.act.o_opart) +
                      ((int64_t)(b * D.Hkv + g) * D.C * grp) * rec;
  uint16_t* out = reinterpret_cast<uint16_t*>(layer_base(P, l) + P.act.o_attn) +
                  (int64_t)b * D.Hq * d + (int64_t)g * grp * d;
  for (int o = threadIdx.x; o < grp * d; o += kConsumers) {
    const int hh = o / d, i = o % d;
    float M = -INFINITY;
    for (int c = 0; c < D.C; ++c)
      M = fmaxf(M, __ldcg(part + ((int64_t)c * grp + hh) * rec));
    float L = 0.f, A = 0.f;
    for (int c = 0; c < D.C; ++c) {
      const float* r = part + ((int64_t)c * grp + hh) * rec;
      const float mc = __ldcg(r);
      const float sc = (mc == -INFINITY) ? 0.f : expf(mc - M);
      L = fmaf(__ldcg(r + 1), sc, L);
      A = fmaf(__ldcg(r + 2 + i), sc, A);
    }
    out[o] = f2bf(A / L);
  }
}

// Greedy argmax over the lm_head tiles' (max, index) pairs; lowest index
// among equal maxima.  Also advances seq_lens (decoder mode).
__device__ void task_argmax(const KernelParams& P, const Smem& S,
                            const TaskDesc& t) {
  const Dims& D = P.dims;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float2* am = reinterpret_cast<const float2*>(global_base(P) +
                                                     P.act.g_amax);
  for (int b = 0; b < D.B; ++b) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = tid; j < D.n_lm_tiles; j += kConsumers) {
      const float2 e = __ldcg(am + (int64_t)b * D.n_lm_tiles + j);
      const int idx = __float_as_int(e.y);
      if (e.x > bv || (e.x == bv && idx < bi)) {
        bv = e.x;
        bi = idx;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      S.scratch[warp] = bv;
      S.scratch[16 + warp] = __int_as_float(bi);
    }
    consumer_sync();
    if (tid == 0) {
      for (int w = 1; w < kConsumerWarps; ++w) {
        const float ov = S.scratch[w];
        const int oi = __float_as_int(S.scratch[16 + w]);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      P.step.next_tokens[b] = (bi == 0x7fffffff) ? 0 : bi;
      if (D.chain_ffn == 0) P.step.seq_lens[b] = __ldcg(P.step.seq_lens + b) + 1;
    }
    consumer_sync();
  }
}

// Bounded wait for a weight page.  On timeout or abort the thread records a
// bail-out in shared memory and carries on without the page (the step's
// result is void by then), so every consumer thread still reaches the same
// barriers and the CTA leaves its loop together.
__device__ __forceinline__ bool wait_page(const KernelParams& P, const Smem& S,
                                          const Ring& ring,
                                          uint64_t deadline) {
  if (S.ctrl[2]) return false;
  uint32_t spins = 0;
  while (!mbar_try_wait(&S.full[ring.slot], ring.phase)) {
    if ((++spins & 1023u) == 0u && (aborted(P) || globaltimer() > deadline)) {
      if (!aborted(P)) raise_error(P, MPK_ERR_TIMEOUT);
      S.ctrl[2] = 1;
      return false;
    }
  }
  return true;
}

// MatMul tile: out[b][row] = sum_k x[b][k] W[row][k] for the task's rows,
// consuming the weight pages the producer streams.  Thread (gbox, r) owns
// row r of column box gbox of every page of a row-block; the four column
// boxes are summed at the end of the row-block.
template <int NB>
__device__ void task_gemv(const KernelParams& P, const Smem& S,
                          const TaskDesc& t, Ring& ring, uint64_t deadline) {
  const Dims& D = P.dims;
  const int tid = threadIdx.x, lane = tid & 31;
  const int B = D.B;
  const Gemv g = gemv_geom(P, t);
  const int n_pages = P.graph.n_pages;
  // x staging: [B][XC] bf16, XC a multiple of the page width
  const int XC = ((kXsBytes / 2 / B) / kPageCols) * kPageCols;
  const int nrb = rb_count(g), nkp = kpages(g);
  int loaded = -1;
  float best_v[NB];
  int best_i[NB];
#pragma unroll
  for (int bb = 0; bb < NB; ++bb) {
    best_v[bb] = -INFINITY;
    best_i[bb] = 0x7fffffff;
  }
  for (int rb = 0; rb < nrb; ++rb) {
    const int len = rb_len(g, rb);
    const int r8 = (len + kBoxRows - 1) / kBoxRows;
    const int prow8 = g.dual ? 2 * r8 : r8;
    const int prows = prow8 * kBoxRows;
    const int gb = tid / prows, r = tid % prows;
    const bool mapped = gb < 4;
    float acc[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) acc[bb] = 0.f;
    for (int x0 = 0; x0 < g.K; x0 += XC) {
      if (x0 != loaded) {
        consumer_sync();
        const int xw = min(XC, g.K - x0);
        const int xpad = ((xw + 63) / 64) * 64;
        for (int bb = 0; bb < B; ++bb) {
          const uint16_t* src = g.src + (int64_t)bb * g.K + x0;
          uint16_t* dst = S.xs + bb * XC;
          for (int i = tid * 8; i < xpad; i += kConsumers * 8) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (i < xw) v = __ldcg(reinterpret_cast<const uint4*>(src + i));
            *reinterpret_cast<uint4*>(dst + i) = v;
          }
        }
        consumer_sync();
        loaded = x0;
      }
      const int cb_end = min(nkp, (x0 + XC) / kPageCols);
      for (int cb = x0 / kPageCols; cb < cb_end; ++cb) {
        const int nbc = min(4, (g.K - cb * kPageCols + 63) / 64);
        const bool have = wait_page(P, S, ring, deadline);
        if (have && mapped && gb < nbc) {
          const uint8_t* rowp = S.pages + (size_t)ring.slot * kPageBytes +
                                ((size_t)(gb * prow8 + (r >> 3)) << 10) +
                                ((r & 7) << 7);
          const uint16_t* xp = S.xs + (cb * kPageCols - x0) + gb * 64;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 wv = *reinterpret_cast<const uint4*>(
                rowp + ((j ^ (r & 7)) << 4));
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
              if (bb < B) {
                const uint4 xv =
                    *reinterpret_cast<const uint4*>(xp + bb * XC + j * 8);
                acc[bb] = dot8(wv, xv, acc[bb]);
              }
            }
          }
        }
        // a page that never arrived (aborted step) is not released, so the
        // producer cannot refill a slot a copy may still be writing
        if (__all_sync(0xffffffffu, have) && lane == 0)
          mbar_arrive(&S.empty[ring.slot]);
        __syncwarp();
        ring.advance(n_pages);
      }
    }
    // reduce the four column boxes of each page row
    if (mapped) {
#pragma unroll
      for (int bb = 0; bb < NB; ++bb)
        if (bb < B) S.red[((gb * prows) + r) * B + bb] = acc[bb];
    }
    consumer_sync();
    const int out_rows = g.dual ? r8 * kBoxRows : prows;
    if (tid < out_rows) {
      const int orow = g.row0 + rb * g.rb_rows + tid;
      const bool valid = tid < len;
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) {
        if (bb < B && valid) {
          float v = 0.f, u = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) v += S.red[((q * prows) + tid) * B + bb];
          if (g.dual) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              u += S.red[((q * prows) + r8 * kBoxRows + tid) * B + bb];
          }
          switch (g.kind) {
            case MPK_TASK_LM_HEAD: {
              P.step.logits[(int64_t)bb * g.N + orow] = v;
              if (v > best_v[bb] || (v == best_v[bb] && orow < best_i[bb])) {
                best_v[bb] = v;
                best_i[bb] = orow;
              }
              break;
            }
            case MPK_TASK_GATEUP: {
              const float gv = round_bf(v), uv = round_bf(u);
              uint16_t* o = reinterpret_cast<uint16_t*>(
                  layer_base(P, g.layer) + P.act.o_act);
              o[(int64_t)bb * g.N + orow] = f2bf(__fmul_rn(silu_f(gv), uv));
              break;
            }
            case MPK_TASK_CHAIN_UP: {
              uint16_t* o = reinterpret_cast<uint16_t*>(layer_base(P, 0) +
                                                        P.act.o_act);
              o[(int64_t)bb * g.N + orow] = f2bf(silu_f(round_bf(v)));
              break;
            }
            default: {
              uint16_t* o;
              if (g.kind == MPK_TASK_QKV)
                o = reinterpret_cast<uint16_t*>(layer_base(P, g.layer) + P.act.o_qkv);
              else if (g.kind == MPK_TASK_O)
                o = reinterpret_cast<uint16_t*>(layer_base(P, g.layer) + P.act.o_o);
              else if (g.kind == MPK_TASK_DOWN)
                o = reinterpret_cast<uint16_t*>(layer_base(P, g.layer) + P.act.o_dout);
              else
                o = reinterpret_cast<uint16_t*>(global_base(P) + P.act.g_z);
              o[(int64_t)bb * g.N + orow] = f2bf(v);
              break;
            }
          }
        }
      }
    }
    consumer_sync();
  }
  if (g.kind == MPK_TASK_LM_HEAD) {
    // tile argmax over threads 0..63 (warps 0 and 1)
    const int warp = tid >> 5;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
      if (bb >= B) break;
      float bv = best_v[bb];
      int bi = best_i[bb];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (lane == 0 && warp < 2) {
        S.scratch[2 * warp] = bv;
        S.scratch[2 * warp + 1] = __int_as_float(bi);
      }
      consumer_sync();
      if (tid == 0) {
        const float ov = S.scratch[2];
        const int oi = __float_as_int(S.scratch[3]);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
        float2* am = reinterpret_cast<float2*>(global_base(P) + P.act.g_amax);
        am[(int64_t)bb * D.n_lm_tiles + t.tile] =
            make_float2(bv, __int_as_float(bi));
      }
      consumer_sync();
    }
  }
}

__device__ void run_task(const KernelParams& P, const Smem& S,
                         const TaskDesc& t, Ring& ring, uint64_t deadline) {
  switch (t.kind) {
    case MPK_TASK_NORM1:
    case MPK_TASK_NORM2:
    case MPK_TASK_FINAL_NORM:
    case MPK_TASK_CHAIN_NORM:
      task_norm(P, S, t);
      break;
    case MPK_TASK_ROPE:
      task_rope(P, S, t);
      break;
    case MPK_TASK_ATTN:
      task_attn(P, S, t);
      break;
    case MPK_TASK_MERGE:
      task_merge(P, S, t);
      break;
    case MPK_TASK_ARGMAX:
      task_argmax(P, S, t);
      break;
    case MPK_TASK_EMPTY:
      break;
    default:
      if (P.dims.B == 1)
        task_gemv<1>(P, S, t, ring, deadline);
      else if (P.dims.B <= 4)
        task_gemv<4>(P, S, t, ring, deadline);
      else if (P.dims.B <= 8)
        task_gemv<8>(P, S, t, ring, deadline);
      else
        task_gemv<16>(P, S, t, ring, deadline);
      break;
  }
}

// ------------------------------------------------------------ queues
__device__ bool ring_push(const KernelParams& P, RingHdr* hdr, uint64_t* slots,
                          uint32_t cap, uint32_t value, uint64_t deadline) {
  const uint32_t pos = atomicAdd(&hdr->tail, 1u);
  uint32_t spins = 0;
  while (pos - ld_acquire(&hdr->head) >= cap) {
    if ((++spins & 255u) == 0u && (aborted(P) || globaltimer() > deadline)) {
      if (!aborted(P)) raise_error(P, MPK_ERR_QUEUE_OVERFLOW);
      return false;
    }
  }
  st_release64(slots + (pos % cap), ((uint64_t)(pos + 1u) << 32) | value);
  return true;
}

__device__ __forceinline__ bool ring_try_pop(RingHdr* hdr, uint64_t* slots,
                                             uint32_t cap, uint32_t& head,
                                             uint32_t& value) {
  const uint64_t v = ld_acquire64(slots + (head % cap));
  if ((uint32_t)(v >> 32) != head + 1u) return false;
  value = (uint32_t)v;
  ++head;
  st_release(&hdr->head, head);
  return true;
}

// Fire `e` (one trigger).  The activating trigger pushes the event to its
// scheduler warp when it has JIT tasks, and runs its empty tasks inline
// (they only trigger their own event).
__device__ void trigger(const KernelParams& P, int e, uint64_t deadline) {
  const DevGraph& G = P.graph;
  const uint32_t epoch = P.step.epoch;
  int stack[16];
  int sp = 0;
  stack[sp++] = e;
  while (sp > 0) {
    const int ev = stack[--sp];
    const EventDesc ed = G.events[ev];
    if (!(ed.flags & (EV_HAS_JIT | EV_HAS_INLINE))) {
      red_release_add(G.counters + ev, 1u);
      continue;
    }
    const uint32_t old = atom_acq_rel_add(G.counters + ev, 1u);
    if (old + 1u != epoch * ed.count) continue;
    if (ed.flags & EV_HAS_JIT) {
      const int s = ev % G.S;
      if (!ring_push(P, G.sched_hdr + s, G.sched_slots + (size_t)s * G.sched_cap,
                     G.sched_cap, (uint32_t)ev, deadline))
        return;
    }
    if (ed.flags & EV_HAS_INLINE) {
      for (int t = ed.first; t <= ed.last; ++t) {
        if (G.tasks[t].launch != MPK_LAUNCH_INLINE) continue;
        if (sp >= 16) {
          raise_error(P, MPK_ERR_QUEUE_OVERFLOW);
          return;
        }
        stack[sp++] = G.tasks[t].trig;
      }
    }
  }
}

__device__ __forceinline__ bool event_done(const KernelParams& P, int e) {
  const uint32_t target = P.step.epoch * P.graph.events[e].count;
  return (int32_t)(ld_relaxed(P.graph.counters + e) - target) >= 0;
}

// ------------------------------------------------------------ roles
__device__ void producer_role(const KernelParams& P, const Smem& S,
                              const int32_t* list, int n, uint64_t deadline) {
  uint32_t issued[16];
  for (int i = 0; i < 16; ++i) issued[i] = 0;
  Ring ring{0, 0};
  const uint64_t policy = evict_first_policy();
  for (int i = 0; i < n; ++i) {
    const TaskDesc t = P.graph.tasks[list[i]];
    if (!is_gemv(t.kind)) continue;
    if (!produce_gemv(P, S, gemv_geom(P, t), ring, issued, deadline, policy)) {
      drain_copies(P, S, issued);
      return;
    }
  }
  // the consumers wait for every page before leaving, so all copies have
  // landed by the time the CTA exits unless the step aborted
  if (aborted(P)) drain_copies(P, S, issued);
}

__device__ void worker_consumers(const KernelParams& P, const Smem& S, int w,
                                 uint64_t deadline) {
  const DevGraph& G = P.graph;
  const int tid = threadIdx.x;
  const int a0 = G.aot_off[w], a1 = G.aot_off[w + 1];
  int ai = a0;
  uint32_t jit_head = 0;
  RingHdr* jh = G.jit_hdr + w;
  uint64_t* js = G.jit_slots + (size_t)w * G.jit_cap;
  if (tid == 0) jit_head = ld_relaxed(&jh->head);
  Ring ring{0, 0};
  int iter = 0;
  uint64_t t_look = 0, t_ready = 0;
  while (true) {
    if (tid == 0) {
      if (G.trace) t_look = globaltimer();
      int cmd = -1;
      uint32_t spins = 0;
      int head_task = (ai < a1) ? G.aot_list[ai] : -1;
      int head_dep = (head_task >= 0) ? G.tasks[head_task].dep : G.end;
      while (!S.ctrl[2]) {
        uint32_t v;
        if (ring_try_pop(jh, js, G.jit_cap, jit_head, v)) {
          cmd = (int)v;
          break;
        }
        if (event_done(P, head_dep)) {
          cmd = head_task;   // -1 when the end event fired
          if (head_task >= 0) ++ai;
          break;
        }
        ++spins;
        if (spins > 32) __nanosleep(spins > 4096 ? 256 : 32);
        if ((spins & 63u) == 0u) {
          if (aborted(P)) break;
          if (globaltimer() > deadline) {
            raise_error(P, MPK_ERR_TIMEOUT);
            break;
          }
        }
      }
      fence_acq_rel_gpu();
      if (G.trace) t_ready = globaltimer();
      S.ctrl[iter & 1] = cmd;
    }
    consumer_sync();
    const int cmd = S.ctrl[iter & 1];
    ++iter;
    if (cmd < 0) break;
    const TaskDesc t = G.tasks[cmd];
    run_task(P, S, t, ring, deadline);
    consumer_sync();
    // only the leader decides to stop (at its next poll), so all consumer
    // threads leave through the same broadcast
    if (tid == 0 && !S.ctrl[2] && !aborted(P)) {
      __threadfence();
      trigger(P, t.trig, deadline);
      if (G.trace) {
        // (task | worker << 32), looked-for, ready, done
        const uint32_t k = atomicAdd(G.trace_count, 1u);
        if (k < G.trace_cap) {
          uint64_t* r = G.trace + 4ull * k;
          r[0] = (uint64_t)(uint32_t)cmd | ((uint64_t)(uint32_t)w << 32);
          r[1] = t_look;
          r[2] = t_ready;
          r[3] = globaltimer();
        }
      }
    }
  }
}

__device__ void scheduler_role(const KernelParams& P, int s,
                               uint64_t deadline) {
  const DevGraph& G = P.graph;
  const int lane = threadIdx.x & 31;
  RingHdr* hdr = G.sched_hdr + s;
  uint64_t* slots = G.sched_slots + (size_t)s * G.sched_cap;
  uint32_t head = (lane == 0) ? ld_relaxed(&hdr->head) : 0;
  uint32_t cursor = (uint32_t)(((int64_t)s * G.W) / G.S);
  uint32_t spins = 0;
  while (true) {
    int e = -1, stop = 0;
    if (lane == 0) {
      uint32_t v;
      if (ring_try_pop(hdr, slots, G.sched_cap, head, v)) {
        e = (int)v;
        fence_acq_rel_gpu();
        spins = 0;
      } else {
        ++spins;
        if (event_done(P, G.end) || aborted(P)) stop = 1;
        if (spins > 32) __nanosleep(spins > 4096 ? 256 : 32);
        if ((spins & 63u) == 0u && globaltimer() > deadline) {
          raise_error(P, MPK_ERR_TIMEOUT);
          stop = 1;
        }
      }
    }
    e = __shfl_sync(0xffffffffu, e, 0);
    stop = __shfl_sync(0xffffffffu, stop, 0);
    if (stop) break;
    if (e < 0) continue;
    const EventDesc ed = G.events[e];
    const int n = ed.last - ed.first + 1;
    for (int i = lane; i < n; i += 32) {
      const int t = ed.first + i;
      if (G.tasks[t].launch != MPK_LAUNCH_JIT) continue;
      const int w = (int)((cursor + (uint32_t)i) % (uint32_t)G.W);
      ring_push(P, G.jit_hdr + w, G.jit_slots + (size_t)w * G.jit_cap,
                G.jit_cap, (uint32_t)t, deadline);
    }
    cursor += (uint32_t)n;
  }
}

// ------------------------------------------------------------ kernels
__device__ __forceinline__ bool setup_smem(const KernelParams& P, uint8_t* raw,
                                           Smem& S) {
  if (smem_addr(raw) & 1023u) {   // uniform: same address for all threads
    if (threadIdx.x == 0) raise_error(P, MPK_ERR_UNSUPPORTED);
    return false;
  }
  S = carve(raw, P.graph.n_pages, P.dims.B);
  if (threadIdx.x == 0) {
    for (int i = 0; i < P.graph.n_pages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsumerWarps);
    }
    S.ctrl[0] = S.ctrl[1] = -1;
    S.ctrl[2] = 0;
    // an earlier step that failed leaves the abort flag up until
    // mpk_reset; read it once per CTA so all threads agree
    S.ctrl[3] = aborted(P) ? 1 : 0;
    fence_proxy_async_smem();
  }
  __syncthreads();
  return S.ctrl[3] == 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    mpk_megakernel(const __grid_constant__ KernelParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint64_t deadline = globaltimer() + P.step.timeout_ns;
  if ((int)blockIdx.x >= P.graph.W) {
    const int warp = threadIdx.x >> 5;
    if (warp >= P.graph.sched_warps_per_sm) return;
    const int s = ((int)blockIdx.x - P.graph.W) * P.graph.sched_warps_per_sm +
                  warp;
    if (s < P.graph.S) scheduler_role(P, s, deadline);
    return;
  }
  Smem S;
  if (!setup_smem(P, smem_raw, S)) return;
  const int w = blockIdx.x;
  if ((threadIdx.x >> 5) == kConsumerWarps) {
    const int a0 = P.graph.aot_off[w], a1 = P.graph.aot_off[w + 1];
    producer_role(P, S, P.graph.aot_list + a0, a1 - a0, deadline);
  } else {
    worker_consumers(P, S, w, deadline);
  }
}

// Kernel-per-operator: block i runs task op_tasks[first + i] with the same
// producer/consumer split; stream order replaces the events.
__global__ void __launch_bounds__(kThreads, 1)
    mpk_kpo_kernel(const __grid_constant__ KernelParams P, int first) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint64_t deadline = globaltimer() + P.step.timeout_ns;
  Smem S;
  if (!setup_smem(P, smem_raw, S)) return;
  const int task = P.graph.op_tasks[first + blockIdx.x];
  if ((threadIdx.x >> 5) == kConsumerWarps) {
    producer_role(P, S, P.graph.op_tasks + first + blockIdx.x, 1, deadline);
  } else {
    Ring ring{0, 0};
    run_task(P, S, P.graph.tasks[task], ring, deadline);
  }
}

// ------------------------------------------------------------ host side
int smem_bytes(int n_pages, int batch) { return smem_bytes_for(n_pages, batch); }

cudaError_t configure_kernels(int smem) {
  cudaError_t e = cudaFuncSetAttribute(
      mpk_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(
      mpk_kpo_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_megakernel(const KernelParams& P, int grid, int smem,
                              cudaStream_t stream) {
  void* args[] = {const_cast<KernelParams*>(&P)};
  return cudaLaunchCooperativeKernel((const void*)mpk_megakernel, dim3(grid),
                                     dim3(kThreads), args, (size_t)smem,
                                     stream);
}

cudaError_t launch_kpo_op(const KernelParams& P, int first, int n_tasks,
                          int smem, cudaStream_t stream) {
  mpk_kpo_kernel<<<n_tasks, kThreads, smem, stream>>>(P, first);
  return cudaGetLastError();
}

int megakernel_max_blocks_per_sm(int smem) {
  int n = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mpk_megakernel, kThreads,
                                                (size_t)smem);
  return n;
}

}  // namespace mpk
