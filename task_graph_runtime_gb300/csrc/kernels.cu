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
//     pipelining: the NEXT tasks' operands stream in while the current task
//     computes, and before the next task's event has fired, because weights
//     (and the KV cache of earlier tokens) never depend on an event;
//   "关键实现细节" 2 -- task descriptors prefetched before dequeue.
//
// GB300 layout of a worker CTA (one per SM, 384 threads = 3 warpgroups):
//   warps 8, 9  -- producers: both walk this worker's AOT task list and
//                  take alternate pages of it (two independent bulk-copy
//                  streams per SM sustain more HBM bandwidth than one).
//                  Weight pages arrive by 1-D bulk copies (cp.async.bulk):
//                  one contiguous copy of up to 32 KB at batch 1, one per
//                  matrix row at batch > 1; AOT attention tasks get their
//                  KV chunk the same way;
//   warps 0..7  -- consumers: poll events and the JIT queue, run task bodies,
//                  release pages, trigger events.
// MatMul tiles run on CUDA cores at batch < 8 and on tensor cores
// (mma.sync m16n8k16, batch as M, 8 weight rows as N) at batch >= 8.
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
constexpr int kProducerWarps = 2;   // two bulk-copy streams per SM
// Three warpgroups: two of consumers, one holding the producers (its other
// two warps only take part in the register hand-over and leave).  Launched
// at kLaunchRegs registers a thread; the producer warpgroup gives registers
// back (setmaxnreg.dec) and the consumer warpgroups take them: 256 * 216 +
// 128 * 72 = 384 * 168.
constexpr int kThreads = kConsumers + 128;
constexpr int kLaunchRegs = 168, kConsumerRegs = 216, kProducerRegs = 72;
static_assert(kConsumers * kConsumerRegs + 128 * kProducerRegs <=
                  kThreads * kLaunchRegs,
              "register hand-over must fit the launch allocation");
constexpr int kMaxRingPages = 8;
constexpr unsigned kFull = 0xffffffffu;

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
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 1-D bulk copy global -> this CTA's shared memory, completion counted in
// bytes on `bar`.  Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src,
                                         uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
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
// 16-byte asynchronous global -> shared copies (one thread's group).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0,
                                        uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr)
      : "memory");
}
// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0,
                                          uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
// acc + sum of 8 products, one fresh partial per 8 columns.
__device__ __forceinline__ float dot8(uint4 w, uint4 x, float acc) {
  float p = bf_lo(w.x) * bf_lo(x.x);
  p = fmaf(bf_hi(w.x), bf_hi(x.x), p);
  p = fmaf(bf_lo(w.y), bf_lo(x.y), p);
  p = fmaf(bf_hi(w.y), bf_hi(x.y), p);
  p = fmaf(bf_lo(w.z), bf_lo(x.z), p);
  p = fmaf(bf_hi(w.z), bf_hi(x.z), p);
  p = fmaf(bf_lo(w.w), bf_lo(x.w), p);
  p = fmaf(bf_hi(w.w), bf_hi(x.w), p);
  return acc + p;
}
__device__ __forceinline__ float silu_f(float z) {
  return z / (1.0f + expf(-z));
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
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

__device__ __forceinline__ bool event_done(const KernelParams& P, int e,
                                           uint32_t epoch) {
  const uint32_t target = epoch * P.graph.events[e].count;
  return (int32_t)(ld_relaxed(P.graph.counters + e) - target) >= 0;
}
// The same with acquire semantics: what the event's triggers wrote before
// triggering is visible to the caller afterwards.
__device__ __forceinline__ bool event_done_acq(const KernelParams& P, int e,
                                               uint32_t epoch) {
  const uint32_t target = epoch * P.graph.events[e].count;
  return (int32_t)(ld_acquire(P.graph.counters + e) - target) >= 0;
}

// ------------------------------------------------------------ shared memory
struct Smem {
  uint8_t* ring;
  uint16_t* xs;       // activation staging (bf16) / attention scratch
  float* res;         // MatMul row results
  uint64_t* full;
  uint64_t* empty;
  volatile int* ctrl; // [0..1] command, [2] bail-out, [3] aborted at entry,
                      // [4] last-chunk flag, [8..10] leader loop state,
                      // [13] JIT stage barrier phases, [14] the step of
                      // this launch the worker is in (multi-step loop)
  TaskDesc* desc;     // [0..1] staged descriptors (slot 2: the fan below)
  uint64_t* times;    // trace: [0] looked-for, [1] ready, [2] operands
                      // staged, [3] last page consumed, [4] body done
  AotRec* head;       // [2] the head AOT record (by queue position parity)
  EventDesc* tev;     // [0..1] triggering event of the staged task
  int32_t* fan;       // [0..1][2] cached fan-out events of the staged task
  uint64_t* jit_bar;  // [2] JIT attention stage barriers
  int2* meta;         // [ring slot] (position, new token's KV page) of the
                      // AOT attention task whose K page is in that slot
  float* scratch;
  int n_pages;
  int page_bytes;
};

__device__ __forceinline__ Smem carve(uint8_t* base, const SmemLayout& L) {
  Smem s;
  s.ring = base;
  s.xs = reinterpret_cast<uint16_t*>(base + L.xs);
  s.res = reinterpret_cast<float*>(base + L.res);
  s.full = reinterpret_cast<uint64_t*>(base + L.bars);
  s.empty = s.full + L.n_pages;
  s.ctrl = reinterpret_cast<volatile int*>(base + L.ctrl);
  s.desc = reinterpret_cast<TaskDesc*>(base + L.ctrl + 64);
  s.times = reinterpret_cast<uint64_t*>(base + L.ctrl + 160);
  s.head = reinterpret_cast<AotRec*>(base + L.ctrl + 224);
  s.tev = reinterpret_cast<EventDesc*>(base + L.ctrl + 352);
  s.meta = reinterpret_cast<int2*>(base + L.ctrl + 384);
  s.fan = reinterpret_cast<int32_t*>(base + L.ctrl + 128);
  s.jit_bar = reinterpret_cast<uint64_t*>(base + L.ctrl + 208);
  s.scratch = reinterpret_cast<float*>(base + L.scratch);
  s.n_pages = L.n_pages;
  s.page_bytes = L.page_bytes;
  return s;
}

// Trace stamp `i` (thread 0, tracing on only).
__device__ __forceinline__ void stamp(const KernelParams& P, const Smem& S,
                                      int i) {
  if (P.graph.trace && threadIdx.x == 0) S.times[i] = globaltimer();
}

// Position in the ring of pages, advanced identically by the producer and
// by every consumer thread.
struct Ring {
  uint32_t slot, phase;
  __device__ __forceinline__ void advance(int n) {
    if (++slot == (uint32_t)n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};
__device__ __forceinline__ uint8_t* page_ptr(const Smem& S, uint32_t slot) {
  return S.ring + (size_t)slot * S.page_bytes;
}

// Bounded wait for a ring page, by every consumer thread (each observes the
// mbarrier phase, which makes the bulk-copied bytes visible to it).  On
// timeout or abort the thread records a bail-out and carries on without the
// page (the step's result is void by then), so all consumer threads still
// reach the same barriers and leave the loop together.
__device__ __forceinline__ bool wait_full(const KernelParams& P,
                                          const Smem& S, const Ring& ring,
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
// Release a page (one arrival per consumer warp).  A page that never arrived
// is not released, so the producer cannot refill a slot that a copy may
// still be writing.
__device__ __forceinline__ void release_page(const Smem& S, Ring& ring,
                                             bool have) {
  if (__all_sync(kFull, have) && (threadIdx.x & 31) == 0)
    mbar_arrive(&S.empty[ring.slot]);
  __syncwarp();
  ring.advance(S.n_pages);
}

// ------------------------------------------------------------ tensors
__device__ __forceinline__ char* layer_base(const KernelParams& P, int l) {
  return P.act.base + (int64_t)l * P.act.layer_stride;
}
__device__ __forceinline__ char* global_base(const KernelParams& P) {
  return P.act.base + P.act.global_block;
}
template <typename T = uint16_t>
__device__ __forceinline__ T* lt(const KernelParams& P, int l, int64_t off) {
  return reinterpret_cast<T*>(layer_base(P, l) + off);
}
__device__ __forceinline__ const uint16_t* layer_w(const KernelParams& P,
                                                   int l, int which) {
  return P.w.layers[l * MPK_LAYER_NTENSORS + which];
}

// ------------------------------------------------------------ MatMul tiles
__device__ __forceinline__ bool is_gemv(int kind) {
  return kind == MPK_TASK_QKV || kind == MPK_TASK_O ||
         kind == MPK_TASK_GATEUP || kind == MPK_TASK_DOWN ||
         kind == MPK_TASK_LM_HEAD || kind == MPK_TASK_CHAIN_UP ||
         kind == MPK_TASK_CHAIN_DOWN;
}

// Geometry of one MatMul task.
// Batch 1: the tile's rows are streamed as contiguous pages (a gate/up
// tile: its gate rows, then its up rows), `pph` pages per half: flat pages
// of 16384 elements, or pages of `rpp` whole rows; row partial sums land in
// S.res[(half * rows + o) * wpr + part].
// Batch > 1: pages of 8 matrix rows (gate/up tiles: 4 gate rows then the
// matching 4 up rows) by at most 2048 columns, column segments outer (one
// segment of every sequence's activation is staged at a time); results land
// in S.res[b * RP + page row].
struct Gemv {
  int kind, layer;
  int row0, rows;       // output rows [row0, row0 + rows)
  int K, N;             // reduction length, output width
  int dual, up_off;
  int b1, rpp, wpr, pph;
  int ngroups, nsegs;
  const uint16_t* W;
};

__device__ Gemv gemv_geom(const KernelParams& P, const TaskDesc& t) {
  const Dims& D = P.dims;
  Gemv g;
  g.kind = t.kind;
  g.layer = t.layer;
  g.row0 = t.row0;
  g.rows = t.row1 - t.row0;
  g.dual = 0;
  g.up_off = 0;
  const int l = t.layer;
  switch (t.kind) {
    case MPK_TASK_QKV:
      g.K = D.h;
      g.N = (D.Hq + 2 * D.Hkv) * D.d;
      g.W = layer_w(P, l, MPK_W_QKV);
      break;
    case MPK_TASK_O:
      g.K = D.Hq * D.d;
      g.N = D.h;
      g.W = layer_w(P, l, MPK_W_O);
      break;
    case MPK_TASK_GATEUP:
      g.K = D.h;
      g.N = D.F;
      g.dual = 1;
      g.up_off = D.F;
      g.W = layer_w(P, l, MPK_W_GATEUP);
      break;
    case MPK_TASK_DOWN:
      g.K = D.F;
      g.N = D.h;
      g.W = layer_w(P, l, MPK_W_DOWN);
      break;
    case MPK_TASK_LM_HEAD:
      g.K = D.h;
      g.N = D.V;
      g.W = P.w.lm_head;
      break;
    case MPK_TASK_CHAIN_UP:
      g.K = D.h;
      g.N = D.chain_ffn;
      g.W = P.w.chain_w1;
      break;
    default:  // MPK_TASK_CHAIN_DOWN
      g.K = D.chain_ffn;
      g.N = D.h;
      g.W = P.w.chain_w2;
      break;
  }
  const int gsize = g.dual ? 4 : kPageRows;
  g.ngroups = (g.rows + gsize - 1) / gsize;
  g.nsegs = (g.K + kSegCols - 1) / kSegCols;
  g.b1 = D.B == 1 ? 1 : 0;
  g.rpp = b1_rows_per_page(g.K);
  g.wpr = b1_warps_per_row(g.K);
  g.pph = (g.rows + g.rpp - 1) / g.rpp;
  return g;
}

__device__ __forceinline__ int gemv_pages(const Gemv& g) {
  return g.b1 ? (g.dual ? 2 : 1) * g.pph : g.ngroups * g.nsegs;
}

// Batch 1: page p of half `half` starts `e0` elements into that half's
// row stream and holds `ne` elements; returns the address of its first one.
__device__ __forceinline__ const uint16_t* b1_page(const Gemv& g, int p,
                                                   int& half, int64_t& e0,
                                                   int& ne) {
  half = p / g.pph;
  const int q = p - half * g.pph;
  const int64_t total = (int64_t)g.rows * g.K;
  e0 = (int64_t)q * g.rpp * g.K;
  const int64_t span = (int64_t)g.rpp * g.K;
  ne = (int)min(span, total - e0);
  return g.W + ((int64_t)(half ? g.up_off : 0) + g.row0) * g.K + e0;
}

// Batch > 1: page p is row group j of column segment s.
__device__ __forceinline__ void page_coords(const Gemv& g, int p, int& j,
                                            int& s) {
  s = p / g.ngroups;
  j = p - s * g.ngroups;
}
// Weight-matrix row held in row i (0..7) of group j's pages.
__device__ __forceinline__ int page_wrow(const Gemv& g, int j, int i,
                                         bool& valid) {
  if (g.dual) {
    const int o = 4 * j + (i & 3);
    valid = o < g.rows;
    return (i < 4 ? 0 : g.up_off) + g.row0 + o;
  }
  const int o = kPageRows * j + i;
  valid = o < g.rows;
  return g.row0 + o;
}

// ------------------------------------------------------------ producer
// Weight page p of a MatMul task: one bulk copy per valid row, issued by
// lanes 0..7 after lane 0 posts the byte count.
__device__ void issue_gemv_page(const Gemv& g, int p, uint8_t* page,
                                uint64_t* bar, uint64_t policy) {
  const int lane = threadIdx.x & 31;
  if (g.b1) {
    // one contiguous copy of n whole rows
    if (lane == 0) {
      int half, ne;
      int64_t e0;
      const uint16_t* src = b1_page(g, p, half, e0, ne);
      const uint32_t bytes = (uint32_t)ne * 2u;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(page, src, bytes, bar, policy);
    }
    return;
  }
  int j, s;
  page_coords(g, p, j, s);
  const int c0 = s * kSegCols;
  const uint32_t bytes = (uint32_t)min(kSegCols, g.K - c0) * 2u;
  bool valid = false;
  int wr = 0;
  if (lane < kPageRows) wr = page_wrow(g, j, lane, valid);
  const uint32_t vmask = __ballot_sync(kFull, valid);
  if (lane == 0) mbar_arrive_expect_tx(bar, __popc(vmask) * bytes);
  __syncwarp();
  if (valid)
    bulk_g2s(page + lane * kPagePitch, g.W + (int64_t)wr * g.K + c0, bytes,
             bar, policy);
}
// Chunk c of (b, g) covers tokens [t0, t1) of the n = seq_len + 1 positions.
__device__ __forceinline__ void chunk_range(int c, int n, int C, int& t0,
                                            int& t1) {
  t0 = (int)(((int64_t)c * n) / C);
  t1 = (int)(((int64_t)(c + 1) * n) / C);
}

// KV chunk of an AOT attention task: the cached tokens [t0, min(t1, pos))
// into the K page (which == 0) or the V page (which == 1) as token-major
// rows of d values, one bulk copy per run of tokens inside one KV page.
// Lane 0 only.
__device__ void issue_attn_page(const KernelParams& P, const TaskDesc& t,
                                int which, uint8_t* page, uint64_t* bar,
                                uint64_t policy, int2* meta) {
  const Dims& D = P.dims;
  const int b = t.b, pos = __ldcg(P.step.seq_lens + b);
  const int n = pos + 1;
  int t0 = 0, t1 = 0;
  const bool ok = pos >= 0 && n <= D.max_ctx;
  if (ok) chunk_range(t.c, n, D.C, t0, t1);
  const int te = ok ? min(min(t1, pos), t0 + kAttnMaxTokens) : 0;
  const int P_ = D.page_size, d = D.d;
  const uint32_t row_bytes = (uint32_t)d * 2u;
  const int32_t* pt = P.step.page_table + (int64_t)b * D.max_pages;
  if (meta) {
    // the consumers read these after the K page's arrival (the arrive
    // below releases them)
    const int pidx = ok ? pos / P_ : D.max_pages;
    *meta = make_int2(pos, pidx < D.max_pages ? __ldg(pt + pidx) : -1);
  }
  const int64_t head_elems = (int64_t)P_ * d;
  const int64_t layer_elems =
      (int64_t)t.layer * P.step.num_pages * D.Hkv * head_elems;
  const uint16_t* pool = which ? P.step.v_pool : P.step.k_pool;
  uint32_t total = 0;
  for (int tok = t0; tok < te;) {
    const int run_end = min(te, (tok / P_ + 1) * P_);
    const int pg = __ldg(pt + tok / P_);
    if (pg >= 0 && pg < P.step.num_pages)
      total += (uint32_t)(run_end - tok) * row_bytes;
    else
      raise_error(P, MPK_ERR_KV_PAGE);
    tok = run_end;
  }
  mbar_arrive_expect_tx(bar, total);
  for (int tok = t0; tok < te;) {
    const int run_end = min(te, (tok / P_ + 1) * P_);
    const int pg = __ldg(pt + tok / P_);
    if (pg >= 0 && pg < P.step.num_pages) {
      const int64_t off = layer_elems + ((int64_t)pg * D.Hkv + t.g) * head_elems +
                          (int64_t)(tok % P_) * d;
      bulk_g2s(page + (size_t)(tok - t0) * row_bytes, pool + off,
               (uint32_t)(run_end - tok) * row_bytes, bar, policy);
    }
    tok = run_end;
  }
}

// After an abort: wait (bounded) until every copy this producer issued has
// landed, so no bulk copy writes into shared memory after the CTA exits.
__device__ void drain_copies(const KernelParams& P, const Smem& S,
                             const uint32_t* issued) {
  if ((threadIdx.x & 31) != 0) return;
  const uint64_t limit = globaltimer() + 200000000ull;  // 200 ms
  for (int s = 0; s < S.n_pages; ++s) {
    if (!(issued[s] & 1u)) continue;
    const uint32_t ph = (issued[s] >> 1) & 1u;
    while (!mbar_try_wait(&S.full[s], ph)) {
      if (globaltimer() > limit) return;
    }
  }
}

// Pages a task takes from the ring (0 for tasks that use none).
__device__ __forceinline__ int ring_pages_of(const KernelParams& P,
                                             const TaskDesc& t, Gemv* g) {
  if (is_gemv(t.kind)) {
    *g = gemv_geom(P, t);
    return gemv_pages(*g);
  }
  if (t.kind == MPK_TASK_ATTN && t.launch == MPK_LAUNCH_AOT) return 2;
  return 0;
}

// Bounded wait for a free ring slot by lane 0; every lane then observes the
// released phase before any copy into the slot is issued.
__device__ __forceinline__ bool wait_empty(const KernelParams& P,
                                           const Smem& S, const Ring& ring,
                                           uint64_t deadline) {
  const int lane = threadIdx.x & 31;
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
  }
  ok = __shfl_sync(kFull, ok, 0);
  if (ok) (void)mbar_try_wait(&S.empty[ring.slot], ring.phase ^ 1u);
  return ok != 0;
}

// Producer warp `pid` of kProducerWarps: walks the task list and issues
// the pages whose global index gp (over the whole list) has
// gp % kProducerWarps == pid.  The ring position advances by one for every
// page, issued here or by the other producer, so page gp lands in slot
// gp % n_pages with phase (gp / n_pages) & 1 -- the order in which the
// consumers take them.
__device__ void producer_role(const KernelParams& P, const Smem& S,
                              const int32_t* list, int n, int steps,
                              uint64_t deadline, int pid) {
  static_assert(kProducerWarps == 2, "page ownership alternates");
  const int lane = threadIdx.x & 31;
  uint32_t issued[kMaxRingPages];
#pragma unroll
  for (int i = 0; i < kMaxRingPages; ++i) issued[i] = 0;
  const uint64_t policy = evict_first_policy();
  Ring ring{0, 0};
  int64_t gp = 0;
  int turn = 0;            // gp % 2
  // the list is walked once per step of the launch; weight pages of the
  // next step stream in while this one ends, but cached K/V (whose position
  // the step before advances) only after that step's end event
  for (int step = 0, i = 0; step < steps; ++i) {
    if (i == n) {
      if (++step == steps) break;
      i = -1;
      continue;
    }
    const TaskDesc t = P.graph.tasks[list[i]];
    Gemv g;
    const int np = ring_pages_of(P, t, &g);
    if (np > 0 && step > 0 && t.kind == MPK_TASK_ATTN) {
      int ok = 1;
      if (lane == 0) {
        uint32_t spins = 0;
        while (!event_done_acq(P, P.graph.end, P.step.epoch + step - 1)) {
          if ((++spins & 255u) == 0u &&
              (aborted(P) || globaltimer() > deadline)) {
            if (!aborted(P)) raise_error(P, MPK_ERR_TIMEOUT);
            ok = 0;
            break;
          }
        }
      }
      if (!__shfl_sync(kFull, ok, 0)) {
        drain_copies(P, S, issued);
        return;
      }
    }
    // batch-1 weight pages: source pointer and length advance linearly
    const bool lin = np > 0 && is_gemv(t.kind) && g.b1;
    const int64_t span = lin ? (int64_t)g.rpp * g.K : 0;
    const int64_t total = (int64_t)g.rows * g.K;
    int64_t e0 = 0;
    int half = 0;
    for (int p = 0; p < np; ++p, ++gp, turn ^= 1, ring.advance(S.n_pages)) {
      const bool mine = turn == pid;
      const int64_t my_e0 = e0;
      const int my_half = half;
      if (lin) {   // advance to the next page of the half (or the next half)
        e0 += span;
        if (e0 >= total) {
          e0 = 0;
          ++half;
        }
      }
      if (!mine) continue;
      if (!wait_empty(P, S, ring, deadline)) {
        drain_copies(P, S, issued);
        return;
      }
      uint8_t* page = page_ptr(S, ring.slot);
      uint64_t* bar = &S.full[ring.slot];
      if (lin) {
        if (lane == 0) {
          const uint32_t bytes = (uint32_t)min(span, total - my_e0) * 2u;
          const uint16_t* src =
              g.W + ((int64_t)(my_half ? g.up_off : 0) + g.row0) * g.K + my_e0;
          mbar_arrive_expect_tx(bar, bytes);
          bulk_g2s(page, src, bytes, bar, policy);
        }
      } else if (is_gemv(t.kind)) {
        issue_gemv_page(g, p, page, bar, policy);
      } else if (lane == 0) {
        issue_attn_page(P, t, p, page, bar, policy,   // p 0: K, 1: V
                        p == 0 ? &S.meta[ring.slot] : nullptr);
      }
      __syncwarp();
      issued[ring.slot] = 1u | (ring.phase << 1);
    }
  }
  // the consumers wait for every page before leaving, so all copies have
  // landed by the time the CTA exits unless the step aborted
  if (aborted(P)) drain_copies(P, S, issued);
}

// ------------------------------------------------------------ x staging
// Where a MatMul tile's activation row comes from.  Norm modes form the
// residual sum (or gather the embedding row), round it to bf16, and RMSNorm
// it with `gain`; tile 0 also stores the residual for later operators.
enum { X_PLAIN = 0, X_NORM_ADD = 1, X_NORM_EMBED = 2 };
struct XSrc {
  int mode;
  const int32_t* tok;     // embedding mode: this step's tokens
  const uint16_t* a;      // plain source, or first addend
  const uint16_t* c;      // second addend
  const uint16_t* gain;
  uint16_t* resid;        // residual output (tile 0 only), else null
};

// Tokens step `step` of the launch embeds: the caller's for step 0, else
// those step - 1 produced.
__device__ __forceinline__ const int32_t* step_tokens(const KernelParams& P,
                                                      int step) {
  return step == 0 ? P.step.tokens
                   : P.step.next_tokens + (int64_t)(step - 1) * P.dims.B;
}

__device__ XSrc x_source(const KernelParams& P, const TaskDesc& t,
                         int step = 0) {
  const Dims& D = P.dims;
  const int l = t.layer;
  const bool res = (t.flags & TASK_F_RESIDUAL) != 0;
  XSrc x{X_PLAIN, step_tokens(P, step), nullptr, nullptr, nullptr, nullptr};
  switch (t.kind) {
    case MPK_TASK_QKV:
      x.gain = layer_w(P, l, MPK_W_LN1);
      if (res) x.resid = lt(P, l, P.act.o_h);
      if (l == 0) {
        x.mode = X_NORM_EMBED;
      } else {
        x.mode = X_NORM_ADD;
        x.a = lt(P, l - 1, P.act.o_hmid);
        x.c = lt(P, l - 1, P.act.o_dout);
      }
      break;
    case MPK_TASK_O:
      x.a = lt(P, l, P.act.o_attn);
      break;
    case MPK_TASK_GATEUP:
      x.mode = X_NORM_ADD;
      x.a = lt(P, l, P.act.o_h);
      x.c = lt(P, l, P.act.o_o);
      x.gain = layer_w(P, l, MPK_W_LN2);
      if (res) x.resid = lt(P, l, P.act.o_hmid);
      break;
    case MPK_TASK_DOWN:
      x.a = lt(P, l, P.act.o_act);
      break;
    case MPK_TASK_LM_HEAD:
      if (D.chain_ffn > 0) {
        x.a = reinterpret_cast<const uint16_t*>(global_base(P) + P.act.g_z);
      } else {
        x.mode = X_NORM_ADD;
        x.a = lt(P, D.L - 1, P.act.o_hmid);
        x.c = lt(P, D.L - 1, P.act.o_dout);
        x.gain = P.w.final_norm;
        if (res) x.resid = lt(P, D.L, P.act.o_h);
      }
      break;
    case MPK_TASK_CHAIN_UP:
      x.mode = X_NORM_EMBED;
      x.gain = P.w.final_norm;
      break;
    default:  // MPK_TASK_CHAIN_DOWN
      x.a = lt(P, 0, P.act.o_act);
      break;
  }
  return x;
}

// Prefetch into L2 the RMSNorm gain of a MatMul task's prologue (a weight,
// independent of any event), so the prologue after the event finds it
// there.  One thread.
__device__ __forceinline__ void prefetch_gain(const KernelParams& P,
                                              const TaskDesc& t) {
  if (!is_gemv(t.kind)) return;
  const XSrc x = x_source(P, t);
  if (x.mode == X_PLAIN) return;
  const char* p = reinterpret_cast<const char*>(x.gain);
  for (int off = 0; off < P.dims.h * 2; off += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off) : "memory");
}

// Pre-norm values of 8 columns [k, k + 8) of sequence b from the raw words
// of the source(s): the embedding row, or the two addends of the residual
// sum (rounded to bf16, as the tensor is).
struct PreRaw {
  uint4 a, c;
};
__device__ __forceinline__ void pre_finish(const XSrc& x, const PreRaw& r,
                                           float (&v)[8]) {
  const uint32_t* pa = &r.a.x;
  const uint32_t* pc = &r.c.x;
  if (x.mode == X_NORM_EMBED) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[2 * q] = bf_lo(pa[q]);
      v[2 * q + 1] = bf_hi(pa[q]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[2 * q] = round_bf(__fadd_rn(bf_lo(pa[q]), bf_lo(pc[q])));
      v[2 * q + 1] = round_bf(__fadd_rn(bf_hi(pa[q]), bf_hi(pc[q])));
    }
  }
}
__device__ __forceinline__ void pre_values(const KernelParams& P,
                                           const XSrc& x, int b, int K, int k,
                                           float (&v)[8]) {
  PreRaw r;
  if (x.mode == X_NORM_EMBED) {
    int tok = __ldcg(x.tok + b);
    tok = min(max(tok, 0), P.dims.V - 1);
    r.a = __ldg(reinterpret_cast<const uint4*>(P.w.embed + (int64_t)tok * K +
                                               k));
    r.c = make_uint4(0, 0, 0, 0);
  } else {
    r.a = __ldcg(reinterpret_cast<const uint4*>(x.a + (int64_t)b * K + k));
    r.c = __ldcg(reinterpret_cast<const uint4*>(x.c + (int64_t)b * K + k));
  }
  pre_finish(x, r, v);
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]),
                    pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
}
// bf16((v * r) * w) for 8 columns (one rounding, the oracle's order).
__device__ __forceinline__ uint4 norm8(const float (&v)[8], float r,
                                       uint4 wv) {
  const uint32_t* pw = &wv.x;
  float o[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    o[2 * q] = __fmul_rn(__fmul_rn(v[2 * q], r), bf_lo(pw[q]));
    o[2 * q + 1] = __fmul_rn(__fmul_rn(v[2 * q + 1], r), bf_hi(pw[q]));
  }
  return pack8(o);
}
__device__ __forceinline__ float rms_factor(float ss, int K, float eps) {
  return 1.0f / sqrtf(ss / (float)K + eps);
}

// Batch 1: all K columns of x go to S.xs as bf16 (chunk c = columns
// 8c .. 8c + 7 at 16-byte word c); the MatMul loop widens them once per tile
// into registers, so the staging costs half the shared memory of fp32 and
// leaves room for one more weight page.
__device__ __forceinline__ void widen8(uint4 v, float4& a, float4& b) {
  a = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
  b = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
}

__device__ void stage_x_b1(const KernelParams& P, const Smem& S,
                           const TaskDesc& t, const Gemv& g) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const XSrc x = x_source(P, t, S.ctrl[14]);
  const int K = g.K, nch = K >> 3;
  uint4* xs = reinterpret_cast<uint4*>(S.xs);
  if (x.mode == X_PLAIN) {
    for (int ch = tid; ch < nch; ch += kConsumers)
      xs[ch] = __ldcg(reinterpret_cast<const uint4*>(x.a) + ch);
    consumer_sync();
    return;
  }
  constexpr int kMaxChunks = 4;  // K <= 8192 for normed operators
  float v[kMaxChunks][8];
  uint4 wv[kMaxChunks];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int ch = tid + k * kConsumers;
    if (ch < nch) {
      wv[k] = __ldg(reinterpret_cast<const uint4*>(x.gain) + ch);
      pre_values(P, x, 0, K, ch * 8, v[k]);
#pragma unroll
      for (int q = 0; q < 8; ++q) ss = fmaf(v[k][q], v[k][q], ss);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) S.scratch[warp] = ss;
  consumer_sync();
  float tot = 0.f;
#pragma unroll
  for (int q = 0; q < kConsumerWarps; ++q) tot += S.scratch[q];
  const float r = rms_factor(tot, K, P.dims.eps);
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int ch = tid + k * kConsumers;
    if (ch < nch) {
      xs[ch] = norm8(v[k], r, wv[k]);
      if (x.resid) reinterpret_cast<uint4*>(x.resid)[ch] = pack8(v[k]);
    }
  }
  consumer_sync();
}

// Batch > 1, norm modes: the RMS factor of every sequence into
// S.scratch[32 + b] (warp w takes sequences w, w + 8, ...); tile 0 stores the
// residual.  The input words are brought into the x buffer (not yet staged)
// with asynchronous 16-byte copies, 1024 columns of every sequence at a
// time, so all of a batch's loads are in flight together; each thread reads
// back only the chunks it copied itself.
__device__ void norm_stats(const KernelParams& P, const Smem& S,
                           const TaskDesc& t, const Gemv& g) {
  const XSrc x = x_source(P, t, S.ctrl[14]);
  if (x.mode == X_PLAIN) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = P.dims.B, K = g.K, nch = K >> 3;
  constexpr int CB = 128;   // chunks (of 8 columns) per sequence per batch
  uint4* ta = reinterpret_cast<uint4*>(S.xs);     // [B][CB]
  uint4* tc = ta + (size_t)B * CB;                 // [B][CB]
  float ss[2] = {0.f, 0.f};   // this lane's share for sequences warp, warp + 8
  for (int c0 = 0; c0 < nch; c0 += CB) {
    for (int q = 0; q < 2; ++q) {
      const int b = warp + q * kConsumerWarps;
      if (b >= B) break;
      const uint16_t* ra;
      if (x.mode == X_NORM_EMBED) {
        int tok = __ldcg(x.tok + b);
        tok = min(max(tok, 0), P.dims.V - 1);
        ra = P.w.embed + (int64_t)tok * K;
      } else {
        ra = x.a + (int64_t)b * K;
      }
      for (int ch = lane; ch < CB && c0 + ch < nch; ch += 32) {
        cp_async16(ta + b * CB + ch, ra + (c0 + ch) * 8);
        if (x.mode != X_NORM_EMBED)
          cp_async16(tc + b * CB + ch, x.c + (int64_t)b * K + (c0 + ch) * 8);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    for (int q = 0; q < 2; ++q) {
      const int b = warp + q * kConsumerWarps;
      if (b >= B) break;
      for (int ch = lane; ch < CB && c0 + ch < nch; ch += 32) {
        PreRaw raw;
        raw.a = ta[b * CB + ch];
        raw.c = x.mode != X_NORM_EMBED ? tc[b * CB + ch] : make_uint4(0, 0, 0, 0);
        float v[8];
        pre_finish(x, raw, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) ss[q] = fmaf(v[k], v[k], ss[q]);
        if (x.resid)
          reinterpret_cast<uint4*>(x.resid + (int64_t)b * K)[c0 + ch] = pack8(v);
      }
    }
  }
  for (int q = 0; q < 2; ++q) {
    const int b = warp + q * kConsumerWarps;
    const float tot = warp_sum(ss[q]);
    if (b < B && lane == 0) S.scratch[32 + b] = rms_factor(tot, K, P.dims.eps);
  }
  consumer_sync();
}

// Batch > 1: stage column segment s of every sequence into S.xs, row b at
// b * kPagePitch bytes; columns up to the next multiple of 16 are zeroed.
// Norm modes: the segment goes in quarters of 512 columns.  Each quarter's
// raw words arrive by asynchronous copies -- the first addend (or the
// embedding row) straight into its place in the row, the second addend
// into a scratch area after the rows -- and are then normalised in place.
constexpr int kSegQuarter = 64;   // chunks (of 8 columns)
__device__ void stage_x_seg(const KernelParams& P, const Smem& S,
                            const TaskDesc& t, const Gemv& g, int s) {
  const XSrc x = x_source(P, t, S.ctrl[14]);
  const int B = P.dims.B, K = g.K;
  const int c0 = s * kSegCols, cols = min(kSegCols, K - c0);
  const int nch = cols >> 3, nch16 = ((cols + 15) >> 4) << 1;
  auto row = [&](int b) {
    return reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(S.xs) +
                                    (size_t)b * kPagePitch);
  };
  consumer_sync();   // every warp is done with the previous segment
  // columns past the segment up to the next multiple of 16: zero
  for (int idx = threadIdx.x; idx < B * (nch16 - nch); idx += kConsumers) {
    const int b = idx / (nch16 - nch), ch = nch + idx % (nch16 - nch);
    row(b)[ch] = make_uint4(0, 0, 0, 0);
  }
  if (x.mode == X_PLAIN) {
    for (int idx = threadIdx.x; idx < B * nch; idx += kConsumers) {
      const int b = idx / nch, ch = idx - b * nch;
      cp_async16(row(b) + ch, x.a + (int64_t)b * K + c0 + ch * 8);
    }
    cp_async_commit();
    cp_async_wait_all();
    consumer_sync();
    return;
  }
  uint4* tmp = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(S.xs) +
                                        (size_t)B * kPagePitch);   // [B][64]
  const bool embed = x.mode == X_NORM_EMBED;
  for (int q0 = 0; q0 < nch; q0 += kSegQuarter) {
    const int nq = min(kSegQuarter, nch - q0);
    for (int idx = threadIdx.x; idx < B * nq; idx += kConsumers) {
      const int b = idx / nq, ch = q0 + idx % nq;
      const int64_t k = c0 + ch * 8;
      if (embed) {
        int tok = __ldcg(x.tok + b);
        tok = min(max(tok, 0), P.dims.V - 1);
        cp_async16(row(b) + ch, P.w.embed + (int64_t)tok * K + k);
      } else {
        cp_async16(row(b) + ch, x.a + (int64_t)b * K + k);
        cp_async16(tmp + b * kSegQuarter + (ch - q0), x.c + (int64_t)b * K + k);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    consumer_sync();
    for (int idx = threadIdx.x; idx < B * nq; idx += kConsumers) {
      const int b = idx / nq, ch = q0 + idx % nq;
      PreRaw raw;
      raw.a = row(b)[ch];
      raw.c = embed ? make_uint4(0, 0, 0, 0) : tmp[b * kSegQuarter + (ch - q0)];
      float v[8];
      pre_finish(x, raw, v);
      row(b)[ch] = norm8(v, S.scratch[32 + b],
                         __ldg(reinterpret_cast<const uint4*>(x.gain + c0) + ch));
    }
    consumer_sync();   // the scratch area is reused by the next quarter
  }
}

// ------------------------------------------------------------ epilogue
// The dot product of output row o (half 1: the up row of a gate/up tile)
// for sequence b, from the body's result buffer: at batch 1 the sum of the
// row's per-warp partials in a fixed order, else S.res[b * RP + page row].
__device__ __forceinline__ float res_get(const Smem& S, const Gemv& g, int b,
                                         int half, int o) {
  if (g.b1) {
    const float* q = S.res + ((size_t)half * g.rows + o) * g.wpr;
    float v = q[0];
    for (int s = 1; s < g.wpr; ++s) v += q[s];
    return v;
  }
  const int RP = g.ngroups * kPageRows;
  const int pr = g.dual ? 8 * (o >> 2) + 4 * half + (o & 3) : o;
  return S.res[b * RP + pr];
}

// Write the operator's output from the row results.
__device__ void gemv_epilogue(const KernelParams& P, const Smem& S,
                              const TaskDesc& t, const Gemv& g) {
  const Dims& D = P.dims;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = D.B, R = g.rows;
  const int l = g.layer;
  for (int idx = tid; idx < B * R; idx += kConsumers) {
    const int b = idx / R, o = idx - b * R;
    const int orow = g.row0 + o;
    if (g.dual) {
      const float gv = round_bf(res_get(S, g, b, 0, o));
      const float uv = round_bf(res_get(S, g, b, 1, o));
      lt(P, l, P.act.o_act)[(int64_t)b * g.N + orow] =
          f2bf(__fmul_rn(silu_f(gv), uv));
      continue;
    }
    const float v = res_get(S, g, b, 0, o);
    switch (g.kind) {
      case MPK_TASK_LM_HEAD:
        P.step.logits[(int64_t)b * g.N + orow] = v;
        break;
      case MPK_TASK_CHAIN_UP:
        lt(P, 0, P.act.o_act)[(int64_t)b * g.N + orow] =
            f2bf(silu_f(round_bf(v)));
        break;
      case MPK_TASK_QKV:
        lt(P, l, P.act.o_qkv)[(int64_t)b * g.N + orow] = f2bf(v);
        break;
      case MPK_TASK_O:
        lt(P, l, P.act.o_o)[(int64_t)b * g.N + orow] = f2bf(v);
        break;
      case MPK_TASK_DOWN:
        lt(P, l, P.act.o_dout)[(int64_t)b * g.N + orow] = f2bf(v);
        break;
      default:  // MPK_TASK_CHAIN_DOWN
        reinterpret_cast<uint16_t*>(global_base(P) +
                                    P.act.g_z)[(int64_t)b * g.N + orow] =
            f2bf(v);
        break;
    }
  }
  if (g.kind != MPK_TASK_LM_HEAD) return;
  // tile argmax (lowest index among equal maxima)
  float2* am = reinterpret_cast<float2*>(global_base(P) + P.act.g_amax);
  if (B == 1) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int o = tid; o < R; o += kConsumers) {
      const float v = res_get(S, g, 0, 0, o);
      if (better(v, g.row0 + o, bv, bi)) {
        bv = v;
        bi = g.row0 + o;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      S.scratch[64 + warp] = bv;
      S.scratch[80 + warp] = __int_as_float(bi);
    }
    consumer_sync();
    if (tid == 0) {
      for (int w = 1; w < kConsumerWarps; ++w) {
        const float ov = S.scratch[64 + w];
        const int oi = __float_as_int(S.scratch[80 + w]);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      am[t.tile] = make_float2(bv, __int_as_float(bi));
    }
    return;
  }
  for (int b = warp; b < B; b += kConsumerWarps) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int o = lane; o < R; o += 32) {
      const float v = res_get(S, g, b, 0, o);
      if (better(v, g.row0 + o, bv, bi)) {
        bv = v;
        bi = g.row0 + o;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0)
      am[(int64_t)b * D.n_lm_tiles + t.tile] =
          make_float2(bv, __int_as_float(bi));
  }
}

// ------------------------------------------------------------ MatMul bodies
// Dot product of one row's chunks [c0, c1) (8 columns each) with the fp32
// x planes (xa: first four columns of each chunk, xb: last four), one warp:
// lane reads chunks lane, lane + 32, ...; paired fp32 FMAs (__ffma2_rn)
// into eight independent partial sums.
__device__ __forceinline__ void fma8(uint4 w, float4 x0, float4 x1, float2& a,
                                     float2& b) {
  a = __ffma2_rn(make_float2(bf_lo(w.x), bf_hi(w.x)), make_float2(x0.x, x0.y), a);
  b = __ffma2_rn(make_float2(bf_lo(w.y), bf_hi(w.y)), make_float2(x0.z, x0.w), b);
  a = __ffma2_rn(make_float2(bf_lo(w.z), bf_hi(w.z)), make_float2(x1.x, x1.y), a);
  b = __ffma2_rn(make_float2(bf_lo(w.w), bf_hi(w.w)), make_float2(x1.z, x1.w), b);
}
__device__ __forceinline__ float row_dot(const uint4* row, const uint4* xs,
                                         int c0, int c1) {
  const int lane = threadIdx.x & 31;
  float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
  int ch = c0 + lane;
  float4 x0, x1, x2, x3;
  for (; ch + 32 < c1; ch += 64) {
    widen8(xs[ch], x0, x1);
    widen8(xs[ch + 32], x2, x3);
    fma8(row[ch], x0, x1, a0, a1);
    fma8(row[ch + 32], x2, x3, a2, a3);
  }
  if (ch < c1) {
    widen8(xs[ch], x0, x1);
    fma8(row[ch], x0, x1, a0, a1);
  }
  return warp_sum(((a0.x + a0.y) + (a1.x + a1.y)) +
                  ((a2.x + a2.y) + (a3.x + a3.y)));
}

// Dot of this lane's NCK chunks row[lane + 32 k] with the x chunks held in
// registers (two float4 halves per chunk), summed over the warp.
template <int NCK>
__device__ __forceinline__ float row_dot_xreg(const uint4* row,
                                              const float4 (&xr)[16]) {
  const int lane = threadIdx.x & 31;
  float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
  uint4 w[NCK > 0 ? NCK : 1];
#pragma unroll
  for (int k = 0; k < NCK; ++k) w[k] = row[lane + 32 * k];
#pragma unroll
  for (int k = 0; k < NCK; ++k) {
    if (k & 1) fma8(w[k], xr[2 * k], xr[2 * k + 1], a2, a3);
    else fma8(w[k], xr[2 * k], xr[2 * k + 1], a0, a1);
  }
  return warp_sum(((a0.x + a0.y) + (a1.x + a1.y)) +
                  ((a2.x + a2.y) + (a3.x + a3.y)));
}

// One batch-1 page of whole rows [i0, i0 + n).  With NCK > 0 this warp's x
// part (NCK 32-chunk strides) is in registers; NCK == 0 reads x from shared
// memory.
template <int NCK>
__device__ __forceinline__ void b1_page_rows(const uint4* pg, float* out,
                                             const Gemv& g, int i0, int n,
                                             bool multi, int part, int nch,
                                             int c0, int c1, const uint4* xs,
                                             const float4 (&xr)[16]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (multi) {
    for (int r = warp; r < n; r += kConsumerWarps) {
      const uint4* row = pg + (size_t)r * nch;
      const float v = NCK > 0 ? row_dot_xreg<NCK>(row, xr)
                              : row_dot(row, xs, 0, nch);
      if (lane == 0) out[i0 + r] = v;
    }
  } else {
    const int r = warp / g.wpr;
    if (r < n) {
      const uint4* row = pg + (size_t)r * nch;
      const float v = NCK > 0 ? row_dot_xreg<NCK>(row + c0, xr)
                              : row_dot(row, xs, c0, c1);
      if (lane == 0) out[(i0 + r) * g.wpr + part] = v;
    }
  }
}

// Batch 1.  Pages hold whole rows.  With 8 or more rows per page warp w
// takes rows w, w + 8, ...; with fewer, each row is split over wpr warps into
// column parts of equal length and warp w always takes part w % wpr.  When
// a warp's part is 1, 2, 4, 6 or 8 strides of 32 chunks, its x values stay
// in registers for the whole tile and the loop reads only the weights from
// shared memory.
template <int NCK>
__device__ void gemv_b1_loop(const KernelParams& P, const Smem& S,
                             const Gemv& g, Ring& ring, uint64_t deadline,
                             bool multi, int part, int nch, int c0, int c1) {
  const int lane = threadIdx.x & 31;
  const uint4* xs = reinterpret_cast<const uint4*>(S.xs);
  float4 xr[16];
#pragma unroll
  for (int k = 0; k < NCK; ++k)
    widen8(xs[c0 + lane + 32 * k], xr[2 * k], xr[2 * k + 1]);
  const int halves = g.dual ? 2 : 1;
  for (int half = 0; half < halves; ++half) {
    float* out = S.res + (size_t)half * g.rows * g.wpr;
    for (int i0 = 0; i0 < g.rows; i0 += g.rpp) {
      const int n = min(g.rpp, g.rows - i0);
      const bool have = wait_full(P, S, ring, deadline);
      if (have)
        b1_page_rows<NCK>(
            reinterpret_cast<const uint4*>(page_ptr(S, ring.slot)), out, g,
            i0, n, multi, part, nch, c0, c1, xs, xr);
      release_page(S, ring, have);
    }
  }
}

__device__ void gemv_b1(const KernelParams& P, const Smem& S,
                        const TaskDesc& t, const Gemv& g, Ring& ring,
                        uint64_t deadline) {
  stage_x_b1(P, S, t, g);
  stamp(P, S, 2);
  const int warp = threadIdx.x >> 5;
  const int nch = g.K >> 3;
  const bool multi = g.rpp >= kPageRows;
  const int part = multi ? 0 : warp % g.wpr;
  const int cpw = multi ? nch : (nch + g.wpr - 1) / g.wpr;
  const int c0 = part * cpw, c1 = min(nch, c0 + cpw);
  const bool even = (cpw & 31) == 0 && (multi || nch % g.wpr == 0);
  switch (even ? cpw >> 5 : 0) {
    case 8: gemv_b1_loop<8>(P, S, g, ring, deadline, multi, part, nch, c0, c1); break;
    case 6: gemv_b1_loop<6>(P, S, g, ring, deadline, multi, part, nch, c0, c1); break;
    case 4: gemv_b1_loop<4>(P, S, g, ring, deadline, multi, part, nch, c0, c1); break;
    case 2: gemv_b1_loop<2>(P, S, g, ring, deadline, multi, part, nch, c0, c1); break;
    case 1: gemv_b1_loop<1>(P, S, g, ring, deadline, multi, part, nch, c0, c1); break;
    default: gemv_b1_loop<0>(P, S, g, ring, deadline, multi, part, nch, c0, c1); break;
  }
  consumer_sync();
  stamp(P, S, 3);
  gemv_epilogue(P, S, t, g);
}

// A tile with more row groups than a body keeps accumulators for cannot be
// built by the host (its row cap); should one arrive anyway, its surplus
// pages are consumed unread and the step reports MPK_ERR_UNSUPPORTED, so the
// ring stays in step with the producer.
__device__ void skip_extra_groups(const KernelParams& P, const Smem& S,
                                  const Gemv& g, int kept, Ring& ring,
                                  uint64_t deadline) {
  if (g.ngroups <= kept) return;
  if (threadIdx.x == 0) raise_error(P, MPK_ERR_UNSUPPORTED);
  for (int j = kept; j < g.ngroups; ++j)
    release_page(S, ring, wait_full(P, S, ring, deadline));
}

// Batch 2..7 on CUDA cores: column segments outer; warp w owns row w of
// every page; up to 8 row groups per tile.
template <int NB>
__device__ void gemv_cc(const KernelParams& P, const Smem& S,
                        const TaskDesc& t, const Gemv& g, Ring& ring,
                        uint64_t deadline) {
  constexpr int kMaxGroups = 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = P.dims.B, RP = g.ngroups * kPageRows;
  norm_stats(P, S, t, g);
  float acc[kMaxGroups][NB];
#pragma unroll
  for (int j = 0; j < kMaxGroups; ++j)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[j][b] = 0.f;
  for (int s = 0; s < g.nsegs; ++s) {
    stage_x_seg(P, S, t, g, s);
    const int nch = min(kSegCols, g.K - s * kSegCols) >> 3;
#pragma unroll
    for (int j = 0; j < kMaxGroups; ++j) {
      if (j < g.ngroups) {
        bool valid;
        page_wrow(g, j, warp, valid);
        const bool have = wait_full(P, S, ring, deadline);
        if (have && valid) {
          const uint4* row = reinterpret_cast<const uint4*>(
              page_ptr(S, ring.slot) + warp * kPagePitch);
          for (int ch = lane; ch < nch; ch += 32) {
            const uint4 wv = row[ch];
#pragma unroll
            for (int b = 0; b < NB; ++b)
              if (b < B)
                acc[j][b] = dot8(wv,
                                 reinterpret_cast<const uint4*>(
                                     reinterpret_cast<const uint8_t*>(S.xs) +
                                     (size_t)b * kPagePitch)[ch],
                                 acc[j][b]);
          }
        }
        release_page(S, ring, have);
      }
    }
    skip_extra_groups(P, S, g, kMaxGroups, ring, deadline);
  }
#pragma unroll
  for (int j = 0; j < kMaxGroups; ++j)
    if (j < g.ngroups)
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (b < B) {
          const float v = warp_sum(acc[j][b]);
          if (lane == 0) S.res[b * RP + j * kPageRows + warp] = v;
        }
  consumer_sync();
  gemv_epilogue(P, S, t, g);
}

// Batch >= 8 on tensor cores: mma.sync m16n8k16 with the sequences as M
// (rows >= batch repeat the last sequence and are discarded) and a page's 8
// weight rows as N.  Column segments outer.  Every warp takes its own
// 256 columns (16 k-steps) of every page, so all 8 warps consume each page
// together and the ring drains as fast as it fills.  At the end the 8
// per-warp partial sums of every output are added in warp order.
__device__ void gemv_mma(const KernelParams& P, const Smem& S,
                         const TaskDesc& t, const Gemv& g, Ring& ring,
                         uint64_t deadline) {
  constexpr int kMaxGroups = 16;
  constexpr int kKS = kSegCols / 16 / kConsumerWarps;   // k-steps a warp
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int B = P.dims.B, RP = g.ngroups * kPageRows;
  norm_stats(P, S, t, g);
  stamp(P, S, 2);
  float acc[kMaxGroups][4];
#pragma unroll
  for (int j = 0; j < kMaxGroups; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
  // ldmatrix row addresses: A = x rows (sequences), B = page rows
  const int arow = min((lane & 7) + ((lane >> 3) & 1) * 8, B - 1);
  const uint32_t a_base = smem_addr(S.xs) + arow * kPagePitch +
                          ((lane >> 4) * 8) * 2 + warp * kKS * 32;
  const uint32_t b_off = (lane & 7) * kPagePitch + ((lane >> 3) * 8) * 2 +
                         warp * kKS * 32;
  const int kq = (lane & 3) * 2;   // this lane's k within an 8-column block
  for (int s = 0; s < g.nsegs; ++s) {
    stage_x_seg(P, S, t, g, s);
    const int cols = min(kSegCols, g.K - s * kSegCols);
    const int nks = min(kKS, ((cols + 15) >> 4) - warp * kKS);   // may be <= 0
    const int kc = cols - warp * kKS * 16;   // columns left from this slice
#pragma unroll
    for (int j = 0; j < kMaxGroups; ++j) {
      if (j < g.ngroups) {
        const bool have = wait_full(P, S, ring, deadline);
        if (have && nks > 0) {
          const uint32_t pb = smem_addr(page_ptr(S, ring.slot)) + b_off;
          // two chains (even and odd k-steps), joined after the page
          float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < kKS; kk += 2) {
            if (kk < nks) {
              uint32_t b0, b1, b2, b3, x0, x1, x2, x3;
              ldsm_x4(pb + kk * 32, b0, b1, b2, b3);
              ldsm_x4(a_base + kk * 32, x0, x1, x2, x3);
              const int kb = kk * 16 + kq;
              if (kb >= kc) b0 = 0u;
              if (kb + 8 >= kc) b1 = 0u;
              mma_16816(e0, x0, x1, x2, x3, b0, b1);
              if (kk + 1 < nks) {
                ldsm_x4(a_base + kk * 32 + 32, x0, x1, x2, x3);
                if (kb + 16 >= kc) b2 = 0u;
                if (kb + 24 >= kc) b3 = 0u;
                mma_16816(e1, x0, x1, x2, x3, b2, b3);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] += e0[e] + e1[e];
        }
        release_page(S, ring, have);
      }
    }
    skip_extra_groups(P, S, g, kMaxGroups, ring, deadline);
  }
  stamp(P, S, 3);
  // per-warp partials [warp][B][RP] in the x buffer (8 * B * 128 floats fit
  // in its B * (kPagePitch + 1024) bytes), once every warp is done with x
  consumer_sync();
  float* part = reinterpret_cast<float*>(S.xs);
  const int BR = B * RP;
  // D fragment: rows (sequences) lane/4 and lane/4 + 8, columns (page rows)
  // (lane % 4) * 2 and + 1
  const int bq = lane >> 2, nq = (lane & 3) * 2;
#pragma unroll
  for (int j = 0; j < kMaxGroups; ++j) {
    if (j < g.ngroups) {
      float* q = part + warp * BR + j * kPageRows + nq;
      if (bq < B) {
        q[bq * RP] = acc[j][0];
        q[bq * RP + 1] = acc[j][1];
      }
      if (bq + 8 < B) {
        q[(bq + 8) * RP] = acc[j][2];
        q[(bq + 8) * RP + 1] = acc[j][3];
      }
    }
  }
  consumer_sync();
  for (int i = threadIdx.x; i < BR; i += kConsumers) {
    float v = part[i];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) v += part[w * BR + i];
    S.res[i] = v;
  }
  consumer_sync();
  gemv_epilogue(P, S, t, g);
}

// ------------------------------------------------------------ attention
// q/k RMSNorm (optional) and rotate-half RoPE of one head: lane l holds
// dims [l*DL, l*DL + DL); the partner of dim i < d/2 is i + d/2, held by
// lane l ^ 16.  Values are rounded to bf16 after the norm and after RoPE.
template <int DL>
__device__ __forceinline__ void rope_head(const KernelParams& P,
                                          const uint16_t* src,
                                          const uint16_t* nw, const float* cs,
                                          bool rot, float (&x)[DL]) {
  const Dims& D = P.dims;
  const int lane = threadIdx.x & 31, d = DL * 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < DL; ++e) {
    x[e] = bf2f(__ldcg(src + lane * DL + e));
    ss = fmaf(x[e], x[e], ss);
  }
  if (!rot) return;
  if (nw) {
    ss = warp_sum(ss);
    const float r = 1.0f / sqrtf(ss / (float)d + D.eps);
#pragma unroll
    for (int e = 0; e < DL; ++e)
      x[e] = round_bf(__fmul_rn(__fmul_rn(x[e], r),
                                bf2f(__ldg(nw + lane * DL + e))));
  }
  const bool lo = lane < 16;
#pragma unroll
  for (int e = 0; e < DL; ++e) {
    const float other = __shfl_xor_sync(kFull, x[e], 16);
    const int i = (lane & 15) * DL + e;
    const float c = __ldg(cs + 2 * i), s = __ldg(cs + 2 * i + 1);
    const float y = lo ? __fsub_rn(__fmul_rn(x[e], c), __fmul_rn(other, s))
                       : __fadd_rn(__fmul_rn(x[e], c), __fmul_rn(other, s));
    x[e] = round_bf(y);
  }
}

// Sum 32 per-lane values across the warp so that lane j ends with the total
// of value j (a transpose-reduce: 31 shuffles for 32 sums).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
  return v[0];
}

__device__ __forceinline__ void load_row(const uint16_t* p, int DLc,
                                         float* out) {
  if (DLc == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    out[0] = bf_lo(u.x);
    out[1] = bf_hi(u.x);
    out[2] = bf_lo(u.y);
    out[3] = bf_hi(u.y);
  } else if (DLc == 2) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    out[0] = bf_lo(u);
    out[1] = bf_hi(u);
  } else {
    out[0] = bf2f(*p);
  }
}
__device__ __forceinline__ void load_row_cg(const uint16_t* p, int DLc,
                                            float* out) {
  if (DLc == 4) {
    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(p));
    out[0] = bf_lo(u.x);
    out[1] = bf_hi(u.x);
    out[2] = bf_lo(u.y);
    out[3] = bf_hi(u.y);
  } else if (DLc == 2) {
    const uint32_t u = __ldcg(reinterpret_cast<const unsigned int*>(p));
    out[0] = bf_lo(u);
    out[1] = bf_hi(u);
  } else {
    out[0] = bf2f(__ldcg(p));
  }
}

// This lane's DL values of a K (or V) row in shared memory, widened.
template <int DL>
__device__ __forceinline__ void smem_row(const uint16_t* row,
                                         float (&out)[DL]) {
  load_row(row + (threadIdx.x & 31) * DL, DL, out);
}

// Online softmax over the tokens [lo, hi) of one shared-memory buffer whose
// row 0 is token `base` (K rows at kb, V rows at vb, d values each), in
// blocks of 32/GRP tokens dealt to the 8 consumer warps (lane j of a block
// scores token j/GRP against head j mod GRP).  The token `newpos` (when
// >= 0) is read from knew/vnew instead.  Updates this warp's (m, l, acc).
template <int DL, int GRP>
__device__ __forceinline__ void attn_tokens(
    const KernelParams& P, const float (&qr)[GRP][DL], const uint16_t* kb,
    const uint16_t* vb, int base, int lo, int hi, int newpos,
    const uint16_t* knew, const uint16_t* vnew, float& m_run, float& l_run,
    float (&acc)[GRP][DL]) {
  constexpr int d = DL * 32, TB = 32 / GRP;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = (hi - lo + TB - 1) / TB;
  for (int blk = warp; blk < nblk; blk += kConsumerWarps) {
    const int t_blk = lo + blk * TB;
    // scores: one K row at a time
    float sv[32];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      const int tok = t_blk + tb;
      float kf[DL];
#pragma unroll
      for (int e = 0; e < DL; ++e) kf[e] = 0.f;
      if (tok < hi)
        smem_row<DL>(tok == newpos ? knew : kb + (size_t)(tok - base) * d, kf);
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        float sc = 0.f;
#pragma unroll
        for (int e = 0; e < DL; ++e) sc = fmaf(qr[h][e], kf[e], sc);
        sv[tb * GRP + h] = sc;
      }
    }
    float sc = reduce_scatter32(sv) * P.dims.attn_scale;
    if (t_blk + lane / GRP >= hi) sc = -INFINITY;
    float mb = sc;
#pragma unroll
    for (int o = GRP; o < 32; o <<= 1)
      mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
    const float m_new = fmaxf(m_run, mb);   // finite: the block's token 0 is
                                            // always valid
    const float corr = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
    const float p = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
    float lb = p;
#pragma unroll
    for (int o = GRP; o < 32; o <<= 1) lb += __shfl_xor_sync(kFull, lb, o);
    l_run = l_run * corr + lb;
    m_run = m_new;
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      const float ch = __shfl_sync(kFull, corr, h);
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[h][e] *= ch;
    }
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      const int tok = t_blk + tb;
      float vf[DL];
#pragma unroll
      for (int e = 0; e < DL; ++e) vf[e] = 0.f;
      if (tok < hi)
        smem_row<DL>(tok == newpos ? vnew : vb + (size_t)(tok - base) * d, vf);
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        const float pth = __shfl_sync(kFull, p, tb * GRP + h);
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[h][e] = fmaf(pth, vf[e], acc[h][e]);
      }
    }
  }
}

// JIT attention streams its cached tokens through two shared-memory stages
// of kJitStageTok tokens (K rows then V rows), filled by bulk copies that
// one consumer thread issues, one per run of tokens inside a KV page.
constexpr int kJitStageTok = 64;
__device__ __host__ __forceinline__ int jit_stage_bytes(int d) {
  return kJitStageTok * d * 2 * 2;   // K and V rows of one stage
}

// Copy the cached tokens [a, e) of (layer l, sequence b, KV head g) into a
// stage (K rows at kdst, V rows at vdst, row 0 = token a); completes on
// `bar`.  Called by the issuing thread alone.  Unmapped pages raise
// MPK_ERR_KV_PAGE and are skipped (their bytes are not expected, so the
// stage still completes).
__device__ void issue_kv_stage(const KernelParams& P, int l, int b, int g,
                               int a, int e, uint8_t* kdst, uint8_t* vdst,
                               uint64_t* bar, uint64_t policy) {
  const Dims& D = P.dims;
  const int P_ = D.page_size, d = D.d;
  const uint32_t row_bytes = (uint32_t)d * 2u;
  const int32_t* pt = P.step.page_table + (int64_t)b * D.max_pages;
  const int64_t head_elems = (int64_t)P_ * d;
  const int64_t layer_elems = (int64_t)l * P.step.num_pages * D.Hkv * head_elems;
  uint32_t total = 0;
  for (int tok = a; tok < e;) {
    const int run_end = min(e, (tok / P_ + 1) * P_);
    const int pg = __ldg(pt + tok / P_);
    if (pg >= 0 && pg < P.step.num_pages)
      total += (uint32_t)(run_end - tok) * row_bytes * 2u;
    else
      raise_error(P, MPK_ERR_KV_PAGE);
    tok = run_end;
  }
  mbar_arrive_expect_tx(bar, total);
  for (int tok = a; tok < e;) {
    const int run_end = min(e, (tok / P_ + 1) * P_);
    const int pg = __ldg(pt + tok / P_);
    if (pg >= 0 && pg < P.step.num_pages) {
      const int64_t off = layer_elems + ((int64_t)pg * D.Hkv + g) * head_elems +
                          (int64_t)(tok % P_) * d;
      const uint32_t bytes = (uint32_t)(run_end - tok) * row_bytes;
      bulk_g2s(kdst + (size_t)(tok - a) * row_bytes, P.step.k_pool + off,
               bytes, bar, policy);
      bulk_g2s(vdst + (size_t)(tok - a) * row_bytes, P.step.v_pool + off,
               bytes, bar, policy);
    }
    tok = run_end;
  }
}

// Merge the 8 warps' (m, l, acc) records of wbuf ([warp][GRP][2 + d]) per
// head: the factors exp(m_w - M) and the sum L are formed once per head
// (S.scratch), then thread i of the head's d outputs sums its column.
// Returns through `emit(h, i, A, L)` for the outputs this thread owns.
template <int GRP, int d, typename Emit>
__device__ __forceinline__ void merge_warps(const Smem& S, const float* wbuf,
                                            Emit emit) {
  constexpr int rec = 2 + d;
  const int tid = threadIdx.x;
  float* fac = S.scratch;                       // [GRP][8]
  float* lsum = S.scratch + GRP * kConsumerWarps;   // [GRP]
  if (tid < GRP) {
    const int h = tid;
    float M = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w)
      M = fmaxf(M, wbuf[(w * GRP + h) * rec]);
    float Ls = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* r = wbuf + (w * GRP + h) * rec;
      const float sc =
          (M == -INFINITY || r[0] == -INFINITY) ? 0.f : expf(r[0] - M);
      fac[h * kConsumerWarps + w] = sc;
      Ls = fmaf(r[1], sc, Ls);
    }
    lsum[h] = Ls;
    // the merged maximum replaces warp 0's for the caller
    S.scratch[GRP * (kConsumerWarps + 1) + h] = M;
  }
  consumer_sync();
  for (int o = tid; o < GRP * d; o += kConsumers) {
    const int h = o / d, i = o - h * d;
    float A = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
      A = fmaf(wbuf[(w * GRP + h) * rec + 2 + i], fac[h * kConsumerWarps + w],
               A);
    emit(h, i, A, lsum[h], S.scratch[GRP * (kConsumerWarps + 1) + h]);
  }
}

// One KV chunk of (sequence b, KV head g): tokens [t0, t1) of the
// n = seq_len + 1 positions.  Prologue: the group's queries (and, for the
// chunk holding the new token, its key and value) get RMSNorm + RoPE; the
// new K/V are appended to the paged cache.  Body: each warp runs an online
// softmax over blocks of 32/GRP tokens for all GRP query heads (lane j of a
// block scores token j/GRP against head j%GRP).  The warps merge into one
// (m, l, acc) partial per head; the last chunk of (b, g) to finish merges
// the C partials (log-sum-exp) into the bf16 attention output.  AOT tasks
// (PRE) read their cached tokens from two ring pages the producer filled
// ahead of time, and the position from the producer's note beside the K
// page; JIT tasks read the paged cache directly.
template <int DL, int GRP, bool PRE>
__device__ void attn_body(const KernelParams& P, const Smem& S,
                          const TaskDesc& t, Ring& ring, uint64_t deadline) {
  constexpr int d = DL * 32, rec = 2 + d;
  const Dims& D = P.dims;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = t.b, g = t.g, l = t.layer, C = D.C;
  // scratch: (JIT) two K/V stages | q [GRP][d] | warp records [8][GRP][rec]
  // | (JIT) the new token's K and V rows (bf16)
  uint8_t* stage0 = reinterpret_cast<uint8_t*>(S.xs);
  float* qf = reinterpret_cast<float*>(stage0 + (PRE ? 0 : 2 * jit_stage_bytes(d)));
  float* wbuf = qf + GRP * d;
  uint16_t* knew = reinterpret_cast<uint16_t*>(wbuf + kConsumerWarps * GRP * rec);
  uint16_t* vnew = knew + d;
  if (!PRE && (int)(reinterpret_cast<uint8_t*>(vnew + d) - stage0) >
                  P.sm.xs_bytes) {
    if (tid == 0) raise_error(P, MPK_ERR_UNSUPPORTED);
    return;
  }
  bool have_k = true, have_v = true;
  uint8_t *kpage = nullptr, *vpage = nullptr;
  Ring kr = ring;
  int pos, page_new = -1;
  if constexpr (PRE) {
    have_k = wait_full(P, S, ring, deadline);
    kpage = page_ptr(S, ring.slot);
    const int2 m = S.meta[ring.slot];
    pos = have_k ? m.x : -1;
    page_new = m.y;
    ring.advance(S.n_pages);
    have_v = wait_full(P, S, ring, deadline);
    vpage = page_ptr(S, ring.slot);
    ring.advance(S.n_pages);
  } else {
    pos = __ldcg(P.step.seq_lens + b);
  }
  const int n = pos + 1;
  int t0 = 0, t1 = 0;
  bool ok = pos >= 0 && n <= D.max_ctx;
  if (ok) {
    chunk_range(t.c, n, C, t0, t1);
    if (PRE) t1 = min(t1, t0 + kAttnMaxTokens);
    if (!PRE) {
      const int pidx = pos / D.page_size;
      if (pidx < D.max_pages)
        page_new = __ldg(P.step.page_table + (int64_t)b * D.max_pages + pidx);
    }
    ok = page_new >= 0 && page_new < P.step.num_pages;
  }
  if (!ok) {
    if (tid == 0 && have_k) raise_error(P, MPK_ERR_KV_PAGE);
    t0 = t1 = 0;
  }
  const bool has_new = ok && t1 == n && t1 > t0;
  // JIT: the cached tokens [t0, ce) stream through two stages; the first two
  // fills go out before the prologue (they do not depend on it), so their
  // latency overlaps the query and RoPE work.  They are issued by lane 0 of
  // the last warp (no query head of its own unless the group has more than
  // 6 heads), which tracks the fills issued and not yet seen complete (bit
  // per stage) and the phase each of them completes.
  const bool issuer = tid == kConsumers - 32;
  const int ce = has_new ? pos : t1;
  const int nsub = PRE ? 0 : (t1 - t0 + kJitStageTok - 1) / kJitStageTok;
  const int sb = jit_stage_bytes(d) / 2;   // K (or V) rows of one stage
  uint64_t* sbar = S.jit_bar;
  uint32_t ph = (uint32_t)S.ctrl[13];
  const uint64_t policy = PRE ? 0ull : evict_first_policy();
  uint32_t pend = 0, pend_ph = 0;
  if (!PRE && issuer) {
    for (int s = 0; s < 2 && s < nsub; ++s) {
      const int a = t0 + s * kJitStageTok;
      issue_kv_stage(P, l, b, g, a, min(ce, a + kJitStageTok),
                     stage0 + s * 2 * sb, stage0 + s * 2 * sb + sb, &sbar[s],
                     policy);
      pend |= 1u << s;
      pend_ph = (pend_ph & ~(1u << s)) | (ph & (1u << s));
    }
  }
  // ---- prologue: queries (and the new key/value) into shared memory
  {
    const uint16_t* qkv = lt(P, l, P.act.o_qkv) +
                          (int64_t)b * (D.Hq + 2 * D.Hkv) * d;
    const float* cs = P.w.rope_cs + (int64_t)(ok ? pos : 0) * (d / 2) * 2;
    const int64_t slot =
        ((((int64_t)l * P.step.num_pages + max(page_new, 0)) * D.Hkv + g) *
             D.page_size +
         (ok ? pos % D.page_size : 0)) *
        d;
    for (int hh = warp; hh < GRP + 2; hh += kConsumerWarps) {
      if (hh >= GRP && !has_new) continue;
      const uint16_t* src;
      const uint16_t* nw = nullptr;
      if (hh < GRP) {
        src = qkv + (int64_t)(g * GRP + hh) * d;
        if (D.qk_norm) nw = layer_w(P, l, MPK_W_QNORM);
      } else if (hh == GRP) {
        src = qkv + (int64_t)(D.Hq + g) * d;
        if (D.qk_norm) nw = layer_w(P, l, MPK_W_KNORM);
      } else {
        src = qkv + (int64_t)(D.Hq + D.Hkv + g) * d;
      }
      float x[DL];
      rope_head<DL>(P, src, nw, cs, hh <= GRP, x);
      if (hh < GRP) {
#pragma unroll
        for (int e = 0; e < DL; ++e) qf[hh * d + lane * DL + e] = x[e];
      } else {
        uint16_t* cache = (hh == GRP ? P.step.k_pool : P.step.v_pool) + slot;
        uint16_t* pg = PRE ? reinterpret_cast<uint16_t*>(
                                 (hh == GRP ? kpage : vpage)) +
                                 (size_t)(pos - t0) * d
                           : nullptr;
        uint16_t* mine = hh == GRP ? knew : vnew;
#pragma unroll
        for (int e = 0; e < DL; ++e) {
          const uint16_t u = f2bf(x[e]);
          cache[lane * DL + e] = u;
          if (PRE) pg[lane * DL + e] = u;
          else mine[lane * DL + e] = u;
        }
      }
    }
    consumer_sync();
  }
  stamp(P, S, 2);
  float qr[GRP][DL];
#pragma unroll
  for (int h = 0; h < GRP; ++h)
#pragma unroll
    for (int e = 0; e < DL; ++e) qr[h][e] = qf[h * d + lane * DL + e];
  // ---- online softmax over this warp's token blocks
  float m_run = -INFINITY, l_run = 0.f;
  float acc[GRP][DL];
#pragma unroll
  for (int h = 0; h < GRP; ++h)
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[h][e] = 0.f;
  if constexpr (PRE) {
    attn_tokens<DL, GRP>(P, qr, reinterpret_cast<const uint16_t*>(kpage),
                         reinterpret_cast<const uint16_t*>(vpage), t0, t0, t1,
                         -1, nullptr, nullptr, m_run, l_run, acc);
  } else {
    // cached tokens [t0, ce) come through the stages; the new token (if
    // this chunk holds it) from knew/vnew
    for (int s = 0; s < nsub; ++s) {
      const int st = s & 1;
      bool got = !S.ctrl[2];
      uint32_t spins = 0;
      while (got && !mbar_try_wait(&sbar[st], (ph >> st) & 1u)) {
        if ((++spins & 1023u) == 0u && (aborted(P) || globaltimer() > deadline)) {
          if (!aborted(P)) raise_error(P, MPK_ERR_TIMEOUT);
          S.ctrl[2] = 1;
          got = false;
        }
      }
      if (got) pend &= ~(1u << st);
      ph ^= 1u << st;
      const int lo = t0 + s * kJitStageTok, hi = min(t1, lo + kJitStageTok);
      if (got)
        attn_tokens<DL, GRP>(
            P, qr, reinterpret_cast<const uint16_t*>(stage0 + st * 2 * sb),
            reinterpret_cast<const uint16_t*>(stage0 + st * 2 * sb + sb), lo,
            lo, hi, has_new ? pos : -1, knew, vnew, m_run, l_run, acc);
      consumer_sync();   // the stage is free again
      if (issuer && s + 2 < nsub && !S.ctrl[2]) {
        const int a = lo + 2 * kJitStageTok;
        issue_kv_stage(P, l, b, g, a, min(ce, a + kJitStageTok),
                       stage0 + st * 2 * sb, stage0 + st * 2 * sb + sb,
                       &sbar[st], policy);
        pend |= 1u << st;
        pend_ph = (pend_ph & ~(1u << st)) | (ph & (1u << st));
      }
    }
    if (issuer) {
      // an abandoned fill still completes (its bytes were expected): wait
      // (bounded) so that no copy lands in shared memory after the task
      const uint64_t lim = globaltimer() + 200000000ull;
      for (int st = 0; st < 2; ++st)
        if (pend & (1u << st))
          while (!mbar_try_wait(&sbar[st], (pend_ph >> st) & 1u) &&
                 globaltimer() < lim) {
          }
      S.ctrl[13] = (int)ph;
    }
  }
  stamp(P, S, 3);
  if constexpr (PRE) {
    // the pages were written through the generic proxy (new token): order
    // that before the producer's next bulk copy into them
    fence_proxy_async_smem();
    release_page(S, kr, have_k);
    release_page(S, kr, have_v);
  }
  // ---- merge the 8 warps into this chunk's partial
#pragma unroll
  for (int h = 0; h < GRP; ++h) {
    float* r = wbuf + (warp * GRP + h) * rec;
    const float mh = __shfl_sync(kFull, m_run, h);
    const float lh = __shfl_sync(kFull, l_run, h);
    if (lane == 0) {
      r[0] = mh;
      r[1] = lh;
    }
#pragma unroll
    for (int e = 0; e < DL; ++e) r[2 + lane * DL + e] = acc[h][e];
  }
  consumer_sync();
  float* part = lt<float>(P, l, P.act.o_opart) +
                (((int64_t)(b * D.Hkv + g) * C) * GRP) * rec;
  float* mine = part + (int64_t)t.c * GRP * rec;
  merge_warps<GRP, d>(S, wbuf, [=](int h, int i, float A, float Ls, float M) {
    mine[h * rec + 2 + i] = A;
    if (i == 0) {
      mine[h * rec] = M;
      mine[h * rec + 1] = Ls;
    }
  });
  __threadfence();
  consumer_sync();
  // ---- the last chunk of (b, g) to finish merges all C partials
  if (tid == 0) {
    uint32_t* cnt = P.graph.merge_cnt + ((int64_t)l * D.B + b) * D.Hkv + g;
    const uint32_t old = atom_acq_rel_add(cnt, 1u);
    const int last = (old + 1u == (uint32_t)C) ? 1 : 0;
    if (last) *reinterpret_cast<volatile uint32_t*>(cnt) = 0u;
    S.ctrl[4] = last;
  }
  consumer_sync();
  if (!S.ctrl[4]) return;
  // warp w merges the partials of chunks w, w + 8, ... (coalesced reads),
  // then the 8 warp results merge as above
  {
    float Mw[GRP], Lw[GRP], Aw[GRP][DL];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      Mw[h] = -INFINITY;
      Lw[h] = 0.f;
#pragma unroll
      for (int e = 0; e < DL; ++e) Aw[h][e] = 0.f;
    }
    // J chunks' partials are loaded before any is merged, so their global
    // reads overlap
    constexpr int J = GRP * (2 + DL) <= 24 ? 3 : 1;
#pragma unroll 1
    for (int c0 = warp; c0 < C; c0 += J * kConsumerWarps) {
      float mc[J][GRP], lc[J][GRP], ac[J][GRP][DL];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = c0 + j * kConsumerWarps;
        const float* rc = part + (int64_t)min(c, C - 1) * GRP * rec;
#pragma unroll
        for (int h = 0; h < GRP; ++h) {
          mc[j][h] = c < C ? __ldcg(rc + h * rec) : -INFINITY;
          lc[j][h] = __ldcg(rc + h * rec + 1);
#pragma unroll
          for (int e = 0; e < DL; ++e)
            ac[j][h][e] = __ldcg(rc + h * rec + 2 + lane * DL + e);
        }
      }
#pragma unroll
      for (int j = 0; j < J; ++j) {
#pragma unroll
        for (int h = 0; h < GRP; ++h) {
          const float Mn = fmaxf(Mw[h], mc[j][h]);
          if (Mn == -INFINITY) continue;
          const float sa = (Mw[h] == -INFINITY) ? 0.f : expf(Mw[h] - Mn);
          const float sc = (mc[j][h] == -INFINITY) ? 0.f : expf(mc[j][h] - Mn);
          Lw[h] = Lw[h] * sa + lc[j][h] * sc;
#pragma unroll
          for (int e = 0; e < DL; ++e)
            Aw[h][e] = Aw[h][e] * sa + ac[j][h][e] * sc;
          Mw[h] = Mn;
        }
      }
    }
    consumer_sync();   // wbuf and the scratch factors are reused
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      float* r = wbuf + (warp * GRP + h) * rec;
      if (lane == 0) {
        r[0] = Mw[h];
        r[1] = Lw[h];
      }
#pragma unroll
      for (int e = 0; e < DL; ++e) r[2 + lane * DL + e] = Aw[h][e];
    }
    consumer_sync();
  }
  uint16_t* out = lt(P, l, P.act.o_attn) + (int64_t)b * D.Hq * d +
                  (int64_t)g * GRP * d;
  merge_warps<GRP, d>(S, wbuf, [=](int h, int i, float A, float Ls, float) {
    out[h * d + i] = f2bf(A / Ls);
  });
}

// JIT attention tasks (batch > 1) as a separate function: its paged-cache
// reads need registers of their own, which would otherwise spill around
// every other task body of the kernel.
template <int DL, int GRP>
__device__ __noinline__ void attn_body_jit(const KernelParams& P,
                                           const Smem& S, const TaskDesc& t,
                                           Ring& ring, uint64_t deadline) {
  attn_body<DL, GRP, false>(P, S, t, ring, deadline);
}

__device__ void task_attn(const KernelParams& P, const Smem& S,
                          const TaskDesc& t, Ring& ring, uint64_t deadline) {
  const int grp = P.dims.Hq / P.dims.Hkv;
  const int dl = P.dims.d / 32;
  const bool pre = t.launch == MPK_LAUNCH_AOT;
#define MPK_ATTN_CASE(G, DL)                                     \
  if (grp == G && dl == DL) {                                    \
    if (pre) attn_body<DL, G, true>(P, S, t, ring, deadline);    \
    else attn_body_jit<DL, G>(P, S, t, ring, deadline);          \
    return;                                                      \
  }
  MPK_ATTN_CASE(1, 1) MPK_ATTN_CASE(1, 2) MPK_ATTN_CASE(1, 4)
  MPK_ATTN_CASE(2, 1) MPK_ATTN_CASE(2, 2) MPK_ATTN_CASE(2, 4)
  MPK_ATTN_CASE(4, 1) MPK_ATTN_CASE(4, 2) MPK_ATTN_CASE(4, 4)
  MPK_ATTN_CASE(8, 1) MPK_ATTN_CASE(8, 2) MPK_ATTN_CASE(8, 4)
#undef MPK_ATTN_CASE
  if (threadIdx.x == 0) raise_error(P, MPK_ERR_UNSUPPORTED);
}

// Greedy argmax over the lm_head tiles' (max, index) pairs; lowest index
// among equal maxima.  Also advances seq_lens (decoder mode).
__device__ void task_argmax(const KernelParams& P, const Smem& S) {
  const Dims& D = P.dims;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float2* am =
      reinterpret_cast<const float2*>(global_base(P) + P.act.g_amax);
  for (int b = 0; b < D.B; ++b) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = tid; j < D.n_lm_tiles; j += kConsumers) {
      const float2 e = __ldcg(am + (int64_t)b * D.n_lm_tiles + j);
      if (better(e.x, __float_as_int(e.y), bv, bi)) {
        bv = e.x;
        bi = __float_as_int(e.y);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      if (better(ov, oi, bv, bi)) {
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
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      P.step.next_tokens[(int64_t)S.ctrl[14] * D.B + b] =
          (bi == 0x7fffffff) ? 0 : bi;
      if (D.chain_ffn == 0)
        P.step.seq_lens[b] = __ldcg(P.step.seq_lens + b) + 1;
    }
    consumer_sync();
  }
}

__device__ void run_task(const KernelParams& P, const Smem& S,
                         const TaskDesc& t, Ring& ring, uint64_t deadline) {
  if (is_gemv(t.kind)) {
    const Gemv g = gemv_geom(P, t);
    const int B = P.dims.B;
    if (B == 1)
      gemv_b1(P, S, t, g, ring, deadline);
    else if (B <= 4)
      gemv_cc<4>(P, S, t, g, ring, deadline);
    else if (B < 8)
      gemv_cc<8>(P, S, t, g, ring, deadline);
    else
      gemv_mma(P, S, t, g, ring, deadline);
    return;
  }
  switch (t.kind) {
    case MPK_TASK_ATTN:
      task_attn(P, S, t, ring, deadline);
      break;
    case MPK_TASK_ARGMAX:
      task_argmax(P, S);
      break;
    default:  // MPK_TASK_EMPTY
      break;
  }
}

// ------------------------------------------------------------ queues
__device__ bool ring_push(const KernelParams& P, RingHdr* hdr, uint64_t* slots,
                          uint32_t cap, uint32_t value, uint64_t deadline) {
  const uint32_t pos = atomicAdd(&hdr->tail, 1u);
  uint32_t spins = 0;
  while ((int32_t)(pos - ld_acquire(&hdr->head)) >= (int32_t)cap) {
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

// Fire `e` (one trigger), whose descriptor `ed0` the caller holds.  The
// activating trigger pushes the event to its scheduler warp when it has JIT
// tasks, and runs its empty tasks inline (they only trigger their own
// event, whose descriptor is read from the graph).
__device__ void trigger(const KernelParams& P, int e, const EventDesc& ed0,
                        const int32_t* fan, uint32_t epoch,
                        uint64_t deadline) {
  const DevGraph& G = P.graph;
  if (ed0.flags & EV_FAN_CACHED) {
    bool fire = ed0.count == 1;
    if (!fire) fire = atom_acq_rel_add(G.counters + e, 1u) + 1u == epoch * ed0.count;
    if (fire) {
      red_release_add(G.counters + fan[0], 1u);
      if (fan[1] >= 0) red_release_add(G.counters + fan[1], 1u);
    }
    return;
  }
  int stack[16];
  int sp = 0;
  int ev = e;
  EventDesc ed = ed0;
  while (true) {
    if (!(ed.flags & (EV_HAS_JIT | EV_HAS_INLINE))) {
      red_release_add(G.counters + ev, 1u);
    } else {
      const uint32_t old = atom_acq_rel_add(G.counters + ev, 1u);
      if (old + 1u == epoch * ed.count) {
        if (ed.flags & EV_HAS_JIT) {
          const int s = ev % G.S;
          if (!ring_push(P, G.sched_hdr + s,
                         G.sched_slots + (size_t)s * G.sched_cap, G.sched_cap,
                         (uint32_t)ev, deadline))
            return;
        }
        if (ed.flags & EV_HAS_INLINE) {
          const int n_in = (int)(ed.flags >> kEvInlineShift);
          for (int t = ed.last - n_in + 1; t <= ed.last; ++t) {
            if (sp >= 16) {
              raise_error(P, MPK_ERR_QUEUE_OVERFLOW);
              return;
            }
            stack[sp++] = G.tasks[t].trig;
          }
        }
      }
    }
    if (sp == 0) return;
    ev = stack[--sp];
    ed = G.events[ev];
  }
}


// ------------------------------------------------------------ roles
// Asynchronous fetch of one AOT record into shared memory (thread 0).
__device__ __forceinline__ void fetch_rec(const AotRec* src, AotRec* dst) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) cp_async16(d + i, s + i);
  cp_async_commit();
}

// Leader-only loop state lives in shared memory (S.ctrl[8..10]) rather than
// in registers that every thread would carry across the task bodies.  The
// head AOT record is fetched asynchronously as soon as the task before it
// is dispatched, so the poll, the dispatch and the trigger read nothing
// from global memory but the event counter.
__device__ void worker_consumers(const KernelParams& P, const Smem& S, int w,
                                 uint64_t deadline) {
  const DevGraph& G = P.graph;
  const int tid = threadIdx.x;
  volatile int* ai_s = S.ctrl + 8;        // queue position of the head record
  volatile int* a1_s = S.ctrl + 9;        // end of this worker's AOT queue
  volatile int* jit_s = S.ctrl + 10;      // JIT ring head
  volatile int* a0_s = S.ctrl + 11;       // queue start (each step walks it)
  volatile int* step_s = S.ctrl + 14;     // step of the launch
  if (tid == 0) {
    const int a0 = G.aot_off[w], a1 = G.aot_off[w + 1];
    *jit_s = (int)ld_relaxed(&G.jit_hdr[w].head);
    *ai_s = a0;
    *a1_s = a1;
    *a0_s = a0;
    *step_s = 0;
    if (a0 < a1) fetch_rec(G.aot_rec + a0, &S.head[a0 & 1]);
  }
  Ring ring{0, 0};
  int iter = 0;
  while (true) {
    const int slot = iter & 1;
    if (tid == 0) {
      if (G.trace) S.times[0] = globaltimer();
      const int ai = *ai_s, step = *step_s;
      const uint32_t epoch = P.step.epoch + (uint32_t)step;
      const bool have_head = ai < *a1_s;
      cp_async_wait_all();
      const AotRec* hr = &S.head[ai & 1];
      int dep;
      uint32_t target;
      if (have_head) {
        prefetch_gain(P, hr->desc);   // warm L2 with the prologue's gain
        dep = hr->desc.dep;
        target = epoch * hr->dep_count;
        if (dep == G.root && step > 0) {
          // the step before must have produced this step's tokens and
          // advanced the sequence lengths
          dep = G.end;
          target = (epoch - 1u) * G.events[G.end].count;
        }
      } else {
        dep = G.end;
        target = epoch * G.events[G.end].count;
      }
      RingHdr* jh = G.jit_hdr + w;
      uint64_t* js = G.jit_slots + (size_t)w * G.jit_cap;
      uint32_t jit_head = (uint32_t)*jit_s;
      int cmd = -1;
      uint32_t spins = 0;
      while (!S.ctrl[2]) {
        uint32_t v;
        if (G.has_jit && ring_try_pop(jh, js, G.jit_cap, jit_head, v)) {
          cmd = (int)v;
          S.desc[slot] = G.tasks[cmd];
          S.tev[slot] = G.events[S.desc[slot].trig];
          S.fan[2 * slot] = S.fan[2 * slot + 1] = -1;
          break;
        }
        // the acquire orders this CTA's later reads after the producers'
        // releasing triggers (passed on to the other threads by the barrier
        // below)
        if ((int32_t)(ld_acquire(G.counters + dep) - target) >= 0) {
          if (have_head) {
            cmd = hr->id;
            S.desc[slot] = hr->desc;
            S.tev[slot] = hr->trig_ev;
            S.fan[2 * slot] = hr->fan[0];
            S.fan[2 * slot + 1] = hr->fan[1];
            *ai_s = ai + 1;
            if (ai + 1 < *a1_s)
              fetch_rec(G.aot_rec + ai + 1, &S.head[(ai + 1) & 1]);
          } else if (step + 1 < P.step.n_steps) {
            // this step has ended: the next one of the launch begins
            const int a0 = *a0_s;
            *step_s = step + 1;
            *ai_s = a0;
            if (a0 < *a1_s) fetch_rec(G.aot_rec + a0, &S.head[a0 & 1]);
            cmd = -2;
          }
          break;
        }
        ++spins;
        if (spins > 64) __nanosleep(spins > 8192 ? 128 : 16);
        if ((spins & 63u) == 0u) {
          if (aborted(P)) break;
          if (globaltimer() > deadline) {
            raise_error(P, MPK_ERR_TIMEOUT);
            break;
          }
        }
      }
      *jit_s = (int)jit_head;
      if (G.trace) {
        S.times[1] = globaltimer();
        S.times[2] = S.times[3] = 0;
      }
      S.ctrl[slot] = cmd;
    }
    consumer_sync();
    const int cmd = S.ctrl[slot];
    ++iter;
    if (cmd == -2) continue;
    if (cmd < 0) break;
    run_task(P, S, S.desc[slot], ring, deadline);
    consumer_sync();
    stamp(P, S, 4);
    // only the leader decides to stop (at its next poll), so all consumer
    // threads leave through the same broadcast
    if (tid == 0 && !S.ctrl[2] && !aborted(P)) {
      // the red.release / atom.acq_rel of the trigger is cumulative: it
      // orders every write of the CTA that the barrier above ordered before
      // this thread
      // a JIT task fires in the step its event fired in (a worker can
      // take one of the next step before it notices this step's end):
      // the dependent event's counter says which; AOT tasks are in the
      // worker's current step
      const TaskDesc& td = S.desc[slot];
      uint32_t epoch = P.step.epoch + (uint32_t)*step_s;
      if (td.launch == MPK_LAUNCH_JIT) {
        const uint32_t c = G.events[td.dep].count;
        if (c > 0) epoch = ld_relaxed(G.counters + td.dep) / c;
      }
      trigger(P, td.trig, S.tev[slot], S.fan + 2 * slot, epoch, deadline);
      if (G.trace) {
        // (task | worker << 32), looked-for, ready, staged, pages done,
        // body done, triggered
        const uint32_t k = atomicAdd(G.trace_count, 1u);
        if (k < G.trace_cap) {
          uint64_t* r = G.trace + 8ull * k;
          r[0] = (uint64_t)(uint32_t)cmd | ((uint64_t)(uint32_t)w << 32);
          r[1] = S.times[0];
          r[2] = S.times[1];
          r[3] = S.times[2];
          r[4] = S.times[3];
          r[5] = S.times[4];
          r[6] = globaltimer();
          r[7] = 0;
        }
      }
    }
  }
  if (tid == 0) cp_async_wait_all();
}

__device__ void scheduler_role(const KernelParams& P, int s,
                               uint64_t deadline) {
  const DevGraph& G = P.graph;
  const int lane = threadIdx.x & 31;
  RingHdr* hdr = G.sched_hdr + s;
  uint64_t* slots = G.sched_slots + (size_t)s * G.sched_cap;
  uint32_t head = (lane == 0) ? ld_relaxed(&hdr->head) : 0;
  uint32_t cursor = (uint32_t)(((int64_t)s * G.W) / G.S);
  // JIT attention chunks differ in length as the sequences do: they are
  // dealt by cost, each worker receiving a run of about `quantum` of the
  // work of one layer (the tokens of all chunks plus a fixed part per task,
  // over the workers), in the order a global cost counter hands out.  The
  // fixed part is the per-chunk time (prologue, merge, trigger, first fill)
  // in units of the time of one token: measured on the batch-16 8B shape
  // as about 10 us against about 0.04 us a token.
  constexpr uint32_t kJitFixedCost = 256;
  unsigned long long quantum = 0;
  if (G.jit_cost && P.step.seq_lens && P.dims.chain_ffn == 0) {   // decoder
    uint64_t tok = 0;
    for (int b = lane; b < P.dims.B; b += 32)
      tok += (uint64_t)max(__ldcg(P.step.seq_lens + b) + 1, 0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tok += __shfl_xor_sync(kFull, tok, o);
    const uint64_t per_layer =
        tok * (uint64_t)P.dims.Hkv +
        (uint64_t)kJitFixedCost * P.dims.B * P.dims.Hkv * P.dims.C;
    quantum = max(per_layer / (uint64_t)G.W, (uint64_t)1);
  }
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
        if (event_done(P, G.end, P.step.epoch + P.step.n_steps - 1) ||
            aborted(P))
          stop = 1;
        if (spins > 32) __nanosleep(spins > 4096 ? 256 : 32);
        if ((spins & 63u) == 0u && globaltimer() > deadline) {
          raise_error(P, MPK_ERR_TIMEOUT);
          stop = 1;
        }
      }
    }
    e = __shfl_sync(kFull, e, 0);
    stop = __shfl_sync(kFull, stop, 0);
    if (stop) break;
    if (e < 0) continue;
    const EventDesc ed = G.events[e];
    const int n = ed.last - ed.first + 1;
    for (int i = lane; i < n; i += 32) {
      const int t = ed.first + i;
      const TaskDesc td = G.tasks[t];
      if (td.launch != MPK_LAUNCH_JIT) continue;
      int w = (int)((cursor + (uint32_t)i) % (uint32_t)G.W);
      if (quantum > 0 && td.kind == MPK_TASK_ATTN) {
        const int pos = __ldcg(P.step.seq_lens + td.b);
        int t0 = 0, t1 = 0;
        if (pos >= 0) chunk_range(td.c, pos + 1, P.dims.C, t0, t1);
        const unsigned long long cost =
            kJitFixedCost + (unsigned long long)max(t1 - t0, 0);
        const unsigned long long at = atomicAdd(G.jit_cost, cost);
        w = (int)(((at + cost / 2) / quantum) % (unsigned long long)G.W);
      }
      ring_push(P, G.jit_hdr + w, G.jit_slots + (size_t)w * G.jit_cap,
                G.jit_cap, (uint32_t)t, deadline);
    }
    cursor += (uint32_t)n;
  }
}

// ------------------------------------------------------------ kernels
__device__ __forceinline__ bool setup_smem(const KernelParams& P, uint8_t* raw,
                                           Smem& S) {
  if (smem_addr(raw) & 127u) {   // uniform: same address for all threads
    if (threadIdx.x == 0) raise_error(P, MPK_ERR_UNSUPPORTED);
    return false;
  }
  S = carve(raw, P.sm);
  if (threadIdx.x == 0) {
    for (int i = 0; i < S.n_pages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsumerWarps);
    }
    S.ctrl[0] = S.ctrl[1] = -1;
    S.ctrl[2] = 0;
    // an earlier step that failed leaves the abort flag up until
    // mpk_reset; read it once per CTA so all threads agree
    S.ctrl[3] = aborted(P) ? 1 : 0;
    S.ctrl[4] = 0;
    mbar_init(&S.jit_bar[0], 1);
    mbar_init(&S.jit_bar[1], 1);
    S.ctrl[13] = 0;   // JIT stage barrier phases
    S.ctrl[14] = 0;   // step of the launch
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
  const int warp = threadIdx.x >> 5;
  if (warp >= kConsumerWarps) {
    regs_dec<kProducerRegs>();
    if (warp >= kConsumerWarps + kProducerWarps) return;
    const int a0 = P.graph.aot_off[w], a1 = P.graph.aot_off[w + 1];
    producer_role(P, S, P.graph.aot_list + a0, a1 - a0, P.step.n_steps,
                  deadline, warp - kConsumerWarps);
  } else {
    regs_inc<kConsumerRegs>();
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
  const int warp = threadIdx.x >> 5;
  if (warp >= kConsumerWarps) {
    regs_dec<kProducerRegs>();
    if (warp >= kConsumerWarps + kProducerWarps) return;
    producer_role(P, S, P.graph.op_tasks + first + blockIdx.x, 1, 1,
                  deadline, warp - kConsumerWarps);
  } else {
    regs_inc<kConsumerRegs>();
    Ring ring{0, 0};
    run_task(P, S, P.graph.tasks[task], ring, deadline);
  }
}

// ------------------------------------------------------------ host side
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
