// Host-side state of a built graph (struct mpk_graph of include/mpk.h),
// shared by the translation units that implement the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "device_abi.h"
#include "mpk.h"
#include "tgraph_builder.h"

namespace mpk_detail {

constexpr uint32_t kJitCap = 1024;
constexpr uint32_t kSchedCap = 4096;
constexpr int kSmemLimit = 232448;   // 227 KB per block on sm_100-class

template <typename T>
struct DevBuf {
  T* p = nullptr;
  size_t n = 0;
  ~DevBuf() { reset(); }
  void reset() {
    if (p) cudaFree(p);
    p = nullptr;
    n = 0;
  }
  cudaError_t alloc(size_t count) {
    reset();
    n = count;
    if (count == 0) return cudaSuccess;
    return cudaMalloc(reinterpret_cast<void**>(&p), count * sizeof(T));
  }
  cudaError_t upload(const std::vector<T>& v) {
    cudaError_t e = alloc(v.size());
    if (e != cudaSuccess || v.empty()) return e;
    return cudaMemcpy(p, v.data(), v.size() * sizeof(T),
                      cudaMemcpyHostToDevice);
  }
};

}  // namespace mpk_detail

using mpk_detail::DevBuf;

struct mpk_graph {
  mpk::BuiltGraph bg;
  uint64_t uid = 0;   // build number, unique within the process
  int num_sched_sms = 4, sched_warps_per_sm = 4, pages_req = 0;
  // export arrays (linear order)
  std::vector<int32_t> x_kind, x_op, x_layer, x_tile, x_row0, x_row1, x_b,
      x_g, x_c, x_pre, op_kind, op_layer, op_n;
  // device encoding
  int device = -1;
  bool encoded = false, bound = false;
  std::vector<mpk::TaskDesc> h_tasks;
  std::vector<mpk::EventDesc> h_events;
  std::vector<int32_t> h_aot, h_aot_off, h_op_tasks, h_op_first;
  std::vector<mpk::AotRec> h_aot_rec;
  DevBuf<mpk::TaskDesc> d_tasks;
  DevBuf<mpk::EventDesc> d_events;
  DevBuf<int32_t> d_aot, d_aot_off, d_op_tasks;
  DevBuf<mpk::AotRec> d_aot_rec;
  DevBuf<uint32_t> d_counters, d_status, d_merge_cnt;
  DevBuf<unsigned long long> d_jit_cost;
  DevBuf<mpk::RingHdr> d_jit_hdr, d_sched_hdr;
  DevBuf<uint64_t> d_jit_slots, d_sched_slots;
  DevBuf<char> d_act;
  DevBuf<const uint16_t*> d_layer_ptrs;
  DevBuf<float> d_rope;
  DevBuf<uint64_t> d_trace;
  DevBuf<uint32_t> d_trace_count;
  mpk::KernelParams params{};
  int smem = 0;
  uint32_t epoch = 0;
  uint64_t timeout_ns = 2000000000ull;
  int mode = MPK_MODE_MEGAKERNEL;
  // captured kernel-per-operator step
  cudaGraphExec_t kpo_exec = nullptr;
  mpk::StepArgs kpo_args{};
  cudaStream_t kpo_stream = nullptr;
  ~mpk_graph() {
    if (kpo_exec) cudaGraphExecDestroy(kpo_exec);
  }
};

