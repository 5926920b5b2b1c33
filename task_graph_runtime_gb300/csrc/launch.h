// Host entry points of kernels.cu (the only translation unit that sees the
// __global__ functions).
#pragma once

#include <cuda_runtime.h>

#include "device_abi.h"

namespace mpk {

cudaError_t configure_kernels(int smem);
cudaError_t launch_megakernel(const KernelParams& P, int grid, int smem,
                              cudaStream_t stream);
cudaError_t launch_kpo_op(const KernelParams& P, int first, int n_tasks,
                          int smem, cudaStream_t stream);
int megakernel_max_blocks_per_sm(int smem);

}  // namespace mpk
