// csa_internal.h -- declarations shared by the translation units of the library
// (not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>

#include "csa_pool.cuh"

namespace csa {

using PoolKernel = void (*)(PoolParams);

// Kernel instantiation for a plan (nullptr if the plan has no instantiation).
PoolKernel fwd_kernel_for(const Plan& pl);
PoolKernel bwd_kernel_for(const Plan& pl);

// Launch helpers (csa_api.cu). note(): records a failing CUDA call for
// csa_last_error_string() and passes the code on. device_sms(): multiprocessor count of a
// device (cached). blocks_per_sm(): resident blocks of `kernel` per SM with `smem` bytes
// of dynamic shared memory (cached; raises the kernel's dynamic shared-memory limit
// once). launch_pdl(): launches `k` as a programmatic dependent of the stream's previous
// kernel.
cudaError_t note(cudaError_t e);
cudaError_t device_sms(int dev, int* sms);
cudaError_t blocks_per_sm(int dev, const void* kernel, int threads, size_t smem, int* blocks);
cudaError_t launch_pdl(const void* k, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args);

}  // namespace csa
