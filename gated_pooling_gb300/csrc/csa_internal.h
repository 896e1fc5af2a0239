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

}  // namespace csa
