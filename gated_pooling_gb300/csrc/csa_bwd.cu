// csa_bwd.cu -- backward instantiations of the pooling kernel (4 columns per thread,
// so that the per-thread dAPE sums fit in registers).
#include "csa_internal.h"

namespace csa {

PoolKernel bwd_kernel_for(const Plan& pl) {
  if (pl.vec != 4) return nullptr;
  if (pl.split) return pl.pp == 8 ? pool_kernel<4, 8, true, true> : nullptr;
  switch (pl.pp) {
    case 1: return pool_kernel<4, 1, true, false>;
    case 2: return pool_kernel<4, 2, true, false>;
    case 4: return pool_kernel<4, 4, true, false>;
    case 8: return pool_kernel<4, 8, true, false>;
    default: return nullptr;
  }
}

}  // namespace csa
