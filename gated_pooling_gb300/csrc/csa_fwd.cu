// csa_fwd.cu -- forward instantiations of the pooling kernel (8 columns per thread).
#include "csa_internal.h"

namespace csa {

PoolKernel fwd_kernel_for(const Plan& pl) {
  if (pl.vec != 8) return nullptr;
  if (pl.split) return pl.pp == 8 ? pool_kernel<8, 8, false, true> : nullptr;
  switch (pl.pp) {
    case 1: return pool_kernel<8, 1, false, false>;
    case 2: return pool_kernel<8, 2, false, false>;
    case 4: return pool_kernel<8, 4, false, false>;
    case 8: return pool_kernel<8, 8, false, false>;
    default: return nullptr;
  }
}

}  // namespace csa
