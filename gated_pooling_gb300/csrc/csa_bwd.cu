// csa_bwd.cu -- backward instantiations of the pooling kernels (generic, long window,
// block streaming with 4 columns per thread so that the per-thread dAPE sums fit in
// registers, split window) and the plan -> kernel choice.
#include "csa_internal.h"
#include "csa_pool_generic.cuh"
#include "csa_pool_long.cuh"
#include "csa_pool_stream.cuh"

namespace csa {

PoolKernel bwd_kernel_for(const Plan& pl) {
  if (pl.generic) return pool_generic_kernel<true>;
  if (pl.longk)
    return pl.sc == 32 ? long_kernel_for<true, 32>(pl.pp, pl.coff == 2)
                       : long_kernel_for<true, 64>(pl.pp, pl.coff == 2);
  if (pl.tma) {
    const int r = pl.pp / pl.coff, coff = pl.coff;
    // one producer warp or all of them (the plan's np)
#define CSA_STREAM_PICK(RR, CC)                                                              \
  if (r == RR && coff == CC)                                                                 \
    return pl.np == 1 ? pool_stream_kernel<CSA_BWD_VEC, CSA_BWD_CONSUMERS, RR, CC, true, 1>             \
                      : pool_stream_kernel<CSA_BWD_VEC, CSA_BWD_CONSUMERS, RR, CC, true,                \
                                           stream_producers(true)>;
    CSA_STREAM_PICK(1, 1)
    CSA_STREAM_PICK(2, 1)
    CSA_STREAM_PICK(4, 1)
    CSA_STREAM_PICK(8, 1)
    CSA_STREAM_PICK(1, 2)
    CSA_STREAM_PICK(2, 2)
    CSA_STREAM_PICK(4, 2)
#undef CSA_STREAM_PICK
    return nullptr;
  }
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
