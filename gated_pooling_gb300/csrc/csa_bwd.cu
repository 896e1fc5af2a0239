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
  if (pl.longk) {
    const bool two = pl.coff == 2;
    switch (pl.pp) {
      case 1: return two ? reinterpret_cast<PoolKernel>(pool_long_kernel<1, CSA_LONG_BWD_GROUPS, 2, true, 64>)
                         : reinterpret_cast<PoolKernel>(pool_long_kernel<1, CSA_LONG_BWD_GROUPS, 1, true, 64>);
      case 2: return two ? reinterpret_cast<PoolKernel>(pool_long_kernel<2, CSA_LONG_BWD_GROUPS, 2, true, 64>)
                         : reinterpret_cast<PoolKernel>(pool_long_kernel<2, CSA_LONG_BWD_GROUPS, 1, true, 64>);
      case 4: return two ? reinterpret_cast<PoolKernel>(pool_long_kernel<4, CSA_LONG_BWD_GROUPS, 2, true, 64>)
                         : reinterpret_cast<PoolKernel>(pool_long_kernel<4, CSA_LONG_BWD_GROUPS, 1, true, 64>);
      case 8: return two ? reinterpret_cast<PoolKernel>(pool_long_kernel<8, CSA_LONG_BWD_GROUPS, 2, true, 64>)
                         : reinterpret_cast<PoolKernel>(pool_long_kernel<8, CSA_LONG_BWD_GROUPS, 1, true, 64>);
      case 16:  // 256-position windows (ratio 128 at coff 2, ratio 256 at coff 1)
        if (pl.sc == 32)
          return two ? reinterpret_cast<PoolKernel>(
                           pool_long_kernel<16, long_groups(true, 256, 32), 2, true, 32>)
                     : reinterpret_cast<PoolKernel>(
                           pool_long_kernel<16, long_groups(true, 256, 32), 1, true, 32>);
        return two ? reinterpret_cast<PoolKernel>(
                         pool_long_kernel<16, long_groups(true, 256, 64), 2, true, 64>)
                   : reinterpret_cast<PoolKernel>(
                         pool_long_kernel<16, long_groups(true, 256, 64), 1, true, 64>);
      default: return nullptr;
    }
  }
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
