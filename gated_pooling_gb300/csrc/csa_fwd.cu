// csa_fwd.cu -- forward instantiations of the pooling kernels (generic, long window,
// register loads, block streaming, split window) and the plan -> kernel choice.
#include "csa_internal.h"
#include "csa_pool_generic.cuh"
#include "csa_pool_long.cuh"
#include "csa_fwd_ldg.cuh"
#include "csa_pool_stream.cuh"

namespace csa {

PoolKernel fwd_kernel_for(const Plan& pl) {
  if (pl.generic) return pool_generic_kernel<false>;
  if (pl.longk)
    return pl.sc == 32 ? long_kernel_for<false, 32>(pl.pp, pl.coff == 2)
                       : long_kernel_for<false, 64>(pl.pp, pl.coff == 2);
  if (pl.ldg) {
    const int r = pl.pp / pl.coff, coff = pl.coff;
#define CSA_LDG_PICK(RR, CC, VV)                                                    \
  if (r == RR && coff == CC && pl.vec == VV)                                        \
    return pool_fwd_ldg_kernel<ldg_threads(RR * CC, VV), RR, CC, VV>;
    CSA_LDG_PICK(1, 1, 4)
    CSA_LDG_PICK(2, 1, 4)
    CSA_LDG_PICK(4, 1, 4)
    CSA_LDG_PICK(8, 1, 4)
    CSA_LDG_PICK(1, 2, 4)
    CSA_LDG_PICK(2, 2, 4)
    CSA_LDG_PICK(4, 2, 4)
    CSA_LDG_PICK(1, 1, 8)
    CSA_LDG_PICK(2, 1, 8)
    CSA_LDG_PICK(1, 2, 8)
#if CSA_LDG_VEC8_MAX_WINDOW >= 4
    CSA_LDG_PICK(4, 1, 8)
    CSA_LDG_PICK(2, 2, 8)
#endif
#undef CSA_LDG_PICK
    return nullptr;
  }
  if (pl.tma) {
    const int r = pl.pp / pl.coff, coff = pl.coff;
    // one producer warp or all of them (the plan's np)
#define CSA_STREAM_PICK(RR, CC)                                                              \
  if (r == RR && coff == CC)                                                                 \
    return pl.np == 1 ? pool_stream_kernel<CSA_FWD_VEC, CSA_FWD_CONSUMERS, RR, CC, false, 1>             \
                      : pool_stream_kernel<CSA_FWD_VEC, CSA_FWD_CONSUMERS, RR, CC, false,                \
                                           stream_producers(false)>;
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
