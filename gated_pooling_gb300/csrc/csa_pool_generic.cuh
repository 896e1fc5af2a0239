// csa_pool_generic.cuh -- pooling kernel for any head dim and naturally aligned pointers
// (the 1-wide path of "Megatron-LM PR #5984", commit "widen the validated envelope to coff
// in {1, 2}": head dims that are not a multiple of the vector width), forward and backward,
// windows of up to CSA_MAX_GENERIC_WINDOW positions.
//
// Same operation and zero ownership as pool_kernel (csa_pool.cuh), in the plainest layout:
// a CTA of 128 threads owns 128 consecutive columns of each half (thread = column j) and a
// contiguous range of output rows. Per row a thread reads its column's window with scalar
// loads (bf16 values and the fp32 ape through the read-only path), takes the max in a
// first pass, the sums in a second and, backward, recomputes the softmax terms in a third
// pass that writes dKV and dScore. The backward's dAPE sums of a thread (one per window
// position) live in shared memory, [position][thread], and become the CTA's partial.
// Used only where the vector kernels cannot run; it is correct for every shape it accepts,
// not fast.
#pragma once

#include "csa_pool.cuh"

namespace csa {

constexpr int kGenericThreads = 128;

__device__ __forceinline__ float bf16_at(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)))
                         << 16);
}
__device__ __forceinline__ void store_bf16(uint16_t* p, float v) {
  *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(pack_bf16x2(v, 0.f) & 0xFFFFu);
}
__device__ __forceinline__ void store_bf16_zero(uint16_t* p) {
  *reinterpret_cast<unsigned short*>(p) = 0;
}

template <bool BWD>
__global__ void __launch_bounds__(kGenericThreads) pool_generic_kernel(const PoolParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  int* sB = reinterpret_cast<int*>(smem);
  // cu_seqlens is cached after the block prefix when the plan left room for it (ape_off
  // past both arrays); with many segments and a long backward window it is read from
  // global memory instead, so that the dAPE sums fit
  const bool cu_cached = p.ape_off >= p.sB_words * 8;
  int* sCu = sB + p.sB_words;
  float* acc = reinterpret_cast<float*>(smem + p.ape_off);  // backward: [W][128] dAPE sums
  auto cu_at = [&](const int s) -> int { return cu_cached ? sCu[s] : __ldg(p.cu + s); };

  const int TC = build_block_prefix(p.cu, p.S, p.r, p.capacity, p.out_rows, p.dev_error, sB,
                                    warp_sums, cu_cached ? sCu : nullptr);
  publish_status(p, TC);
  if (TC < 0) return;
  // (no early launch of the stream's next kernel: it starts when this grid ends, which
  // measured faster than a trigger after the map build, e.g. 1 x 8192 d128 backward 13.3
  // -> 11.6 us, the long-window step 87.0 -> 84.2 us)

  const int tid = threadIdx.x;
  const int r = p.r, d = p.d, C = p.C, W = p.W;
  const bool two = p.coff == 2;
  const int j = blockIdx.x * kGenericThreads + tid;  // this thread's column in each half
  const bool col_ok = j < d;
  const int g = blockIdx.y;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);

  // window position w of a row whose own block starts at token `base`: token, column, ape
  auto tok_of = [&](int base, int w) { return two ? base - r + w : base + w; };
  auto col_of = [&](int w) { return (two && w >= r) ? d + j : j; };
  auto arow_of = [&](int w) { return (two && w >= r) ? w - r : w; };

  if constexpr (BWD) {
    for (int w = 0; w < W; ++w) acc[w * kGenericThreads + tid] = 0.f;
    if (col_ok) {
      // zeros of segments shorter than ratio whose block offset lies in this row group,
      // and of this row group's share of the rows outside [cu[0], cu[S]), this column
      auto zero_row = [&](int64_t t) {
        store_bf16_zero(p.dkv + t * C + j);
        store_bf16_zero(p.dscore + t * C + j);
        if (two) {
          store_bf16_zero(p.dkv + t * C + d + j);
          store_bf16_zero(p.dscore + t * C + d + j);
        }
      };
      const int s_lo = lower_bound_prefix(sB, 0, p.S, o0);
      const int s_hi = (g == p.R - 1) ? p.S : lower_bound_prefix(sB, s_lo, p.S, o1);
      for (int s = s_lo; s < s_hi; ++s) {
        const int a = cu_at(s), b = cu_at(s + 1);
        if (b - a < r)
          for (int t = a; t < b; ++t) zero_row(t);
      }
      const int64_t c_first = cu_at(0);
      const int64_t c_last = cu_at(p.S);
      const int64_t npad = c_first + (p.capacity - c_last);
      const int64_t q0 = static_cast<int64_t>(g) * npad / p.R;
      const int64_t q1 = static_cast<int64_t>(g + 1) * npad / p.R;
      for (int64_t q = q0; q < q1; ++q) zero_row(q < c_first ? q : c_last + (q - c_first));
    }
  }

  if (col_ok && o1 > o0) {
    int s = find_segment(sB, p.S, o0);
    for (int o = o0; o < o1; ++o) {
      s = advance_segment(sB, s, o);
      const int b = o - sB[s];
      const int n = sB[s + 1] - sB[s];
      const int base = cu_at(s) + b * r;
      const int w0 = (two && b == 0) ? r : 0;  // first block: no previous half
      auto x_at = [&](int w) {
        const int64_t off = static_cast<int64_t>(tok_of(base, w)) * C + col_of(w);
        return fmaf(bf16_at(p.score + off), kLog2e,
                    __ldg(p.ape + static_cast<int64_t>(arow_of(w)) * C + col_of(w)) * kLog2e);
      };
      float m = -INFINITY;
      for (int w = w0; w < W; ++w) m = fmaxf(m, x_at(w));
      float z = 0.f, a = 0.f;
      for (int w = w0; w < W; ++w) {
        const float e = fast_exp2(x_at(w) - m);
        z += e;
        a = fmaf(e, bf16_at(p.kv + static_cast<int64_t>(tok_of(base, w)) * C + col_of(w)), a);
      }
      const float rz = rcp_nr(z);
      const float oc = a * rz;
      if constexpr (!BWD) {
        store_bf16(p.out + static_cast<int64_t>(o) * d + j, oc);
      } else {
        const float qg = rz * bf16_at(p.dout + static_cast<int64_t>(o) * d + j);
        for (int w = w0; w < W; ++w) {
          const int64_t off = static_cast<int64_t>(tok_of(base, w)) * C + col_of(w);
          const float kk = fast_exp2(x_at(w) - m) * qg;
          const float t = kk * (bf16_at(p.kv + off) - oc);
          acc[w * kGenericThreads + tid] += t;
          store_bf16(p.dkv + off, kk);
          store_bf16(p.dscore + off, t);
        }
        if (b == n - 1) {  // zeros owned by a segment's last block
          if (two)
            for (int k = 0; k < r; ++k) {
              const int64_t offz = static_cast<int64_t>(base + k) * C + j;
              store_bf16_zero(p.dkv + offz);
              store_bf16_zero(p.dscore + offz);
            }
          for (int t = cu_at(s) + n * r, te = cu_at(s + 1); t < te; ++t) {
            const int64_t offz = static_cast<int64_t>(t) * C + j;
            store_bf16_zero(p.dkv + offz);
            store_bf16_zero(p.dscore + offz);
            if (two) {
              store_bf16_zero(p.dkv + offz + d);
              store_bf16_zero(p.dscore + offz + d);
            }
          }
        }
      }
    }
  }

  if constexpr (BWD) {  // this thread's dAPE sums are the CTA's partial for its column
    if (col_ok) {
      float* dst = p.partial + static_cast<int64_t>(g) * r * C;
      for (int w = 0; w < W; ++w)
        dst[static_cast<int64_t>(arow_of(w)) * C + col_of(w)] = acc[w * kGenericThreads + tid];
    }
  }
}

}  // namespace csa
