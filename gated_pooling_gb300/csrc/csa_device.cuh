// csa_device.cuh -- device helpers of the GB300 CSA/HCA compressor pooling:
// bf16 packing, streaming vector loads/stores, and the THD index map (cu_seqlens ->
// per-segment block prefix in shared memory -> segment of an output row).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)

// ---------------------------------------------------------------------------------
// bf16 <-> fp32. A 32-bit word holds two bf16 values, the lower column in the low half.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> two bf16 (round to nearest even), lower column in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x with the hardware approximation (relative error about 2^-22; x = -inf gives 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------
// Vector IO: NW 32-bit words (NW = 2: 8 bytes, NW = 4: 16 bytes). Streaming loads are
// read once (evict first, no L1 allocation); ape goes through the read-only path.
// ---------------------------------------------------------------------------------
template <int NW>
__device__ __forceinline__ void load_stream(uint32_t (&v)[NW], const uint16_t* p);

template <>
__device__ __forceinline__ void load_stream<4>(uint32_t (&v)[4], const uint16_t* p) {
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "l"(p));
}
template <>
__device__ __forceinline__ void load_stream<2>(uint32_t (&v)[2], const uint16_t* p) {
  asm volatile("ld.global.cs.v2.u32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "l"(p));
}

template <int NW>
__device__ __forceinline__ void store_stream(uint16_t* p, const uint32_t (&v)[NW]);

template <>
__device__ __forceinline__ void store_stream<4>(uint16_t* p, const uint32_t (&v)[4]) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
template <>
__device__ __forceinline__ void store_stream<2>(uint16_t* p, const uint32_t (&v)[2]) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v[0]), "r"(v[1]) : "memory");
}

template <int NW>
__device__ __forceinline__ void store_zero(uint16_t* p) {
  uint32_t z[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) z[i] = 0u;
  store_stream<NW>(p, z);
}

// VEC consecutive fp32 ape values (VEC = 4 or 8), 16-byte aligned.
template <int VEC>
__device__ __forceinline__ void load_ape(float (&a)[VEC], const float* p) {
#pragma unroll
  for (int i = 0; i < VEC; i += 4) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(p + i));
    a[i] = t.x;
    a[i + 1] = t.y;
    a[i + 2] = t.z;
    a[i + 3] = t.w;
  }
}

// ---------------------------------------------------------------------------------
// THD index map
// ---------------------------------------------------------------------------------

// Exclusive block-wide prefix sum of `val` (blockDim.x <= 1024). `total` receives the
// block's sum. `warp_sums` is 32 ints of shared memory. All threads must call it.
__device__ __forceinline__ int block_exclusive_scan(int val, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int x = val;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31 || threadIdx.x == blockDim.x - 1) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = x - val + (wid > 0 ? warp_sums[wid - 1] : 0);
  total = warp_sums[nw - 1];
  __syncthreads();
  return excl;
}

// Builds the block prefix sB[s] = sum_{s' < s} floor(L_s' / ratio), s = 0..S, in shared
// memory and returns total_comp = sB[S]. Checks cu_seqlens (cu[0] >= 0, non-decreasing,
// cu[S] <= capacity) and total_comp <= out_rows; on failure thread 0 writes the code to
// *dev_error (if given) and every thread gets -1. Every thread of the block must call it.
__device__ __forceinline__ int build_block_prefix(const int32_t* __restrict__ cu, int S,
                                                  int ratio, int64_t capacity, int64_t out_rows,
                                                  int32_t* dev_error, int* sB, int* warp_sums) {
  int carry = 0;
  int bad = 0;
  if (threadIdx.x == 0) {
    const int c0 = __ldg(cu);
    const int cS = __ldg(cu + S);
    bad = (c0 < 0 || static_cast<int64_t>(cS) > capacity) ? 1 : 0;
  }
  for (int base = 0; base < S; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int n = 0;
    if (s < S) {
      const int a = __ldg(cu + s);
      const int b = __ldg(cu + s + 1);
      if (b < a) bad = 1;
      else n = (b - a) / ratio;
    }
    int chunk_total;
    const int excl = block_exclusive_scan(n, warp_sums, chunk_total);
    if (s < S) sB[s] = carry + excl;
    carry += chunk_total;
  }
  if (threadIdx.x == 0) sB[S] = carry;
  bad = __syncthreads_or(bad);
  int code = 0;
  if (bad) code = 1;                                       // CSA_DEVERR_CU_SEQLENS
  else if (static_cast<int64_t>(carry) > out_rows) code = 2;  // CSA_DEVERR_OUT_ROWS
  if (code != 0) {
    if (threadIdx.x == 0 && dev_error != nullptr) *reinterpret_cast<volatile int32_t*>(dev_error) = code;
    return -1;
  }
  return carry;
}

// Segment of output row o (0 <= o < sB[S]): the largest s with sB[s] <= o. Segments
// without blocks share their sB value with the next segment and are skipped.
__device__ __forceinline__ int find_segment(const int* sB, int S, int o) {
  int lo = 0, hi = S;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sB[mid] <= o) lo = mid;
    else hi = mid;
  }
  return lo;
}

// First s in [lo, hi) with sB[s] >= v (hi if none).
__device__ __forceinline__ int lower_bound_prefix(const int* sB, int lo, int hi, int v) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sB[mid] < v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

}  // namespace csa
