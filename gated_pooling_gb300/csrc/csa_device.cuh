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

// 1/z to within about one ulp: hardware approximation plus one Newton step.
__device__ __forceinline__ float rcp_nr(float z) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
  const float e = fmaf(-z, r, 1.f);
  return fmaf(r, e, r);
}

// 2^x for the softmax weights. By default the hardware approximation (relative error about
// 2^-22; x = -inf gives 0); built with CSA_FAST_EXP2=0, CUDA's exp2f. Both stay within the
// parity tolerance; the approximation measured faster (the numbers are kept with the
// kernel notes).
#ifndef CSA_FAST_EXP2
#define CSA_FAST_EXP2 1
#endif
__device__ __forceinline__ float fast_exp2(float x) {
#if CSA_FAST_EXP2
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
#else
  return exp2f(x);
#endif
}

// ---------------------------------------------------------------------------------
// Vector IO: NW 32-bit words (NW = 1, 2 or 4: 4, 8 or 16 bytes). Streaming loads are
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
template <>
__device__ __forceinline__ void load_stream<1>(uint32_t (&v)[1], const uint16_t* p) {
  asm volatile("ld.global.cs.u32 %0, [%1];" : "=r"(v[0]) : "l"(p));
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
template <>
__device__ __forceinline__ void store_stream<1>(uint16_t* p, const uint32_t (&v)[1]) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v[0]) : "memory");
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

// Programmatic dependent launch. The kernels are launched as programmatic dependents of
// the previous kernel of their stream; pdl_wait (the first thing the map builders do,
// before any global memory access) holds them until that grid has completed and its
// memory is visible. It returns at once when the kernel was launched normally. No kernel
// of this library triggers its own dependents early (measured slower): the next kernel
// starts when the grid ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Builds the block prefix sB[s] = sum_{s' < s} floor(L_s' / ratio), s = 0..S, in shared
// memory and returns total_comp = sB[S]. Checks cu_seqlens (cu[0] >= 0, non-decreasing,
// cu[S] <= capacity) and total_comp <= out_rows; on failure thread 0 writes the code to
// *dev_error (if given) and every thread gets -1. Every thread of the block must call it.
__device__ __forceinline__ int build_block_prefix(const int32_t* __restrict__ cu, int S,
                                                  int ratio, int64_t capacity, int64_t out_rows,
                                                  int32_t* dev_error, int* sB, int* warp_sums,
                                                  int* sCu = nullptr) {
  pdl_wait();  // the previous kernel's results (cu_seqlens, inputs) are visible after this
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
      if (sCu != nullptr) sCu[s] = a;
      if (b < a) bad = 1;
      else n = (b - a) / ratio;
    }
    int chunk_total;
    const int excl = block_exclusive_scan(n, warp_sums, chunk_total);
    if (s < S) sB[s] = carry + excl;
    carry += chunk_total;
  }
  if (threadIdx.x == 0) {
    sB[S] = carry;
    if (sCu != nullptr) sCu[S] = __ldg(cu + S);
  }
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

// Segment of row o given the segment `s` of an earlier row (rows visited in increasing
// order): advances past segments that end at or before o.
__device__ __forceinline__ int advance_segment(const int* sB, int s, int o) {
  while (sB[s + 1] <= o) ++s;
  return s;
}

// First s in [lo, hi) with sB[s] > v (hi if none).
__device__ __forceinline__ int upper_bound_prefix(const int* sB, int lo, int hi, int v) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (sB[mid] <= v) lo = mid + 1;
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

// ---------------------------------------------------------------------------------
// Packed pairs of fp32 (two adjacent columns) for the sm_100-family f32x2 arithmetic:
// every lane is an IEEE round-to-nearest fp32 operation, two per instruction.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// A word of two bf16 (lower column in the low half) as an f32 pair (exact).
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// An f32 pair rounded to two bf16 (nearest even) in one word.
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t v) { return pack_bf16x2(f2_lo(v), f2_hi(v)); }
// Neumaier's compensated summation step (Neumaier 1974): s + c carries the running sum
// with the rounding error of every addition kept in c.
__device__ __forceinline__ void neumaier_add(float& s, float& c, float x) {
  const float t = s + x;
  c += (fabsf(s) >= fabsf(x)) ? ((s - t) + x) : ((x - t) + s);
  s = t;
}

// max of three fp32 (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace csa

namespace csa {

// ---------------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, 1-D) completing on shared-memory mbarriers.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// counted against `bar`'s transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte shared-memory load that the compiler may not merge with an earlier load of the
// same address (keeps re-reads from turning into long-lived registers).
__device__ __forceinline__ uint4 lds128_fresh(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// NW 32-bit words from shared memory (16, 8 or 4 bytes, aligned). The _fresh form is never
// merged with an earlier load of the same address.
template <int NW>
__device__ __forceinline__ void lds_words(uint32_t (&v)[NW], const void* p) {
  if constexpr (NW == 4) {
    const uint4 t = *reinterpret_cast<const uint4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else if constexpr (NW == 1) {
    v[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(p);
    v[0] = t.x; v[1] = t.y;
  }
}
template <int NW>
__device__ __forceinline__ void lds_words_fresh(uint32_t (&v)[NW], const void* p) {
  if constexpr (NW == 4) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(smem_addr(p)));
  } else if constexpr (NW == 1) {
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v[0]) : "r"(smem_addr(p)));
  } else {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(smem_addr(p)));
  }
}

// L2 policy for data read exactly once (evict first): keeps the stream from displacing
// other lines and raised bulk-copy streaming bandwidth on GB300 by about 10%.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_load with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with `parity` of `bar` to complete, giving up after about `limit`
// SM clock cycles (returns false then). No wait in this library is unbounded. The
// pipeline waits take the call's limit (PoolParams::wait_cycles, kWaitCycles unless a
// test shortened it); the waits that let a stopping CTA's own copies land before it
// exits always take kWaitCycles.
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at GB300 clocks
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

// Copies in flight when a CTA stops early. A CTA must not exit while a bulk copy into its
// shared memory is in flight. On the normal path its consumers wait for every copy, so
// the producers leave without waiting. A thread whose wait ran out stops the pipeline
// (stop_pipeline: sets the CTA's stop word), and then the copies already issued must still
// land. A producer that is done publishes how far it issued and then reads the stop word
// (producer_sees_stop); a stopping thread sets the stop word and then reads the published
// counts. Each side fences (sequentially consistent, CTA scope) between its store and its
// load, so at least one of them sees the other's store: a producer that sees the stop
// waits for its own copies, and a stopping thread that sees a producer's count waits for
// that producer's copies. (A producer whose count is not published yet sees the stop.)
__device__ __forceinline__ bool producer_sees_stop(int* issued_word, int issued, int* stop) {
  *reinterpret_cast<volatile int*>(issued_word) = issued;
  __threadfence_block();
  return *reinterpret_cast<volatile int*>(stop) != 0;
}
__device__ __forceinline__ void stop_pipeline(int* stop, int32_t* dev_error) {
  *reinterpret_cast<volatile int*>(stop) = 1;
  if (dev_error != nullptr) *reinterpret_cast<volatile int32_t*>(dev_error) = 3;  // timeout
  __threadfence_block();
}
__device__ __forceinline__ int read_issued(const int* issued_word) {
  return *reinterpret_cast<const volatile int*>(issued_word);
}


// Release store / acquire load of a shared-memory word (CTA scope): the row a ring slot
// was last armed for, written by the producer warp that armed it.
__device__ __forceinline__ void st_release_shared(int* p, int v) {
  asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
// Waits until *p == v; gives up (false) when *stop is set or after about `limit` cycles.
__device__ __forceinline__ bool wait_shared_eq(const int* p, int v, const int* stop,
                                               long long limit) {
  if (ld_acquire_shared(p) == v) return true;
  const long long t0 = clock64();
  while (ld_acquire_shared(p) != v)
    if (*reinterpret_cast<const volatile int*>(stop) != 0 || clock64() - t0 > limit) return false;
  return true;
}

}  // namespace csa
