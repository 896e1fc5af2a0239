// csa_kpool.cu -- KPool, the DSA indexer's key pooling ("Megatron-LM PR #8835", the KPool
// commits: an FP32 softmax of a gate over pools of P consecutive keys, the pool grid
// restarting at each segment's first valid key; optional key-dtype compression, which casts
// the softmax weights to bf16 before multiplying and reducing).
//
// The pooling reads every key and gate once and writes one bf16 row per pool: it is bound
// by HBM bandwidth (per pool and column: 4P bytes read, 2 written). Two kernels:
//  * vector (d % 8 == 0, P <= 8, 16-byte aligned tensors): a thread owns 8 columns of a
//    pool and loads the pool's P 16-byte pieces of key and gate itself (evict-first), the
//    next pool's loads in flight while one is computed; it works through the 8 columns a
//    pair at a time with the f32x2 instructions. Persistent CTAs own contiguous pool ranges,
//    split over their row slots.
//  * scalar (anything else): a thread owns one column of a pool and walks the pool's keys
//    (max; weights, normaliser and sum; compressed: the bf16 products), re-reading from L1.
// Both build the pool prefix (pools per segment, prefix sums, first valid keys) in shared
// memory first, and check cu_seqlens and the leads there.
#include <climits>
#include <cstdint>

#include "csa_compressor.h"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kKpThreads = 256;

struct KPoolParams {
  const uint16_t* key;
  const uint16_t* gate;
  const int32_t* cu;
  const int32_t* lead;  // or nullptr
  uint16_t* out;
  int32_t* dev_error;
  int64_t capacity;
  int64_t out_rows;
  int S, P, d;
  int V;      // vector kernel: 8-column chunks per row (d / 8)
  int slots;  // vector kernel: rows computed at once per CTA (threads / V)
  int R;      // CTAs (row groups)
  int sB_words;
};

// Pool prefix: sB[s] = pools of the segments before s (s = 0..S) and sF[s] = first valid
// key of segment s, in shared memory. Returns the pool count, or -1 after thread 0 wrote
// a code to *dev_error: CSA_DEVERR_CU_SEQLENS (cu[0] < 0, decreasing, or past capacity),
// CSA_DEVERR_LEAD (a negative lead), CSA_DEVERR_OUT_ROWS (more pools than out_rows).
// Every thread of the block must call it. Waits for the stream's previous grid first.
__device__ int build_pool_prefix(const KPoolParams& p, int* sB, int* sF, int* warp_sums) {
  pdl_wait();
  int carry = 0;
  int bad_cu = 0, bad_lead = 0;
  if (threadIdx.x == 0) {
    const int c0 = __ldg(p.cu);
    const int cS = __ldg(p.cu + p.S);
    bad_cu = (c0 < 0 || static_cast<int64_t>(cS) > p.capacity) ? 1 : 0;
  }
  for (int base = 0; base < p.S; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int n = 0;
    if (s < p.S) {
      const int a = __ldg(p.cu + s);
      const int b = __ldg(p.cu + s + 1);
      const int l = p.lead != nullptr ? __ldg(p.lead + s) : 0;
      if (b < a) {
        bad_cu = 1;
      } else if (l < 0) {
        bad_lead = 1;
      } else {
        const int64_t first = static_cast<int64_t>(a) + l;
        sF[s] = first < b ? static_cast<int>(first) : b;
        n = first < b ? (b - static_cast<int>(first)) / p.P : 0;
      }
    }
    int chunk_total;
    const int excl = block_exclusive_scan(n, warp_sums, chunk_total);
    if (s < p.S) sB[s] = carry + excl;
    carry += chunk_total;
  }
  if (threadIdx.x == 0) sB[p.S] = carry;
  bad_cu = __syncthreads_or(bad_cu);
  bad_lead = __syncthreads_or(bad_lead);
  int code = 0;
  if (bad_cu) code = CSA_DEVERR_CU_SEQLENS;
  else if (bad_lead) code = CSA_DEVERR_LEAD;
  else if (static_cast<int64_t>(carry) > p.out_rows) code = CSA_DEVERR_OUT_ROWS;
  if (code != 0) {
    if (threadIdx.x == 0 && p.dev_error != nullptr)
      *reinterpret_cast<volatile int32_t*>(p.dev_error) = code;
    return -1;
  }
  return carry;
}

// ---------------------------------------------------------------------------------------
// Vector kernel. PT: the largest pool it holds in registers (P <= PT at run time).
// ---------------------------------------------------------------------------------------
template <int PT, bool COMPRESS>
__global__ void __launch_bounds__(kKpThreads, PT <= 2 ? 3 : (PT <= 4 ? 2 : 1))
    kpool_vec_kernel(const KPoolParams p) {
  constexpr int NW = 4;  // 32-bit words (bf16 column pairs) per thread: 8 columns
  extern __shared__ __align__(16) int smem[];
  __shared__ int warp_sums[32];
  int* sB = smem;
  int* sF = sB + p.sB_words;
  const int TC = build_pool_prefix(p, sB, sF, warp_sums);
  if (TC < 0) return;
  // (no early launch of the stream's next kernel: measured slower, as for the pooling)

  const int g = blockIdx.x;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);
  const int nrows = o1 - o0;
  const int tid = threadIdx.x;
  const int rs = tid / p.V;  // row slot
  const int c0 = (tid % p.V) * 8;
  if (rs >= p.slots || rs >= nrows) return;
  const int P = p.P;

  int seg = find_segment(sB, p.S, o0 + rs);
  auto fetch = [&](const int j, uint32_t (&kw)[PT][NW], uint32_t (&gw)[PT][NW]) {
    const int o = o0 + j;
    seg = advance_segment(sB, seg, o);
    const int64_t t0 = static_cast<int64_t>(sF[seg]) + static_cast<int64_t>(o - sB[seg]) * P;
#pragma unroll
    for (int i = 0; i < PT; ++i) {
      if (i < P) {
        const int64_t off = (t0 + i) * p.d + c0;
        load_stream<NW>(kw[i], p.key + off);
        load_stream<NW>(gw[i], p.gate + off);
      }
    }
  };

  const uint64_t kL2 = f2_pack(kLog2e, kLog2e);
  auto compute = [&](const int j, const uint32_t (&kw)[PT][NW], const uint32_t (&gw)[PT][NW]) {
    uint32_t ow[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {  // one column pair at a time
      uint64_t x[PT];
#pragma unroll
      for (int i = 0; i < PT; ++i)
        if (i < P) x[i] = f2_mul(bf2_to_f2(gw[i][q]), kL2);  // gate * log2 e
      float mlo = f2_lo(x[0]), mhi = f2_hi(x[0]);
#pragma unroll
      for (int i = 1; i < PT; ++i) {
        if (i < P) {
          mlo = fmaxf(mlo, f2_lo(x[i]));
          mhi = fmaxf(mhi, f2_hi(x[i]));
        }
      }
      const uint64_t nm = f2_pack(-mlo, -mhi);
      uint64_t z = 0ull;
#pragma unroll
      for (int i = 0; i < PT; ++i) {
        if (i < P) {
          const uint64_t dd = f2_add(x[i], nm);
          x[i] = f2_pack(fast_exp2(f2_lo(dd)), fast_exp2(f2_hi(dd)));  // e = 2^(x - m)
          z = f2_add(z, x[i]);
        }
      }
      const uint64_t rz = f2_pack(rcp_nr(f2_lo(z)), rcp_nr(f2_hi(z)));
      uint64_t a = 0ull;
      if constexpr (!COMPRESS) {
#pragma unroll
        for (int i = 0; i < PT; ++i)
          if (i < P) a = f2_fma(x[i], bf2_to_f2(kw[i][q]), a);
        ow[q] = f2_to_bf2(f2_mul(a, rz));
      } else {
        // weights cast to bf16, each product cast to bf16 (the fp32 product of two bf16
        // values is exact), the products summed in fp32 and the sum cast to bf16
#pragma unroll
        for (int i = 0; i < PT; ++i) {
          if (i < P) {
            const uint64_t pb = bf2_to_f2(f2_to_bf2(f2_mul(x[i], rz)));
            a = f2_add(a, bf2_to_f2(f2_to_bf2(f2_mul(pb, bf2_to_f2(kw[i][q])))));
          }
        }
        ow[q] = f2_to_bf2(a);
      }
    }
    store_stream<NW>(p.out + static_cast<int64_t>(o0 + j) * p.d + c0, ow);
  };

  // two register buffers: the next row's loads are in flight while one is computed
  uint32_t kb[2][PT][NW], gb[2][PT][NW];
  fetch(rs, kb[0], gb[0]);
  for (int j = rs; j < nrows;) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (j < nrows) {
        const int jn = j + p.slots;
        if (jn < nrows) fetch(jn, kb[b ^ 1], gb[b ^ 1]);
        compute(j, kb[b], gb[b]);
        j += p.slots;
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Scalar kernel: any pool size, head dim and (natural) alignment.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_at(const uint16_t* p, int64_t i) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p) + i))
                         << 16);
}
__device__ __forceinline__ float round_bf16(float x) {
  return __uint_as_float(pack_bf16x2(x, 0.f) << 16);
}

template <bool COMPRESS>
__global__ void __launch_bounds__(kKpThreads) kpool_scalar_kernel(const KPoolParams p) {
  extern __shared__ __align__(16) int smem[];
  __shared__ int warp_sums[32];
  int* sB = smem;
  int* sF = sB + p.sB_words;
  const int TC = build_pool_prefix(p, sB, sF, warp_sums);
  if (TC < 0) return;

  const int g = blockIdx.x;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);
  const int64_t items = static_cast<int64_t>(o1 - o0) * p.d;
  const int P = p.P;
  for (int64_t it = threadIdx.x; it < items; it += blockDim.x) {
    const int o = o0 + static_cast<int>(it / p.d);
    const int j = static_cast<int>(it % p.d);
    const int s = find_segment(sB, p.S, o);
    const int64_t t0 = static_cast<int64_t>(sF[s]) + static_cast<int64_t>(o - sB[s]) * P;
    const int64_t base = t0 * p.d + j;
    float m = -INFINITY;
    for (int i = 0; i < P; ++i) m = fmaxf(m, bf16_at(p.gate, base + static_cast<int64_t>(i) * p.d) * kLog2e);
    float z = 0.f, a = 0.f;
    for (int i = 0; i < P; ++i) {
      const int64_t k = base + static_cast<int64_t>(i) * p.d;
      const float e = fast_exp2(bf16_at(p.gate, k) * kLog2e - m);
      z += e;
      if constexpr (!COMPRESS) a = fmaf(e, bf16_at(p.key, k), a);
    }
    const float rz = rcp_nr(z);
    float y;
    if constexpr (!COMPRESS) {
      y = a * rz;
    } else {
      y = 0.f;
      for (int i = 0; i < P; ++i) {
        const int64_t k = base + static_cast<int64_t>(i) * p.d;
        const float e = fast_exp2(bf16_at(p.gate, k) * kLog2e - m);  // the same e as above
        y += round_bf16(round_bf16(e * rz) * bf16_at(p.key, k));
      }
    }
    const uint32_t w = pack_bf16x2(y, 0.f);
    reinterpret_cast<unsigned short*>(p.out)[static_cast<int64_t>(o) * p.d + j] =
        static_cast<unsigned short>(w & 0xFFFFu);
  }
}

using KPoolKernel = void (*)(KPoolParams);

KPoolKernel vec_kernel_for(int P, bool compress) {
  if (P <= 2) return compress ? kpool_vec_kernel<2, true> : kpool_vec_kernel<2, false>;
  if (P <= 4) return compress ? kpool_vec_kernel<4, true> : kpool_vec_kernel<4, false>;
  return compress ? kpool_vec_kernel<8, true> : kpool_vec_kernel<8, false>;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" int64_t csa_kpool_total(const int32_t* cu_seqlens_host, const int32_t* lead_host,
                                   int32_t S, int32_t pool) {
  if (cu_seqlens_host == nullptr || S < 0 || pool < 1) return -1;
  int64_t total = 0;
  for (int s = 0; s < S; ++s) {
    const int64_t a = cu_seqlens_host[s], b = cu_seqlens_host[s + 1];
    const int64_t l = lead_host != nullptr ? lead_host[s] : 0;
    if (b < a || l < 0) return -1;
    if (b - a > l) total += (b - a - l) / pool;
  }
  return total;
}

extern "C" csa_status_t csa_kpool_fwd(const void* key, const void* gate, const int32_t* cu_seqlens,
                                      const int32_t* lead, int32_t S, int32_t pool, int32_t d,
                                      int64_t capacity, void* out, int64_t out_rows,
                                      int32_t compress, int32_t* dev_error, csa_stream_t stream) {
  if (S < 0 || pool < 1 || d < 1 || capacity < 0 || out_rows < 0 ||
      (compress != 0 && compress != 1))
    return CSA_ERR_INVALID_VALUE;
  if (S > CSA_MAX_SEGMENTS || pool > CSA_KPOOL_MAX_POOL) return CSA_ERR_UNSUPPORTED;
  if (capacity > CSA_MAX_ELEMS / d || out_rows > CSA_MAX_ELEMS / d) return CSA_ERR_UNSUPPORTED;
  if (cu_seqlens == nullptr) return CSA_ERR_INVALID_VALUE;
  if (capacity > 0 && (key == nullptr || gate == nullptr)) return CSA_ERR_INVALID_VALUE;
  if (out_rows > 0 && out == nullptr) return CSA_ERR_INVALID_VALUE;
  if (!aligned_to(key, 2) || !aligned_to(gate, 2) || !aligned_to(out, 2) ||
      !aligned_to(cu_seqlens, 4) || !aligned_to(lead, 4) || !aligned_to(dev_error, 4))
    return CSA_ERR_INVALID_VALUE;
  if (S == 0) return CSA_OK;  // no segment, no pool: nothing to enqueue

  KPoolParams p{};
  p.key = static_cast<const uint16_t*>(key);
  p.gate = static_cast<const uint16_t*>(gate);
  p.cu = cu_seqlens;
  p.lead = lead;
  p.out = static_cast<uint16_t*>(out);
  p.dev_error = dev_error;
  p.capacity = capacity;
  p.out_rows = out_rows;
  p.S = S;
  p.P = pool;
  p.d = d;
  p.sB_words = ((S + 1) + 3) & ~3;
  const bool vec = d % 8 == 0 && d / 8 <= kKpThreads && pool <= 8 && aligned_to(key, 16) &&
                   aligned_to(gate, 16) && aligned_to(out, 16);
  KPoolKernel k;
  if (vec) {
    k = vec_kernel_for(pool, compress != 0);
    p.V = d / 8;
    p.slots = kKpThreads / p.V;
  } else {
    k = compress != 0 ? kpool_scalar_kernel<true> : kpool_scalar_kernel<false>;
    p.V = 0;
    p.slots = 0;
  }
  const size_t smem = static_cast<size_t>(2 * p.sB_words) * sizeof(int);
  int dev = 0, sms = 0, bps = 0;
  if (note(cudaGetDevice(&dev)) != cudaSuccess) return CSA_ERR_CUDA;
  if (device_sms(dev, &sms) != cudaSuccess) return CSA_ERR_CUDA;
  if (blocks_per_sm(dev, reinterpret_cast<const void*>(k), kKpThreads, smem, &bps) !=
      cudaSuccess)
    return CSA_ERR_CUDA;
  if (bps < 1) return CSA_ERR_UNSUPPORTED;
  const int64_t want = static_cast<int64_t>(sms) * bps;
  const int64_t cap = out_rows > 0 ? out_rows : 1;
  p.R = static_cast<int>(want < cap ? want : cap);
  void* args[] = {&p};
  if (launch_pdl(reinterpret_cast<const void*>(k), dim3(p.R), dim3(kKpThreads), smem,
                 reinterpret_cast<cudaStream_t>(stream), args) != cudaSuccess)
    return CSA_ERR_CUDA;
  return CSA_OK;
}
