// csa_fwd_ldg.cuh -- forward pooling through register loads, for windows of up to 8
// positions (same operation as csa_pool_stream.cuh; "Megatron-LM PR #5984", commit "CSA:
// add fused Compressor forward+backward CuTe-DSL kernels").
//
// The forward reads ~95% of its bytes. For short windows and narrow rows the bulk-copy
// pipeline's per-row and start-up costs dominate (a stage per row of a few KB), so this
// variant keeps everything in registers: each thread
// owns one chunk of VEC columns of a row (both halves at coff=2) and loads, per row, the
// 2*W pieces of its window (kv and score) itself: 16-byte pieces (8 columns) for windows
// of up to 2 positions, 8-byte pieces (4 columns) for longer windows, whose buffers keep
// more rows in flight at 8 bytes. The loads of the thread's next
// PF rows are in flight while a row is computed (a ring of PF + 1 register buffers; PF is
// larger for shorter windows, whose buffers are smaller), so that enough bytes are in
// flight to cover the memory latency. CTAs are persistent (one per SM, or two) and own a
// contiguous range of rows, split over their row slots.
#pragma once

#include "csa_pool.cuh"

namespace csa {

template <int NT, int R, int COFF, int VEC>
__global__ void __launch_bounds__(NT, CSA_LDG_CTAS) pool_fwd_ldg_kernel(const PoolParams p) {
  static_assert(VEC == 4 || VEC == 8, "chunks of 4 or 8 columns");
  constexpr int NW = VEC / 2;  // 32-bit words (column pairs) per piece
  constexpr int NQ = VEC / 4;  // ape float4s per chunk
  constexpr int W = R * COFF;
  constexpr bool TWO = COFF == 2;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  int* sB = reinterpret_cast<int*>(smem);
  int* sCu = sB + p.sB_words;
  float4* sA = reinterpret_cast<float4*>(smem + p.ape_off);  // [W][V][NQ] float4, x log2(e)

  const int TC = build_block_prefix(p.cu, p.S, R, p.capacity, p.out_rows, p.dev_error, sB,
                                    warp_sums, sCu);
  publish_status(p, TC);
  if (TC < 0) return;

  const int tid = threadIdx.x;
  const int d = p.d, C = p.C, V = p.V;
  const int g = blockIdx.y;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);
  const int nrows = o1 - o0;

  for (int it = tid; it < W * V * NQ; it += NT) {
    const int w = it / (V * NQ);
    const int ch = (it / NQ) % V;
    const bool prev = TWO && w < R;
    const int arow = (TWO && !prev) ? w - R : w;
    const int col = ((TWO && !prev) ? d : 0) + ch * VEC + (it % NQ) * 4;
    float4 a = __ldg(reinterpret_cast<const float4*>(p.ape + static_cast<int64_t>(arow) * C + col));
    a.x *= kLog2e;
    a.y *= kLog2e;
    a.z *= kLog2e;
    a.w *= kLog2e;
    sA[it] = a;
  }
  __syncthreads();

  const int rs = tid / V;
  const int vl = tid % V;
  const int c0 = vl * VEC;
  if (rs >= p.slots || rs >= nrows) return;
  const uint64_t kL2 = f2_pack(kLog2e, kLog2e);

  // window of row o for this chunk: kv and score words of the W positions (masked
  // positions of a segment's first block stay zero and are flagged by has_prev = false)
  int seg = find_segment(sB, p.S, o0 + rs);
  auto fetch = [&](const int j, uint32_t (&kv)[W][NW], uint32_t (&sc)[W][NW], bool& has_prev) {
    const int o = o0 + j;
    seg = advance_segment(sB, seg, o);
    const int b = o - sB[seg];
    has_prev = TWO && b >= 1;
    const int64_t own = (static_cast<int64_t>(sCu[seg]) + static_cast<int64_t>(b) * R) * C +
                        (TWO ? d : 0) + c0;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const bool prev = TWO && i < R;
      if (prev && !has_prev) {
#pragma unroll
        for (int q = 0; q < NW; ++q) kv[i][q] = sc[i][q] = 0u;
        continue;
      }
      const int64_t off = prev ? own - d - static_cast<int64_t>(R - i) * C
                               : own + static_cast<int64_t>(TWO ? i - R : i) * C;
      load_stream<NW>(kv[i], p.kv + off);
      load_stream<NW>(sc[i], p.score + off);
    }
  };

  // rows in flight ahead of the one being computed (16-byte pieces: one row fewer, for the
  // same bytes in flight)
#ifndef CSA_LDG_PF4
#define CSA_LDG_PF4 2  // rows ahead for windows of 4 positions
#endif
#ifndef CSA_LDG_PF4_V8
#define CSA_LDG_PF4_V8 1  // the same with 16-byte pieces
#endif
  constexpr int PF = W >= 8 ? 1 : (W >= 4 ? (VEC == 8 ? CSA_LDG_PF4_V8 : CSA_LDG_PF4) : (VEC == 8 ? 2 : 3));
  uint32_t kv[PF + 1][W][NW], sc[PF + 1][W][NW];
  bool hp[PF + 1];
#pragma unroll
  for (int k = 0; k < PF; ++k) {
    hp[k] = false;
    if (rs + k * p.slots < nrows) fetch(rs + k * p.slots, kv[k], sc[k], hp[k]);
  }
  hp[PF] = false;

  auto compute = [&](const int j, const uint32_t (&kvb)[W][NW], const uint32_t (&scb)[W][NW],
                     const bool has_prev) {
    uint64_t x[W][NW];
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const bool prev = TWO && i < R;
      if (prev && !has_prev) {
#pragma unroll
        for (int q = 0; q < NW; ++q) x[i][q] = f2_pack(-INFINITY, -INFINITY);
        continue;
      }
      uint64_t a2[NW];
#pragma unroll
      for (int q4 = 0; q4 < NQ; ++q4) {
        const float4 a = sA[(i * V + vl) * NQ + q4];
        a2[2 * q4] = f2_pack(a.x, a.y);
        a2[2 * q4 + 1] = f2_pack(a.z, a.w);
      }
#pragma unroll
      for (int q = 0; q < NW; ++q) x[i][q] = f2_fma(bf2_to_f2(scb[i][q]), kL2, a2[q]);
    }
    uint64_t nm[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      float mlo = f2_lo(x[0][q]), mhi = f2_hi(x[0][q]);
#pragma unroll
      for (int i = 1; i + 1 < W; i += 2) {
        mlo = fmax3(mlo, f2_lo(x[i][q]), f2_lo(x[i + 1][q]));
        mhi = fmax3(mhi, f2_hi(x[i][q]), f2_hi(x[i + 1][q]));
      }
      if constexpr (W % 2 == 0 && W > 1) {
        mlo = fmaxf(mlo, f2_lo(x[W - 1][q]));
        mhi = fmaxf(mhi, f2_hi(x[W - 1][q]));
      }
      nm[q] = f2_pack(-mlo, -mhi);
    }
    uint64_t zz[2][NW], AA[2][NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) zz[0][q] = zz[1][q] = AA[0][q] = AA[1][q] = 0ull;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const bool prev = TWO && i < R;
      if (prev && !has_prev) continue;
#pragma unroll
      for (int q = 0; q < NW; ++q) {
        const uint64_t dd = f2_add(x[i][q], nm[q]);
        const uint64_t e2 = f2_pack(fast_exp2(f2_lo(dd)), fast_exp2(f2_hi(dd)));
        zz[i & 1][q] = f2_add(zz[i & 1][q], e2);
        AA[i & 1][q] = f2_fma(e2, bf2_to_f2(kvb[i][q]), AA[i & 1][q]);
      }
    }
    uint32_t ow[NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const uint64_t z = f2_add(zz[0][q], zz[1][q]);
      const uint64_t A = f2_add(AA[0][q], AA[1][q]);
      ow[q] = f2_to_bf2(f2_mul(A, f2_pack(rcp_nr(f2_lo(z)), rcp_nr(f2_hi(z)))));
    }
    store_stream<NW>(p.out + static_cast<int64_t>(o0 + j) * d + c0, ow);
  };

  // step b computes buffer b and refills buffer (b + PF) mod (PF + 1) with the row PF
  // slots ahead (the buffer the previous step consumed); the unrolled steps keep every
  // buffer index a constant
  for (int j = rs; j < nrows;) {
#pragma unroll
    for (int b = 0; b <= PF; ++b) {
      if (j < nrows) {
        const int jn = j + PF * p.slots;
        const int bn = (b + PF) % (PF + 1);
        if (jn < nrows) fetch(jn, kv[bn], sc[bn], hp[bn]);
        compute(j, kv[b], sc[b], hp[b]);
        j += p.slots;
      }
    }
  }
}

}  // namespace csa
