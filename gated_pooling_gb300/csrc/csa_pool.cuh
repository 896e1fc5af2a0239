// csa_pool.cuh -- the general (split-window) pooling kernel of the GB300 CSA/HCA
// compressor, forward and backward, and the launch geometry of every pooling kernel (the
// specialised ones are csa_pool_stream.cuh, csa_fwd_ldg.cuh, csa_pool_long.cuh and
// csa_pool_generic.cuh; csa_api.cu picks one per call).
//
// Operation ("Megatron-LM PR #5984", commit "CSA: add fused Compressor
// forward+backward CuTe-DSL kernels"): per output row (one block of ratio tokens of
// one THD segment) and column j < d, gather the window (coff=2: previous block at
// column j, own block at column d+j; coff=1: own block at column j), add ape, take a
// float32 softmax over the window positions, and sum kv with those weights; the
// backward applies the softmax Jacobian, writes every dKV/dScore slot exactly once
// (zeros where no window reads, commit "fold dKV/dScore zero-init into the backward
// kernel") and sums dAPE without atomics.
//
// Work decomposition (one design for all window sizes):
//   * A column "chunk" is VEC consecutive columns of one half (d/VEC chunks per half).
//     A thread owns one chunk -- the same chunk in both halves at coff=2 -- and PP
//     window positions (position group pg), for every row it visits. Window sizes
//     W = coff*ratio > PP are split across P = ceil(W/PP) position groups whose
//     per-column softmax partials (max, sum, weighted sum) are merged through shared
//     memory in a fixed order.
//   * A CTA is 256 threads = `slots` row slots x P groups x Vs chunks. gridDim.x = K
//     column slices of Vs chunks, gridDim.y = R row groups; row group g owns output
//     rows [g*TC/R, (g+1)*TC/R) (TC = total_comp, computed on the device), so every CTA
//     gets the same number of rows to within one.
//   * Every CTA rebuilds the segment -> block prefix from cu_seqlens into shared memory
//     (the THD index map) and binary-searches it per row.
//   * The ape values of the CTA's column slice are staged once in shared memory,
//     pre-multiplied by log2(e): the softmax runs in base 2 (x' = score*log2e + ape').
//   * Backward: per-thread dAPE sums stay in registers across rows; at the end the
//     CTA adds its row slots in a fixed order and writes one partial per row group;
//     a second kernel adds the R partials in a fixed order. No atomics anywhere.
//   * Zero ownership (backward): the thread that processes a segment's last block
//     zeroes that block's first-half columns (coff=2) and the segment's tail; segments
//     with no block are zeroed by the row group whose row range holds their block
//     offset; rows outside [cu[0], cu[S]) are split evenly across row groups.
#pragma once

#include <algorithm>

#include "csa_device.cuh"

namespace csa {

constexpr int kThreads = 256;

struct PoolParams {
  const uint16_t* kv;     // bf16 [capacity, C]
  const uint16_t* score;  // bf16 [capacity, C]
  const float* ape;       // fp32 [r, C]
  const int32_t* cu;      // int32 [S+1]
  const uint16_t* dout;   // bf16 [out_rows, d]   (backward)
  uint16_t* out;          // bf16 [out_rows, d]   (forward)
  uint16_t* dkv;          // bf16 [capacity, C]   (backward)
  uint16_t* dscore;       // bf16 [capacity, C]   (backward)
  float* partial;         // fp32 [R, r, C]       (backward)
  int32_t* status;        // backward: the call's status word in the workspace (see below)
  int32_t* dev_error;
  long long wait_cycles;  // bound of each pipeline mbarrier wait, in SM clock cycles
  int withhold_row;       // test hook: the producer of CTA (0, 0) never issues the copies of
                          // this row of its range (-1: off), so that its waits run out
  int64_t capacity;
  int64_t out_rows;
  int S, r, coff, d, C, W;
  int P;      // position groups
  int V;      // chunks per half = d / VEC
  int Vs;     // chunks per CTA column slice
  int slots;  // row slots per CTA
  int R;      // row groups = gridDim.y
  int sB_words;  // ints reserved for the block prefix (>= S+1, multiple of 4)
  // block-streaming kernel (csa_pool_stream.cuh) only
  int depth;        // stages in the ring
  int stage_bytes;  // bytes per stage
  int ape_off;      // byte offsets in dynamic shared memory: staged ape,
  int pre_off;      //   the block before the first row (left half),
  int ring_off;     //   the ring of stages,
  int bar_off;      //   the mbarriers (full [(np+1) depth], empty [depth], the previous
                    //   block's), then the rows the slots were armed for (np > 1)
  int box_rows;     // long windows: tokens per tensor box
  int np;           // block-streaming kernel: producer warps that stream rows
};

// Backward: CTA (0, 0) records in the workspace's status word whether the call's
// cu_seqlens and out_rows were valid (0) or not (1). The dAPE reduction reads it after
// the pooling grid has completed and leaves dAPE untouched unless it is 0, so a rejected
// call writes no output at all. Every CTA computes the same TC, so one writer suffices.
__device__ __forceinline__ void publish_status(const PoolParams& p, int TC) {
  if (p.status != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    *p.status = TC < 0 ? 1 : 0;
}

// Zeroes rows [row0, row0+nrows) of dKV and dScore over this CTA's column slice (both
// halves at coff=2, or only the first half with `first_half_only`). Cooperative over the
// threads t0, t0 + nt, ... (the whole CTA by default).
template <int NW>
__device__ __forceinline__ void zero_rows(const PoolParams& p, int64_t row0, int64_t nrows,
                                          int slice_chunks, int t0 = -1, int nt = 0,
                                          bool first_half_only = false) {
  constexpr int VEC = 2 * NW;
  if (t0 < 0) {
    t0 = threadIdx.x;
    nt = blockDim.x;
  }
  const int per_row = slice_chunks * (first_half_only ? 1 : p.coff);
  const int64_t items = nrows * per_row;
  for (int64_t it = t0; it < items; it += nt) {
    const int64_t row = row0 + it / per_row;
    const int rem = static_cast<int>(it % per_row);
    const int half = rem / slice_chunks;
    const int ch = blockIdx.x * p.Vs + rem % slice_chunks;
    const int64_t off = row * p.C + half * p.d + ch * VEC;
    store_zero<NW>(p.dkv + off);
    store_zero<NW>(p.dscore + off);
  }
}

// VEC: columns per chunk (8 forward, 4 backward). PP: window positions per thread.
// SPLIT: windows span several position groups (P > 1).
// (8-position backward: one CTA per SM, so that its window, weights and dAPE sums stay in
// registers without spills)
template <int VEC, int PP, bool BWD, bool SPLIT>
__global__ void __launch_bounds__(kThreads, (BWD && PP >= 8) ? 1 : 2) pool_kernel(const PoolParams p) {
  constexpr int NW = VEC / 2;  // 32-bit words per chunk
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  int* sB = reinterpret_cast<int*>(smem);
  float* sA = reinterpret_cast<float*>(sB + p.sB_words);   // [W][Vs*VEC], x log2(e)
  float* sX = sA + p.W * p.Vs * VEC;                        // merge area / dAPE reduction

  const int TC = build_block_prefix(p.cu, p.S, p.r, p.capacity, p.out_rows, p.dev_error, sB,
                                    warp_sums);
  publish_status(p, TC);
  if (TC < 0) return;
  // (no early launch of the stream's next kernel: it starts when this grid ends, which
  // measured faster than a trigger after the map build, e.g. 1 x 8192 d128 backward 13.3
  // -> 11.6 us, the long-window step 87.0 -> 84.2 us)

  const int tid = threadIdx.x;
  const int r = p.r, d = p.d, C = p.C;
  const bool two = p.coff == 2;
  const int slice_w = p.Vs * VEC;  // columns per half in this slice (full slices)
  const int slice_chunks = min(p.Vs, p.V - static_cast<int>(blockIdx.x) * p.Vs);

  // Stage ape of this column slice, all window positions, scaled by log2(e).
  for (int it = tid; it < p.W * p.Vs * (VEC / 4); it += blockDim.x) {
    const int w = it / (p.Vs * (VEC / 4));
    const int c4 = (it % (p.Vs * (VEC / 4))) * 4;     // column inside the slice
    const int ch = blockIdx.x * p.Vs + c4 / VEC;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ch < p.V) {
      const bool prev = two && w < r;
      const int arow = (two && !prev) ? w - r : w;
      const int col = ((two && !prev) ? d : 0) + blockIdx.x * slice_w + c4;
      a = __ldg(reinterpret_cast<const float4*>(p.ape + static_cast<int64_t>(arow) * C + col));
    }
    float* dst = sA + w * slice_w + c4;
    dst[0] = a.x * kLog2e;
    dst[1] = a.y * kLog2e;
    dst[2] = a.z * kLog2e;
    dst[3] = a.w * kLog2e;
  }

  const int tps = p.Vs * p.P;
  const int slot = tid / tps;
  const bool worker = slot < p.slots;
  const int vl = tid % p.Vs;
  const int pg = SPLIT ? (tid / p.Vs) % p.P : 0;
  const int chunk = blockIdx.x * p.Vs + vl;
  const bool col_ok = worker && chunk < p.V;
  const int c0 = chunk * VEC;

  const int g = blockIdx.y;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);

  if constexpr (BWD) {
    // Segments shorter than ratio: claimed by the row group whose range holds sB[s].
    const int s_lo = lower_bound_prefix(sB, 0, p.S, o0);
    const int s_hi = (g == p.R - 1) ? p.S : lower_bound_prefix(sB, s_lo, p.S, o1);
    for (int s = s_lo; s < s_hi; ++s) {
      const int a = __ldg(p.cu + s);
      const int b = __ldg(p.cu + s + 1);
      if (b - a < r && b > a) zero_rows<NW>(p, a, b - a, slice_chunks);
    }
    // Rows outside [cu[0], cu[S]): an even share per row group.
    const int64_t c_first = __ldg(p.cu);
    const int64_t c_last = __ldg(p.cu + p.S);
    const int64_t npad = c_first + (p.capacity - c_last);
    const int64_t q0 = static_cast<int64_t>(g) * npad / p.R;
    const int64_t q1 = static_cast<int64_t>(g + 1) * npad / p.R;
    const int64_t h0 = min(q1, c_first);                 // [q0, h0): rows before cu[0]
    if (h0 > q0) zero_rows<NW>(p, q0, h0 - q0, slice_chunks);
    const int64_t t0 = max(q0, c_first), t1 = q1;        // indices past cu[0] map to cu[S]+
    if (t1 > t0) zero_rows<NW>(p, c_last + (t0 - c_first), t1 - t0, slice_chunks);
  }
  __syncthreads();  // sA ready

  float acc[PP][VEC];  // backward: dAPE sums of this thread's positions and columns
#pragma unroll
  for (int i = 0; i < PP; ++i)
#pragma unroll
    for (int c = 0; c < VEC; ++c) acc[i][c] = 0.f;

  const int span = o1 - o0;
  const int n_iter = (span + p.slots - 1) / p.slots;  // uniform over the CTA
  for (int iter = 0; iter < n_iter; ++iter) {
    const int o = o0 + iter * p.slots + slot;
    const bool active = col_ok && o < o1;

    int s = 0, b = 0, n = 1, cs = 0, ce = 0;
    if (active) {
      s = find_segment(sB, p.S, o);
      b = o - sB[s];
      n = sB[s + 1] - sB[s];
      cs = __ldg(p.cu + s);
      ce = __ldg(p.cu + s + 1);
    }
    const int base = cs + b * r;

    // ---- gather the window slice of this thread --------------------------------
    uint32_t kvw[PP][NW], scw[PP][NW];
    int off[PP];
    int aoff[PP];
    bool valid[PP];
#pragma unroll
    for (int i = 0; i < PP; ++i) {
      const int w = pg * PP + i;
      const bool prev = two && w < r;
      const int wo = (two && !prev) ? w - r : w;  // position inside the block read
      bool v = active && w < p.W;
      if (prev) v = v && b >= 1;
      const int tok = prev ? base - r + w : base + wo;
      const int col = ((two && !prev) ? d : 0) + c0;
      valid[i] = v;
      off[i] = tok * C + col;
      aoff[i] = w * slice_w + vl * VEC;
      if (v) {
        load_stream<NW>(kvw[i], p.kv + off[i]);
        load_stream<NW>(scw[i], p.score + off[i]);
      } else {
#pragma unroll
        for (int q = 0; q < NW; ++q) kvw[i][q] = scw[i][q] = 0u;
      }
    }
    uint32_t gw[NW];
    if constexpr (BWD) {
      if (active) {
        load_stream<NW>(gw, p.dout + static_cast<int64_t>(o) * d + c0);
      } else {
#pragma unroll
        for (int q = 0; q < NW; ++q) gw[q] = 0u;
      }
    }

    // ---- per-column softmax over this thread's positions (base 2) --------------
    float m_loc[VEC], z_loc[VEC], a_loc[VEC];
    float e[PP][VEC];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      float x0[PP], x1[PP];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int i = 0; i < PP; ++i) {
        if (valid[i]) {
          const float2 a = *reinterpret_cast<const float2*>(sA + aoff[i] + 2 * q);
          x0[i] = fmaf(bf16_lo(scw[i][q]), kLog2e, a.x);
          x1[i] = fmaf(bf16_hi(scw[i][q]), kLog2e, a.y);
          mx0 = fmaxf(mx0, x0[i]);
          mx1 = fmaxf(mx1, x1[i]);
        } else {
          x0[i] = x1[i] = -INFINITY;
        }
      }
      float z0 = 0.f, z1 = 0.f, s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < PP; ++i) {
        float e0 = 0.f, e1 = 0.f;
        if (valid[i]) {
          e0 = fast_exp2(x0[i] - mx0);
          e1 = fast_exp2(x1[i] - mx1);
        }
        z0 += e0;
        z1 += e1;
        s0 = fmaf(e0, bf16_lo(kvw[i][q]), s0);
        s1 = fmaf(e1, bf16_hi(kvw[i][q]), s1);
        e[i][2 * q] = e0;
        e[i][2 * q + 1] = e1;
      }
      m_loc[2 * q] = mx0;
      m_loc[2 * q + 1] = mx1;
      z_loc[2 * q] = z0;
      z_loc[2 * q + 1] = z1;
      a_loc[2 * q] = s0;
      a_loc[2 * q + 1] = s1;
    }

    // ---- merge across position groups (fixed order) ----------------------------
    float M[VEC], Z[VEC], A[VEC];
    if constexpr (SPLIT) {
      // partials: [3][blockDim][VEC]; finals: [3][slots*Vs][VEC]
      float* pm = sX;
      float* pz = pm + kThreads * VEC;
      float* pa = pz + kThreads * VEC;
      float* fm = pa + kThreads * VEC;
      const int nfin = p.slots * p.Vs * VEC;
      float* fz = fm + nfin;
      float* fa = fz + nfin;
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        pm[tid * VEC + c] = m_loc[c];
        pz[tid * VEC + c] = z_loc[c];
        pa[tid * VEC + c] = a_loc[c];
      }
      __syncthreads();
      if (worker) {
        for (int c = pg; c < VEC; c += p.P) {
          float mm = -INFINITY, zz = 0.f, aa = 0.f;
          for (int k = 0; k < p.P; ++k) {
            const int src = (slot * p.P + k) * p.Vs + vl;
            const float mk = pm[src * VEC + c];
            if (mk == -INFINITY) continue;
            const float mn = fmaxf(mm, mk);
            const float so = fast_exp2(mm - mn);  // 0 while mm is -inf
            const float sn = fast_exp2(mk - mn);
            zz = __fadd_rn(__fmul_rn(zz, so), __fmul_rn(pz[src * VEC + c], sn));
            aa = __fadd_rn(__fmul_rn(aa, so), __fmul_rn(pa[src * VEC + c], sn));
            mm = mn;
          }
          const int dst = (slot * p.Vs + vl) * VEC + c;
          fm[dst] = mm;
          fz[dst] = zz;
          fa[dst] = aa;
        }
      }
      __syncthreads();
      if (worker) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          const int src = (slot * p.Vs + vl) * VEC + c;
          M[c] = fm[src];
          Z[c] = fz[src];
          A[c] = fa[src];
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        M[c] = m_loc[c];
        Z[c] = z_loc[c];
        A[c] = a_loc[c];
      }
    }

    if constexpr (!BWD) {
      if (active && pg == 0) {
        uint32_t ow[NW];
#pragma unroll
        for (int q = 0; q < NW; ++q) ow[q] = pack_bf16x2(A[2 * q] / Z[2 * q], A[2 * q + 1] / Z[2 * q + 1]);
        store_stream<NW>(p.out + static_cast<int64_t>(o) * d + c0, ow);
      }
    } else {
      // ---- softmax Jacobian: dKV = p*g, dScore = p*g*(kv - out) ------------------
      float oc[VEC], qc[VEC], gc[VEC];
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        oc[c] = A[c] / Z[c];
        const float scale = SPLIT ? fast_exp2(m_loc[c] - M[c]) : 1.f;
        qc[c] = __fdiv_rn(scale, Z[c]);
        gc[c] = (c & 1) ? bf16_hi(gw[c >> 1]) : bf16_lo(gw[c >> 1]);
      }
#pragma unroll
      for (int i = 0; i < PP; ++i) {
        if (!valid[i]) continue;
        uint32_t dk[NW], ds[NW];
#pragma unroll
        for (int q = 0; q < NW; ++q) {
          const float v0 = bf16_lo(kvw[i][q]), v1 = bf16_hi(kvw[i][q]);
          const float k0 = (e[i][2 * q] * qc[2 * q]) * gc[2 * q];
          const float k1 = (e[i][2 * q + 1] * qc[2 * q + 1]) * gc[2 * q + 1];
          const float t0 = k0 * (v0 - oc[2 * q]);
          const float t1 = k1 * (v1 - oc[2 * q + 1]);
          acc[i][2 * q] += t0;
          acc[i][2 * q + 1] += t1;
          dk[q] = pack_bf16x2(k0, k1);
          ds[q] = pack_bf16x2(t0, t1);
        }
        store_stream<NW>(p.dkv + off[i], dk);
        store_stream<NW>(p.dscore + off[i], ds);
      }
      // ---- zeros owned by a segment's last block -----------------------------------
      if (active && b == n - 1) {
        if (two)  // first-half columns of the last block's own tokens
          for (int k = pg; k < r; k += p.P) {
            const int64_t offz = static_cast<int64_t>(base + k) * C + c0;
            store_zero<NW>(p.dkv + offz);
            store_zero<NW>(p.dscore + offz);
          }
        const int tail0 = cs + n * r;  // the segment's tail tokens, every half
        for (int k = pg; k < ce - tail0; k += p.P) {
          const int64_t offz = static_cast<int64_t>(tail0 + k) * C + c0;
          store_zero<NW>(p.dkv + offz);
          store_zero<NW>(p.dscore + offz);
          if (two) {
            store_zero<NW>(p.dkv + offz + d);
            store_zero<NW>(p.dscore + offz + d);
          }
        }
      }
    }
  }

  if constexpr (BWD) {
    // ---- dAPE: add the row slots in a fixed order, one partial per row group -------
    float* red = sX;  // [PP*VEC][kThreads]
    if (p.slots > 1) {
      __syncthreads();
#pragma unroll
      for (int i = 0; i < PP; ++i)
#pragma unroll
        for (int c = 0; c < VEC; ++c) red[(i * VEC + c) * kThreads + tid] = acc[i][c];
      // slots added pairwise in a fixed tree (slot q absorbs slot q + h, h = the powers
      // of two below the slot count, largest first): each thread adds into its own entries
      const int ns = p.slots;
      int h = 1;
      while (2 * h < ns) h *= 2;
      for (; h >= 1; h /= 2) {
        __syncthreads();
        if (slot < h && slot + h < ns)
#pragma unroll
          for (int iv = 0; iv < PP * VEC; ++iv)
            red[iv * kThreads + tid] += red[iv * kThreads + tid + h * tps];
      }
      __syncthreads();
      if (slot == 0) {
#pragma unroll
        for (int i = 0; i < PP; ++i)
#pragma unroll
          for (int c = 0; c < VEC; ++c) acc[i][c] = red[(i * VEC + c) * kThreads + tid];
      }
    }
    if (slot == 0 && col_ok) {
      float* dst = p.partial + static_cast<int64_t>(g) * r * C;
#pragma unroll
      for (int i = 0; i < PP; ++i) {
        const int w = pg * PP + i;
        if (w >= p.W) continue;
        const bool prev = two && w < r;
        const int arow = (two && !prev) ? w - r : w;
        const int col = ((two && !prev) ? d : 0) + c0;
        float* q = dst + static_cast<int64_t>(arow) * C + col;
#pragma unroll
        for (int c = 0; c < VEC; c += 4)
          *reinterpret_cast<float4*>(q + c) = make_float4(acc[i][c], acc[i][c + 1], acc[i][c + 2], acc[i][c + 3]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// Launch planning (host)
// ------------------------------------------------------------------------------------
struct Plan {
  int vec = 0, pp = 0, P = 0, V = 0, Vs = 0, slots = 0, K = 0, R = 0, sB_words = 0;
  size_t smem = 0;
  bool split = false;
  bool tma = false;  // block-streaming kernel (bulk copies) for windows of <= 8 positions
  bool ldg = false;  // forward through register loads (csa_fwd_ldg.cuh)
  bool longk = false;  // long windows through 2-D tensor copies (csa_pool_long.cuh)
  bool generic = false;  // any head dim / alignment, scalar (csa_pool_generic.cuh)
  int box_rows = 0;    // long windows: tokens per tensor box
  int sc = 64;         // long windows: columns per CTA slice (64, or 32)
  int coff = 0;
  int threads = kThreads;
  int np = 1;  // block-streaming kernel: producer warps that stream rows
  int depth = 0, stage_bytes = 0, ape_off = 0, pre_off = 0, ring_off = 0, bar_off = 0;
};

inline int positions_per_thread(int W) { return W >= 5 ? 8 : (W >= 3 ? 4 : W); }

// Row groups R of a plan (grid = K column slices x R): as many as fill the SMs' resident
// CTAs (sms x bps) once over the K slices, rounded down -- rounding up would leave the last
// few CTAs to run in a second wave after the rest, nearly doubling the time when K does not
// divide that count -- at least 1 and at most the row count (and 65535, the grid's y
// limit). The generic kernel's many small CTAs take at most one row group per SM, so that
// its dAPE partials need no more workspace than the vector kernels'.
inline int row_groups(const Plan& pl, int sms, int bps, int64_t out_rows) {
  int64_t want = static_cast<int64_t>(sms) * bps / (pl.K > 0 ? pl.K : 1);
  if (want < 1) want = 1;
  if (pl.generic && want > sms) want = sms;
  const int64_t cap = out_rows > 0 ? out_rows : 1;
  int64_t R = want < cap ? want : cap;
  if (R < 1) R = 1;
  if (R > 65535) R = 65535;
  return static_cast<int>(R);
}

// Geometry that does not depend on the device.
inline Plan plan_shape(bool bwd, int S, int r, int coff, int d) {
  Plan pl;
  pl.vec = bwd ? 4 : 8;
  const int W = coff * r;
  pl.pp = positions_per_thread(W);
  pl.P = (W + pl.pp - 1) / pl.pp;
  pl.split = pl.P > 1;
  pl.V = d / pl.vec;
  pl.Vs = std::min(pl.V, 32);
  if (pl.split) pl.Vs = std::min(pl.Vs, std::max(1, kThreads / pl.P));
  const int tps = pl.Vs * pl.P;
  pl.slots = std::max(1, kThreads / tps);
  pl.K = (pl.V + pl.Vs - 1) / pl.Vs;
  pl.sB_words = ((S + 1) + 3) & ~3;
  size_t x = 0;
  if (pl.split)
    x = std::max(x, (size_t)(3 * kThreads * pl.vec + 3 * pl.slots * pl.Vs * pl.vec) * sizeof(float));
  if (bwd) x = std::max(x, (size_t)kThreads * pl.pp * pl.vec * sizeof(float));
  pl.smem = (size_t)pl.sB_words * sizeof(int) + (size_t)W * pl.Vs * pl.vec * sizeof(float) + x;
  return pl;
}

// Block-streaming kernel shape: columns per thread and consumer threads, per direction.
// The backward keeps 4 columns per thread so that its per-thread dAPE sums and softmax
// weights stay in registers.
// CTAs per SM, per direction: one by default (two forward CTAs, each with half the ring,
// measured no faster; two backward CTAs run short of registers).
#ifndef CSA_STREAM_FWD_CTAS
#define CSA_STREAM_FWD_CTAS 1
#endif
#ifndef CSA_STREAM_BWD_CTAS
#define CSA_STREAM_BWD_CTAS 1
#endif
// Consumers plus producer warps per CTA (and the backward's zero warp): 8 consumer warps
// + 4 producer warps forward, + 3 producer warps + the zero warp backward: 12 warps, three
// per SM sub-partition, leave 168 registers per thread (no spills; a 13th warp would cut
// that to 128). One warp issues about one bulk copy per quarter microsecond on GB300
// whatever its size, so the rows of stages below CSA_STREAM_ONE_PRODUCER_BYTES are dealt
// to several producer warps; larger stages keep one.
#ifndef CSA_STREAM_FWD_PRODUCERS
#define CSA_STREAM_FWD_PRODUCERS 4
#endif
#ifndef CSA_STREAM_BWD_PRODUCERS
#define CSA_STREAM_BWD_PRODUCERS 3
#endif
#ifndef CSA_STREAM_ONE_PRODUCER_BYTES
#define CSA_STREAM_ONE_PRODUCER_BYTES (8 * 1024)
#endif
constexpr int stream_producers(bool bwd) {
  return bwd ? CSA_STREAM_BWD_PRODUCERS : CSA_STREAM_FWD_PRODUCERS;
}
#ifndef CSA_FWD_VEC
#define CSA_FWD_VEC 8
#endif
#ifndef CSA_FWD_CONSUMERS
#define CSA_FWD_CONSUMERS 256
#endif
#ifndef CSA_BWD_VEC
#define CSA_BWD_VEC 4
#endif
#ifndef CSA_BWD_CONSUMERS
#define CSA_BWD_CONSUMERS 256
#endif

#ifndef CSA_FWD_LDG
#define CSA_FWD_LDG 1      // forward windows <= 8 through register loads
#endif
#ifndef CSA_LDG_THREADS
#define CSA_LDG_THREADS 512
#endif
// 8-position windows keep two rows of 32 words each in registers per thread: 384 threads
// (168 registers each) instead of 512 (128 each, which spilled)
#ifndef CSA_LDG_THREADS_W8
#define CSA_LDG_THREADS_W8 384
#endif
// 16-byte pieces (8 columns a thread, 256 threads a CTA) for windows of up to
// CSA_LDG_VEC8_MAX_WINDOW positions when d % 8 == 0: windows of 1-2 positions measured
// 25% faster with them (4x16384 r2 c1 d512 forward 42.7 -> 32.1 us; 35.2 at 384 threads),
// 4-position windows 3-13% slower (fewer rows or fewer threads in flight, to fit the
// registers)
#ifndef CSA_LDG_VEC8_MAX_WINDOW
#define CSA_LDG_VEC8_MAX_WINDOW 2
#endif
#ifndef CSA_LDG_THREADS_V8
#define CSA_LDG_THREADS_V8 256
#endif
constexpr int ldg_vec(int window, int d) {
  return (window <= CSA_LDG_VEC8_MAX_WINDOW && d % 8 == 0) ? 8 : 4;
}
constexpr int ldg_threads(int window, int vec) {
  return window >= 8 ? CSA_LDG_THREADS_W8 : (vec == 8 ? CSA_LDG_THREADS_V8 : CSA_LDG_THREADS);
}
#ifndef CSA_LDG_CTAS
#define CSA_LDG_CTAS 1
#endif

// ratio/coff pairs the block-streaming kernel is instantiated for (window <= 8).
inline bool stream_window_supported(int r, int coff) {
  if (coff == 2) return r == 1 || r == 2 || r == 4;
  return r == 1 || r == 2 || r == 4 || r == 8;
}

// Block-streaming kernel geometry: one CTA per SM, NC consumers + a producer warp, as many
// stages as shared memory holds (<= 64), at least `slots + 2`. Returns false when the shape
// does not fit it.
inline bool plan_stream(bool bwd, int S, int r, int coff, int d, size_t smem_limit, Plan* out) {
  if (!stream_window_supported(r, coff)) return false;
  const int W = coff * r;
  const int vec = bwd ? CSA_BWD_VEC : CSA_FWD_VEC;
  const int nc = bwd ? CSA_BWD_CONSUMERS : CSA_FWD_CONSUMERS;
  if (d % vec != 0) return false;
  Plan pl;
  pl.tma = true;
  pl.coff = coff;
  pl.vec = vec;
  pl.pp = W;
  pl.P = 1;
  pl.V = d / vec;
  if (pl.V > nc) return false;
  pl.Vs = pl.V;
  pl.K = 1;
  pl.slots = nc / pl.V;
  pl.sB_words = ((S + 1) + 3) & ~3;
  const size_t C = (size_t)coff * d;
  pl.stage_bytes = (int)(2 * r * C * 2 + (bwd ? (size_t)d * 2 : 0));
  const size_t ape_off = (size_t)pl.sB_words * 8;  // block prefix + cu_seqlens
  const size_t pre_off = ape_off + (size_t)W * d * 4;
  const size_t ring_off = (pre_off + (coff == 2 ? 2 * (size_t)r * C * 2 : 0) + 127) & ~(size_t)127;
  const size_t red = bwd ? (size_t)W * vec * nc * 4 : 0;
  // CTAs per SM share the SM's 228 KiB (1 KiB reserved per CTA)
  const int ctas = bwd ? CSA_STREAM_BWD_CTAS : CSA_STREAM_FWD_CTAS;
  smem_limit = std::min<size_t>(smem_limit, (228 * 1024) / ctas - 1024 - 256);
  if (smem_limit <= ring_off + 64) return false;
  // one producer warp for stages of 8 KB or more (it keeps the copy engine busy on its
  // own; more warps measured slower there), all of them for smaller stages
  const int np = pl.stage_bytes >= CSA_STREAM_ONE_PRODUCER_BYTES ? 1 : stream_producers(bwd);
  // per stage: the stage, np + 1 full barriers, the empty barrier (+ the armed-row word)
  const size_t per_slot = (size_t)(np + 2) * 8 + (np > 1 ? 4 : 0);
  size_t depth = std::min<size_t>(64, (smem_limit - ring_off - 8) / (pl.stage_bytes + per_slot));
  while (depth >= 3 && ring_off + std::max(depth * pl.stage_bytes, red) + depth * per_slot + 8 >
                           smem_limit)
    --depth;
  depth -= depth % np;  // every slot belongs to one producer warp
  if (depth < 3 || depth < (size_t)np) return false;
  if ((size_t)pl.slots + 2 > depth) pl.slots = (int)depth - 2;  // keep the ring ahead of the consumers
  pl.depth = (int)depth;
  pl.np = np;
  pl.threads = nc + 32 * np + (bwd ? 32 : 0);  // + producers (+ zero warp)
  pl.ape_off = (int)ape_off;
  pl.pre_off = (int)pre_off;
  pl.ring_off = (int)ring_off;
  pl.bar_off = (int)(ring_off + std::max(depth * pl.stage_bytes, red));
  pl.smem = (size_t)pl.bar_off + depth * per_slot + 8;  // + the previous block's barrier
  *out = pl;
  return true;
}

// Register-load forward geometry: 4 columns per thread, CSA_LDG_THREADS threads per CTA,
// rows split over NT/(d/4) row slots. Returns false when the shape does not fit it.
// Measured on GB300: register loads win for windows of <= 4 positions and for narrow rows
// (d < 512), where the bulk-copy pipeline's start-up dominates; the block-streaming kernel
// wins for 8-position windows of wide rows (the headline ratio=4 coff=2 d=512 pack).
#ifndef CSA_FWD_LDG_MAX_WINDOW
#define CSA_FWD_LDG_MAX_WINDOW 4
#endif
#ifndef CSA_FWD_LDG_BELOW_D
#define CSA_FWD_LDG_BELOW_D 512
#endif
inline bool fwd_prefers_ldg(int r, int coff, int d) {
  return coff * r <= CSA_FWD_LDG_MAX_WINDOW || d < CSA_FWD_LDG_BELOW_D;
}

inline bool plan_fwd_ldg(int S, int r, int coff, int d, size_t smem_limit, Plan* out) {
  if (!CSA_FWD_LDG || !stream_window_supported(r, coff) || d % 4 != 0) return false;
  if (!fwd_prefers_ldg(r, coff, d)) return false;
  Plan pl;
  pl.ldg = true;
  pl.coff = coff;
  pl.vec = ldg_vec(coff * r, d);
  pl.pp = coff * r;
  pl.P = 1;
  pl.V = d / pl.vec;
  const int nt = ldg_threads(coff * r, pl.vec);
  if (pl.V > nt) return false;
  pl.Vs = pl.V;
  pl.K = 1;
  pl.slots = nt / pl.V;
  pl.sB_words = ((S + 1) + 3) & ~3;
  pl.ape_off = pl.sB_words * 8;
  pl.smem = (size_t)pl.ape_off + (size_t)coff * r * d * 4;
  if (pl.smem > smem_limit) return false;
  pl.threads = nt;
  *out = pl;
  return true;
}

// Long-window geometry (csa_pool_long.cuh): W = coff*ratio in {16, 32, 64, 128, 256} and d
// a multiple of the slice width sc (64 columns per half, 16 chunks of 4; 32 for
// 256-position windows). A stage holds the [W x sc] kv and score tiles (tile rows of 2·sc
// bytes, 1024-byte aligned for the 2·sc-byte swizzle; at coff=2 the own half starts at
// tile row ratio, a multiple of 8), the backward adds the dout slice in a ring of its own.
// Tensor boxes (loads, and the backward's stores) are [ratio tokens x sc columns].
constexpr int kLongSliceCols = 64;  // columns per half in a long-window CTA slice

// Consumer groups of 8 warps in the long-window kernel (csa_pool_long.cuh) on 64-column
// slices, per direction.
#ifndef CSA_LONG_FWD_GROUPS
#define CSA_LONG_FWD_GROUPS 3
#endif
#ifndef CSA_LONG_BWD_GROUPS
#define CSA_LONG_BWD_GROUPS 2
#endif

// Columns per CTA slice of the long-window kernel: 64, or 32 where the head dim is not a
// multiple of 64 or 64-column slices would give the SMs fewer than 16 rows each (the pages'
// 65k-token r128 coff 2 d128 example: 512 rows of 64 KB per slice, 6.7 per SM). Narrower
// slices give each CTA twice the rows, half as large, so that the pipeline's fill and
// drain weigh less: that example's step 60.7 -> 53.2 us; with 27 rows per SM (d512) the
// 64-column slices stay 2% faster. (CSA_LONG_SC = 32 or 64 forces one width.)
#ifndef CSA_LONG_SC
#define CSA_LONG_SC 0
#endif
inline int long_slice_cols(int W, int d, int64_t out_rows, int sms) {
  (void)W;
  if (CSA_LONG_SC != 0) return CSA_LONG_SC;
  if (d % 64 != 0) return 32;
  const int64_t rows_per_sm = out_rows * (d / 64) / (sms > 0 ? sms : 1);
  return rows_per_sm < 16 ? 32 : kLongSliceCols;
}

// Consumer groups of the long-window kernel for a window of W positions. On 64-column
// slices a 256-position window has 64 KB stages, of which only two or three fit, so two
// groups do not take alternate rows there: both take every row, each half of its positions
// (the position split), which the backward runs (r128c2 d128: 57.6 -> 54.4 us; the forward
// measured slower with it, 20.5 -> 21.1 us, and runs one group). On 32-column slices the
// groups have 4 warps and take alternate rows.
#ifndef CSA_LONG_W256_FWD_GROUPS
#define CSA_LONG_W256_FWD_GROUPS 1
#endif
#ifndef CSA_LONG_W256_BWD_GROUPS
#define CSA_LONG_W256_BWD_GROUPS 2
#endif
#ifndef CSA_LONG32_FWD_GROUPS
#define CSA_LONG32_FWD_GROUPS 3  // forward groups of 4 warps on 32-column slices, W < 256
#endif
// 256-position windows on 32-column slices: three groups, with ape in shared memory (the
// forward keeps x' in registers): r128c2 d128 forward 16.6 -> 14.9 us, backward 35.5 ->
// 32.2 us against two groups (whose forward keeps ape in registers too). At coff 1 the
// backward's three groups would spill and it keeps two.
#ifndef CSA_LONG32_W256_FWD_GROUPS
#define CSA_LONG32_W256_FWD_GROUPS 3
#endif
#ifndef CSA_LONG32_W256_BWD_GROUPS
#define CSA_LONG32_W256_BWD_GROUPS 3
#endif
#ifndef CSA_LONG32_BWD_GROUPS
#define CSA_LONG32_BWD_GROUPS 2  // backward groups of 4 warps on 32-column slices, W < 256
#endif
constexpr int long_groups(bool bwd, int W, int sc, int coff) {
  return W >= 256 ? (sc == 32 ? (bwd ? (coff == 2 ? CSA_LONG32_W256_BWD_GROUPS : 2)
                                     : CSA_LONG32_W256_FWD_GROUPS)
                              : (bwd ? CSA_LONG_W256_BWD_GROUPS : CSA_LONG_W256_FWD_GROUPS))
                  : (bwd ? (sc == 32 ? CSA_LONG32_BWD_GROUPS : CSA_LONG_BWD_GROUPS)
                         : (sc == 32 ? CSA_LONG32_FWD_GROUPS : CSA_LONG_FWD_GROUPS));
}
// The position split: two groups on a 64-column slice of a 256-position window.
// (the split measured slower for shorter windows, whose lanes then keep the softmax terms
// in registers: long_r128_d512 backward 56.1 -> 58.3 us, 64-position windows up to +60%)
#ifndef CSA_LONG_PS_MIN_WINDOW
#define CSA_LONG_PS_MIN_WINDOW 256
#endif
constexpr bool long_position_split(int W, int ng, int sc) {
  return ng == 2 && W >= CSA_LONG_PS_MIN_WINDOW && sc == 64;
}
// The forward keeps a lane's ape in registers where its consumers have 8 warps (registers
// for 168 a thread) or split the positions; otherwise ape sits in shared memory.
constexpr bool long_ape_in_regs(bool bwd, int W, int ng, int sc) {
  return !bwd && (ng * sc * 4 <= 256 || long_position_split(W, ng, sc));
}

#ifndef CSA_LONG_W256
#define CSA_LONG_W256 1  // 256-position windows on the long-window kernel (else the split kernel)
#endif
// sc: columns per slice (long_slice_cols).
inline bool plan_long(bool bwd, int S, int r, int coff, int d, int sc, size_t smem_limit,
                      Plan* out) {
  const int W = coff * r;
  if (!(W == 16 || W == 32 || W == 64 || W == 128 || (CSA_LONG_W256 && W == 256))) return false;
  if ((sc != 64 && sc != 32) || d % sc != 0) return false;
  Plan pl;
  pl.longk = true;
  pl.coff = coff;
  pl.vec = 4;
  pl.pp = W / 16;
  pl.P = 16;
  pl.V = d / 4;
  pl.Vs = sc / 4;
  pl.K = d / sc;
  pl.sc = sc;
  pl.slots = 1;
  pl.box_rows = r;
  pl.sB_words = ((S + 1) + 3) & ~3;
  const int ng = long_groups(bwd, W, sc, coff);
  const bool ape_smem = !long_ape_in_regs(bwd, W, ng, sc);
  const size_t ape_off = ((size_t)pl.sB_words * 8 + 15) & ~(size_t)15;
  // the position split's column max and sums exchange ([3][2 groups][sc columns] floats)
  // sits just below the ring
  const size_t xch = long_position_split(W, ng, sc) ? (size_t)3 * 2 * sc * 4 : 0;
  const size_t ring_off =
      ape_off + (ape_smem ? (size_t)(sc / 4) * (W + 4) * 16 : 0) + xch;
  pl.stage_bytes = 2 * W * sc * 2;
  // + the dout slice and 4 mbarriers (backward: two full, empty, done), 3 (forward)
  const size_t per_stage = (size_t)pl.stage_bytes + (bwd ? (size_t)sc * 2 + 32 : 24);
  if (smem_limit < ring_off + 1024 + 2 * per_stage) return false;
  const size_t depth = std::min<size_t>(16, (smem_limit - ring_off - 1024) / per_stage);
  // every consumer group needs a stage of its own (the groups of the position split share
  // theirs)
  if (depth <= (size_t)(long_position_split(W, ng, sc) ? 1 : ng)) return false;
  pl.depth = (int)depth;
  pl.threads = ng * sc * 4 + (bwd ? 96 : 32);  // + producer warp (+ store and zero warps)
  pl.ape_off = (int)ape_off;
  pl.ring_off = (int)ring_off;
  pl.smem = ring_off + 1024 + depth * per_stage;
  *out = pl;
  return true;
}

// Generic geometry (csa_pool_generic.cuh): 128 threads = 128 columns of each half per CTA,
// grid = ceil(d/128) column slices x R row groups; the backward keeps W x 128 fp32 dAPE
// sums in shared memory. Returns false for windows above the generic limit.
constexpr int kGenericMaxWindow = 256;
inline bool plan_generic(bool bwd, int S, int r, int coff, int d, size_t smem_limit, Plan* out) {
  const int W = coff * r;
  if (W > kGenericMaxWindow) return false;
  Plan pl;
  pl.generic = true;
  pl.coff = coff;
  pl.vec = 1;
  pl.pp = W;
  pl.P = 1;
  pl.V = d;
  pl.Vs = 128;
  pl.K = (d + 127) / 128;
  pl.slots = 1;
  pl.sB_words = ((S + 1) + 3) & ~3;
  // block prefix, cu_seqlens (cached when it fits: with many segments and a long backward
  // window the kernel reads it from global memory), then the backward's dAPE sums
  const size_t sums = bwd ? (size_t)W * 128 * 4 : 0;
  size_t ape_off = ((size_t)pl.sB_words * 8 + 15) & ~(size_t)15;
  if (ape_off + sums > smem_limit) ape_off = ((size_t)pl.sB_words * 4 + 15) & ~(size_t)15;
  pl.ape_off = (int)ape_off;
  pl.smem = ape_off + sums;
  if (pl.smem > smem_limit) return false;
  pl.threads = 128;
  *out = pl;
  return true;
}

// The plan of a call, in order of preference: forward windows of <= 8 positions (or
// narrow rows) take the register-load kernel, other windows of <= 8 positions the
// block-streaming kernel, windows of 16..256 positions the tensor-copy kernel (`tensor_maps`:
// the driver's tensor-map encoder is available), everything else the split kernel; shapes
// or pointers the vector kernels cannot take (`fast` false) go to the generic kernel.
// Returns false for a generic shape that does not fit. make_plan (csa_api.cu) adds the
// kernel and the row groups.
inline bool choose_plan(bool bwd, int S, int r, int coff, int d, int64_t out_rows, int sms,
                        bool fast, bool tensor_maps, size_t smem_limit, Plan* pl) {
  if (!fast) return plan_generic(bwd, S, r, coff, d, smem_limit, pl);
  if (!bwd && plan_fwd_ldg(S, r, coff, d, smem_limit, pl)) return true;
  if (plan_stream(bwd, S, r, coff, d, smem_limit, pl)) return true;
  if (tensor_maps &&
      plan_long(bwd, S, r, coff, d, long_slice_cols(coff * r, d, out_rows, sms), smem_limit, pl))
    return true;
  *pl = plan_shape(bwd, S, r, coff, d);
  return true;
}

}  // namespace csa
