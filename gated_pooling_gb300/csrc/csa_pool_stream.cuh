// csa_pool_stream.cuh -- block-streaming pooling kernel for windows of up to 8 positions
// (ratio 1, 2, 4 at coff=2 and up to ratio 8 at coff=1): the backward of all of them and
// the forward of 8-position windows on wide rows (the headline ratio=4 coff=2 d=512
// pack; shorter windows and narrow rows go forward through csa_fwd_ldg.cuh).
//
// Same operation and zero ownership as pool_kernel (csa_pool.cuh). One CTA per SM owns a
// contiguous range of output rows [o0, o1). Output row o is block b of segment s; its R
// tokens are R consecutive rows of kv/score, so the block's full-width rows are ONE
// contiguous range of R*C bf16 values. Producer warps stream, for each row of the range,
// that block of kv and of score (and, backward, the dout row) into a ring of
// shared-memory stages with 1-D bulk asynchronous copies (TMA), completing on the
// row's `full` mbarrier. For small stages the rows are dealt round robin to several
// producer warps, since one warp issues about one bulk copy per quarter microsecond. The window of
// row o is the left half of stage o-1 (previous block, coff=2) and the right half of
// stage o (own block; the whole stage at coff=1), so every consumed byte crosses HBM
// once. A stage is released (`empty` mbarrier) once rows o and o+1 have read it; ring
// slots and phases are running counters. The block before o0 (read by row o0 when it is
// not a segment's first block) is fetched once, left half only, into a buffer laid out
// like a stage, its row copies issued by producer warp 0's lanes together. The mbarriers
// are set up before the index map is read.
//
// Consumers (NC threads): a thread owns one chunk of VEC columns of a row, the same
// chunk in both halves; NC/(d/VEC) rows are computed at once (row j -> row slot j mod
// slots). Columns are processed in pairs with the f32x2 instructions. ratio and coff are
// template parameters, so the window layout is static. No thread holds data in flight
// in registers; every wait is bounded. The backward has one more warp, which writes the
// zeros of segments shorter than ratio and of the padding rows while the others stream.
#pragma once

#include <type_traits>

#include "csa_pool.cuh"

namespace csa {

// NP: producer warps (1 for large stages, stream_producers(BWD) for small ones; the block
// has exactly NP of them, so that a one-producer launch keeps the registers and code of a
// one-producer block).
template <int VEC, int NC, int R, int COFF, bool BWD, int NP>
__global__ void __launch_bounds__(NC + 32 * NP + (BWD ? 32 : 0),
                                  BWD ? CSA_STREAM_BWD_CTAS : CSA_STREAM_FWD_CTAS)
    pool_stream_kernel(const PoolParams p) {
  constexpr int NW = VEC / 2;               // 32-bit words (= column pairs) per chunk
  // ape values per shared-memory vector: pairs in the forward (two 8-byte reads per
  // position measured slightly faster than one 16-byte read), quads in the backward
  constexpr int AW = (VEC >= 4 && BWD) ? 4 : 2;
  constexpr int NA = VEC / AW;              // ape vectors per chunk
  constexpr int W = R * COFF;
  constexpr bool TWO = COFF == 2;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  __shared__ int s_abort;
  __shared__ int s_issued[NP];  // a finished producer warp's next row (-1: not finished)
  int* sB = reinterpret_cast<int*>(smem);                     // block prefix [S+1]
  int* sCu = sB + p.sB_words;                                  // cu_seqlens [S+1]
  const float* sA = reinterpret_cast<const float*>(smem + p.ape_off);  // [W][NA][V] x AW
  unsigned char* pre = smem + p.pre_off;  // block before the first row: kv, score [R][C]
  unsigned char* stages = smem + p.ring_off;
  // Row j's stage is slot j mod depth, released on empty[j mod depth]; its `full` barrier
  // is full[j mod K depth], K = NP + 1 sets of depth barriers. A phase-parity wait cannot
  // tell a barrier's phase from the one two phases back, so the barrier's previous row,
  // j - K depth, must have landed whenever a consumer waits for row j. It has: the
  // consumer finished row j - NP slots, a row of the same producer warp (NP slots is a
  // multiple of NP), so that warp had armed its rows up to there, among them row
  // j - NP depth, and before arming that row it waited until the consumers had handed
  // back row j - K depth, which they do only after it landed. The same holds for the
  // previous stage's barrier, row j - 1 (row j - NP slots read stage j - NP slots - 1, or,
  // as a segment's first block, waited for its arming before releasing it). One producer
  // arms in order, and K = 2 follows the same way.
  constexpr int K = NP + 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);  // [K depth]
  uint64_t* empty = full + K * p.depth;                             // [depth]
  uint64_t* pre_bar = empty + p.depth;
  // several producer warps: the row each slot was last armed for (a segment's first block
  // waits for its previous row's arming before releasing that stage)
  int* slot_row = reinterpret_cast<int*>(pre_bar + 1);

  const int tid = threadIdx.x;
  const int d = p.d, C = p.C, V = p.V;

  using ApeVec = typename std::conditional<AW == 4, float4, float2>::type;
  auto ape_src = [&](const int it) {
    const int w = it / (NA * V);
    const int h = (it / V) % NA;
    const int ch = it % V;
    const bool prev = TWO && w < R;
    const int arow = (TWO && !prev) ? w - R : w;
    const int col = ((TWO && !prev) ? d : 0) + ch * VEC + AW * h;
    return reinterpret_cast<const ApeVec*>(p.ape + static_cast<int64_t>(arow) * C + col);
  };
  // mbarriers, one per thread, before the map is read: their set-up does not depend on it.
  // The CTA-scope proxy fence makes them visible to the bulk-copy engine; the barriers
  // inside the block prefix make them visible to the other threads.
  for (int i = tid; i < (K + 1) * p.depth + 1; i += blockDim.x) {
    if (i < K * p.depth) mbar_init(&full[i], 1);
    else if (i < (K + 1) * p.depth) mbar_init(&empty[i - K * p.depth], COFF * V);
    else mbar_init(pre_bar, 1);
    fence_proxy_async_smem();
  }
  if (NP > 1 && tid < p.depth) slot_row[tid] = -1;
  if (tid == 0) s_abort = 0;
  if (tid < NP) s_issued[tid] = -1;

  // (the block prefix ends with a barrier: the mbarriers are ready after it)
  const int TC = build_block_prefix(p.cu, p.S, R, p.capacity, p.out_rows, p.dev_error, sB,
                                    warp_sums, sCu);
  publish_status(p, TC);
  if (TC < 0) return;
  // (no early launch of the stream's next kernel: it starts when this grid ends, which
  // measured faster than a trigger after the map build, e.g. 1 x 8192 d128 backward 13.3
  // -> 11.6 us, the long-window step 87.0 -> 84.2 us)

  const int g = blockIdx.y;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);
  const int nrows = o1 - o0;
  const int kv_bytes = R * C * 2;  // one block of kv (or score), full width
  const int stage_g = 2 * kv_bytes;

  // does row o0 read a previous block (coff = 2 and not a segment's first block)?
  bool need_pre = false;
  if (TWO && nrows > 0) {
    const int s = find_segment(sB, p.S, o0);
    need_pre = o0 > sB[s];
  }

  // test hook: the first CTA's producer skips this row's copies (the stage never fills)
  const int withheld = (blockIdx.x == 0 && blockIdx.y == 0) ? p.withhold_row : -1;
  // Waits until the copies that producer warp q issued before its row jn have landed (the
  // slots of its rows before jn - depth were handed back, so those have), and, for warp
  // 0, the previous block's copies.
  auto drain = [&](const int q, const int jn) {
    for (int k = jn - NP; k >= 0 && k >= jn - p.depth; k -= NP)
      if (k != withheld)
        mbar_wait_bounded(&full[k % (K * p.depth)],
                          static_cast<uint32_t>((k / (K * p.depth)) & 1), kWaitCycles);
    if (q == 0 && need_pre) mbar_wait_bounded(pre_bar, 0, kWaitCycles);
  };
  // A wait ran out: stop the pipeline, then wait for the copies of the producer warps that
  // are done (the others see the stop and wait for their own; producer_sees_stop).
  auto stop_and_drain = [&]() {
    stop_pipeline(&s_abort, p.dev_error);
    for (int q = 0; q < NP; ++q) {
      const int jn = read_issued(&s_issued[q]);
      if (jn >= 0) drain(q, jn);
    }
  };

  // row j's full barrier and phase parity from its slot and lap = (j / depth) mod 2K
  auto fbar = [&](const int slot, const uint32_t lap) {
    return &full[slot + static_cast<int>(lap >= K ? lap - K : lap) * p.depth];
  };
  auto fpar = [](const uint32_t lap) { return lap >= K ? 1u : 0u; };
  auto next_lap = [](const uint32_t lap) { return lap + 1 == 2 * K ? 0u : lap + 1; };

  uint64_t acc[W][NW];  // backward: dAPE sums, column pairs
#pragma unroll
  for (int i = 0; i < W; ++i)
#pragma unroll
    for (int q = 0; q < NW; ++q) acc[i][q] = 0ull;

  if (tid >= NC) {
    // ------------------------------ producers -----------------------------------------
    // NP producer warps; lane 0 of warp pw streams the rows j = pw, pw + NP, ... into ring
    // slots j mod depth (depth is a multiple of NP, so every slot has one producer). A warp
    // has one bulk copy in issue at a time (about a quarter of a microsecond each on GB300),
    // so for small stages several warps issue side by side; large stages keep the copy
    // engine busy from one warp, and the plan uses one.
    // Warp 0's lanes first issue the previous block's 2*R row copies together. (Warp NP:
    // the backward's zero warp.)
    const int pw = (tid - NC) >> 5;
    const int lane = (tid - NC) & 31;
    const uint64_t pol = l2_evict_first_policy();
    if (pw == 0 && need_pre) {
      const int s = find_segment(sB, p.S, o0);
      if (lane == 0) mbar_arrive_expect_tx(pre_bar, static_cast<uint32_t>(2 * R * d * 2));
      __syncwarp();
      if (lane < 2 * R) {
        const int w = lane % R;
        const bool sc = lane >= R;
        const int64_t off = static_cast<int64_t>(sCu[s] + (o0 - sB[s] - 1) * R + w) * C;
        bulk_load_hint(pre + (sc ? kv_bytes : 0) + w * C * 2, (sc ? p.score : p.kv) + off,
                       d * 2, pre_bar, pol);
      }
    }
    if (BWD && pw == NP) {
      // the zero warp (backward): the zeros of segments shorter than ratio and of this row
      // group's share of the padding rows, written while the consumers stream
      const int s_lo = lower_bound_prefix(sB, 0, p.S, o0);
      const int s_hi = (g == p.R - 1) ? p.S : lower_bound_prefix(sB, s_lo, p.S, o1);
      for (int s2 = s_lo; s2 < s_hi; ++s2) {
        const int a = sCu[s2];
        const int b = sCu[s2 + 1];
        if (b - a < R && b > a) zero_rows<NW>(p, a, b - a, V, lane, 32);
      }
      const int64_t c_first = sCu[0];
      const int64_t c_last = sCu[p.S];
      const int64_t npad = c_first + (p.capacity - c_last);
      const int64_t q0 = static_cast<int64_t>(g) * npad / p.R;
      const int64_t q1 = static_cast<int64_t>(g + 1) * npad / p.R;
      const int64_t h0 = min(q1, c_first);
      if (h0 > q0) zero_rows<NW>(p, q0, h0 - q0, V, lane, 32);
      const int64_t t0 = max(q0, c_first), t1 = q1;
      if (t1 > t0) zero_rows<NW>(p, c_last + (t0 - c_first), t1 - t0, V, lane, 32);
    }
    if (pw < NP && lane == 0) {
      int s = nrows > pw ? find_segment(sB, p.S, o0 + pw) : 0;
      int j = pw;
      int slot = pw;     // j % depth
      uint32_t lap = 0;  // (j / depth) mod 2K
      for (; j < nrows; j += NP) {
        // the slot's previous row, j - depth, has been handed back (its `empty` phase)
        // ((j / depth) - 1) & 1 = (lap & 1) ^ 1, 2K being even
        if (j >= p.depth && !mbar_wait_bounded(&empty[slot], (lap & 1u) ^ 1u, p.wait_cycles)) {
          stop_and_drain();
          break;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        const int o = o0 + j;
        s = advance_segment(sB, s, o);
        uint64_t* fb = fbar(slot, lap);
        if constexpr (NP > 1) st_release_shared(&slot_row[slot], j);
        if (j != withheld) {  // test hook: a withheld stage never fills
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(stage_g + (BWD ? d * 2 : 0)));
          const int base = sCu[s] + (o - sB[s]) * R;
          unsigned char* st = stages + static_cast<size_t>(slot) * p.stage_bytes;
          const int64_t off = static_cast<int64_t>(base) * C;
          bulk_load_hint(st, p.kv + off, kv_bytes, fb, pol);
          bulk_load_hint(st + kv_bytes, p.score + off, kv_bytes, fb, pol);
          if constexpr (BWD)
            bulk_load_hint(st + stage_g, p.dout + static_cast<int64_t>(o) * d, d * 2, fb, pol);
        }
        slot += NP;
        if (slot >= p.depth) {
          slot -= p.depth;
          lap = next_lap(lap);
        }
      }
      // done: on the normal path the consumers wait for every copy issued here; after a
      // stop this warp waits for its own, unless a stopping thread has seen them
      if (producer_sees_stop(&s_issued[pw], j, &s_abort)) drain(pw, j);
    }
  } else {
    // ------------------------------ consumers -----------------------------------------
    // While the first stages are in flight: stage ape (scaled by log2 e) as
    // [w][h][chunk] vectors of AW values (a chunk's vectors are V apart).
    {
      ApeVec* dstA = reinterpret_cast<ApeVec*>(smem + p.ape_off);
      auto put = [&](const int it, ApeVec a) {
        a.x *= kLog2e;
        a.y *= kLog2e;
        if constexpr (AW == 4) {
          a.z *= kLog2e;
          a.w *= kLog2e;
        }
        dstA[it] = a;
      };
      for (int it = tid; it < W * NA * V; it += NC) put(it, __ldg(ape_src(it)));
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory");  // consumers only

    const int rs = tid / V;  // row slot
    const int vl = tid % V;  // chunk
    const int c0 = vl * VEC;
    const uint64_t kL2 = f2_pack(kLog2e, kLog2e);
    if (rs < p.slots && rs < nrows) {
      int s = find_segment(sB, p.S, o0 + rs);
      // stage of row j and its phase parity, advanced by `slots` rows per iteration
      // (slots < depth), and the same for row j - 1
      int slot = rs;  // rs < slots < depth
      uint32_t lap = 0;  // (j / depth) mod 2K, as the producers count it
      for (int j = rs; j < nrows; j += p.slots) {
        const int pslot = slot == 0 ? p.depth - 1 : slot - 1;
        const uint32_t plap = slot != 0 ? lap : lap == 0 ? 2 * K - 1 : lap - 1;
        const int o = o0 + j;
        s = advance_segment(sB, s, o);
        const int b = o - sB[s];
        const int n = sB[s + 1] - sB[s];
        const int cs = sCu[s];
        const int base = cs + b * R;
        const bool has_prev = TWO && b >= 1;
        bool ok = mbar_wait_bounded(fbar(slot, lap), fpar(lap), p.wait_cycles);
        // kv chunk of the own block's first token; score sits kv_bytes further, rows are C2
        // bytes apart. The previous block (coff=2) uses the same layout (its own stage, or
        // the block fetched before the first row).
        const int C2 = C * 2;
        const unsigned char* own_kv =
            stages + static_cast<size_t>(slot) * p.stage_bytes + ((TWO ? d : 0) + c0) * 2;
        const unsigned char* prev_kv = nullptr;
        if (has_prev) {
          if (j == 0) {
            ok = ok && mbar_wait_bounded(pre_bar, 0, p.wait_cycles);
            prev_kv = pre + c0 * 2;
          } else {
            ok = ok && mbar_wait_bounded(fbar(pslot, plap), fpar(plap), p.wait_cycles);
            prev_kv = stages + static_cast<size_t>(pslot) * p.stage_bytes + c0 * 2;
          }
        }
        if (!ok) {  // a copy wait ran out: stop, and say so
          stop_and_drain();
          break;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;

        // x' = score*log2e + ape*log2e for window position i (column pairs)
        uint64_t x[W][NW];
        auto load_x = [&](const int i, const unsigned char* kvp) {
          uint32_t sw[NW];
          lds_words<NW>(sw, kvp + kv_bytes);
          uint64_t a2[NW];
#pragma unroll
          for (int h = 0; h < NA; ++h) {
            if constexpr (AW == 4) {
              const float4 a = reinterpret_cast<const float4*>(sA)[(i * NA + h) * V + vl];
              a2[2 * h] = f2_pack(a.x, a.y);
              a2[2 * h + 1] = f2_pack(a.z, a.w);
            } else {
              const float2 a = reinterpret_cast<const float2*>(sA)[(i * NA + h) * V + vl];
              a2[h] = f2_pack(a.x, a.y);
            }
          }
#pragma unroll
          for (int q = 0; q < NW; ++q) x[i][q] = f2_fma(bf2_to_f2(sw[q]), kL2, a2[q]);
        };
        if constexpr (TWO) {
          if (has_prev) {
#pragma unroll
            for (int i = 0; i < R; ++i) load_x(i, prev_kv + i * C2);
          } else {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
              for (int q = 0; q < NW; ++q) x[i][q] = f2_pack(-INFINITY, -INFINITY);
          }
        }
#pragma unroll
        for (int w = 0; w < R; ++w) load_x(W - R + w, own_kv + w * C2);

        // negated column max, pairs
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

        // e = 2^(x' - m); Z = sum e and A = sum e*kv, as two interleaved partial sums
        uint64_t zz[2][NW], AA[2][NW];
#pragma unroll
        for (int q = 0; q < NW; ++q) zz[0][q] = zz[1][q] = AA[0][q] = AA[1][q] = 0ull;
        auto acc_e = [&](const int i, const unsigned char* kvp) {
          uint32_t kw[NW];
          lds_words<NW>(kw, kvp);
#pragma unroll
          for (int q = 0; q < NW; ++q) {
            const uint64_t dd = f2_add(x[i][q], nm[q]);
            const uint64_t e2 = f2_pack(fast_exp2(f2_lo(dd)), fast_exp2(f2_hi(dd)));
            zz[i & 1][q] = f2_add(zz[i & 1][q], e2);
            AA[i & 1][q] = f2_fma(e2, bf2_to_f2(kw[q]), AA[i & 1][q]);
            x[i][q] = e2;  // x now holds e
          }
        };
        if constexpr (TWO) {
          if (has_prev) {
#pragma unroll
            for (int i = 0; i < R; ++i) acc_e(i, prev_kv + i * C2);
          } else {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
              for (int q = 0; q < NW; ++q) x[i][q] = 0ull;
          }
        }
#pragma unroll
        for (int w = 0; w < R; ++w) acc_e(W - R + w, own_kv + w * C2);
        uint64_t A[NW];
        float rz[VEC];
#pragma unroll
        for (int q = 0; q < NW; ++q) {
          const uint64_t z = f2_add(zz[0][q], zz[1][q]);
          A[q] = f2_add(AA[0][q], AA[1][q]);
          rz[2 * q] = rcp_nr(f2_lo(z));
          rz[2 * q + 1] = rcp_nr(f2_hi(z));
        }

        if constexpr (!BWD) {
          uint32_t ow[NW];
#pragma unroll
          for (int q = 0; q < NW; ++q)
            ow[q] = f2_to_bf2(f2_mul(A[q], f2_pack(rz[2 * q], rz[2 * q + 1])));
          store_stream<NW>(p.out + static_cast<int64_t>(o) * d + c0, ow);
        } else {
          // p*g = e * (g / Z); dScore = p*g*(kv - out)
          uint32_t gw[NW];
          lds_words<NW>(gw, stages + static_cast<size_t>(slot) * p.stage_bytes + stage_g + c0 * 2);
          uint64_t noc[NW], qg[NW];
#pragma unroll
          for (int q = 0; q < NW; ++q) {
            noc[q] = f2_mul(A[q], f2_pack(-rz[2 * q], -rz[2 * q + 1]));
            qg[q] = f2_mul(bf2_to_f2(gw[q]), f2_pack(rz[2 * q], rz[2 * q + 1]));
          }
          const int64_t row_off = static_cast<int64_t>(base) * C + c0;  // own block, first half
          auto grad = [&](const int i, const unsigned char* kvp, int64_t goff) {
            uint32_t kw[NW];
            lds_words_fresh<NW>(kw, kvp);
            uint32_t dk[NW], ds[NW];
#pragma unroll
            for (int q = 0; q < NW; ++q) {
              const uint64_t k2 = f2_mul(x[i][q], qg[q]);
              const uint64_t t2 = f2_mul(k2, f2_add(bf2_to_f2(kw[q]), noc[q]));
              acc[i][q] = f2_add(acc[i][q], t2);
              dk[q] = f2_to_bf2(k2);
              ds[q] = f2_to_bf2(t2);
            }
            store_stream<NW>(p.dkv + goff, dk);
            store_stream<NW>(p.dscore + goff, ds);
          };
          if constexpr (TWO) {
            if (has_prev) {
#pragma unroll
              for (int i = 0; i < R; ++i)
                grad(i, prev_kv + i * C2, row_off - static_cast<int64_t>(R - i) * C);
            }
          }
#pragma unroll
          for (int w = 0; w < R; ++w)
            grad(W - R + w, own_kv + w * C2, row_off + static_cast<int64_t>(w) * C + (TWO ? d : 0));
          if (b == n - 1) {  // zeros owned by a segment's last block
            if constexpr (TWO) {
#pragma unroll
              for (int k = 0; k < R; ++k) {
                store_zero<NW>(p.dkv + row_off + static_cast<int64_t>(k) * C);
                store_zero<NW>(p.dscore + row_off + static_cast<int64_t>(k) * C);
              }
            }
            const int ce = sCu[s + 1];
            for (int t = cs + n * R; t < ce; ++t) {
              const int64_t offz = static_cast<int64_t>(t) * C + c0;
              store_zero<NW>(p.dkv + offz);
              store_zero<NW>(p.dscore + offz);
              if (TWO) {
                store_zero<NW>(p.dkv + offz + d);
                store_zero<NW>(p.dscore + offz + d);
              }
            }
          }
        }
        // release the own stage and (coff=2) the previous one, which row o-1 also read. A
        // segment's first block has not read the previous stage; its arrival there counts
        // toward row j - 1's phase only once row j - 1 is armed (its producer waited for
        // that slot's earlier phase). One producer arms in order, so row j armed means row
        // j - 1 armed; with several, the first block waits for row j - 1's arming.
        mbar_arrive(&empty[slot]);
        if (TWO && j >= 1) {
          if (NP > 1 && !has_prev && !wait_shared_eq(&slot_row[pslot], j - 1, &s_abort,
                                                    p.wait_cycles)) {
            stop_and_drain();
            break;
          }
          mbar_arrive(&empty[pslot]);
        }
        slot += p.slots;
        if (slot >= p.depth) {
          slot -= p.depth;
          lap = next_lap(lap);
        }
      }
    }
  }

  if constexpr (BWD) {
    // dAPE: add the row slots of each chunk in a fixed order, one partial per row group
    __syncthreads();
    float* red = reinterpret_cast<float*>(stages);  // [W*VEC][NC]
    if (tid < NC) {
#pragma unroll
      for (int i = 0; i < W; ++i)
#pragma unroll
        for (int q = 0; q < NW; ++q) {
          red[(i * VEC + 2 * q) * NC + tid] = f2_lo(acc[i][q]);
          red[(i * VEC + 2 * q + 1) * NC + tid] = f2_hi(acc[i][q]);
        }
    }
    // the row slots of every (position, column) added pairwise in a fixed tree (slot q
    // absorbs slot q + h, h = the powers of two below the slot count, largest first; each
    // thread adds into its own entries): log2(slots) short steps instead of a serial sum
    // over the slots (narrow rows have up to ~60 of them)
    const int ns = p.slots;
    int h = 1;
    while (2 * h < ns) h *= 2;
    const int rs = tid / V;  // this thread's row slot (its column of red is tid)
    for (; ns > 1 && h >= 1; h /= 2) {
      __syncthreads();
      if (tid < NC && rs < h && rs + h < ns)
#pragma unroll
        for (int iv = 0; iv < W * VEC; ++iv) red[iv * NC + tid] += red[iv * NC + tid + h * V];
    }
    __syncthreads();
    if (tid < V) {
      const int c0 = tid * VEC;
      float* dst = p.partial + static_cast<int64_t>(g) * R * C;
#pragma unroll
      for (int i = 0; i < W; ++i) {
        float sum[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) sum[c] = red[(i * VEC + c) * NC + tid];
        const bool prev = TWO && i < R;
        const int arow = (TWO && !prev) ? i - R : i;
        const int col = ((TWO && !prev) ? d : 0) + c0;
        float* q = dst + static_cast<int64_t>(arow) * C + col;
#pragma unroll
        for (int h = 0; h < NA; ++h) {
          if constexpr (AW == 4)
            *reinterpret_cast<float4*>(q + 4 * h) =
                make_float4(sum[4 * h], sum[4 * h + 1], sum[4 * h + 2], sum[4 * h + 3]);
          else
            *reinterpret_cast<float2*>(q + 2 * h) = make_float2(sum[2 * h], sum[2 * h + 1]);
        }
      }
    }
  }
}

}  // namespace csa
