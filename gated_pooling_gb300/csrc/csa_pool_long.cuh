// csa_pool_long.cuh -- pooling kernel for long windows (W = coff*ratio in {16, 32, 64, 128,
// 256}; e.g. the ratio=128 family of "Megatron-LM PR #5984", commit "add dedicated
// ratio=128 kernels", at coff 1 and 2), forward and backward, for head dims that are
// multiples of the slice width SC.
//
// Same operation and zero ownership as pool_kernel (csa_pool.cuh). A CTA owns a slice of SC
// columns per half (64, or 32 where the head dim is not a multiple of 64 or the SMs would
// get few rows each: narrower slices give each CTA twice the rows, half as large;
// long_slice_cols in csa_pool.cuh) and a contiguous range of output rows. For each row a
// producer warp loads the slice's window with 2-D tensor-map bulk copies (TMA, 2·SC-byte
// swizzle): one box of [ratio tokens x SC columns] per tensor per block half (at coff=2
// the previous block at the slice's first-half columns, the own block at its second-half
// columns), plus the dout slice in the backward, into a ring of shared-memory stages
// completing on mbarriers. The backward writes each slot's dKV and dScore over the kv and
// score values it has consumed in the stage (every slot has exactly one reader and
// writer), and a store warp copies the finished tiles out with tensor-map bulk stores,
// whole tile rows at a time, and hands the stage back to the producer as soon as they have
// been read out. A zero warp writes meanwhile the zeros of short segments, of the rows
// outside [cu[0], cu[S]), and of the segments whose last block is a row of the CTA (that
// block's own first-half columns at coff=2, and the segment's tail).
//
// Consumers are NG groups of SC/8 warps; group h takes the rows h, h+NG, ... of the CTA's
// range (more groups keep more warps in flight where registers allow), except in the
// position split of 256-position windows on 64-column slices, where both groups take every
// row, each half of its positions. Warp wi of a group owns the 8 columns [8wi, 8wi+8) of
// the slice; its lane (pg = lane / 2, ch = lane % 2) owns 4 of them and the window
// positions pg, pg+16, pg+32, ... A column's max and its sums (sum e, sum e*kv) are
// reduced over the 16 position lanes with xor shuffles; the adds of a butterfly are
// commutative, so all 16 lanes end with the same bits and the result is the same on every
// run. Groups never wait for each other (the position split's two groups excepted): a
// stage is released once the threads of its group have arrived on its `empty` barrier.
// The swizzle puts the 8 rows that each half-warp reads at once on disjoint banks. The ape
// values of a thread's slots are kept in registers (forwards of 8 consumer warps, and the
// position split) or in shared memory; in the backward the registers hold the thread's
// dAPE sums, which the groups add in a fixed order into the CTA's partial at the end. With
// several backward groups, or 16 positions per lane, the softmax terms are recomputed from
// the staged tile in each pass instead of being kept in registers. All waits are bounded.
#pragma once

#include <cuda.h>

#include "csa_pool.cuh"

namespace csa {


__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Shared -> global tensor-map bulk store of one box, tracked by the issuing thread's bulk
// groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y,
                                             const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   map),
               "r"(x), "r"(y), "r"(smem_addr(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void sts_words2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(smem_addr(p)), "r"(a), "r"(b) : "memory");
}

// Byte offset of (tile row y, 16-byte chunk c) in a tile of SC-column rows written with the
// 2·SC-byte swizzle (tile base on a 1024-byte boundary): 128-byte rows keep chunk c at
// c ^ (y mod 8), 64-byte rows at c ^ ((y / 2) mod 4) (the swizzle XORs address bits 4-6,
// resp. 4-5, with bits 7-9, resp. 7-8).
template <int SC>
__device__ __forceinline__ int swz(int y, int c) {
  if constexpr (SC == 64) return y * 128 + ((c ^ (y & 7)) << 4);
  return y * 64 + ((c ^ ((y >> 1) & 3)) << 4);
}

// Named barrier `id` over n threads that also ANDs a predicate over them: every thread
// gets the same answer.
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Column-pair arithmetic of the consumers: packed f32x2 instructions (PK), or the same
// operations on each fp32 of the pair, which the compiler is free to schedule and contract
// (a product and a sum into one fma) as scalar code.
template <bool PK>
__device__ __forceinline__ uint64_t c2_fma(uint64_t a, uint64_t b, uint64_t c) {
  if constexpr (PK) return f2_fma(a, b, c);
  return f2_pack(fmaf(f2_lo(a), f2_lo(b), f2_lo(c)), fmaf(f2_hi(a), f2_hi(b), f2_hi(c)));
}
template <bool PK>
__device__ __forceinline__ uint64_t c2_add(uint64_t a, uint64_t b) {
  if constexpr (PK) return f2_add(a, b);
  return f2_pack(f2_lo(a) + f2_lo(b), f2_hi(a) + f2_hi(b));
}
template <bool PK>
__device__ __forceinline__ uint64_t c2_mul(uint64_t a, uint64_t b) {
  if constexpr (PK) return f2_mul(a, b);
  return f2_pack(f2_lo(a) * f2_lo(b), f2_hi(a) * f2_hi(b));
}

template <int PP, int NG, int COFF, bool BWD, int SC>
__global__ void __launch_bounds__(NG * SC * 4 + (BWD ? 96 : 32), 1)
    pool_long_kernel(const PoolParams p, const __grid_constant__ CUtensorMap tm_kv,
                     const __grid_constant__ CUtensorMap tm_sc,
                     const __grid_constant__ CUtensorMap tm_dkv,
                     const __grid_constant__ CUtensorMap tm_dsc) {
  constexpr int VEC = 4, NW = 2;
  static_assert(SC == 64 || SC == 32, "slices of 64 or 32 columns");
  constexpr int W = 16 * PP;      // window positions
  constexpr int RB = SC * 2;      // bytes of a tile row (one token of the slice)
  constexpr int kTile = W * RB;   // one tensor's window in a stage
  constexpr int kPos = 16 * RB;   // tile bytes between a lane's positions pg + 16 i
  constexpr int GT = SC * 4;      // threads of a consumer group (SC / 8 warps)
  constexpr int NCT = NG * GT;    // consumer threads
  static_assert(NG >= 1 && (!BWD || NG <= 4), "the dAPE combine handles up to four groups");
  // the position split (two groups on a 64-column slice of a 256-position window): both
  // groups take every row, group g the positions [128 g, 128 g + 128) (the previous block,
  // then the own block), and they merge the column max and the sums through shared memory;
  // otherwise the groups take alternate rows
  constexpr bool kPS = long_position_split(W, NG, SC);
  constexpr int PPG = kPS ? PP / 2 : PP;  // positions per lane in a row
  constexpr int RSTEP = kPS ? 1 : NG;     // rows a group advances per iteration
  constexpr bool kApReg = long_ape_in_regs(BWD, W, NG, SC);  // a lane's ape in registers
  // packed f32x2 arithmetic where it measured faster: the forward of 256-position windows,
  // whose 8 consumer warps are bound by instruction issue (r128c2 d128 forward 20.5 -> 18.1
  // us on 64-column slices); elsewhere it measured slower (up to +15 % for 64-position
  // backwards)
#ifndef CSA_LONG_PACKED
#define CSA_LONG_PACKED 1  // 0: never, 1: 256-position forwards, 2: every instantiation
#endif
  constexpr bool kPk = CSA_LONG_PACKED == 2 || (CSA_LONG_PACKED == 1 && !BWD && PP >= 16);
  // later passes recompute the softmax terms from the staged tile instead of keeping them in
  // registers: in the backward when several groups share the registers or a lane owns 16
  // positions, and in the position split when a lane owns 8 (its forward keeps ape in
  // registers instead)
  constexpr bool kRecomp = kPS ? PPG >= 8 : (BWD && (NG > 1 || PP >= 16));
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  __shared__ int s_abort;
  __shared__ int s_issued;  // the finished producer's row count (-1: not finished)
  int* sB = reinterpret_cast<int*>(smem);
  int* sCu = sB + p.sB_words;
  // stages start on a 1024-byte boundary (the swizzle pattern); the plan reserves the slack
  unsigned char* stages =
      smem + p.ring_off + ((1024u - (smem_addr(smem + p.ring_off) & 1023u)) & 1023u);
  unsigned char* gring = stages + static_cast<size_t>(p.depth) * p.stage_bytes;  // dout
  // row j's stage is slot j mod depth and its `full` barrier full[j mod 2 depth]: the
  // producer arms rows in order, so a group at row j, having seen row j - NG land, knows
  // row j - depth was armed, which waited until slot j - 2 depth was handed back; that row
  // has landed, so a phase-parity wait on full[j mod 2 depth] is exact (with depth
  // barriers, a slow copy of row j - depth would alias row j's phase)
  uint64_t* full = reinterpret_cast<uint64_t*>(gring + (BWD ? p.depth * SC * 2 : 0));
  uint64_t* empty = full + 2 * p.depth;
  uint64_t* done = empty + p.depth;  // backward: a group has written the stage's gradients

  const int tid = threadIdx.x;
  // mbarriers, one per thread, before the map is read (their set-up does not depend on
  // it): the CTA-scope proxy fence makes them visible to the bulk-copy engine, the
  // barriers inside the block prefix to the other threads
  {
    const int nb = (BWD ? 4 : 3) * p.depth;
    for (int t = tid; t < nb; t += blockDim.x) {
      const int k = t / p.depth;
      if (k < 2) mbar_init(&full[t], 1);
      else if (k == 2) mbar_init(&empty[t - 2 * p.depth], BWD ? 1 : (kPS ? NCT : GT));
      else mbar_init(&done[t - 3 * p.depth], kPS ? NCT : GT);  // (bwd empty: store warp)
      fence_proxy_async_smem();
    }
    if (tid == 0) {
      s_abort = 0;
      s_issued = -1;
    }
  }
  const int TC = build_block_prefix(p.cu, p.S, p.r, p.capacity, p.out_rows, p.dev_error, sB,
                                    warp_sums, sCu);
  publish_status(p, TC);
  if (TC < 0) return;
  // (no early launch of the stream's next kernel: it starts when this grid ends, which
  // measured faster than a trigger after the map build, e.g. 1 x 8192 d128 backward 13.3
  // -> 11.6 us, the long-window step 87.0 -> 84.2 us)

  const int r = p.r, d = p.d, C = p.C;
  constexpr bool two = COFF == 2;
  const int col0 = blockIdx.x * SC;  // first column of the slice (in a half)
  const int g = blockIdx.y;
  const int o0 = static_cast<int>(static_cast<int64_t>(g) * TC / p.R);
  const int o1 = static_cast<int>(static_cast<int64_t>(g + 1) * TC / p.R);
  const int nrows = o1 - o0;
  // test hook: the first CTA's producer skips this row's copies (the stage never fills)
  const int withheld = (blockIdx.x == 0 && blockIdx.y == 0) ? p.withhold_row : -1;
  // Waits until the copies of the rows before jn have landed (the slots of rows before
  // jn - depth were handed back, so those have).
  auto drain = [&](const int jn) {
    for (int k = max(0, jn - p.depth); k < jn; ++k)
      if (k != withheld)
        mbar_wait_bounded(&full[k % (2 * p.depth)],
                          static_cast<uint32_t>((k / (2 * p.depth)) & 1), kWaitCycles);
  };
  // A wait ran out: stop the pipeline, then wait for the producer's copies if it is done
  // (if not, it sees the stop and waits for them itself; producer_sees_stop).
  auto stop_and_drain = [&]() {
    stop_pipeline(&s_abort, p.dev_error);
    const int jn = read_issued(&s_issued);
    if (jn >= 0) drain(jn);
  };

  if (tid >= NCT) {
    if constexpr (BWD) {
      // ---------------------------- store warp ----------------------------------------
      if (tid == NCT + 32) {
        int s = nrows > 0 ? find_segment(sB, p.S, o0) : 0;
        bool bad = false;
        int slot = 0;     // stage of row j
        uint32_t ph = 0;  // (j / depth) & 1
        for (int j = 0; j < nrows; ++j, slot = slot + 1 == p.depth ? 0 : slot + 1, ph ^= slot == 0) {
          if (!mbar_wait_bounded(&done[slot], ph, p.wait_cycles) ||
              *reinterpret_cast<volatile int*>(&s_abort)) {
            bad = true;
            break;
          }
          const int o = o0 + j;
          s = advance_segment(sB, s, o);
          const int base = sCu[s] + (o - sB[s]) * r;
          const unsigned char* st = stages + static_cast<size_t>(slot) * p.stage_bytes;
          if (two && o > sB[s]) {  // previous block, first-half columns
            tma_store_2d(&tm_dkv, col0, base - r, st);
            tma_store_2d(&tm_dsc, col0, base - r, st + kTile);
          }
          const int yo = two ? r * RB : 0;
          const int x = (two ? d : 0) + col0;
          tma_store_2d(&tm_dkv, x, base, st + yo);
          tma_store_2d(&tm_dsc, x, base, st + kTile + yo);
          bulk_commit();
          // hand the stage back as soon as its tiles have been read (the next row's
          // gradients are still being computed: nothing else waits for this warp), so that
          // the producer refills it while the consumers work on the next row
          bulk_wait_read<0>();
          mbar_arrive(&empty[slot]);
        }
        bulk_wait_all();
        if (bad) stop_and_drain();
      }
    }
    if (BWD && tid >= NCT + 64) {
      // the zero warp: the zeros of short segments and of this row group's share of the
      // rows outside [cu[0], cu[S]), over this slice, while the consumers run
      const int zt = tid - NCT - 64;
      const int s_lo = lower_bound_prefix(sB, 0, p.S, o0);
      const int s_hi = (g == p.R - 1) ? p.S : lower_bound_prefix(sB, s_lo, p.S, o1);
      for (int s = s_lo; s < s_hi; ++s) {
        const int a = sCu[s], b = sCu[s + 1];
        if (b - a < r && b > a) zero_rows<NW>(p, a, b - a, SC / VEC, zt, 32);
      }
      // segments whose last block is a row of this group (sB[s+1] - 1 in [o0, o1)): the
      // first-half columns of that block's own tokens (coff=2; no next block reads them)
      // and the segment's tail tokens
      const int t_lo = upper_bound_prefix(sB, 1, p.S + 1, o0);
      const int t_hi = upper_bound_prefix(sB, t_lo, p.S + 1, o1);
      for (int t = t_lo; t < t_hi; ++t) {
        const int s = t - 1;
        const int n = sB[t] - sB[s];
        if (n < 1) continue;
        const int cs = sCu[s], ce = sCu[t];
        if (two) zero_rows<NW>(p, cs + (n - 1) * r, r, SC / VEC, zt, 32, true);
        if (ce > cs + n * r) zero_rows<NW>(p, cs + n * r, ce - cs - n * r, SC / VEC, zt, 32);
      }
      const int64_t c_first = sCu[0];
      const int64_t c_last = sCu[p.S];
      const int64_t npad = c_first + (p.capacity - c_last);
      const int64_t q0 = static_cast<int64_t>(g) * npad / p.R;
      const int64_t q1 = static_cast<int64_t>(g + 1) * npad / p.R;
      const int64_t h0 = min(q1, c_first);
      if (h0 > q0) zero_rows<NW>(p, q0, h0 - q0, SC / VEC, zt, 32);
      const int64_t t0 = max(q0, c_first), t1 = q1;
      if (t1 > t0) zero_rows<NW>(p, c_last + (t0 - c_first), t1 - t0, SC / VEC, zt, 32);
    }
    // ------------------------------ producer ------------------------------------------
    if (tid == NCT) {
      const uint64_t pol = l2_evict_first_policy();
      int s = nrows > 0 ? find_segment(sB, p.S, o0) : 0;
      int j = 0;
      int slot = 0;      // j % depth
      uint32_t lap = 0;  // (j / depth) % 4: full barrier slot + (lap & 1) depth, parity lap >> 1
      for (; j < nrows;
           ++j, slot = slot + 1 == p.depth ? 0 : slot + 1, lap = (lap + (slot == 0)) & 3u) {
        if (j >= p.depth && !mbar_wait_bounded(&empty[slot], (lap & 1u) ^ 1u, p.wait_cycles)) {
          stop_pipeline(&s_abort, p.dev_error);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        const int o = o0 + j;
        s = advance_segment(sB, s, o);
        if (j == withheld) continue;  // test hook: this stage never fills
        const int b = o - sB[s];
        const int base = sCu[s] + b * r;
        const bool has_prev = two && b >= 1;
        unsigned char* st = stages + static_cast<size_t>(slot) * p.stage_bytes;
        uint64_t* fb = &full[slot + ((lap & 1u) ? p.depth : 0)];
        const int boxes = has_prev ? 2 : 1;
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(boxes * r * RB * 2 + (BWD ? SC * 2 : 0)));
        if (has_prev) {  // previous block, first-half columns -> tile rows [0, r)
          tma_load_2d(st, &tm_kv, col0, base - r, fb, pol);
          tma_load_2d(st + kTile, &tm_sc, col0, base - r, fb, pol);
        }
        // own block -> tile rows [r, 2r) at coff=2 (second-half columns), [0, r) at coff=1
        const int yo = two ? r * RB : 0;
        const int x = (two ? d : 0) + col0;
        tma_load_2d(st + yo, &tm_kv, x, base, fb, pol);
        tma_load_2d(st + kTile + yo, &tm_sc, x, base, fb, pol);
        if constexpr (BWD)
          bulk_load_hint(gring + slot * SC * 2, p.dout + static_cast<int64_t>(o) * d + col0, SC * 2,
                         fb, pol);
      }
      // done: on the normal path the consumers wait for every copy issued here; after a
      // stop the producer waits for them, unless a stopping thread has seen them
      if (producer_sees_stop(&s_issued, j, &s_abort)) drain(j);
    }
    return;
  }

  // ------------------------------ consumers -------------------------------------------
  const int grp = tid / GT;
  const int lane = tid & 31;
  const int wi = (tid % GT) >> 5;  // 16-byte chunk of the slice row (8 columns)
  const int pg = lane >> 1;              // position lane
  const int ch = lane & 1;               // which 4 columns of the chunk
  const int cl = wi * 8 + ch * 4;        // first column of this thread inside the slice

  // ape of this thread's slots, scaled by log2 e: registers (column pairs), or shared memory
  // as [4-column group][position] float4 (written by group 0; groups W + 4 apart, so that
  // the two column groups of a quarter-warp fall on different banks)
  uint64_t ap[kApReg ? PPG : 1][NW];
  float4* sAp = reinterpret_cast<float4*>(smem + p.ape_off) + (wi * 2 + ch) * (W + 4);
  if (kApReg || grp == 0) {
#pragma unroll
    for (int ii = 0; ii < (kApReg ? PPG : PP); ++ii) {
      const int i = (kApReg && kPS ? grp * PPG : 0) + ii;
      const int w = pg + 16 * i;
      const bool prev = two && w < r;
      const int arow = (two && !prev) ? w - r : w;
      const int col = ((two && !prev) ? d : 0) + col0 + cl;
      float4 a = __ldg(reinterpret_cast<const float4*>(p.ape + static_cast<int64_t>(arow) * C + col));
      a.x *= kLog2e;
      a.y *= kLog2e;
      a.z *= kLog2e;
      a.w *= kLog2e;
      if constexpr (kApReg) {
        ap[ii][0] = f2_pack(a.x, a.y);
        ap[ii][1] = f2_pack(a.z, a.w);
      } else {
        sAp[w] = a;
      }
    }
  }
  if constexpr (!kApReg) asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");  // ape staged

  // ape' of the lane's position index ii (window position w) as two column pairs. (16
  // positions per lane: the shared-memory reads are volatile, so that the compiler does not
  // hoist all positions' reads ahead and run out of registers.)
  auto ape_at = [&](const int ii, const int w, uint64_t (&a2)[NW]) {
    if constexpr (kApReg) {
      a2[0] = ap[ii][0];
      a2[1] = ap[ii][1];
    } else {
      uint4 t;
      if constexpr (PP >= 16) {
        t = lds128_fresh(sAp + w);
      } else {
        const float4 f = sAp[w];
        t = make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z),
                       __float_as_uint(f.w));
      }
      a2[0] = (static_cast<uint64_t>(t.y) << 32) | t.x;
      a2[1] = (static_cast<uint64_t>(t.w) << 32) | t.z;
    }
  };

  uint64_t acc[BWD ? PPG : 1][NW];  // backward dAPE sums of this thread's slots (column pairs)
  const int ib = kPS ? grp * PPG : 0;  // this group's first position index (pg + 16 ib)
  // the position split's exchange of the groups' column max and sums (just below the ring)
  float (*s_xm)[SC] =
      reinterpret_cast<float (*)[SC]>(smem + p.ring_off - (kPS ? 3 * 2 * SC * 4 : 0));
  float (*s_xz)[SC] = s_xm + 2;
  float (*s_xa)[SC] = s_xm + 4;
#pragma unroll
  for (int i = 0; i < (BWD ? PPG : 1); ++i) acc[i][0] = acc[i][1] = 0ull;
  const uint64_t kL2 = f2_pack(kLog2e, kLog2e);
  // With packed arithmetic (kPk) the column max takes two positions per instruction where a
  // pair of position indices
  // (ii even) is valid or invalid as a whole: positions pg + 16 i are in the previous half
  // exactly when i < ratio / 16, an even number unless the window has 32 positions over two
  // halves (with one half of 8 positions the split even depends on the lane).
  constexpr int kStep = (kPk && PPG >= 2 && !(COFF == 2 && PP <= 2)) ? 2 : 1;

  // this thread's tile offset for position pg + 16 i is sw0 + kPos i: the swizzle depends on
  // the tile row only through its low three bits, which are those of pg
  const int sw0 = swz<SC>(pg, wi) + ch * 8;
  const int j0 = kPS ? 0 : grp;
  int s = nrows > j0 ? find_segment(sB, p.S, o0 + j0) : 0;
  // stage of row j and its lap (j / depth) % 4, advanced by RSTEP rows per iteration (RSTEP
  // < depth): the new slot is below RSTEP exactly when it wrapped
  int slot = j0;
  uint32_t lap = 0;
  for (int j = j0; j < nrows; j += RSTEP,
           slot = slot + RSTEP >= p.depth ? slot + RSTEP - p.depth : slot + RSTEP,
           lap = (lap + (slot < RSTEP)) & 3u) {
    const int o = o0 + j;
    s = advance_segment(sB, s, o);
    const int b = o - sB[s];
    const bool has_prev = two && b >= 1;
    const bool ok =
        mbar_wait_bounded(&full[slot + ((lap & 1u) ? p.depth : 0)], lap >> 1, p.wait_cycles);
    if constexpr (kPS) {
      // both groups work on this row and meet at its exchanges: they decide together
      if (!ok) stop_and_drain();
      if (!bar_and(2, NCT, ok && *reinterpret_cast<volatile int*>(&s_abort) == 0)) break;
    } else {
      if (!__all_sync(0xFFFFFFFFu, ok)) {  // a copy wait ran out: stop, and say so
        stop_and_drain();
        break;
      }
      if (__any_sync(0xFFFFFFFFu, *reinterpret_cast<volatile int*>(&s_abort) != 0)) break;
    }
    unsigned char* st = stages + static_cast<size_t>(slot) * p.stage_bytes;

    // x' = score*log2e + ape' at this thread's slots, as two column pairs; invalid (first
    // block, previous half) slots are skipped. With kRecomp the later passes read the slots
    // again instead of keeping x' (and e) in registers.
    auto x_at = [&](const int ii, const int i, const int w, uint64_t (&x)[NW]) {
      uint32_t sw[NW];
      if constexpr (PP >= 16) lds_words_fresh<NW>(sw, st + kTile + sw0 + i * kPos);
      else lds_words<NW>(sw, st + kTile + sw0 + i * kPos);
      uint64_t a2[NW];
      ape_at(ii, w, a2);
#pragma unroll
      for (int q = 0; q < NW; ++q) x[q] = c2_fma<kPk>(bf2_to_f2(sw[q]), kL2, a2[q]);
    };
    uint64_t e[kRecomp ? 1 : PPG][NW];
    float m[VEC] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int ii = 0; ii < PPG; ii += kStep) {
      const int i = ib + ii;
      const int w = pg + 16 * i;
      if (two && w < r && !has_prev) continue;
      uint64_t x[kStep][NW];
#pragma unroll
      for (int h = 0; h < kStep; ++h) {
        x_at(ii + h, i + h, w + 16 * h, x[h]);
        if constexpr (!kRecomp) {
          e[ii + h][0] = x[h][0];
          e[ii + h][1] = x[h][1];
        }
      }
#pragma unroll
      for (int q = 0; q < NW; ++q) {
        if constexpr (kStep == 2) {
          m[2 * q] = fmax3(m[2 * q], f2_lo(x[0][q]), f2_lo(x[1][q]));
          m[2 * q + 1] = fmax3(m[2 * q + 1], f2_hi(x[0][q]), f2_hi(x[1][q]));
        } else {
          m[2 * q] = fmaxf(m[2 * q], f2_lo(x[0][q]));
          m[2 * q + 1] = fmaxf(m[2 * q + 1], f2_hi(x[0][q]));
        }
      }
    }
#pragma unroll
    for (int k = 2; k < 32; k <<= 1)
#pragma unroll
      for (int c = 0; c < VEC; ++c) m[c] = fmaxf(m[c], __shfl_xor_sync(0xFFFFFFFFu, m[c], k));
    if constexpr (kPS) {  // the column max over both halves (exact: the same in both groups)
      if (pg == 0)
#pragma unroll
        for (int c = 0; c < VEC; ++c) s_xm[grp][cl + c] = m[c];
      asm volatile("bar.sync 2, %0;" ::"n"(NCT) : "memory");
#pragma unroll
      for (int c = 0; c < VEC; ++c) m[c] = fmaxf(m[c], s_xm[grp ^ 1][cl + c]);
    }
    const uint64_t nm[NW] = {f2_pack(-m[0], -m[1]), f2_pack(-m[2], -m[3])};
    // e = 2^(x' - m) of a slot's column pairs
    auto exp_at = [&](const uint64_t (&x)[NW], uint64_t (&ec)[NW]) {
#pragma unroll
      for (int q = 0; q < NW; ++q) {
        const uint64_t dd = c2_add<kPk>(x[q], nm[q]);
        ec[q] = f2_pack(fast_exp2(f2_lo(dd)), fast_exp2(f2_hi(dd)));
      }
    };

    // two accumulation chains per column (one in the backward, which is short of registers)
    constexpr int NCH = BWD ? 1 : 2;
    uint64_t z[2][NW], a[2][NW];
#pragma unroll
    for (int q = 0; q < NW; ++q) z[0][q] = z[1][q] = a[0][q] = a[1][q] = 0ull;
#pragma unroll
    for (int ii = 0; ii < PPG; ++ii) {
      const int i = ib + ii;
      const int w = pg + 16 * i;
      if (two && w < r && !has_prev) continue;
      uint32_t kw[NW];
      if constexpr (PP >= 16) lds_words_fresh<NW>(kw, st + sw0 + i * kPos);
      else lds_words<NW>(kw, st + sw0 + i * kPos);
      uint64_t x[NW], ec[NW];
      if constexpr (kRecomp) {
        x_at(ii, i, w, x);
      } else {
        x[0] = e[ii][0];
        x[1] = e[ii][1];
      }
      exp_at(x, ec);
#pragma unroll
      for (int q = 0; q < NW; ++q) {
        if constexpr (!kRecomp) e[ii][q] = ec[q];
        z[ii % NCH][q] = c2_add<kPk>(z[ii % NCH][q], ec[q]);
        a[ii % NCH][q] = c2_fma<kPk>(ec[q], bf2_to_f2(kw[q]), a[ii % NCH][q]);
      }
    }
    float Z[VEC], A[VEC];
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const uint64_t zq = c2_add<kPk>(z[0][q], z[1][q]);
      const uint64_t aq = c2_add<kPk>(a[0][q], a[1][q]);
      Z[2 * q] = f2_lo(zq);
      Z[2 * q + 1] = f2_hi(zq);
      A[2 * q] = f2_lo(aq);
      A[2 * q + 1] = f2_hi(aq);
    }
#pragma unroll
    for (int k = 2; k < 32; k <<= 1)
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        Z[c] += __shfl_xor_sync(0xFFFFFFFFu, Z[c], k);
        A[c] += __shfl_xor_sync(0xFFFFFFFFu, A[c], k);
      }
    if constexpr (kPS) {  // both halves' sums, added in group order: the same bits in both
      if (pg == 0)
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          s_xz[grp][cl + c] = Z[c];
          s_xa[grp][cl + c] = A[c];
        }
      asm volatile("bar.sync 2, %0;" ::"n"(NCT) : "memory");
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        Z[c] = s_xz[0][cl + c] + s_xz[1][cl + c];
        A[c] = s_xa[0][cl + c] + s_xa[1][cl + c];
      }
    }
    float rz[VEC], oc[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      rz[c] = rcp_nr(Z[c]);
      oc[c] = A[c] * rz[c];
    }
    if constexpr (!BWD) {
      if (pg == 0 && (!kPS || grp == 0)) {
        uint32_t ow[NW] = {pack_bf16x2(oc[0], oc[1]), pack_bf16x2(oc[2], oc[3])};
        store_stream<NW>(p.out + static_cast<int64_t>(o) * d + col0 + cl, ow);
      }
    } else {
      uint32_t gw[NW];
      lds_words<NW>(gw, gring + slot * SC * 2 + cl * 2);
      const uint64_t qg[NW] = {f2_pack(rz[0] * bf16_lo(gw[0]), rz[1] * bf16_hi(gw[0])),
                               f2_pack(rz[2] * bf16_lo(gw[1]), rz[3] * bf16_hi(gw[1]))};
      const uint64_t noc[NW] = {f2_pack(-oc[0], -oc[1]), f2_pack(-oc[2], -oc[3])};
#pragma unroll
      for (int ii = 0; ii < PPG; ++ii) {
        const int i = ib + ii;
        const int w = pg + 16 * i;
        const bool prev = two && w < r;
        if (prev && !has_prev) continue;
        uint32_t kw[NW];
        lds_words_fresh<NW>(kw, st + sw0 + i * kPos);
        uint64_t ei[NW];
        if constexpr (kRecomp) {
          uint64_t x[NW];
          x_at(ii, i, w, x);
          exp_at(x, ei);
        } else {
          ei[0] = e[ii][0];
          ei[1] = e[ii][1];
        }
        uint64_t kk[NW], t[NW];
#pragma unroll
        for (int q = 0; q < NW; ++q) {
          kk[q] = c2_mul<kPk>(ei[q], qg[q]);
          t[q] = c2_mul<kPk>(kk[q], c2_add<kPk>(bf2_to_f2(kw[q]), noc[q]));
          acc[ii][q] = c2_add<kPk>(acc[ii][q], t[q]);
        }
        // dKV and dScore replace the kv and score values of this slot in the stage
        sts_words2(st + sw0 + i * kPos, f2_to_bf2(kk[0]), f2_to_bf2(kk[1]));
        sts_words2(st + kTile + sw0 + i * kPos, f2_to_bf2(t[0]), f2_to_bf2(t[1]));
      }
      // (the zeros owned by a segment's last block are written by the zero warp)
    }
    if constexpr (BWD) {
      fence_proxy_async_smem();  // the stage's new contents, to the bulk-store engine
      mbar_arrive(&done[slot]);
    } else {
      mbar_arrive(&empty[slot]);
    }
  }

  if constexpr (BWD) {
    // the CTA's dAPE partial for this thread's slots: group 0's sums, then group 1's (with
    // the position split each group owns its positions' slots)
    if constexpr (NG >= 2 && !kPS) {
      // group h's sums pass through the ape area to group 0, which adds them in group order
      for (int h = 1; h < NG; ++h) {
        // ape, or the previous group's sums, no longer read
        asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");
        if (grp == h)
#pragma unroll
          for (int i = 0; i < PP; ++i)
            sAp[pg + 16 * i] = make_float4(f2_lo(acc[i][0]), f2_hi(acc[i][0]),
                                           f2_lo(acc[i][1]), f2_hi(acc[i][1]));
        asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");
        if (grp == 0)
#pragma unroll
          for (int i = 0; i < PP; ++i) {
            const float4 o1v = sAp[pg + 16 * i];
            acc[i][0] = c2_add<kPk>(acc[i][0], f2_pack(o1v.x, o1v.y));
            acc[i][1] = c2_add<kPk>(acc[i][1], f2_pack(o1v.z, o1v.w));
          }
      }
      if (grp != 0) return;
    }
    float* dst = p.partial + static_cast<int64_t>(g) * r * C;
#pragma unroll
    for (int ii = 0; ii < PPG; ++ii) {
      const int w = pg + 16 * (ib + ii);
      const bool prev = two && w < r;
      const int arow = (two && !prev) ? w - r : w;
      const int col = ((two && !prev) ? d : 0) + col0 + cl;
      *reinterpret_cast<float4*>(dst + static_cast<int64_t>(arow) * C + col) =
          make_float4(f2_lo(acc[ii][0]), f2_hi(acc[ii][0]), f2_lo(acc[ii][1]), f2_hi(acc[ii][1]));
    }
  }
}

// The long-window kernel for pp positions per lane (W = 16 pp), coff and a slice width, as
// the plain kernel pointer the launcher takes (its tensor-map arguments are passed by the
// launch's argument array).
template <bool BWD, int SC>
void (*long_kernel_for(int pp, bool two))(PoolParams) {
  using K = void (*)(PoolParams);
#define CSA_LONG_PICK(PP)                                                                   \
  return two ? reinterpret_cast<K>(pool_long_kernel<PP, long_groups(BWD, 16 * PP, SC, 2), 2, BWD, SC>) \
             : reinterpret_cast<K>(pool_long_kernel<PP, long_groups(BWD, 16 * PP, SC, 1), 1, BWD, SC>)
  switch (pp) {
    case 1: CSA_LONG_PICK(1);
    case 2: CSA_LONG_PICK(2);
    case 4: CSA_LONG_PICK(4);
    case 8: CSA_LONG_PICK(8);
    case 16: CSA_LONG_PICK(16);  // ratio 128 at coff 2, ratio 256 at coff 1
    default: return nullptr;
  }
#undef CSA_LONG_PICK
}

}  // namespace csa
