// Host-side checks of the launch planning (no GPU needed): the geometry the plan functions
// of csa_pool.cuh produce for a sweep of shapes must fit the device limits and the layout
// the kernels index, every plan the library can choose must have a kernel instantiation,
// and the row-group rule must never spill CTAs into a second wave. Built with nvcc against
// the library's objects and run by tests/test_plan.py; prints "ok <checks>" or the failures.
#include <cstdio>
#include <cstdlib>

#include "csa_internal.h"

namespace {

int failures = 0;
long checks = 0;

void expect(bool cond, const char* what, int W, int coff, int d, int bwd, long extra = 0) {
  ++checks;
  if (!cond) {
    if (failures < 40)
      std::printf("FAIL %s (W=%d coff=%d d=%d bwd=%d x=%ld)\n", what, W, coff, d, bwd, extra);
    ++failures;
  }
}

// GB300: 227 KB of shared memory per block (opt-in); the library keeps 256 bytes for the
// kernels' static shared memory.
constexpr size_t kOptin = 232448;
constexpr size_t kLimit = kOptin - 256;
constexpr int kSms = 152;

void check_long(int bwd, int r, int coff, int d, int64_t out_rows) {
  const int W = r * coff;
  const int sc = csa::long_slice_cols(W, d, out_rows, kSms);
  expect(sc == 32 || sc == 64, "slice width is 32 or 64", W, coff, d, bwd, sc);
  if (d % 64 != 0) expect(sc == 32, "head dims off a multiple of 64 take 32 columns", W, coff, d, bwd);
  csa::Plan pl;
  if (!csa::plan_long(bwd, 3, r, coff, d, sc, kLimit, &pl)) return;
  const int ng = csa::long_groups(bwd, W, sc, coff);
  const bool split = csa::long_position_split(W, ng, sc);
  expect(d % sc == 0 && pl.K * sc == d, "slices cover the head dim", W, coff, d, bwd, sc);
  expect(pl.Vs * 4 == sc, "slice chunks", W, coff, d, bwd, sc);
  expect(pl.smem <= kLimit, "shared memory within the limit", W, coff, d, bwd, (long)pl.smem);
  expect(pl.depth >= 2 && pl.depth <= 16, "ring depth", W, coff, d, bwd, pl.depth);
  expect(pl.depth > (split ? 1 : ng), "a stage per consumer group", W, coff, d, bwd, pl.depth);
  expect(pl.threads % 32 == 0 && pl.threads <= 1024, "block size", W, coff, d, bwd, pl.threads);
  expect(pl.threads == ng * sc * 4 + (bwd ? 96 : 32), "block = groups + service warps", W, coff,
         d, bwd, pl.threads);
  expect(pl.stage_bytes == 2 * W * sc * 2, "stage holds the kv and score tiles", W, coff, d, bwd);
  expect(pl.stage_bytes % 1024 == 0, "stages keep the swizzle alignment", W, coff, d, bwd,
         pl.stage_bytes);
  expect(r <= 256, "tensor box rows <= 256", W, coff, d, bwd, r);
  expect((sc * 2) % 16 == 0, "tensor x offsets on 16 bytes", W, coff, d, bwd, sc);
  expect(pl.box_rows == r, "box rows = ratio", W, coff, d, bwd, pl.box_rows);
  // the ape area (shared-memory ape: one float4 per 4-column group and position, groups
  // W + 4 apart) and the position split's exchange lie between ape_off and ring_off
  const bool ape_smem = !csa::long_ape_in_regs(bwd, W, ng, sc);
  const size_t ape = ape_smem ? (size_t)(sc / 4) * (W + 4) * 16 : 0;
  const size_t xch = split ? (size_t)3 * 2 * sc * 4 : 0;
  expect((size_t)pl.ape_off + ape + xch <= (size_t)pl.ring_off, "ape area below the ring", W,
         coff, d, bwd);
  expect((size_t)pl.ape_off >= (size_t)pl.sB_words * 8, "ape area above the map", W, coff, d,
         bwd);
  const size_t per_stage = (size_t)pl.stage_bytes + (bwd ? (size_t)sc * 2 + 32 : 24);
  expect((size_t)pl.ring_off + 1024 + pl.depth * per_stage == pl.smem,
         "ring, 1 KB alignment slack, dout slices and barriers", W, coff, d, bwd);
}

void check_stream(int bwd, int r, int coff, int d) {
  csa::Plan pl;
  if (!csa::plan_stream(bwd, 3, r, coff, d, kLimit, &pl)) return;
  const int W = r * coff;
  expect(pl.smem <= kLimit, "stream: shared memory within the limit", W, coff, d, bwd,
         (long)pl.smem);
  expect(pl.depth >= 3 && pl.depth % pl.np == 0, "stream: ring depth", W, coff, d, bwd,
         pl.depth);
  expect(pl.slots + 2 <= pl.depth, "stream: the ring stays ahead of the row slots", W, coff, d,
         bwd, pl.slots);
  expect(pl.threads % 32 == 0 && pl.threads <= 1024, "stream: block size", W, coff, d, bwd,
         pl.threads);
  expect(pl.V * pl.vec == d && pl.slots >= 1, "stream: a row's chunks", W, coff, d, bwd);
  expect(pl.ring_off % 128 == 0, "stream: ring alignment", W, coff, d, bwd, pl.ring_off);
  expect(pl.stage_bytes % 16 == 0, "stream: bulk copies of 16-byte multiples", W, coff, d, bwd,
         pl.stage_bytes);
}

void check_ldg(int r, int coff, int d) {
  csa::Plan pl;
  if (!csa::plan_fwd_ldg(3, r, coff, d, kLimit, &pl)) return;
  const int W = r * coff;
  expect(pl.vec == 4 || pl.vec == 8, "ldg: chunks of 4 or 8 columns", W, coff, d, 0, pl.vec);
  if (pl.vec == 8) expect(W <= 4 && d % 8 == 0, "ldg: 16-byte pieces for short windows", W, coff, d, 0);
  expect(pl.V * pl.vec == d && pl.slots >= 1 && pl.slots * pl.V <= pl.threads,
         "ldg: a row's chunks fit the block", W, coff, d, 0, pl.slots);
  expect(pl.smem <= kLimit, "ldg: shared memory within the limit", W, coff, d, 0, (long)pl.smem);
  expect(pl.threads % 32 == 0 && pl.threads <= 1024, "ldg: block size", W, coff, d, 0,
         pl.threads);
}

// Every shape within the header's limits has a plan: the generic kernel for windows of up
// to 256 positions at any segment count, the split kernel (plan_shape, always chosen last)
// within the shared-memory limit for windows of up to 2048.
void check_envelope() {
  for (int S : {1, 1000, 16384})
    for (int bwd = 0; bwd < 2; ++bwd)
      for (int coff = 1; coff <= 2; ++coff)
        for (int r = 1; r * coff <= 2048; r *= 2) {
          const int W = r * coff;
          for (int d : {8, 13, 64, 512, 4096}) {
            if (W <= 256) {
              csa::Plan pg;
              expect(csa::plan_generic(bwd, S, r, coff, d, kLimit, &pg), "generic plan exists",
                     W, coff, d, bwd, S);
              expect(pg.smem <= kLimit && (size_t)pg.ape_off >= (size_t)pg.sB_words * 4,
                     "generic: block prefix, then the sums, within the limit", W, coff, d, bwd,
                     S);
            }
            if (d % 8 == 0) {
              const csa::Plan ps = csa::plan_shape(bwd, S, r, coff, d);
              expect(ps.smem <= kLimit, "split: shared memory within the limit", W, coff, d, bwd,
                     S);
            }
          }
        }
}

// Every shape within the header's limits gets a plan from choose_plan (the library's own
// choice) and that plan a kernel: a plan without an instantiation would make a valid call
// return CSA_ERR_UNSUPPORTED.
void check_dispatch() {
  for (int fast = 0; fast < 2; ++fast)
    for (int bwd = 0; bwd < 2; ++bwd)
      for (int S : {1, 3, 16384})
        for (int coff = 1; coff <= 2; ++coff)
          for (int r : {1, 2, 3, 4, 5, 8, 16, 32, 64, 128, 256, 512, 1024, 2048}) {
            const int W = r * coff;
            if (W > 2048 || (!fast && W > 256)) continue;
            for (int d : {8, 13, 16, 24, 32, 64, 96, 128, 160, 192, 264, 512, 1024, 2048}) {
              if (fast && d % 8 != 0) continue;
              for (int64_t rows : {1L, 512L, 100000L}) {
                csa::Plan pl;
                const bool ok = csa::choose_plan(bwd, S, r, coff, d, rows, kSms, fast != 0, true,
                                                 kLimit, &pl);
                expect(ok, "a plan for every shape within the limits", W, coff, d, bwd, S);
                if (!ok) continue;
                const csa::PoolKernel k = bwd ? csa::bwd_kernel_for(pl) : csa::fwd_kernel_for(pl);
                expect(k != nullptr, "a kernel for every plan", W, coff, d, bwd, S);
                expect(pl.smem <= kLimit, "the chosen plan's shared memory", W, coff, d, bwd, S);
              }
            }
          }
}

void check_row_groups() {
  for (int generic = 0; generic < 2; ++generic)
    for (int bps = 1; bps <= 4; ++bps)
      for (int K = 1; K <= 700; K += (K < 40 ? 1 : 37))
        for (int64_t rows : {0L, 1L, 7L, 151L, 152L, 4096L, 1000000L}) {
          csa::Plan pl;
          pl.K = K;
          pl.generic = generic != 0;
          const int R = csa::row_groups(pl, kSms, bps, rows);
          expect(R >= 1, "row groups >= 1", 0, 0, K, bps, R);
          expect(R <= (rows > 0 ? rows : 1), "row groups <= rows", 0, 0, K, bps, R);
          if (K <= kSms * bps)
            expect((int64_t)R * K <= (int64_t)kSms * bps, "one wave of CTAs", 0, 0, K, bps, R);
          if (rows >= 1000000 && !generic)
            expect(R == (K <= kSms * bps ? kSms * bps / K : 1), "the SMs filled", 0, 0, K, bps,
                   R);
          if (generic) expect(R <= kSms, "generic: a row group per SM at most", 0, 0, K, bps, R);
        }
}

}  // namespace

int main() {
  const int ratios[] = {1, 2, 3, 4, 5, 8, 16, 32, 64, 128, 256, 1024};
  const int dims[] = {8, 16, 24, 32, 64, 96, 128, 160, 192, 256, 512, 1024, 2048};
  for (int bwd = 0; bwd < 2; ++bwd)
    for (int r : ratios)
      for (int coff = 1; coff <= 2; ++coff)
        for (int d : dims) {
          for (int64_t rows : {1L, 64L, 512L, 4096L, 100000L}) check_long(bwd, r, coff, d, rows);
          check_stream(bwd, r, coff, d);
          if (!bwd) check_ldg(r, coff, d);
        }
  // the slice-width rule: 32 columns while 64-column slices give the SMs fewer than 16 rows
  expect(csa::long_slice_cols(256, 128, 512, kSms) == 32, "few rows: 32 columns", 256, 2, 128,
         0);
  expect(csa::long_slice_cols(256, 512, 512, kSms) == 64, "many rows: 64 columns", 256, 2, 512,
         0);
  expect(csa::long_slice_cols(128, 96, 100000, kSms) == 32, "d96: 32 columns", 128, 1, 96, 0);
  check_row_groups();
  check_envelope();
  check_dispatch();
  if (failures) {
    std::printf("%d of %ld checks failed\n", failures, checks);
    return 1;
  }
  std::printf("ok %ld\n", checks);
  return 0;
}
