// csa_oracle.cpp -- plain fp64 CPU definition of the CSA/HCA KV-compressor
// gated-softmax pooling over THD-packed ragged sequences, forward and backward.
//
// TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's CPU
// baseline may load or call this code. It shares nothing with the CUDA library:
// no headers, no helpers, no tables. It is written to be checked by eye against
// the definition, not to be fast: plain nested loops over segments, blocks,
// columns and window positions, all arithmetic in double.
//
// Sources (cited by page title and section):
//  * "Megatron-LM PR #5984", commit "CSA: add fused Compressor forward+backward
//    CuTe-DSL kernels": one fused region per direction over THD packs. It gathers
//    each block's window, adds the positional embedding (ape) to the scores, applies
//    the overlapping-window transform, takes a float32 softmax over the window
//    positions, sums kv weighted by that softmax and casts the sum to bf16.
//  * same page, commit "fold dKV/dScore zero-init into the backward kernel": the
//    backward writes every dKV/dScore position. Slots that no window reads hold
//    exact zeros: at coff=2 the first-half columns of each segment's last block,
//    each segment's tail tokens (seqlen mod ratio), every token of a segment
//    shorter than ratio, and every row past cu_seqlens[S]. dAPE is a sum over
//    blocks.
//  * same page, commit "widen the validated envelope to coff in {1, 2}": at coff=1
//    a block's window is just its own ratio tokens and every position is valid.
//  * "cudnn-frontend PR #710" (ratio=2): position-in-block indexing, the masking of
//    the first block's previous half, the tails and the short segments are all
//    defined for any ratio >= 1.
// Column/half assignment at coff=2: the previous block's tokens contribute their
// columns [0,d) and the block's own tokens their columns [d,2d), each with the ape
// row of the token's position inside its own block and the same ape column. This
// is the plainest reading the first-half zero class supports: the last block's
// own first-half columns are unread because there is no following block.
//
// Readings where the pages are silent:
//  * The bf16 cast's backward is the identity: gradients use the unrounded output.
//  * Masked (first block, coff=2) positions take no part in the softmax (weight 0).
//  * Rows outside [cu_seqlens[0], cu_seqlens[S]) get zero gradients.
//  * Unconsumed slots are +0.0 (bit pattern 0x0000).
//  * All roundings to bf16 and to fp32 are round-to-nearest-even.
//
// Parity pins (tests/test_oracle_pins.py): brute-force predicate evaluator on tiny
// packs, closed form for total_comp, uniform-score and shift invariants, softmax
// Jacobian identities, the ratio=1 identity, central finite differences, and a
// hand-derived golden pack (tests/golden/).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

double bf16_bits_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Round a double to the nearest bf16 (8 significant bits, fp32 exponent range,
// subnormals down to 2^-133), ties to even, in one step (no detour via fp32).
uint16_t double_to_bf16_bits(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const bool neg = std::signbit(x);
  if (x == 0.0) return neg ? 0x8000 : 0x0000;
  if (std::isinf(x)) return neg ? 0xFF80 : 0x7F80;
  int e = 0;
  std::frexp(x, &e);                         // |x| in [2^(e-1), 2^e)
  int q = e - 8;                             // spacing of bf16 numbers in that binade
  if (q < -133) q = -133;                    // subnormal spacing
  const double y = std::ldexp(x, -q);        // exact: power-of-two scaling
  const double r = std::nearbyint(y);        // round half to even (default mode)
  const double v = std::ldexp(r, q);
  if (std::fabs(v) >= std::ldexp(1.0, 128)) return neg ? 0xFF80 : 0x7F80;
  const float f = static_cast<float>(v);     // exact: v has <= 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return static_cast<uint16_t>(u >> 16);
}

// Error codes shared by every entry point of the oracle.
enum { ORACLE_OK = 0, ORACLE_BAD_ARGS = 1, ORACLE_BAD_CU = 2, ORACLE_OUT_ROWS = 3,
       ORACLE_DOUBLE_WRITE = 4, ORACLE_BAD_LEAD = 5 };

int check_args(const int32_t* cu, int S, int ratio, int coff, int d, int64_t capacity) {
  if (cu == nullptr || S < 0 || ratio < 1 || (coff != 1 && coff != 2) || d < 1 ||
      capacity < 0)
    return ORACLE_BAD_ARGS;
  if (cu[0] < 0) return ORACLE_BAD_CU;
  for (int s = 0; s < S; ++s)
    if (cu[s + 1] < cu[s]) return ORACLE_BAD_CU;
  if (static_cast<int64_t>(cu[S]) > capacity) return ORACLE_BAD_CU;
  return ORACLE_OK;
}

int64_t count_blocks(const int32_t* cu, int S, int ratio) {
  int64_t total = 0;
  for (int s = 0; s < S; ++s) total += (cu[s + 1] - cu[s]) / ratio;
  return total;
}

// The output rows in order: row o is block `b` of the segment starting at token `c`.
struct BlockRef {
  int64_t c;
  int64_t b;
};

std::vector<BlockRef> list_blocks(const int32_t* cu, int S, int ratio) {
  std::vector<BlockRef> rows;
  for (int s = 0; s < S; ++s) {
    const int64_t n = (cu[s + 1] - cu[s]) / ratio;
    for (int64_t b = 0; b < n; ++b) rows.push_back({cu[s], b});
  }
  return rows;
}

// Runs fn(t, begin, end) for t = 0..nthreads-1 over contiguous, nearly equal ranges of
// [0, rows) (output rows, or slots), on nthreads threads (the calling thread when
// nthreads is 1).
template <typename Fn>
void over_row_ranges(int64_t rows, int nthreads, Fn fn) {
  if (nthreads <= 1) {
    fn(0, int64_t{0}, rows);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t)
    pool.emplace_back(fn, t, rows * t / nthreads, rows * (t + 1) / nthreads);
  for (std::thread& th : pool) th.join();
}

// One valid position of a pooling window: the token row and column it reads in
// kv/score (and writes in dKV/dScore), and the flat index of its ape element.
struct WindowPos {
  int64_t token;
  int64_t col;
  int64_t ape_index;
};

// Window of block b (0-based) of the segment starting at token c, for output
// column j < d. coff=1: the block's own ratio tokens at column j, ape row = the
// position inside the block. coff=2: positions 0..ratio-1 are the previous block's
// tokens at column j (absent for the first block), positions ratio..2*ratio-1 are
// the block's own tokens at column d+j; ape row = the token's position inside its
// own block, ape column = the column read.
void window_of(int64_t c, int64_t b, int ratio, int coff, int d, int64_t j,
               std::vector<WindowPos>& win) {
  const int64_t C = static_cast<int64_t>(coff) * d;
  win.clear();
  if (coff == 1) {
    for (int w = 0; w < ratio; ++w) {
      const int64_t t = c + b * ratio + w;
      win.push_back({t, j, static_cast<int64_t>(w) * C + j});
    }
    return;
  }
  if (b >= 1) {
    for (int w = 0; w < ratio; ++w) {
      const int64_t t = c + (b - 1) * ratio + w;
      win.push_back({t, j, static_cast<int64_t>(w) * C + j});
    }
  }
  for (int w = 0; w < ratio; ++w) {
    const int64_t t = c + b * ratio + w;
    win.push_back({t, d + j, static_cast<int64_t>(w) * C + d + j});
  }
}

// Softmax statistics of one window, in double.
struct WindowStats {
  std::vector<double> x;  // score + ape
  std::vector<double> v;  // kv
  std::vector<double> p;  // softmax weights
  double m = 0.0;         // max of x
  double o = 0.0;         // sum_w p_w v_w (unrounded output)
};

void window_stats(const uint16_t* kv, const uint16_t* score, const float* ape, int64_t C,
                  const std::vector<WindowPos>& win, WindowStats& st) {
  const size_t n = win.size();
  st.x.resize(n);
  st.v.resize(n);
  st.p.resize(n);
  for (size_t i = 0; i < n; ++i) {
    const int64_t flat = win[i].token * C + win[i].col;
    st.x[i] = bf16_bits_to_double(score[flat]) + static_cast<double>(ape[win[i].ape_index]);
    st.v[i] = bf16_bits_to_double(kv[flat]);
  }
  st.m = st.x[0];
  for (size_t i = 1; i < n; ++i)
    if (st.x[i] > st.m) st.m = st.x[i];
  double z = 0.0;
  for (size_t i = 0; i < n; ++i) {
    st.p[i] = std::exp(st.x[i] - st.m);
    z += st.p[i];
  }
  for (size_t i = 0; i < n; ++i) st.p[i] /= z;
  st.o = 0.0;
  for (size_t i = 0; i < n; ++i) st.o += st.p[i] * st.v[i];
}

// First-order size of the rounding error an fp32 evaluation of the same window
// can make in the output, in units of the fp32 unit roundoff: the summands'
// magnitudes plus the spread of kv around the output weighted by how far each
// weight's exponent argument is from zero (the absolute error of an fp32
// exponent argument is proportional to |x| + |m|). The weights' own errors enter
// only through kv - out, since the normalisation makes them sum to one.
// These masses are the tolerance machinery of the parity tests, not part of the
// operation; tests/test_oracle_pins.py pins them to hand-derived closed forms and
// to a plain float32 re-evaluation of every window.
double output_error_mass(const WindowStats& st) {
  double a = 0.0;
  for (size_t i = 0; i < st.p.size(); ++i)
    a += st.p[i] * (std::fabs(st.v[i]) +
                    std::fabs(st.v[i] - st.o) * (1.0 + std::fabs(st.x[i]) + std::fabs(st.m)));
  return a;
}

// Forward over nthreads threads, each taking a contiguous range of output rows (the
// per-element arithmetic is the same whatever the thread count).
int fwd_impl(const uint16_t* kv, const uint16_t* score, const float* ape,
             const int32_t* cu_seqlens, int S, int ratio, int coff, int d, int64_t capacity,
             int64_t out_rows, uint16_t* out_bf16, double* out_f64, double* out_err,
             int nthreads) {
  int rc = check_args(cu_seqlens, S, ratio, coff, d, capacity);
  if (rc != ORACLE_OK) return rc;
  if (kv == nullptr || score == nullptr || ape == nullptr || out_bf16 == nullptr)
    return ORACLE_BAD_ARGS;
  if (count_blocks(cu_seqlens, S, ratio) > out_rows) return ORACLE_OUT_ROWS;
  const int64_t C = static_cast<int64_t>(coff) * d;
  const std::vector<BlockRef> rows = list_blocks(cu_seqlens, S, ratio);
  over_row_ranges(static_cast<int64_t>(rows.size()), nthreads,
                  [&](int, int64_t o_begin, int64_t o_end) {
    std::vector<WindowPos> win;
    WindowStats st;
    for (int64_t o = o_begin; o < o_end; ++o) {
      for (int64_t j = 0; j < d; ++j) {
        window_of(rows[o].c, rows[o].b, ratio, coff, d, j, win);
        window_stats(kv, score, ape, C, win, st);
        out_bf16[o * d + j] = double_to_bf16_bits(st.o);
        if (out_f64 != nullptr) out_f64[o * d + j] = st.o;
        if (out_err != nullptr) out_err[o * d + j] = output_error_mass(st);
      }
    }
  });
  return ORACLE_OK;
}

// Backward over nthreads threads (contiguous output-row ranges). Every slot is read by
// at most one window position, so the threads write disjoint slots; each thread sums its
// rows' dAPE terms, and the thread sums are added in thread order at the end (with one
// thread: the plain sum over rows in order).
int bwd_impl(const uint16_t* kv, const uint16_t* score, const float* ape,
             const int32_t* cu_seqlens, const uint16_t* dout, int S, int ratio, int coff, int d,
             int64_t capacity, int64_t out_rows, uint16_t* dkv_bf16, uint16_t* dscore_bf16,
             double* dape_f64, double* dkv_f64, double* dscore_f64, float* dape_f32,
             int32_t* owners, double* dkv_err, double* dscore_err, double* dape_err,
             double* dape_abs, int nthreads) {
  int rc = check_args(cu_seqlens, S, ratio, coff, d, capacity);
  if (rc != ORACLE_OK) return rc;
  if (kv == nullptr || score == nullptr || ape == nullptr || dkv_bf16 == nullptr ||
      dscore_bf16 == nullptr || dape_f64 == nullptr)
    return ORACLE_BAD_ARGS;
  const int64_t total = count_blocks(cu_seqlens, S, ratio);
  if (total > out_rows) return ORACLE_OUT_ROWS;
  if (total > 0 && dout == nullptr) return ORACLE_BAD_ARGS;
  const int64_t C = static_cast<int64_t>(coff) * d;
  const int64_t slots = capacity * C;
  const int64_t napes = static_cast<int64_t>(ratio) * C;
  if (nthreads < 1) nthreads = 1;

  // Every slot starts as an exact +0; consumed slots are overwritten below.
  std::vector<double> gkv(static_cast<size_t>(slots), 0.0);
  std::vector<double> gsc(static_cast<size_t>(slots), 0.0);
  std::vector<double> gsc_err(dscore_err != nullptr ? static_cast<size_t>(slots) : 0, 0.0);
  std::vector<double> gkv_err(dkv_err != nullptr ? static_cast<size_t>(slots) : 0, 0.0);
  std::vector<int32_t> count(static_cast<size_t>(slots), 0);
  // per-thread dAPE sums: value, error mass, absolute terms
  std::vector<std::vector<double>> t_dape(nthreads, std::vector<double>(napes, 0.0));
  std::vector<std::vector<double>> t_err(nthreads, std::vector<double>(napes, 0.0));
  std::vector<std::vector<double>> t_abs(nthreads, std::vector<double>(napes, 0.0));

  const std::vector<BlockRef> rows = list_blocks(cu_seqlens, S, ratio);
  over_row_ranges(static_cast<int64_t>(rows.size()), nthreads,
                  [&](int t, int64_t o_begin, int64_t o_end) {
    std::vector<WindowPos> win;
    WindowStats st;
    std::vector<double>& my_dape = t_dape[t];
    std::vector<double>& my_err = t_err[t];
    std::vector<double>& my_abs = t_abs[t];
    for (int64_t o = o_begin; o < o_end; ++o) {
      for (int64_t j = 0; j < d; ++j) {
        window_of(rows[o].c, rows[o].b, ratio, coff, d, j, win);
        window_stats(kv, score, ape, C, win, st);
        const double g = bf16_bits_to_double(dout[o * d + j]);
        const double oerr = output_error_mass(st);
        for (size_t i = 0; i < win.size(); ++i) {
          const int64_t flat = win[i].token * C + win[i].col;
          // d out / d kv_w = p_w ; d out / d x_w = p_w (kv_w - out)  (softmax Jacobian)
          const double dk = st.p[i] * g;
          const double ds = st.p[i] * g * (st.v[i] - st.o);
          gkv[flat] = dk;
          gsc[flat] = ds;
          count[flat] += 1;
          my_dape[win[i].ape_index] += ds;
          // error masses (units of the fp32 unit roundoff): a weight p*g carries the
          // error of its exponent argument, |x| + |m|, plus a rounding; dScore adds the
          // error of kv - out, which is the output's
          const double xm = 1.0 + std::fabs(st.x[i]) + std::fabs(st.m);
          const double err = std::fabs(st.p[i] * g) * (std::fabs(st.v[i] - st.o) * xm + oerr);
          if (dscore_err != nullptr) gsc_err[flat] = err;
          if (dkv_err != nullptr) gkv_err[flat] = std::fabs(dk) * xm;
          my_err[win[i].ape_index] += err + std::fabs(ds);
          my_abs[win[i].ape_index] += std::fabs(ds);
        }
      }
    }
  });

  for (int64_t i = 0; i < napes; ++i) {
    double v = 0.0, e = 0.0, a = 0.0;
    for (int t = 0; t < nthreads; ++t) {
      v += t_dape[t][i];
      e += t_err[t][i];
      a += t_abs[t][i];
    }
    dape_f64[i] = v;
    if (dape_err != nullptr) dape_err[i] = e;
    if (dape_abs != nullptr) dape_abs[i] = a;
  }
  // every slot rounded (and its owner count checked), over slot ranges per thread
  std::vector<int> twice(nthreads, 0);
  over_row_ranges(slots, nthreads, [&](int t, int64_t i0, int64_t i1) {
    for (int64_t i = i0; i < i1; ++i) {
      if (count[i] > 1) twice[t] = 1;
      dkv_bf16[i] = double_to_bf16_bits(gkv[i]);
      dscore_bf16[i] = double_to_bf16_bits(gsc[i]);
      if (dkv_f64 != nullptr) dkv_f64[i] = gkv[i];
      if (dscore_f64 != nullptr) dscore_f64[i] = gsc[i];
      if (owners != nullptr) owners[i] = count[i];
      if (dscore_err != nullptr) dscore_err[i] = gsc_err[i];
      if (dkv_err != nullptr) dkv_err[i] = gkv_err[i];
    }
  });
  for (int t = 0; t < nthreads; ++t)
    if (twice[t]) return ORACLE_DOUBLE_WRITE;
  if (dape_f32 != nullptr)
    for (int64_t i = 0; i < napes; ++i) dape_f32[i] = static_cast<float>(dape_f64[i]);
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------------
// KPool: the DSA indexer's key pooling ("Megatron-LM PR #8835", the KPool commits: the
// commit that adds "dsa_indexer_kpool_key_dtype_compression" and the explicit-mask pool
// origin, and the one that squashes the tail-less certificate fix and the empty-query
// guard; KPool selection itself is NVIDIA#8287 there).
//
// Keys of one segment are grouped into pools of P consecutive keys ("pooled keys on the
// grid [0:4], [4:8], ..."), the grid starting at the segment's first valid key: packed
// pooling resets at every segment, and the pool origin is the first valid key of each
// sample. A pool becomes one pooled key: per column, an FP32 softmax of the gate over
// the pool's keys weights the keys ("FP32 pool softmax").
//  * default: the weighted sum is taken in FP32 and cast to bf16 once ("the FP32
//    weighted reduction and BF16 output of the existing KPool implementation");
//  * key-dtype compression: the FP32 softmax is cast to the key dtype (bf16) before
//    multiplying and reducing: each weight is rounded to bf16, each weight x key
//    product to bf16, and their sum is cast to bf16.
// Keys after the last complete pool of a segment (its incomplete tail) form no pool:
// tail selection appends those keys individually, which is part of the selection, not
// of the pooling. Readings where the page is silent:
//  * the gate has the keys' shape [tokens, d]: one softmax per pool and column (the
//    gate has a key axis; a per-key gate is the case of equal columns);
//  * the FP32 softmax weight is the exact weight rounded to fp32; its cast to bf16,
//    the products and the final cast round to nearest even;
//  * the sum of the bf16 products is formed exactly (compensated) and rounded once;
//  * the first valid key of segment s is cu_seqlens[s] + lead[s] (lead >= 0; a lead at
//    or past the segment's end leaves it without pools).

// The pools in output order: pool o starts at token start[o].
std::vector<int64_t> list_pools(const int32_t* cu, const int32_t* lead, int S, int P) {
  std::vector<int64_t> start;
  for (int s = 0; s < S; ++s) {
    const int64_t first = static_cast<int64_t>(cu[s]) + (lead != nullptr ? lead[s] : 0);
    const int64_t valid = static_cast<int64_t>(cu[s + 1]) - first;
    const int64_t n = valid > 0 ? valid / P : 0;
    for (int64_t b = 0; b < n; ++b) start.push_back(first + b * P);
  }
  return start;
}

int check_kpool_args(const int32_t* cu, const int32_t* lead, int S, int P, int d,
                     int64_t capacity) {
  const int rc = check_args(cu, S, P, 1, d, capacity);
  if (rc != ORACLE_OK) return rc;
  if (lead != nullptr)
    for (int s = 0; s < S; ++s)
      if (lead[s] < 0) return ORACLE_BAD_LEAD;
  return ORACLE_OK;
}

// One pool and column: weights, pooled value in both modes, error mass and slack.
struct PoolColumn {
  double o = 0.0;      // the pooled value before its final bf16 cast
  double err = 0.0;    // first-order fp32 error mass (units of the fp32 unit roundoff)
  double slack = 0.0;  // compression: absolute change a different bf16 weight could make
};

// Weights of an fp32 evaluation are only close to the exact ones: the half-width of the
// interval an fp32 weight can land in, in units of the fp32 unit roundoff, is taken as
// 8 x p x (P + 6 + 2(|x_i| + |m|) + 2 max_j(|x_j| + |m|)): the exponent argument's
// absolute error (~ |x| + |m|, in the exponent of each term and of the normaliser), the
// exponential's and the reciprocal's roundings and the P-term normaliser sum. Where that
// interval holds a bf16 rounding boundary, the compressed weight is not decided by the
// arithmetic, and the slack is the largest change the other choice makes to the pooled
// value (pins in tests/test_kpool_oracle.py).
PoolColumn pool_column(const uint16_t* key, const uint16_t* gate, int64_t start, int P, int d,
                       int64_t j, bool compress) {
  std::vector<double> x(P), v(P), p(P);
  for (int i = 0; i < P; ++i) {
    const int64_t flat = (start + i) * d + j;
    x[i] = bf16_bits_to_double(gate[flat]);
    v[i] = bf16_bits_to_double(key[flat]);
  }
  double m = x[0];
  for (int i = 1; i < P; ++i)
    if (x[i] > m) m = x[i];
  double z = 0.0;
  for (int i = 0; i < P; ++i) {
    p[i] = std::exp(x[i] - m);
    z += p[i];
  }
  for (int i = 0; i < P; ++i) p[i] /= z;
  PoolColumn r;
  if (!compress) {
    for (int i = 0; i < P; ++i) r.o += p[i] * v[i];
    for (int i = 0; i < P; ++i)
      r.err += p[i] * (std::fabs(v[i]) + std::fabs(v[i] - r.o) * (1.0 + std::fabs(x[i]) + std::fabs(m)));
    return r;
  }
  double xspread = 0.0;
  for (int i = 0; i < P; ++i) xspread = std::max(xspread, std::fabs(x[i]) + std::fabs(m));
  const double u32 = std::ldexp(1.0, -24);
  double abs_sum = 0.0;
  double comp = 0.0;  // Neumaier compensation: the P-term sum of products, exact here
  for (int i = 0; i < P; ++i) {
    const double pf = static_cast<double>(static_cast<float>(p[i]));       // FP32 weight
    const double pb = bf16_bits_to_double(double_to_bf16_bits(pf));         // cast to bf16
    const double prod = bf16_bits_to_double(double_to_bf16_bits(pb * v[i]));  // bf16 product
    const double t = r.o + prod;
    comp += std::fabs(r.o) >= std::fabs(prod) ? (r.o - t) + prod : (prod - t) + r.o;
    r.o = t;
    abs_sum += std::fabs(prod);
    const double half = 8.0 * u32 * p[i] *
                        (P + 6.0 + 2.0 * (std::fabs(x[i]) + std::fabs(m)) + 2.0 * xspread);
    // bf16 rounding is monotone: the ends of the interval give the extreme choices
    double worst = 0.0;
    for (const double q : {p[i] - half, p[i] + half}) {
      const double qb =
          bf16_bits_to_double(double_to_bf16_bits(static_cast<double>(static_cast<float>(q))));
      const double alt = bf16_bits_to_double(double_to_bf16_bits(qb * v[i]));
      if (qb != pb) worst = std::max(worst, std::fabs(alt - prod));
    }
    r.slack += worst;
  }
  r.o += comp;
  // the kernel adds the P products in fp32: at most (P - 1) roundings of partial sums
  r.err = P * abs_sum;
  return r;
}

int kpool_impl(const uint16_t* key, const uint16_t* gate, const int32_t* cu, const int32_t* lead,
               int S, int P, int d, int64_t capacity, int64_t out_rows, int compress,
               uint16_t* out_bf16, double* out_f64, double* out_err, double* out_slack,
               int nthreads) {
  int rc = check_kpool_args(cu, lead, S, P, d, capacity);
  if (rc != ORACLE_OK) return rc;
  if (compress != 0 && compress != 1) return ORACLE_BAD_ARGS;
  const std::vector<int64_t> pools = list_pools(cu, lead, S, P);
  if (static_cast<int64_t>(pools.size()) > out_rows) return ORACLE_OUT_ROWS;
  if (!pools.empty() && (key == nullptr || gate == nullptr || out_bf16 == nullptr))
    return ORACLE_BAD_ARGS;
  over_row_ranges(static_cast<int64_t>(pools.size()), nthreads < 1 ? 1 : nthreads,
                  [&](int, int64_t o_begin, int64_t o_end) {
    for (int64_t o = o_begin; o < o_end; ++o)
      for (int64_t j = 0; j < d; ++j) {
        const PoolColumn r = pool_column(key, gate, pools[o], P, d, j, compress != 0);
        out_bf16[o * d + j] = double_to_bf16_bits(r.o);
        if (out_f64 != nullptr) out_f64[o * d + j] = r.o;
        if (out_err != nullptr) out_err[o * d + j] = r.err;
        if (out_slack != nullptr) out_slack[o * d + j] = r.slack;
      }
  });
  return ORACLE_OK;
}

}  // namespace

extern "C" {

// total_comp = sum over segments of floor(seqlen / ratio); -1 on bad arguments.
int64_t csa_oracle_total_comp(const int32_t* cu_seqlens, int S, int ratio) {
  if (cu_seqlens == nullptr || S < 0 || ratio < 1) return -1;
  for (int s = 0; s < S; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
  return count_blocks(cu_seqlens, S, ratio);
}

// Per output row o < out_rows: {segment, block inside segment, first token of the
// block}; rows at or past total_comp get {-1, -1, -1}.
int csa_oracle_map_blocks(const int32_t* cu_seqlens, int S, int ratio, int64_t out_rows,
                          int32_t* seg_blk_base) {
  if (cu_seqlens == nullptr || S < 0 || ratio < 1 || out_rows < 0 ||
      (out_rows > 0 && seg_blk_base == nullptr))
    return ORACLE_BAD_ARGS;
  for (int64_t i = 0; i < out_rows * 3; ++i) seg_blk_base[i] = -1;
  int64_t o = 0;
  for (int s = 0; s < S; ++s) {
    const int64_t n = (cu_seqlens[s + 1] - cu_seqlens[s]) / ratio;
    for (int64_t b = 0; b < n; ++b, ++o) {
      if (o >= out_rows) return ORACLE_OUT_ROWS;
      seg_blk_base[o * 3 + 0] = s;
      seg_blk_base[o * 3 + 1] = static_cast<int32_t>(b);
      seg_blk_base[o * 3 + 2] = static_cast<int32_t>(cu_seqlens[s] + b * ratio);
    }
  }
  return ORACLE_OK;
}

// Forward. kv, score: bf16 bit patterns [capacity, coff*d]; ape: fp32 [ratio, coff*d];
// out_bf16: [out_rows, d] (rows past total_comp are left untouched).
// Optional (may be NULL): out_f64 (unrounded outputs), out_err (error mass, see
// output_error_mass).
int csa_oracle_fwd(const uint16_t* kv, const uint16_t* score, const float* ape,
                   const int32_t* cu_seqlens, int S, int ratio, int coff, int d,
                   int64_t capacity, int64_t out_rows, uint16_t* out_bf16, double* out_f64,
                   double* out_err) {
  return fwd_impl(kv, score, ape, cu_seqlens, S, ratio, coff, d, capacity, out_rows, out_bf16,
                  out_f64, out_err, 1);
}

// Backward. dout: bf16 bits [out_rows, d]. Writes every element of dkv_bf16 and
// dscore_bf16 ([capacity, coff*d]) and dape_f64 ([ratio, coff*d], the sum over all
// blocks, overwritten). Optional (may be NULL): dkv_f64/dscore_f64 (unrounded),
// dape_f32 (dape rounded to fp32), owners (int32 [capacity, coff*d]: how many
// window positions read the slot; must be 0 or 1), dkv_err, dscore_err and dape_err
// (first-order fp32 error masses in units of the fp32 unit roundoff), dape_abs (sum
// of the absolute values of the terms of each dAPE entry).
int csa_oracle_bwd(const uint16_t* kv, const uint16_t* score, const float* ape,
                   const int32_t* cu_seqlens, const uint16_t* dout, int S, int ratio, int coff,
                   int d, int64_t capacity, int64_t out_rows, uint16_t* dkv_bf16,
                   uint16_t* dscore_bf16, double* dape_f64, double* dkv_f64, double* dscore_f64,
                   float* dape_f32, int32_t* owners, double* dkv_err, double* dscore_err,
                   double* dape_err, double* dape_abs) {
  return bwd_impl(kv, score, ape, cu_seqlens, dout, S, ratio, coff, d, capacity, out_rows,
                  dkv_bf16, dscore_bf16, dape_f64, dkv_f64, dscore_f64, dape_f32, owners,
                  dkv_err, dscore_err, dape_err, dape_abs, 1);
}

// The forward and backward on nthreads host threads (contiguous output-row ranges per
// thread), for timing the oracle on all host cores. Same results as the single-thread
// entry points (dAPE up to the order of its final additions). Returns ORACLE_BAD_ARGS
// for nthreads < 1.
int csa_oracle_fwd_threads(const uint16_t* kv, const uint16_t* score, const float* ape,
                           const int32_t* cu_seqlens, int S, int ratio, int coff, int d,
                           int64_t capacity, int64_t out_rows, uint16_t* out_bf16,
                           int nthreads) {
  if (nthreads < 1) return ORACLE_BAD_ARGS;
  return fwd_impl(kv, score, ape, cu_seqlens, S, ratio, coff, d, capacity, out_rows, out_bf16,
                  nullptr, nullptr, nthreads);
}

int csa_oracle_bwd_threads(const uint16_t* kv, const uint16_t* score, const float* ape,
                           const int32_t* cu_seqlens, const uint16_t* dout, int S, int ratio,
                           int coff, int d, int64_t capacity, int64_t out_rows,
                           uint16_t* dkv_bf16, uint16_t* dscore_bf16, double* dape_f64,
                           int nthreads) {
  if (nthreads < 1) return ORACLE_BAD_ARGS;
  return bwd_impl(kv, score, ape, cu_seqlens, dout, S, ratio, coff, d, capacity, out_rows,
                  dkv_bf16, dscore_bf16, dape_f64, nullptr, nullptr, nullptr, nullptr, nullptr,
                  nullptr, nullptr, nullptr, nthreads);
}

// Host threads the machine offers (std::thread::hardware_concurrency; at least 1).
int csa_oracle_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n == 0 ? 1 : static_cast<int>(n);
}

// Round doubles to bf16 bit patterns (exposed so the pins can test the rounding).
void csa_oracle_round_bf16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_bits(x[i]);
}

// KPool: number of pools (sum over segments of floor((seqlen - lead) / P), segments
// whose lead reaches their end contributing none); -1 on bad arguments.
int64_t csa_oracle_kpool_total(const int32_t* cu_seqlens, const int32_t* lead, int S, int P) {
  if (cu_seqlens == nullptr || S < 0 || P < 1) return -1;
  for (int s = 0; s < S; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s] || (lead != nullptr && lead[s] < 0)) return -1;
  return static_cast<int64_t>(list_pools(cu_seqlens, lead, S, P).size());
}

// KPool forward. key, gate: bf16 bit patterns [capacity, d]; lead: int32 [S] or NULL
// (zeros); out_bf16: [out_rows, d] (rows past the pool count are left untouched);
// compress: 0 = FP32 weighted sum, 1 = key-dtype compression. Optional (may be NULL):
// out_f64 (value before the final cast), out_err (error mass, units of the fp32 unit
// roundoff), out_slack (compression: absolute change an undecided bf16 weight could
// make). nthreads >= 1 host threads over contiguous pool ranges (same results).
int csa_oracle_kpool_fwd(const uint16_t* key, const uint16_t* gate, const int32_t* cu_seqlens,
                         const int32_t* lead, int S, int P, int d, int64_t capacity,
                         int64_t out_rows, int compress, uint16_t* out_bf16, double* out_f64,
                         double* out_err, double* out_slack, int nthreads) {
  if (nthreads < 1) return ORACLE_BAD_ARGS;
  return kpool_impl(key, gate, cu_seqlens, lead, S, P, d, capacity, out_rows, compress,
                    out_bf16, out_f64, out_err, out_slack, nthreads);
}

}  // extern "C"
