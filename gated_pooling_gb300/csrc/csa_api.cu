// csa_api.cu -- the C ABI of the GB300 CSA/HCA compressor pooling: argument checks,
// launch planning, the index-map test hook and the fixed-order dAPE reduction.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <atomic>
#include <mutex>
#include <type_traits>
#include <vector>

#include <cuda.h>

#include "csa_compressor.h"
#include "csa_internal.h"

namespace csa {
namespace {

// Every launch runs on the current device. Multiprocessor counts and occupancies are
// looked up once per (device, kernel, shared-memory size).
struct OccEntry {
  int dev;
  const void* kernel;
  int threads;
  size_t smem;
  int blocks;
};
std::mutex g_mu;
std::vector<OccEntry> g_occ;
std::vector<int> g_sms;
std::vector<std::pair<int, const void*>> g_attr_set;
thread_local cudaError_t t_last_error = cudaSuccess;
// Test hook state (csa_compressor_test_hooks): the pipeline wait bound and the withheld row.
std::atomic<long long> g_wait_cycles{kWaitCycles};
std::atomic<int> g_withhold_row{-1};

}  // namespace

// Records a failing CUDA call for csa_last_error_string() and passes the code on.
cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess) t_last_error = e;
  return e;
}

cudaError_t device_sms(int dev, int* sms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < static_cast<int>(g_sms.size()) && g_sms[dev] > 0) {
    *sms = g_sms[dev];
    return cudaSuccess;
  }
  int n = 0;
  cudaError_t e = note(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
  if (e != cudaSuccess) return e;
  if (dev >= static_cast<int>(g_sms.size())) g_sms.resize(dev + 1, 0);
  g_sms[dev] = n;
  *sms = n;
  return cudaSuccess;
}

// Blocks of `kernel` resident per SM with `smem` bytes of dynamic shared memory (0 if
// it cannot run at all). Raises the kernel's dynamic shared-memory limit once.
cudaError_t blocks_per_sm(int dev, const void* kernel, int threads, size_t smem, int* blocks) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (const OccEntry& e : g_occ)
    if (e.dev == dev && e.kernel == kernel && e.threads == threads && e.smem == smem) {
      *blocks = e.blocks;
      return cudaSuccess;
    }
  bool attr = false;
  for (const auto& a : g_attr_set) attr = attr || (a.first == dev && a.second == kernel);
  if (!attr) {
    // The dynamic limit may reach the opt-in maximum less the kernel's static shared memory.
    int optin = 0;
    cudaError_t e = note(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = note(cudaFuncGetAttributes(&fa, kernel));
    if (e != cudaSuccess) return e;
    const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
    e = note(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn));
    if (e != cudaSuccess) return e;
    g_attr_set.emplace_back(dev, kernel);
  }
  int n = 0;
  cudaError_t e = note(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem));
  if (e != cudaSuccess) return e;
  g_occ.push_back({dev, kernel, threads, smem, n});
  *blocks = n;
  return cudaSuccess;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 2-D tensor maps for the long-window kernel, encoded through the driver entry point the
// runtime hands out (no link against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// bf16 matrix [rows, cols] (row stride cols), boxes of [box_rows, box_cols] written to
// shared memory with the (box_cols * 2)-byte swizzle (box_cols 64 or 32).
bool encode_bf16_map(CUtensorMap* map, const void* base, int64_t rows, int cols, int box_cols,
                     int box_rows) {
  if (box_cols != 64 && box_cols != 32) return false;
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols),
                              static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

csa_status_t check_sizes(int32_t S, int32_t ratio, int32_t coff, int32_t d, int64_t capacity,
                         int64_t out_rows) {
  if (S < 0 || ratio < 1 || d < 1 || capacity < 0 || out_rows < 0) return CSA_ERR_INVALID_VALUE;
  if (coff != 1 && coff != 2) return CSA_ERR_UNSUPPORTED;
  if (S > CSA_MAX_SEGMENTS) return CSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(coff) * ratio > CSA_MAX_WINDOW) return CSA_ERR_UNSUPPORTED;
  const int64_t C = static_cast<int64_t>(coff) * d;
  if (C > INT_MAX / 8) return CSA_ERR_UNSUPPORTED;
  if (capacity > 0 && capacity > INT_MAX / C) return CSA_ERR_UNSUPPORTED;
  if (out_rows > 0 && out_rows > INT_MAX / d) return CSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(ratio) * C > INT_MAX) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

static_assert(kGenericMaxWindow == CSA_MAX_GENERIC_WINDOW, "generic window limit");

// Backward workspace: the fp32 dAPE partials [R, ratio, coff*d], then (at the next 16-byte
// boundary) the call's status word that the pooling kernel writes and the reduction reads.
size_t partial_bytes(const Plan& pl, int32_t ratio, int32_t coff, int32_t d) {
  return (static_cast<size_t>(pl.R) * ratio * coff * d * sizeof(float) + 15) & ~static_cast<size_t>(15);
}
size_t workspace_need(const Plan& pl, int32_t ratio, int32_t coff, int32_t d) {
  return partial_bytes(pl, ratio, coff, d) + 16;
}

// Plan plus the device-dependent row-group count R. `fast`: d % 8 == 0 and every pointer
// 16-byte aligned (the vector kernels); otherwise the generic scalar kernel.
csa_status_t make_plan(bool bwd, int32_t S, int32_t ratio, int32_t coff, int32_t d,
                       int64_t out_rows, bool fast, Plan* pl, PoolKernel* kernel) {
  int dev = 0, sms = 0, bps = 0, optin = 0;
  if (note(cudaGetDevice(&dev)) != cudaSuccess) return CSA_ERR_CUDA;
  if (device_sms(dev, &sms) != cudaSuccess) return CSA_ERR_CUDA;
  if (note(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
      cudaSuccess)
    return CSA_ERR_CUDA;
  const size_t limit = static_cast<size_t>(optin) - 256;  // static shared memory headroom
  if (!choose_plan(bwd, S, ratio, coff, d, out_rows, sms, fast, encode_fn() != nullptr, limit,
                   pl))
    return CSA_ERR_UNSUPPORTED;
  *kernel = bwd ? bwd_kernel_for(*pl) : fwd_kernel_for(*pl);
  if (*kernel == nullptr) return CSA_ERR_UNSUPPORTED;
  if (blocks_per_sm(dev, reinterpret_cast<const void*>(*kernel), pl->threads, pl->smem, &bps) !=
      cudaSuccess)
    return CSA_ERR_CUDA;
  if (bps < 1) return CSA_ERR_UNSUPPORTED;  // shared memory of the plan does not fit
  pl->R = row_groups(*pl, sms, bps, out_rows);
  return CSA_OK;
}

PoolParams base_params(const Plan& pl, const void* kv, const void* score, const float* ape,
                       const int32_t* cu, int32_t S, int32_t ratio, int32_t coff, int32_t d,
                       int64_t capacity, int64_t out_rows, int32_t* dev_error) {
  PoolParams p{};
  p.kv = static_cast<const uint16_t*>(kv);
  p.score = static_cast<const uint16_t*>(score);
  p.ape = ape;
  p.cu = cu;
  p.dev_error = dev_error;
  p.capacity = capacity;
  p.out_rows = out_rows;
  p.S = S;
  p.r = ratio;
  p.coff = coff;
  p.d = d;
  p.C = coff * d;
  p.W = coff * ratio;
  p.P = pl.P;
  p.V = pl.V;
  p.Vs = pl.Vs;
  p.slots = pl.slots;
  p.R = pl.R;
  p.sB_words = pl.sB_words;
  p.depth = pl.depth;
  p.stage_bytes = pl.stage_bytes;
  p.ape_off = pl.ape_off;
  p.pre_off = pl.pre_off;
  p.ring_off = pl.ring_off;
  p.bar_off = pl.bar_off;
  p.box_rows = pl.box_rows;
  p.np = pl.np;
  p.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
  p.withhold_row = g_withhold_row.load(std::memory_order_relaxed);
  return p;
}

}  // namespace

// Every pooling kernel is launched as a programmatic dependent of the stream's previous
// kernel (it waits for that grid inside build_block_prefix before touching memory).
#ifndef CSA_PDL_POOL
#define CSA_PDL_POOL 1
#endif
cudaError_t launch_pdl(const void* k, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = CSA_PDL_POOL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return note(cudaLaunchKernelExC(&cfg, k, args));
}

namespace {

csa_status_t launch(PoolKernel k, const Plan& pl, PoolParams& p, cudaStream_t stream) {
  if (pl.longk) {
    // tensor maps over kv and score [capacity, C]; with no rows any aligned address will
    // do (nothing is copied)
    // (the backward also stores dKV and dScore through maps; the forward gets copies of
    // the input maps in those places and never uses them)
    CUtensorMap mkv, msc, mdkv, mdsc;
    const int sw = 4 * pl.Vs;  // the slice: 64 (or 32) columns = one 128 (64)-byte swizzle row
    const void* kv = p.kv != nullptr ? static_cast<const void*>(p.kv) : p.ape;
    const void* sc = p.score != nullptr ? static_cast<const void*>(p.score) : p.ape;
    const void* dkv = p.dkv != nullptr ? static_cast<const void*>(p.dkv) : kv;
    const void* dsc = p.dscore != nullptr ? static_cast<const void*>(p.dscore) : sc;
    if (!encode_bf16_map(&mkv, kv, p.capacity, p.C, sw, pl.box_rows) ||
        !encode_bf16_map(&msc, sc, p.capacity, p.C, sw, pl.box_rows) ||
        !encode_bf16_map(&mdkv, dkv, p.capacity, p.C, sw, pl.box_rows) ||
        !encode_bf16_map(&mdsc, dsc, p.capacity, p.C, sw, pl.box_rows))
      return CSA_ERR_CUDA;
    void* args[] = {&p, &mkv, &msc, &mdkv, &mdsc};
    const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(k), dim3(pl.K, pl.R),
                                     dim3(pl.threads), pl.smem, stream, args);
    return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
  }
  void* args[] = {&p};
  const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(k), dim3(pl.K, pl.R),
                                   dim3(pl.threads), pl.smem, stream, args);
  return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

// dAPE = (accumulate ? dAPE : 0) + sum over row groups g = 0..R-1 of partial[g]. A block
// covers COLS entries (one per lane group) with SPLIT thread groups; group k adds the
// contiguous row-group range [k*R/SPLIT, (k+1)*R/SPLIT) (loaded kReduceBatch at a time, so
// the loads overlap) with compensated fp32 sums; the range sums are then combined pairwise
// in a fixed tree. SPLIT follows R (about five partials per group, ten when R is small),
// COLS is 16 when there are few entries (more blocks); both measured on GB300. The result
// is the same bits on every run. Launched as a programmatic dependent of the pooling
// kernel: it waits for that grid's results.
constexpr int kReduceBatch = 12;  // partials a thread has in flight at once
// A non-zero status word (the pooling kernel found cu_seqlens or out_rows invalid) leaves
// dAPE untouched.
template <int SPLIT, int COLS>
__global__ void __launch_bounds__(COLS * SPLIT)
    dape_reduce_kernel(const float* __restrict__ partial, int R, int n, float* __restrict__ dape,
                       int accumulate, const int32_t* __restrict__ status) {
  constexpr int kReduceSplit = SPLIT;
  constexpr int kReduceCols = COLS;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // read with the partials (only the final write depends on it)
  const int32_t call_status = *reinterpret_cast<const volatile int32_t*>(status);
  __shared__ float s_sum[kReduceSplit][kReduceCols];
  __shared__ float s_cmp[kReduceSplit][kReduceCols];
  const int lane = threadIdx.x % kReduceCols;
  const int k = threadIdx.x / kReduceCols;
  const int e = blockIdx.x * kReduceCols + lane;
  const int g_lo = static_cast<int>(static_cast<int64_t>(k) * R / kReduceSplit);
  const int g_hi = static_cast<int>(static_cast<int64_t>(k + 1) * R / kReduceSplit);
  float s = 0.f, c = 0.f;
  if (e < n) {
    // kReduceBatch partials in flight at a time, added in ascending g
    for (int g0 = g_lo; g0 < g_hi; g0 += kReduceBatch) {
      float v[kReduceBatch];
#pragma unroll
      for (int u = 0; u < kReduceBatch; ++u)
        v[u] = g0 + u < g_hi ? __ldg(partial + static_cast<int64_t>(g0 + u) * n + e) : 0.f;
#pragma unroll
      for (int u = 0; u < kReduceBatch; ++u)
        if (g0 + u < g_hi) neumaier_add(s, c, v[u]);
    }
  }
  s_sum[k][lane] = s;
  s_cmp[k][lane] = c;
  // the range sums, combined pairwise in a fixed tree (ranges k and k + h, h = SPLIT/2,
  // SPLIT/4, ..., 1), carrying each side's compensation
  for (int h = kReduceSplit / 2; h >= 1; h /= 2) {
    __syncthreads();
    if (k < h) {
      float t = s_sum[k][lane], tc = s_cmp[k][lane];
      neumaier_add(t, tc, s_sum[k + h][lane]);
      neumaier_add(t, tc, s_cmp[k + h][lane]);
      s_sum[k][lane] = t;
      s_cmp[k][lane] = tc;
    }
  }
  __syncthreads();
  if (k == 0 && e < n && call_status == 0) {
    float t = 0.f, tc = 0.f;
    if (accumulate) neumaier_add(t, tc, dape[e]);
    neumaier_add(t, tc, s_sum[0][lane]);
    neumaier_add(t, tc, s_cmp[0][lane]);
    dape[e] = t + tc;
  }
}

__global__ void map_blocks_kernel(const int32_t* __restrict__ cu, int S, int ratio,
                                  int64_t capacity, int64_t out_rows, int32_t* __restrict__ out,
                                  int32_t* dev_error) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_sums[32];
  int* sB = reinterpret_cast<int*>(smem);
  const int TC = build_block_prefix(cu, S, ratio, capacity, out_rows, dev_error, sB, warp_sums);
  if (TC < 0) return;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < out_rows;
       o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int32_t v0 = -1, v1 = -1, v2 = -1;
    if (o < TC) {
      const int s = find_segment(sB, S, static_cast<int>(o));
      const int b = static_cast<int>(o) - sB[s];
      v0 = s;
      v1 = b;
      v2 = __ldg(cu + s) + b * ratio;
    }
    out[3 * o + 0] = v0;
    out[3 * o + 1] = v1;
    out[3 * o + 2] = v2;
  }
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" {

const char* csa_status_string(int status) {
  switch (status) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_VALUE: return "CSA_ERR_INVALID_VALUE: null, negative or misaligned argument";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: coff not in {1,2}, or a size limit exceeded";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: workspace missing or smaller than csa_compressor_bwd_workspace_bytes";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    default: return "unknown csa status";
  }
}

const char* csa_last_error_string(void) {
  return t_last_error == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(t_last_error);
}

int64_t csa_compressor_total_comp(const int32_t* cu, int32_t S, int32_t ratio) {
  if (cu == nullptr || S < 0 || ratio < 1) return -1;
  int64_t t = 0;
  for (int32_t s = 0; s < S; ++s) {
    if (cu[s + 1] < cu[s]) return -1;
    t += (cu[s + 1] - cu[s]) / ratio;
  }
  return t;
}

csa_status_t csa_compressor_fwd(const void* kv, const void* score, const float* ape,
                                const int32_t* cu_seqlens, int32_t S, int32_t ratio,
                                int32_t coff, int32_t d, int64_t capacity, void* out,
                                int64_t out_rows, int32_t* dev_error, csa_stream_t stream) {
  csa_status_t st = check_sizes(S, ratio, coff, d, capacity, out_rows);
  if (st != CSA_OK) return st;
  if (cu_seqlens == nullptr || ape == nullptr) return CSA_ERR_INVALID_VALUE;
  if (capacity > 0 && (kv == nullptr || score == nullptr)) return CSA_ERR_INVALID_VALUE;
  if (out_rows > 0 && out == nullptr) return CSA_ERR_INVALID_VALUE;
  if (!aligned_to(kv, 2) || !aligned_to(score, 2) || !aligned_to(ape, 4) || !aligned_to(out, 2))
    return CSA_ERR_INVALID_VALUE;
  const bool fast = d % 8 == 0 && aligned16(kv) && aligned16(score) && aligned16(ape) &&
                    aligned16(out);
  if (!fast && coff * ratio > CSA_MAX_GENERIC_WINDOW) return CSA_ERR_UNSUPPORTED;
  Plan pl;
  PoolKernel k;
  st = make_plan(false, S, ratio, coff, d, out_rows, fast, &pl, &k);
  if (st != CSA_OK) return st;
  PoolParams p = base_params(pl, kv, score, ape, cu_seqlens, S, ratio, coff, d, capacity,
                             out_rows, dev_error);
  p.out = static_cast<uint16_t*>(out);
  return launch(k, pl, p, reinterpret_cast<cudaStream_t>(stream));
}

size_t csa_compressor_bwd_workspace_bytes(int32_t S, int32_t ratio, int32_t coff, int32_t d,
                                          int64_t capacity, int64_t out_rows) {
  if (check_sizes(S, ratio, coff, d, capacity, out_rows) != CSA_OK) return 0;
  // enough for whichever kernel the call's pointers select
  size_t need = 0;
  for (int fast = 0; fast < 2; ++fast) {
    if (fast && d % 8 != 0) continue;
    if (!fast && coff * ratio > CSA_MAX_GENERIC_WINDOW) continue;
    Plan pl;
    PoolKernel k;
    if (make_plan(true, S, ratio, coff, d, out_rows, fast != 0, &pl, &k) != CSA_OK) continue;
    need = std::max(need, workspace_need(pl, ratio, coff, d));
  }
  return need;
}

csa_status_t csa_compressor_bwd(const void* kv, const void* score, const float* ape,
                                const int32_t* cu_seqlens, const void* dout, int32_t S,
                                int32_t ratio, int32_t coff, int32_t d, int64_t capacity,
                                int64_t out_rows, void* dkv, void* dscore, float* dape,
                                int32_t accumulate_dape, void* workspace, size_t workspace_bytes,
                                int32_t* dev_error, csa_stream_t stream) {
  csa_status_t st = check_sizes(S, ratio, coff, d, capacity, out_rows);
  if (st != CSA_OK) return st;
  if (cu_seqlens == nullptr || ape == nullptr || dape == nullptr) return CSA_ERR_INVALID_VALUE;
  if (capacity > 0 && (kv == nullptr || score == nullptr || dkv == nullptr || dscore == nullptr))
    return CSA_ERR_INVALID_VALUE;
  if (out_rows > 0 && dout == nullptr) return CSA_ERR_INVALID_VALUE;
  if (!aligned_to(kv, 2) || !aligned_to(score, 2) || !aligned_to(ape, 4) ||
      !aligned_to(dout, 2) || !aligned_to(dkv, 2) || !aligned_to(dscore, 2) ||
      !aligned_to(dape, 4) || !aligned_to(workspace, 4))
    return CSA_ERR_INVALID_VALUE;
  const bool fast = d % 8 == 0 && aligned16(kv) && aligned16(score) && aligned16(ape) &&
                    aligned16(dout) && aligned16(dkv) && aligned16(dscore) && aligned16(dape) &&
                    aligned16(workspace);
  if (!fast && coff * ratio > CSA_MAX_GENERIC_WINDOW) return CSA_ERR_UNSUPPORTED;
  Plan pl;
  pl.R = 1;  // no plan has fewer row groups: smaller workspaces are rejected before planning
  if (workspace == nullptr || workspace_bytes < workspace_need(pl, ratio, coff, d))
    return CSA_ERR_WORKSPACE;
  PoolKernel k;
  st = make_plan(true, S, ratio, coff, d, out_rows, fast, &pl, &k);
  if (st != CSA_OK) return st;
  const size_t need = workspace_need(pl, ratio, coff, d);
  if (workspace == nullptr || workspace_bytes < need) return CSA_ERR_WORKSPACE;
  PoolParams p = base_params(pl, kv, score, ape, cu_seqlens, S, ratio, coff, d, capacity,
                             out_rows, dev_error);
  p.dout = static_cast<const uint16_t*>(dout);
  p.dkv = static_cast<uint16_t*>(dkv);
  p.dscore = static_cast<uint16_t*>(dscore);
  p.partial = static_cast<float*>(workspace);
  p.status = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) +
                                        partial_bytes(pl, ratio, coff, d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = launch(k, pl, p, s);
  if (st != CSA_OK) return st;
  const float* part = static_cast<const float*>(workspace);
  int n = ratio * coff * d;
  int R = pl.R;
  int acc = accumulate_dape != 0;
  const int32_t* status = p.status;
  void* rargs[] = {&part, &R, &n, &dape, &acc, &status};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // thread groups per block: the power of two nearest above R/5 (R/10 when R is below 32),
  // at most 32; 16 entries per block when 32-entry blocks would be fewer than 64
  const int per = R < 32 ? 10 : 5;
  int split = 1;
  while (split < 32 && split * per < R) split *= 2;
  const bool narrow = (n + 31) / 32 < 64;
  const int cols = narrow ? 16 : 32;
  auto pick = [&](auto c) -> const void* {
    constexpr int C = decltype(c)::value;
    return split == 1    ? reinterpret_cast<const void*>(dape_reduce_kernel<1, C>)
           : split == 2  ? reinterpret_cast<const void*>(dape_reduce_kernel<2, C>)
           : split == 4  ? reinterpret_cast<const void*>(dape_reduce_kernel<4, C>)
           : split == 8  ? reinterpret_cast<const void*>(dape_reduce_kernel<8, C>)
           : split == 16 ? reinterpret_cast<const void*>(dape_reduce_kernel<16, C>)
                         : reinterpret_cast<const void*>(dape_reduce_kernel<32, C>);
  };
  const void* rk = narrow ? pick(std::integral_constant<int, 16>{})
                          : pick(std::integral_constant<int, 32>{});
  cfg.gridDim = dim3((n + cols - 1) / cols);
  cfg.blockDim = dim3(cols * split);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      note(cudaLaunchKernelExC(&cfg, rk, rargs));
  return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

csa_status_t csa_compressor_test_hooks(int64_t wait_cycles, int32_t withhold_row) {
  if (wait_cycles < 0 || (wait_cycles > 0 && wait_cycles < CSA_TEST_MIN_WAIT_CYCLES) ||
      wait_cycles > kWaitCycles)
    return CSA_ERR_INVALID_VALUE;
  g_wait_cycles.store(wait_cycles == 0 ? kWaitCycles : wait_cycles, std::memory_order_relaxed);
  g_withhold_row.store(withhold_row < 0 ? -1 : withhold_row, std::memory_order_relaxed);
  return CSA_OK;
}

csa_status_t csa_compressor_map_blocks(const int32_t* cu_seqlens, int32_t S, int32_t ratio,
                                       int64_t capacity, int64_t out_rows, int32_t* seg_blk_base,
                                       int32_t* dev_error, csa_stream_t stream) {
  if (cu_seqlens == nullptr || S < 0 || ratio < 1 || capacity < 0 || out_rows < 0)
    return CSA_ERR_INVALID_VALUE;
  if (out_rows > 0 && seg_blk_base == nullptr) return CSA_ERR_INVALID_VALUE;
  if (S > CSA_MAX_SEGMENTS || out_rows > INT_MAX / 3) return CSA_ERR_UNSUPPORTED;
  const int64_t blocks64 = (out_rows + kThreads - 1) / kThreads;
  const int blocks = blocks64 < 1 ? 1 : (blocks64 > 1024 ? 1024 : static_cast<int>(blocks64));
  const size_t smem = static_cast<size_t>((S + 1 + 3) & ~3) * sizeof(int);
  int dev = 0, bps = 0;
  if (note(cudaGetDevice(&dev)) != cudaSuccess) return CSA_ERR_CUDA;
  if (blocks_per_sm(dev, reinterpret_cast<const void*>(map_blocks_kernel), kThreads, smem, &bps) !=
      cudaSuccess)
    return CSA_ERR_CUDA;
  void* args[] = {const_cast<int32_t**>(&cu_seqlens), &S, &ratio, &capacity, &out_rows,
                  &seg_blk_base, &dev_error};
  const cudaError_t e = note(cudaLaunchKernel(reinterpret_cast<const void*>(map_blocks_kernel),
                                              dim3(blocks), dim3(kThreads), args, smem,
                                              reinterpret_cast<cudaStream_t>(stream)));
  return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

}  // extern "C"
