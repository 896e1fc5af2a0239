// csa_noalloc.cu -- backward pooling for callers that cannot allocate device memory.
//
// csa_compressor_bwd needs a caller-provided device workspace for its dAPE partial sums.
// Some callers cannot call cudaMalloc at the point where they run the backward: code
// running inside a custom allocator or memory-pool callback (where allocating would
// re-enter the allocator), runtimes whose memory is reserved up front and handed out
// by a framework the caller does not control, and plugin hosts that forbid device
// allocation by plugins. csa_compressor_bwd_noalloc serves them: its scratch is a
// file-scope __device__ array of CSA_NOALLOC_SCRATCH_BYTES bytes that exists on every
// GPU that loads this library, for as long as the process keeps the library loaded.
//
// Setup: the first call on a device (with that device current) looks up the array's
// device address with cudaGetSymbolAddress and remembers it for that device; this first
// call should come before any stream capture. The array is shared by every call on a
// device and keeps the last call's contents; nothing in it needs to start at zero (the
// backward writes every partial it later reads). Calls whose work overlaps on the GPU
// (different streams, or different host threads, on the same device) race on the array.
// This file allocates nothing and calls no allocating routine.
#include <mutex>

#include "csa_compressor.h"
#include "csa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[CSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" csa_status_t csa_compressor_bwd_noalloc(const void* kv, const void* score,
                                                   const float* ape, const int32_t* cu_seqlens,
                                                   const void* dout, int32_t S, int32_t ratio,
                                                   int32_t coff, int32_t d, int64_t capacity,
                                                   int64_t out_rows, void* dkv, void* dscore,
                                                   float* dape, int32_t accumulate_dape,
                                                   int32_t* dev_error, csa_stream_t stream) {
  const size_t need = csa_compressor_bwd_workspace_bytes(S, ratio, coff, d, capacity, out_rows);
  if (need == 0) {
    // Bad sizes: let the regular entry point report the precise status.
    return csa_compressor_bwd(kv, score, ape, cu_seqlens, dout, S, ratio, coff, d, capacity,
                              out_rows, dkv, dscore, dape, accumulate_dape, nullptr, 0,
                              dev_error, stream);
  }
  if (need > static_cast<size_t>(CSA_NOALLOC_SCRATCH_BYTES)) return CSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA_ERR_CUDA;
  return csa_compressor_bwd(kv, score, ape, cu_seqlens, dout, S, ratio, coff, d, capacity,
                            out_rows, dkv, dscore, dape, accumulate_dape, scratch,
                            static_cast<size_t>(CSA_NOALLOC_SCRATCH_BYTES), dev_error, stream);
}
