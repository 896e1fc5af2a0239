/*
 * csa_compressor.h -- C ABI of the GB300 (sm_103a) CSA/HCA KV-compressor
 * gated-softmax pooling over THD-packed ragged sequences.
 *
 * The operation (pages "Megatron-LM PR #5984", commit "CSA: add fused Compressor
 * forward+backward CuTe-DSL kernels", and "cudnn-frontend PR #710"):
 *
 *   A pack holds S segments; segment s covers tokens [cu_seqlens[s], cu_seqlens[s+1]).
 *   A segment of length L has floor(L / ratio) blocks of ratio consecutive tokens,
 *   starting at the segment's first token; its last L mod ratio tokens belong to no
 *   block. Output rows are the blocks of all segments in order (total_comp rows).
 *   For block b of a segment and output column j < d, the window is:
 *     coff=1: the block's own ratio tokens at column j;
 *     coff=2: the previous block's ratio tokens at column j (absent for b = 0)
 *             followed by the block's own ratio tokens at column d + j.
 *   Each position adds ape[q, column read] to its score, q = the token's position in
 *   its own block. A float32 softmax over the window positions weights kv, and the
 *   weighted sum is rounded to bf16: out[row, j].
 *   The backward gives dKV = p * dout and dScore = p * dout * (kv - out) at every slot
 *   a window reads (out unrounded), +0 at every slot no window reads (the last
 *   block's first-half columns at coff=2, tails, segments shorter than ratio, rows
 *   outside [cu_seqlens[0], cu_seqlens[S])), and dAPE[q, col] = the sum of the
 *   unrounded dScore terms that used ape[q, col].
 *
 * Conventions common to every entry point
 *   - Every buffer belongs to the caller. The library allocates nothing, never
 *     synchronises, and never reads device memory from the host.
 *   - Work is enqueued on `stream` (NULL: the legacy default stream) of the current
 *     device; calls return as soon as it is enqueued. The kernels are launched as
 *     programmatic dependents of the stream's previous kernel: they may start while it
 *     finishes, but read and write nothing before it has completed, so stream order
 *     holds exactly as for ordinary launches (also inside CUDA graphs).
 *   - bf16 tensors are row-major and contiguous, fp32 tensors (ape, dape, workspace) too.
 *     Pointers need their natural alignment (2 bytes for bf16, 4 for fp32). The fast
 *     kernels run when d is a multiple of 8 and every pointer is 16-byte aligned; any
 *     other shape takes a scalar kernel, which accepts windows (coff * ratio) of up to
 *     CSA_MAX_GENERIC_WINDOW positions.
 *   - Host-side argument checks return a status and enqueue nothing. Problems that
 *     only the device can see (cu_seqlens decreasing, negative or past capacity;
 *     more blocks than out_rows) make the kernels write a code to *dev_error (when
 *     dev_error is not NULL), skip all output writes, and finish normally; outputs are
 *     then unspecified. The library never clears *dev_error.
 *   - Results are bitwise reproducible run to run (no atomics anywhere).
 */
#ifndef CSA_COMPRESSOR_H_
#define CSA_COMPRESSOR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* csa_stream_t;

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_VALUE = 1, /* NULL pointer, negative size, misaligned pointer */
  CSA_ERR_UNSUPPORTED = 2,   /* coff not in {1,2}, size limits below */
  CSA_ERR_WORKSPACE = 3,     /* backward workspace NULL or smaller than the query's size */
  CSA_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} csa_status_t;

/* Codes the kernels write to *dev_error. */
#define CSA_DEVERR_CU_SEQLENS 1 /* cu_seqlens[0] < 0, decreasing, or cu_seqlens[S] > capacity */
#define CSA_DEVERR_OUT_ROWS 2   /* total_comp > out_rows */
#define CSA_DEVERR_TIMEOUT 3    /* a wait for an asynchronous copy gave up (about 2 s); the
                                   kernel stopped early, outputs (dAPE included) are
                                   incomplete */
#define CSA_DEVERR_LEAD 4       /* KPool: a negative lead */

/* Limits checked on the host (CSA_ERR_UNSUPPORTED beyond them). */
#define CSA_MAX_SEGMENTS 16384   /* S */
#define CSA_MAX_WINDOW 2048      /* coff * ratio */
#define CSA_MAX_GENERIC_WINDOW 256 /* coff * ratio when d % 8 != 0 or a pointer is not 16-byte aligned */
#define CSA_MAX_ELEMS 2147483647 /* capacity*coff*d and out_rows*d must stay below 2^31 */
#define CSA_KPOOL_MAX_POOL 1024  /* KPool pool size */

/* Text for a status code (static storage). */
const char* csa_status_string(int status);

/* Text of the last CUDA runtime error a call of this library met on the calling host
 * thread (why a call returned CSA_ERR_CUDA); static storage. */
const char* csa_last_error_string(void);

/* total_comp = sum over s of floor((cu[s+1] - cu[s]) / ratio), from a HOST copy of
 * cu_seqlens [S+1]. Returns -1 when cu_seqlens is NULL, S < 0, ratio < 1 or the
 * offsets decrease. Definition: "Megatron-LM PR #5984", commit "fold dKV/dScore
 * zero-init into the backward kernel" (tails are seqlen mod ratio). */
int64_t csa_compressor_total_comp(const int32_t* cu_seqlens_host, int32_t S, int32_t ratio);

/* Forward pooling ("Megatron-LM PR #5984", commit "CSA: add fused Compressor
 * forward+backward CuTe-DSL kernels"; coff=1 per commit "widen the validated
 * envelope to coff in {1, 2}"; any ratio >= 1 per "cudnn-frontend PR #710").
 *   kv, score   bf16 [capacity, coff*d] (device)
 *   ape         fp32 [ratio, coff*d] (device)
 *   cu_seqlens  int32 [S+1] (device), non-decreasing, cu_seqlens[S] <= capacity
 *   out         bf16 [out_rows, d] (device); rows >= total_comp are not written
 *   dev_error   int32 (device) or NULL
 * S = 0 or out_rows = 0 with no block is a valid no-op. */
csa_status_t csa_compressor_fwd(const void* kv, const void* score, const float* ape,
                                const int32_t* cu_seqlens, int32_t S, int32_t ratio,
                                int32_t coff, int32_t d, int64_t capacity, void* out,
                                int64_t out_rows, int32_t* dev_error, csa_stream_t stream);

/* Bytes of device workspace csa_compressor_bwd needs for these sizes on the current
 * device: per-row-group dAPE partial sums (reduced in a fixed order) and a 16-byte status
 * block through which the pooling kernel tells the reduction whether the call's
 * cu_seqlens were valid. 0 on bad sizes. */
size_t csa_compressor_bwd_workspace_bytes(int32_t S, int32_t ratio, int32_t coff, int32_t d,
                                          int64_t capacity, int64_t out_rows);

/* Backward pooling ("Megatron-LM PR #5984", commits "CSA: add fused Compressor
 * forward+backward CuTe-DSL kernels" and "fold dKV/dScore zero-init into the
 * backward kernel"). Inputs as for the forward, plus
 *   dout        bf16 [out_rows, d] (device); rows >= total_comp are not read
 *   dkv, dscore bf16 [capacity, coff*d] (device): EVERY element is written
 *   dape        fp32 [ratio, coff*d] (device): accumulate_dape = 0 stores the sum,
 *               1 adds it to the current contents; left untouched when the device
 *               rejects cu_seqlens or out_rows
 *   workspace   device scratch of at least csa_compressor_bwd_workspace_bytes(...)
 *               bytes (CSA_ERR_WORKSPACE otherwise), 16-byte aligned for the vector
 *               kernels; contents on entry do not matter
 * Two kernels are enqueued: the pooling backward and a fixed-order dAPE reduction. */
csa_status_t csa_compressor_bwd(const void* kv, const void* score, const float* ape,
                                const int32_t* cu_seqlens, const void* dout, int32_t S,
                                int32_t ratio, int32_t coff, int32_t d, int64_t capacity,
                                int64_t out_rows, void* dkv, void* dscore, float* dape,
                                int32_t accumulate_dape, void* workspace, size_t workspace_bytes,
                                int32_t* dev_error, csa_stream_t stream);

/* Size of the device scratch array csa_compressor_bwd_noalloc uses (4 MiB per GPU). */
#define CSA_NOALLOC_SCRATCH_BYTES (4 << 20)

/* Backward pooling for callers that cannot allocate device memory when they run it --
 * for example code running inside an allocator or memory-pool callback (allocating there
 * would re-enter the allocator), or a plugin in a host that reserves all device memory up
 * front. The pages describe no such entry point; it is this library's addition. Same
 * arguments and results as csa_compressor_bwd, without the workspace: the dAPE partial
 * sums go to a file-scope device array of CSA_NOALLOC_SCRATCH_BYTES bytes that every GPU
 * loading the library holds until the process unloads it. Nothing is allocated.
 *   - Sizes whose workspace (csa_compressor_bwd_workspace_bytes) exceeds
 *     CSA_NOALLOC_SCRATCH_BYTES are rejected with CSA_ERR_UNSUPPORTED, enqueueing nothing.
 *   - The first call on a device (that device current) looks up the array's device
 *     address once; make that first call before any stream capture.
 *   - All calls on a device share the array, which keeps the last call's contents
 *     (nothing in it needs to start at zero). Calls whose GPU work overlaps -- on
 *     different streams or host threads of the same device -- race on it: order them. */
csa_status_t csa_compressor_bwd_noalloc(const void* kv, const void* score, const float* ape,
                                        const int32_t* cu_seqlens, const void* dout, int32_t S,
                                        int32_t ratio, int32_t coff, int32_t d, int64_t capacity,
                                        int64_t out_rows, void* dkv, void* dscore, float* dape,
                                        int32_t accumulate_dape, int32_t* dev_error,
                                        csa_stream_t stream);

/* Smallest non-zero wait bound csa_compressor_test_hooks accepts, in SM clock cycles. */
#define CSA_TEST_MIN_WAIT_CYCLES 1000000

/* Test hook for the bounded waits: lets a test make a pipeline wait run out without any
 * fault. The pages have no counterpart; it is this library's own.
 *   wait_cycles   bound of every later pooling launch's pipeline waits, in SM clock
 *                 cycles (CSA_TEST_MIN_WAIT_CYCLES .. about 2 s); 0 restores the default
 *                 of about 2 s
 *   withhold_row  >= 0: in every later launch of a bulk-copy kernel (the block-streaming
 *                 and long-window kernels), the producer of CTA (0, 0) skips the copies
 *                 of row `withhold_row` of its row range, so the waits for that stage run
 *                 out, the kernel writes CSA_DEVERR_TIMEOUT to *dev_error, lets its own
 *                 copies land and returns; < 0: off (the default)
 * Process-wide; applies to calls made after it returns, from any host thread.
 * CSA_ERR_INVALID_VALUE for a bound outside the range above. */
csa_status_t csa_compressor_test_hooks(int64_t wait_cycles, int32_t withhold_row);

/* Index map only (the THD segment/block mapping the pooling kernels use), for
 * checking it bit for bit: for every output row o < out_rows writes
 * seg_blk_base[3*o .. 3*o+2] = {segment, block inside the segment, first token of the
 * block}, or {-1, -1, -1} when o >= total_comp. seg_blk_base: int32 [out_rows, 3],
 * device. Reads cu_seqlens on the device like the pooling kernels. */
csa_status_t csa_compressor_map_blocks(const int32_t* cu_seqlens, int32_t S, int32_t ratio,
                                       int64_t capacity, int64_t out_rows, int32_t* seg_blk_base,
                                       int32_t* dev_error, csa_stream_t stream);

/* ------------------------------------------------------------------------------------
 * KPool: the DSA indexer's key pooling ("Megatron-LM PR #8835", the KPool commits: the
 * one adding dsa_indexer_kpool_key_dtype_compression and the explicit-mask pool origin,
 * and the one with the empty-query guard; KPool selection is NVIDIA#8287 there).
 *
 *   Segment s covers keys [cu_seqlens[s], cu_seqlens[s+1]); its first valid key is
 *   f = cu_seqlens[s] + lead[s] (lead NULL: 0). Its keys from f on are grouped into
 *   pools of `pool` consecutive keys, the grid restarting at every segment; the
 *   fewer-than-pool keys after its last complete pool form no pool (tail selection, which
 *   appends them individually, is part of the selection, not of this pooling). Output
 *   rows are the pools of all segments in order (csa_kpool_total rows).
 *   For a pool and column j < d: an FP32 softmax of gate[t, j] over the pool's keys t
 *   weights key[t, j]:
 *     compress = 0: out = bf16(sum_t p_t key[t, j]), the sum in fp32;
 *     compress = 1 (key-dtype compression): each weight is cast to bf16 before
 *       multiplying and reducing: out = bf16(sum_t bf16(bf16(p_t) * key[t, j])), the sum
 *       of the bf16 products in fp32.
 *   Forward only: the selection that consumes the pooled keys records no gradient.
 * ------------------------------------------------------------------------------------ */

/* Number of pools: sum over s of floor(max(0, cu[s+1] - cu[s] - lead[s]) / pool), from
 * HOST copies of cu_seqlens [S+1] and lead [S] (lead may be NULL). Returns -1 when
 * cu_seqlens is NULL, S < 0, pool < 1, the offsets decrease or a lead is negative. */
int64_t csa_kpool_total(const int32_t* cu_seqlens_host, const int32_t* lead_host, int32_t S,
                        int32_t pool);

/* KPool forward.
 *   key, gate   bf16 [capacity, d] (device)
 *   cu_seqlens  int32 [S+1] (device), non-decreasing, cu_seqlens[S] <= capacity
 *   lead        int32 [S] (device), >= 0, or NULL (every segment starts at cu_seqlens[s];
 *               a lead at or past the segment's end leaves it without pools)
 *   pool        1 .. CSA_KPOOL_MAX_POOL
 *   out         bf16 [out_rows, d] (device); rows >= the pool count are not written
 *   compress    0 or 1 (see above)
 *   dev_error   int32 (device) or NULL: CSA_DEVERR_CU_SEQLENS, CSA_DEVERR_LEAD or
 *               CSA_DEVERR_OUT_ROWS (more pools than out_rows); nothing is written then
 * The vector kernel runs when d is a multiple of 8, pool <= 8 and key, gate and out are
 * 16-byte aligned; anything else takes a scalar kernel. One kernel is enqueued (none when
 * S = 0). Status codes as for the compressor. */
csa_status_t csa_kpool_fwd(const void* key, const void* gate, const int32_t* cu_seqlens,
                           const int32_t* lead, int32_t S, int32_t pool, int32_t d,
                           int64_t capacity, void* out, int64_t out_rows, int32_t compress,
                           int32_t* dev_error, csa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA_COMPRESSOR_H_ */
