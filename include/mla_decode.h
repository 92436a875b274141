/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) paged MLA decode library.
 *
 * Operation. Multi-head Latent Attention decode over a paged latent KV cache:
 * for every request b < B and query head h < H, with L = seq_lens[b],
 *
 *   row_t   = kv_cache[block_table[b][t / block_size]][t % block_size][0:576]
 *   s_t     = sm_scale * ( q_nope[b,h,:] . row_t[0:512] + q_pe[b,h,:] . row_t[512:576] )
 *   lse     = ln sum_t exp(s_t)                      (natural log, sm_scale included)
 *   out     = sum_t exp(s_t - lse) * row_t[0:512]    (V is the first 512 latent columns)
 *
 * Sources: "SM100 Cutlass MLA decode with unrestricted num_heads (< 128) for
 * DeepSeek TP" (vLLM PR #20769), opening post (fewer than 128 query heads) and
 * bot summary (heads padded to 128 inside the kernel; KV split across blocks
 * and SMs with a reduction kernel that combines the partial results; a tile
 * scheduler; TMA and warp specialisation), plus the review thread (workspace
 * sized by an op, allocated per instance by the caller, uninitialised memory
 * is fine, sized for the decode batch only); "[Kernel] Flashinfer MLA
 * (trtllm-gen) decode kernel integration" (vLLM PR #21078), E2E Benchmark
 * (paged cache with --block-size 32) and Kernel-only microbenchmark
 * (bs = 512 and bs = 1 decode latency).
 *
 * Conventions shared by every call below:
 *  - All tensors are dense, row-major, owned by the caller. Device pointers
 *    point to memory of the device that was current when the plan was made.
 *  - bf16 tensors are passed as void* (IEEE bfloat16 bit patterns).
 *  - A stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).
 *  - Nothing here allocates device memory except mla_decode_plan (its small
 *    work list). The workspace is caller-owned and needs no initialisation.
 *  - The library loads on any machine; calls that need an sm_103 GPU return
 *    MLA_ERR_UNSUPPORTED_DEVICE elsewhere (a missing-symbol import failure on
 *    older GPUs is what the PR #20769 thread reports; this ABI avoids it).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,         /* bad shape, pointer, alignment or value */
  MLA_ERR_UNSUPPORTED_DEVICE = 2,  /* no sm_103 device current */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < mla_plan_workspace_bytes */
  MLA_ERR_CUDA = 4,                /* a CUDA runtime call failed (launch, alloc, copy) */
  MLA_ERR_DEVICE_FAULT = 5         /* the kernels flagged bad input (see mla_check_device_error) */
} mla_status_t;

/* Device-side error bits reported through mla_check_device_error. */
#define MLA_DEVERR_BAD_BLOCK 1u      /* a block_table entry outside [0, num_blocks) */
#define MLA_DEVERR_SEQLEN_MISMATCH 2u /* device seq_lens[b] differs from the plan's */
#define MLA_DEVERR_TIMEOUT 4u        /* an internal wait gave up (kernel returned early) */

typedef struct mla_plan_s* mla_plan_t; /* opaque; owned by the library */

/* Planner options; zero-initialise and set what you need. */
typedef struct {
  int num_clusters;   /* 0: query the device for co-resident CTA pairs; > 0: use this many */
  int force_splits;   /* 0: automatic; > 0: split every request into this many KV chunks
                         (testing aid; chunks are whole 96-token tiles, empty ones dropped) */
  int host_only;      /* nonzero: build the schedule on the host only (no device upload,
                         no device query unless num_clusters == 0); such a plan can be
                         inspected but not passed to mla_decode */
  int lengths_are_bounds; /* nonzero: seq_lens_host are upper bounds. The schedule (pairs,
                         splits, workspace) is built for the bounds, and on every call the
                         kernels read each request's length L from the device seq_lens
                         (0 <= L <= bound; a larger L raises MLA_DEVERR_SEQLEN_MISMATCH and
                         is clamped to the bound). The launch then does not depend on the
                         lengths: one mla_decode captured in a CUDA graph can be replayed
                         as the lengths change, with no plan update between replays. */
  int q_len;          /* query tokens per request (0 or 1: one; more: speculative decoding).
                         The request's length L counts them as its last q_len tokens and
                         query token j attends to its first L - q_len + 1 + j tokens (each
                         L must be 0 or at least q_len). q_nope, q_pe, out and lse then have
                         a q_len dimension after B: [B, q_len, H, ...]; the q_len * H query
                         rows of a request share its latent KV and are processed as one
                         request with q_len * H heads (at most 1024). */
} mla_plan_options_t;

/*
 * mla_decode_plan — the split-KV scheduler ("tile scheduler" of PR #20769's
 * bot summary; per-decode-batch sizing of its review thread).
 *
 * Reads seq_lens_host[B] (host memory, int32, each 0 <= L <= max_blocks *
 * block_size), chooses how many KV chunks each request is split into and
 * which CTA pair processes each chunk (longest first), and sizes the
 * workspace. Launches no kernel. Copies the schedule (a few KB) to device
 * memory owned by the plan, on the current device.
 * Arguments: B >= 1 requests; 1 <= H <= 1024 query heads, processed in head
 * groups of 128 (one MMA M tile each; each group reads the request's KV once;
 * a group of fewer than 128 heads is padded inside the kernel, never in
 * memory); block_size in {16, 32, 64, 128}; max_blocks >= 1 is the row length
 * of block_table.
 * On success *plan_out receives a new plan (free it with mla_plan_destroy).
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_CUDA.
 */
mla_status_t mla_decode_plan(int B, int H, const int32_t* seq_lens_host, int block_size,
                             int max_blocks, mla_plan_t* plan_out);

/* Same as mla_decode_plan with explicit options (opts may be NULL). */
mla_status_t mla_decode_plan_ex(int B, int H, const int32_t* seq_lens_host, int block_size,
                                int max_blocks, const mla_plan_options_t* opts,
                                mla_plan_t* plan_out);

/*
 * Rebuild an existing plan for new lengths with the same B, H, block_size and
 * max_blocks, reusing its device allocation when large enough. The upload is
 * an asynchronous copy on `stream` from pinned host memory held by the plan
 * (two buffers used in turn), so a decode enqueued later on the same stream
 * sees the new schedule. The call never synchronises the device: when the
 * schedule outgrows the plan's device buffer, a larger one is allocated, the
 * error word is carried over by a copy on `stream`, and the old buffer is
 * kept until mla_plan_destroy. It waits on the host only for the upload made
 * two updates earlier. Do not update a plan while a decode that uses it may
 * still be running on another stream. Errors as mla_decode_plan.
 */
mla_status_t mla_plan_update(mla_plan_t plan, const int32_t* seq_lens_host, void* stream);

/* Workspace bytes mla_decode needs for this plan (0 if no request is split). */
size_t mla_plan_workspace_bytes(mla_plan_t plan);

/* Introspection (tests, logging). Return -1 on a bad argument. */
int mla_plan_num_splits(mla_plan_t plan, int b);  /* KV chunks of request b */
int mla_plan_num_work_items(mla_plan_t plan);     /* chunks over all requests */
int mla_plan_num_clusters(mla_plan_t plan);       /* CTA pairs launched */
/* Work item i: request, first token, end token, partial slot (-1: writes
 * out/lse directly) and the CTA pair that runs it. */
int mla_plan_work_item(mla_plan_t plan, int i, int32_t* b, int32_t* t0, int32_t* t1,
                       int32_t* slot, int32_t* cluster);
/* Query rows [*h_begin, *h_end) of work item i: its head group (128 rows, or
 * the rest for the last group). A request's rows are its heads (j * H + h for
 * query token j with several query tokens). */
int mla_plan_work_item_heads(mla_plan_t plan, int i, int32_t* h_begin, int32_t* h_end);

/*
 * mla_decode — one decode step over the paged latent cache.
 *
 *  q_nope       device bf16 [B, H, 512]   16-byte aligned ([B, q_len, H, 512]
 *               for a plan with q_len > 1; likewise q_pe, out and lse)
 *  q_pe         device bf16 [B, H, 64]    16-byte aligned
 *  kv_cache     device bf16 [num_blocks, block_size, 576]; each row is 512
 *               c_kv columns then 64 k_pe columns; 16-byte aligned
 *  num_blocks   rows of the block pool (>= 1)
 *  block_table  device int32 [B, max_blocks]; entry p of request b names the
 *               physical block of its tokens [p*block_size, (p+1)*block_size).
 *               Entries past a request's last page are never read.
 *  seq_lens     device int32 [B]; must equal the host copy the plan was built
 *               from (a mismatch raises MLA_DEVERR_SEQLEN_MISMATCH)
 *  sm_scale     softmax scale applied to q.k (e.g. 1/sqrt(192))
 *  out          device bf16 [B, H, 512], 16-byte aligned (written)
 *  lse          device fp32 [B, H] (written): natural-log log-sum-exp of the
 *               scaled scores; -inf and out = 0 for a request with L = 0
 *  workspace    device memory of at least mla_plan_workspace_bytes(plan)
 *               bytes, 256-byte aligned, contents ignored (may be NULL if 0)
 *  stream       cudaStream_t as void*
 *
 * Asynchronous: returns after enqueueing the decode kernel (and, when some
 * request is split, the combine kernel) on `stream`. Enqueues nothing else, so
 * it can be captured in a CUDA graph. Block ids outside [0, num_blocks) are
 * detected on the device: the affected rows are read as zeros and an error
 * bit is raised (no trap); see mla_check_device_error.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED_DEVICE,
 * MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_CUDA.
 */
mla_status_t mla_decode(mla_plan_t plan, const void* q_nope, const void* q_pe,
                        const void* kv_cache, int64_t num_blocks, const int32_t* block_table,
                        const int32_t* seq_lens, float sm_scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_fp8 — mla_decode over an FP8 latent cache, the "fp8 KV cache"
 * the pages' deployments serve with ("[Kernel][DSV4.1] Fuse MXFP8 wo_b GEMM
 * with sequence-parallel reduce-scatter" (vLLM PR #57428), serving command
 * with --kv-cache-dtype fp8; "Support DS conv-state layout in fused KDA
 * decode kernel" (vLLM PR #53396), E2E setup). The pages name the cache type
 * only; the element format and the scale below are the readings taken.
 *
 *  kv_cache_fp8 device uint8 [num_blocks, block_size, 576], 16-byte aligned:
 *               OCP E4M3 bytes (sign, 4 exponent bits with bias 7, 3
 *               mantissa bits; no infinities, S.1111.111 is NaN), same row
 *               layout as the bf16 cache (512 c_kv then 64 k_pe columns)
 *  kv_scale     per-tensor scale, finite and > 0: element (blk, slot, d)
 *               stands for kv_scale * e4m3(kv_cache_fp8[blk][slot][d])
 *
 * Every other argument, the plan (any plan mla_decode accepts), the outputs
 * and the errors are those of mla_decode; MLA_ERR_INVALID_ARG also for a bad
 * kv_scale. Computation: K and V are multiplied in 8-bit on the tensor core;
 * q (bf16) and the softmax weights enter those products as two E4M3 terms
 * each, about the 8 significant bits of bf16, and the cache scale is applied
 * in fp32. Reads 576 bytes per cached token instead of 1152.
 */
mla_status_t mla_decode_fp8(mla_plan_t plan, const void* q_nope, const void* q_pe,
                            const void* kv_cache_fp8, float kv_scale, int64_t num_blocks,
                            const int32_t* block_table, const int32_t* seq_lens, float sm_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Sparse (top-k) decode: each request attends only to a selected list of its
 * tokens, the "FlashInfer sparse MLA" attention backend named by "[Kernel]
 * [DSV4.1] Fuse MXFP8 wo_b GEMM with sequence-parallel reduce-scatter" (vLLM
 * PR #57428), serving command. The page names the backend only; the readings
 * taken: topk_indices[b][i] (i < topk) are logical token positions of
 * request b, shared by all its query heads; an entry outside [0, L) is
 * padding and is skipped; an entry listed twice is attended twice; one query
 * token per request. The token selection itself (the indexer) is upstream.
 *
 * mla_sparse_plan — plan for B requests of H query heads with topk entries
 * each (1 <= topk <= 2^20; opts as for mla_decode_plan_ex, q_len 0 or 1;
 * lengths_are_bounds is implied). The plan serves any lists and lengths, so
 * a sparse decode can be captured in a CUDA graph and replayed; it cannot be
 * passed to mla_plan_update, mla_decode, mla_decode_fp8 or
 * mla_decode_no_alloc. mla_plan_workspace_bytes includes the row lists
 * below (B * topk int32, plus B counts).
 * Errors: as mla_decode_plan_ex.
 */
mla_status_t mla_sparse_plan(int B, int H, int topk, const mla_plan_options_t* opts,
                             mla_plan_t* plan_out);

/*
 * mla_decode_sparse — one sparse decode step. A small kernel turns each
 * request's list into the cache rows of its valid entries (in list order)
 * and their count, in the workspace; the decode kernel then copies those
 * rows straight from the paged cache (16-byte asynchronous copies), each
 * request's length being its number of valid entries.
 *
 *  q_nope, q_pe, out, lse, sm_scale, stream   as for mla_decode ([B, H, ...])
 *  kv_cache      device cache [num_blocks, block_size, 576]: bf16 when
 *                kv_fp8 = 0, E4M3 bytes with per-tensor scale kv_scale when
 *                kv_fp8 = 1 (as for mla_decode_fp8); 16-byte aligned
 *  block_size    16, 32, 64 or 128; num_blocks * block_size < 2^31 - 64
 *                (cache rows are 32-bit indices); block_table device int32
 *                [B, max_blocks]; seq_lens device int32 [B] (the lengths L
 *                the list entries are checked against; L <= max_blocks *
 *                block_size is the caller's to keep, as for mla_decode: an
 *                entry whose page lies past the table is skipped)
 *  topk_indices  device int32 [B, topk]
 *  workspace     device memory of at least mla_plan_workspace_bytes(plan)
 *                bytes, 256-byte aligned (always needed: it holds the
 *                row lists)
 *
 * Asynchronous, two or three kernels on `stream` (row lists, decode, and the
 * combine when the plan splits). A selected token whose block id lies
 * outside [0, num_blocks) is skipped and raises MLA_DEVERR_BAD_BLOCK.
 * Errors: MLA_ERR_INVALID_ARG (also for a plan not made by
 * mla_sparse_plan), MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_WORKSPACE_TOO_SMALL,
 * MLA_ERR_CUDA.
 */
mla_status_t mla_decode_sparse(mla_plan_t plan, const void* q_nope, const void* q_pe,
                               const void* kv_cache, int kv_fp8, float kv_scale,
                               int64_t num_blocks, int block_size, const int32_t* block_table,
                               int max_blocks, const int32_t* seq_lens,
                               const int32_t* topk_indices, float sm_scale, void* out, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device memory behind mla_decode_no_alloc (32 MiB). */
#define MLA_NO_ALLOC_SCRATCH_BYTES (((size_t)32) << 20)

/*
 * mla_decode_no_alloc — mla_decode for callers that cannot allocate device
 * memory at decode time. The method's sources have no counterpart: it exists
 * for serving engines whose caching allocator already holds nearly all of
 * HBM, so that a cudaMalloc outside the pool fails or fragments it, and for
 * host threads that must not wait on the device-wide synchronisation that
 * cudaMalloc and cudaFree can bring. (Each call copies the work list from
 * pageable host memory, and such a copy may hold the calling thread until
 * the driver has staged it; it does not wait for the device.)
 *
 * Same computation, kernels and argument rules as mla_decode (bf16 cache),
 * with three differences:
 *  - No workspace argument. The split partials and a copy of the plan's work
 *    list live in one fixed array of MLA_NO_ALLOC_SCRATCH_BYTES inside the
 *    library's device image. Every GPU that loads the library holds it until
 *    the process exits.
 *  - The plan may be host-only (mla_decode_plan_ex with host_only = 1, so
 *    that planning allocates no device memory either). Each call copies the
 *    plan's work list from host memory into the scratch on `stream`.
 *  - err_bits (device uint32, required) receives this call's MLA_DEVERR_*
 *    bits: the call zeroes it, then the kernels OR into it. Read it after the
 *    stream has reached the end of the call. mla_check_device_error does not
 *    see this call's errors.
 *
 * The call allocates nothing: no cudaMalloc, no cudaFree, no pinned memory.
 * Its first call on each device looks up the scratch's device address (and
 * sets the kernel attributes mla_decode also needs). It refuses a stream
 * that is being captured into a CUDA graph (MLA_ERR_INVALID_ARG): its
 * work-list copies read the plan's host memory, which a later
 * mla_plan_update or mla_plan_destroy may change or free before a replay.
 *
 * Every call on a device shares the one scratch array, which keeps what the
 * last call left there. Calls whose work may overlap on the GPU (different
 * streams, or several threads) race on it and corrupt each other's results:
 * order them on one stream or synchronise between them.
 *
 * Errors: those of mla_decode; MLA_ERR_INVALID_ARG also for a NULL err_bits
 * and for a capturing stream; MLA_ERR_WORKSPACE_TOO_SMALL when the plan's
 * work list plus its split partials (mla_plan_workspace_bytes) need more
 * than MLA_NO_ALLOC_SCRATCH_BYTES; such a plan must use mla_decode.
 */
mla_status_t mla_decode_no_alloc(mla_plan_t plan, const void* q_nope, const void* q_pe,
                                 const void* kv_cache, int64_t num_blocks,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 float sm_scale, void* out, float* lse, uint32_t* err_bits,
                                 void* stream);

/*
 * mla_check_device_error — synchronise `stream`, read and clear the plan's
 * device error word (sticky across decodes since the last check). Writes the
 * MLA_DEVERR_* bits to *bits_out (may be NULL) and returns
 * MLA_ERR_DEVICE_FAULT if any bit was set, MLA_OK otherwise, MLA_ERR_CUDA if
 * a CUDA call failed.
 */
mla_status_t mla_check_device_error(mla_plan_t plan, void* stream, uint32_t* bits_out);

/* Free a plan and its device memory (synchronises its device). NULL is ok. */
void mla_plan_destroy(mla_plan_t plan);

/* Static description of a status code. */
const char* mla_status_string(mla_status_t status);

/* 1 if the current device can run mla_decode, 0 otherwise. */
int mla_device_supported(void);

/*
 * mla_selftest_wait_timeout — health check of the error path that every
 * decode relies on when one of its waits cannot complete. The method's
 * sources have no counterpart (they describe no failure detection beyond
 * retries in CI).
 *
 * One warp of a one-block kernel waits, through the same bounded wait routine
 * the decode roles use, on a shared-memory barrier that nothing ever
 * completes. After the wait limit (2e9 SM cycles, about a second) every thread
 * gives up, and the kernel sets MLA_DEVERR_TIMEOUT in a device word that is
 * copied to *bits_out. No trap and no fault is involved: the device stays
 * usable, and a decode issued afterwards runs normally.
 *
 * stream: a cudaStream_t (NULL = the legacy default stream); the call
 * synchronises it and takes about a second. bits_out: host memory, receives
 * the MLA_DEVERR_* bits (MLA_DEVERR_TIMEOUT when the wait gave up as
 * designed). The call allocates and frees 4 bytes of device memory.
 *
 * Errors: MLA_ERR_INVALID_ARG if bits_out is NULL, MLA_ERR_UNSUPPORTED_DEVICE
 * off sm_103, MLA_ERR_CUDA if an allocation, launch or copy fails.
 */
mla_status_t mla_selftest_wait_timeout(void* stream, uint32_t* bits_out);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
