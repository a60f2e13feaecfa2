/*
 * gqa_decode.h -- C ABI of libgqadecode.so, the GB300 (sm_103a) decode-step
 * attention core of the Gemma-4-31B text decoder.
 *
 * Operation (gemma-4-31B Model Spec, "Compute-graph nodes" table, the two
 * `attn.core` rows; tensor shapes from "Tensors of the main nodes", `attn.core`
 * row; masks and append-before-attend from the "Gemma 4 31B-it Text
 * Architecture" page, "Compact form"):
 *
 *   for each sequence b < B and query head h < H, with g = H / KVH and
 *   kvh = floor(h / g):
 *     attended positions  A_b = [lo_b, L_b),  L_b = seq_lens[b],
 *                         lo_b = max(0, L_b - window) if window > 0, else 0
 *     o[b,h,:] = sum_{s in A_b} w_s * v[b,s,kvh,:],
 *     w_s      = exp(<q[b,h,:], k[b,s,kvh,:]>) / sum_{s' in A_b} exp(<q[b,h,:], k[b,s',kvh,:]>)
 *
 *   The attention scale is exactly 1 (no 1/sqrt(D)) and there is no logit
 *   soft-cap (the Model Spec applies its soft-cap to the final logits only).
 *   seq_lens[b] counts the current token, whose K/V row is already in the cache
 *   (the query sits at position L_b - 1).  An empty range (L_b == 0) gives o = 0.
 *
 *   Supported geometries (the two attn.core rows):
 *     slidingDecodeGQA: H = 32, KVH = 16, D = 256, window = 1024 (any window >= 0 accepted)
 *     decodeGQA:        H = 32, KVH =  4, D = 512, window = 0    (any window >= 0 accepted)
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is DEVICE memory of the current CUDA device, owned by
 *     the caller.  The library keeps no pointer past the call.
 *   - bf16 means IEEE bfloat16 (1-8-7), row-major, densely packed, 16-byte
 *     aligned base address.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  Host-side
 *     argument checks happen before anything is enqueued; a failed check
 *     returns an error and enqueues nothing.
 *   - Data-dependent problems are not trapped.  seq_lens and block tables live on
 *     the device and are never read by the host: a length outside
 *     [0, capacity] is clamped into it, and a block-table entry outside [0, P)
 *     on an attended page turns that sequence's output into NaN.  Both raise a
 *     bit in the device status word (gqa_device_status).
 *   - Results are deterministic: the same inputs on the same GPU model give
 *     bit-identical outputs (no floating-point atomics).
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (cudaStream_t is `struct CUstream_st *`). */
typedef struct CUstream_st *gqa_stream_t;

typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, size out of the shape domain */
    GQA_ERR_UNSUPPORTED = 2,      /* (H, KVH, D) is not one of the two attn.core geometries */
    GQA_ERR_WORKSPACE = 3,        /* caller workspace smaller than gqa_workspace_size() */
    GQA_ERR_CUDA = 4              /* a CUDA runtime/driver call failed (launch, allocation, ...) */
} gqa_status_t;

typedef enum {
    GQA_OUT_BF16 = 0, /* o written as bf16 (round to nearest even from the fp32 result) */
    GQA_OUT_F32 = 1   /* o written as fp32 */
} gqa_out_dtype_t;

/* Bits of the device status word (see gqa_device_status). */
#define GQA_DEVICE_WAIT_TIMEOUT 1u /* a pipeline wait gave up after ~2 s; outputs invalid */
#define GQA_DEVICE_BAD_PAGE 2u     /* an attended block-table entry was outside [0, P) */
#define GQA_DEVICE_BAD_LENGTH 4u   /* a seq_lens entry was outside [0, capacity] and was clamped */

/* Limits of the shape domain (Model Spec, "At a glance" table, Shape domain row:
 * B in [1, 256], S in [1, 262144], page size 16). */
#define GQA_MAX_BATCH 256
#define GQA_MAX_SEQ 262144
#define GQA_PAGE_SIZE 16

/*
 * Bytes of device scratch that one call with these sizes needs when the caller
 * supplies the workspace (split-softmax partials, per-(b,kvh) arrival counters
 * and the device status word).  The bound depends on B, H, KVH and D only; S and
 * window are accepted so callers can pass the full call shape.  Returns 0 when
 * the arguments are outside the supported domain (the matching gqa_decode call
 * would fail its argument check).  Pure host arithmetic: no CUDA call.
 */
size_t gqa_workspace_size(int B, int max_seq, int H, int KVH, int D, int window);

/*
 * Prepare a caller-owned workspace for first use: zero-fills `workspace_bytes`
 * bytes on `stream`.  Required once before the first gqa_decode* call that uses
 * the workspace, and again after gqa_device_status reported a nonzero word.
 * Every completed call leaves the workspace ready for the next one.
 */
gqa_status_t gqa_workspace_init(void *workspace, size_t workspace_bytes, gqa_stream_t stream);

/*
 * attn.core over a contiguous KV cache.
 *
 *   q         bf16 [B, H, D]
 *   k, v      bf16 [B, S, KVH, D]; row s of sequence b is cache position s.
 *             k and v may alias (both are only read).
 *   seq_lens  int32 [B] (device), L_b in [0, S]
 *   window    0 = full history (decodeGQA); > 0 = the last `window` positions
 *             (slidingDecodeGQA uses 1024)
 *   out       [B, H, D], bf16 or fp32 per out_dtype; must not overlap the inputs
 *   workspace device scratch of at least gqa_workspace_size(B, S, H, KVH, D, window)
 *             bytes, prepared by gqa_workspace_init; NULL = use a library-owned
 *             per-device buffer (grown on demand with cudaMalloc, which
 *             synchronises the device; calls that share it must not run
 *             concurrently on different streams)
 *
 * Only positions in [lo_b, L_b) are read from k and v; q, k, v, seq_lens are
 * never written.  B == 0 is a valid empty batch: GQA_OK, nothing enqueued.
 * Errors: GQA_ERR_INVALID_ARGUMENT (null or non-16-byte-aligned pointer,
 * B outside [0, 256], S outside [1, 262144], window < 0, unknown out_dtype),
 * GQA_ERR_UNSUPPORTED, GQA_ERR_WORKSPACE, GQA_ERR_CUDA.
 */
gqa_status_t gqa_decode(const void *q, const void *k, const void *v, const int32_t *seq_lens,
                        int B, int S, int H, int KVH, int D, int window, void *out,
                        gqa_out_dtype_t out_dtype, void *workspace, size_t workspace_bytes,
                        gqa_stream_t stream);

/*
 * attn.core over a paged KV cache (16-position pages, Model Spec "At a glance",
 * Shape domain row).
 *
 *   q                 bf16 [B, H, D]
 *   k_pages, v_pages  bf16 [P, 16, KVH, D]: page p, slot j holds one cache
 *                     position for every KV head
 *   block_table       int32 [B, max_pages] (device): position s of sequence b is
 *                     slot s % 16 of page block_table[b, s / 16].  Only the
 *                     entries of pages that hold attended positions are read;
 *                     the rest may hold anything (e.g. -1).
 *   seq_lens          int32 [B] (device), L_b in [0, 16 * max_pages]
 *   page_size         must be 16
 *   other arguments   as for gqa_decode
 *
 * Errors as for gqa_decode, plus GQA_ERR_INVALID_ARGUMENT for P < 1,
 * max_pages < 1, 16 * max_pages > 262144, or page_size != 16.
 */
gqa_status_t gqa_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                              const int32_t *block_table, const int32_t *seq_lens, int B, int P,
                              int max_pages, int page_size, int H, int KVH, int D, int window,
                              void *out, gqa_out_dtype_t out_dtype, void *workspace,
                              size_t workspace_bytes, gqa_stream_t stream);

/*
 * Read and clear the device status word of a workspace (NULL = the library-owned
 * workspace of the current device).  Synchronises `stream`, then stores the OR
 * of the GQA_DEVICE_* bits raised by the calls since the last read into *flags.
 * When the word is nonzero the workspace is re-zeroed before returning.
 */
gqa_status_t gqa_device_status(void *workspace, uint32_t *flags, gqa_stream_t stream);

/*
 * gqa_decode without any allocation, for callers that cannot allocate device
 * memory during a call: for example a plugin layer that is handed only the
 * tensors of one operator, or a runtime whose device memory all belongs to a
 * fixed pool.  gqa_decode needs a workspace the caller supplies or the library
 * allocates (cudaMalloc); this call instead uses one fixed device array of
 * GQA_NOALLOC_SCRATCH_BYTES bytes, built into the library.  Every GPU that
 * loads the library holds that array until the process exits.
 *
 * No counterpart on the reference pages: it is an interface convenience of
 * this library, computing exactly what gqa_decode computes.
 *
 * Arguments, layouts and errors are those of gqa_decode, without the workspace.
 * In addition it returns GQA_ERR_WORKSPACE, enqueueing nothing, when the call
 * needs more scratch than the array holds.  The need is at least
 *   (grid + B*KVH) * g * (D + 2) * 4 bytes plus about 16*B*KVH + 1 KB,
 * where grid = the device's SM count; what is left holds partials of up to
 * min(8*grid, 2048) dynamically scheduled chunks, the slots gqa_decode always
 * has.  Fewer slots leave the result unchanged up to rounding but balance the
 * load across SMs less well.  On a 152-SM GB300 the array covers every
 * slidingDecodeGQA call (B <= 256, all 1216 slots) and decodeGQA calls with
 * B <= 216 (about 860 of the 1216 slots at B = 1, 740 at B = 32).
 *
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  It does the following:
 *   - Its first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and the SM count.  Make
 *     that first call before any stream capture.
 *   - Every call clears the array's claim counter with a 64-byte
 *     cudaMemsetAsync on `stream`.
 * All calls on a device share the one array, and it keeps the last call's
 * contents.  Calls whose kernels overlap on the GPU (different streams) race on
 * it; serialise them.  The array has its own device status word, which
 * collects the GQA_DEVICE_* bits of every call until gqa_noalloc_status reads
 * and clears it (gqa_device_status reads workspaces only).
 */
#define GQA_NOALLOC_SCRATCH_BYTES (16u << 20)

gqa_status_t gqa_decode_noalloc(const void *q, const void *k, const void *v,
                                const int32_t *seq_lens, int B, int S, int H, int KVH, int D,
                                int window, void *out, gqa_out_dtype_t out_dtype,
                                gqa_stream_t stream);

/*
 * Read and clear the device status word of gqa_decode_noalloc's fixed array on the
 * current device: synchronises `stream`, stores the OR of the GQA_DEVICE_* bits
 * raised by gqa_decode_noalloc calls since the last read into *flags, and zeroes
 * the word when it was nonzero.  Allocates nothing.  Errors: GQA_ERR_INVALID_ARGUMENT
 * for a NULL flags pointer, GQA_ERR_CUDA for a failed CUDA call.
 */
gqa_status_t gqa_noalloc_status(uint32_t *flags, gqa_stream_t stream);

/*
 * Decode over a window-capped ring-buffer cache.  Each sliding layer of the
 * retrofit on the "Retrofit Plan: Gemma 4 31B IT -> Progressive Multi-Scale SWA
 * with Block Attention Residuals" page keeps its own KV cache, capped at its
 * window (§3.3 "Progressive Window Assignment", windows 1024/2048/4096/8192;
 * §7.3: the cache grows with the window, not with the sequence).
 *
 *   k, v   bf16 [B, C, KVH, D] contiguous; position s of sequence b is held in
 *          row s mod C (the caller writes the new token there before the call)
 *   C      ring length, 1 <= C <= GQA_MAX_SEQ
 *   window attended positions [max(0, L - window), L), 1 <= window <= C, so
 *          every one of them is still in the ring
 * seq_lens[b] = L is the sequence's length, which may exceed C; it is clamped
 * to [0, GQA_MAX_SEQ] (GQA_DEVICE_BAD_LENGTH when clamped).  Everything else --
 * q, out, workspace, stream, geometries, errors -- is as for gqa_decode; a C or
 * window outside the ranges above returns GQA_ERR_INVALID_ARGUMENT.  The same
 * workspace size serves (it does not depend on C).
 */
gqa_status_t gqa_decode_ring(const void *q, const void *k, const void *v,
                             const int32_t *seq_lens, int B, int C, int H, int KVH, int D,
                             int window, void *out, gqa_out_dtype_t out_dtype, void *workspace,
                             size_t workspace_bytes, gqa_stream_t stream);

/*
 * decodeGQA over a single K=V cache: only the values are cached, and the kernel
 * derives each key from its value.  On the global layers keys and values come
 * from the same projection (gemma-4-31B Model Spec, "What to watch for": values
 * = keys; "Gemma 4 31B-it Text Architecture", decoder listing: V = v_norm(K_raw),
 * K = rope(k_norm(K_raw))).  Both norms divide K_raw by the same root mean
 * square, so the key of the cached value row v at position s is
 *     k = rope(w_k * v, s)
 * with the global layers' rope (Model Spec, `attn.rope` row for layers 5, 11,
 * ..., 59): the pairs (i, i + 256), i < 64, rotated by s * 1e6^(-2i/512),
 * k[i] = x[i] cos - x[i+256] sin, k[i+256] = x[i+256] cos + x[i] sin, every other
 * coordinate unchanged.  Then the attention core is decodeGQA's, full history.
 * Reads half the bytes of separate K and V caches.
 *
 *   q          bf16 [B, 32, 512] (already normed and rotated at its position)
 *   v          bf16 [B, S, 4, 512] contiguous; row s is position s
 *   v_pages    bf16 [P, 16, 4, 512] (paged form); position s of sequence b is
 *              slot s % 16 of page block_table[b][s / 16]
 *   w_k        bf16 [512], the layer's k_norm weight (device memory)
 * Only the decodeGQA geometry (H = 32, KVH = 4, D = 512) is accepted; the
 * slidingDecodeGQA geometry returns GQA_ERR_UNSUPPORTED (its layers project
 * separate values).  Everything else is as for gqa_decode / gqa_decode_paged
 * with window = 0.
 */
gqa_status_t gqa_decode_keqv(const void *q, const void *v, const void *w_k,
                             const int32_t *seq_lens, int B, int S, int H, int KVH, int D,
                             void *out, gqa_out_dtype_t out_dtype, void *workspace,
                             size_t workspace_bytes, gqa_stream_t stream);

gqa_status_t gqa_decode_keqv_paged(const void *q, const void *v_pages, const void *w_k,
                                   const int32_t *block_table, const int32_t *seq_lens, int B,
                                   int P, int max_pages, int page_size, int H, int KVH, int D,
                                   void *out, gqa_out_dtype_t out_dtype, void *workspace,
                                   size_t workspace_bytes, gqa_stream_t stream);

/*
 * Decode-step producer: the nodes ahead of the attention core, fused, for one new
 * token per sequence.  "Gemma 4 31B-it Text Architecture", decoder listing:
 * Q = rope(q_norm(Q)), K = rope(k_norm(K_raw)), V = v_norm(V_raw) with V_raw =
 * K_raw on the global layers, and the new K/V appended to the cache before
 * attention.  gemma-4-31B Model Spec rows: attn.qk_norm (per head
 * x / sqrt(mean(x^2) + 1e-6) * w), attn.v_norm (the same without w), attn.rope
 * (pairs (i, i + D/2) rotated by pos * theta^(-2i/D): 128 pairs, theta 1e4 on
 * slidingDecodeGQA layers; 64 pairs, theta 1e6 on decodeGQA layers).
 *
 *   q_raw     bf16 [B, H, D]        projections of the new token (device)
 *   k_raw     bf16 [B, KVH, D]
 *   v_raw     bf16 [B, KVH, D], or NULL on a global layer with one K=V cache:
 *             then v = v_norm(k_raw) is written to v_cache and k_cache is unused
 *             (gqa_decode_keqv derives the keys)
 *   w_q, w_k  bf16 [D], the q_norm and k_norm weights
 *   seq_lens  int32 [B] (device): lengths AFTER the append; the new token sits at
 *             position L - 1.  Sequences with L < 1 are skipped.
 *   q_out     bf16 [B, H, D]: the attention core's q
 *   gqa_prepare_decode: k_cache, v_cache bf16 [B, rows, KVH, D]; the token goes
 *             to row L - 1 (ring = 0; skipped when L > rows) or row (L - 1) mod
 *             rows (ring = 1, the window-capped cache of gqa_decode_ring)
 *   gqa_prepare_decode_paged: page pools [P, 16, KVH, D]; the token goes to slot
 *             (L - 1) % 16 of page block_table[b][(L - 1) / 16]; a page id outside
 *             [0, P) skips the write (the decode call then reports it)
 * Outputs are rounded to bf16 (round to nearest even) from fp32 arithmetic; the
 * rotation angles are reduced mod 2 pi in fp64.  One kernel launch on `stream`,
 * with programmatic dependent launch so a decode call right behind it overlaps its
 * start.  Errors: GQA_ERR_UNSUPPORTED for other geometries (or v_raw = NULL on a
 * sliding geometry), GQA_ERR_INVALID_ARGUMENT for null or misaligned pointers
 * (16 bytes; 4 for the weights, seq_lens and the block table) and bad sizes,
 * GQA_ERR_CUDA for a failed launch.
 */
gqa_status_t gqa_prepare_decode(const void *q_raw, const void *k_raw, const void *v_raw,
                                const void *w_q, const void *w_k, const int32_t *seq_lens, int B,
                                int H, int KVH, int D, void *q_out, void *k_cache, void *v_cache,
                                int rows, int ring, gqa_stream_t stream);

gqa_status_t gqa_prepare_decode_paged(const void *q_raw, const void *k_raw, const void *v_raw,
                                      const void *w_q, const void *w_k,
                                      const int32_t *block_table, const int32_t *seq_lens, int B,
                                      int P, int max_pages, int page_size, int H, int KVH, int D,
                                      void *q_out, void *k_pages, void *v_pages,
                                      gqa_stream_t stream);

/*
 * Multi-query decode: T new tokens per sequence attend in one call (speculative
 * decoding's draft tokens, or a short chunk of prefill).  "Gemma 4 31B-it Text
 * Architecture", "Inference behavior: Prefill, Cache, and Long Context" and
 * "Compact form": the step's positions are past_seen_tokens + arange(T), the new
 * K/V rows are appended before attention, and every query keeps its own mask
 * (keys s <= t on full layers, t - 1024 < s <= t on sliding layers).  With L_b =
 * seq_lens[b] the length AFTER the append, query t (0 <= t < T) sits at position
 * p = L_b - T + t and attends to
 *     [max(0, p + 1 - window), p + 1)   (window > 0), or [0, p + 1)   (window 0);
 * a query at a negative position (L_b < T - t) attends to nothing and gets o = 0.
 * Each cached K/V row is read once for all T * g query rows of its KV head.
 *
 *   q         bf16 [B, T, H, D]: token t's heads at q[b, t]
 *   k, v      bf16 [B, S, KVH, D] (gqa_decode_mq) or page pools [P, 16, KVH, D] with
 *             block_table [B, max_pages] (gqa_decode_mq_paged), as for gqa_decode
 *             and gqa_decode_paged; only rows of attended positions are used
 *   T         1 .. GQA_MAX_QUERIES_SLIDING (slidingDecodeGQA geometry) or
 *             1 .. GQA_MAX_QUERIES_GLOBAL (decodeGQA geometry)
 *   out       [B, T, H, D], bf16 or fp32 per out_dtype
 *   workspace at least gqa_workspace_size_mq(B, T, H, KVH, D) bytes, prepared by
 *             gqa_workspace_init; NULL = the library-owned per-device buffer
 * Everything else -- seq_lens, window, errors, status bits -- is as for gqa_decode
 * and gqa_decode_paged; a T outside its range returns GQA_ERR_INVALID_ARGUMENT.  A
 * block-table entry outside [0, P) turns into NaN the outputs of exactly the
 * queries whose attended range covers that page.  Rows outside a sequence's
 * attended range are never used; a non-finite value inside it may reach every
 * query of that sequence (the P.V product multiplies it by a zero weight).
 * T >= 2 runs on the tcgen05 tensor cores: scores and P.V as 128-position mma
 * with TMEM accumulators.  T = 1 is a single-token decode and runs on gqa_decode's
 * kernel.
 */
#define GQA_MAX_QUERIES_SLIDING 8
#define GQA_MAX_QUERIES_GLOBAL 4

size_t gqa_workspace_size_mq(int B, int T, int H, int KVH, int D);

gqa_status_t gqa_decode_mq(const void *q, const void *k, const void *v, const int32_t *seq_lens,
                           int B, int T, int S, int H, int KVH, int D, int window, void *out,
                           gqa_out_dtype_t out_dtype, void *workspace, size_t workspace_bytes,
                           gqa_stream_t stream);

gqa_status_t gqa_decode_mq_paged(const void *q, const void *k_pages, const void *v_pages,
                                 const int32_t *block_table, const int32_t *seq_lens, int B,
                                 int T, int P, int max_pages, int page_size, int H, int KVH,
                                 int D, int window, void *out, gqa_out_dtype_t out_dtype,
                                 void *workspace, size_t workspace_bytes, gqa_stream_t stream);

/*
 * Host-side check of the device-resident inputs, for tests and debugging: the
 * caller copies seq_lens (and the block table) to host memory and passes them
 * here.  The decode calls never read these arrays on the host (they stay on the
 * device and the kernel clamps a bad length and turns a bad page into NaN
 * output, raising a GQA_DEVICE_* bit); this reports the same conditions
 * synchronously.
 *
 *   seq_lens     host int32 [B]
 *   capacity     S for a contiguous cache, 16 * max_pages for a paged one
 *   window       0 = full history, > 0 = last `window` positions
 *   block_table  host int32 [B, max_pages], or NULL for a contiguous cache
 *   P            pages in the pool (paged only)
 *   first_bad    optional: index b of the first bad sequence, or -1
 *
 * A sequence is bad when its length lies outside [0, capacity], or (paged)
 * when a page covering one of its attended positions [lo, L) lies outside
 * [0, P).  Entries past the last attended page are not looked at.  Returns
 * GQA_OK when no sequence is bad, GQA_ERR_INVALID_ARGUMENT otherwise or for bad
 * sizes (B outside [0, GQA_MAX_BATCH], capacity < 1, window < 0, NULL seq_lens
 * with B > 0, max_pages or P < 1 on a paged check).
 */
gqa_status_t gqa_check_inputs_host(const int32_t *seq_lens, int B, int capacity, int window,
                                   const int32_t *block_table, int max_pages, int P,
                                   int *first_bad);

/*
 * Which kernel a gqa_decode_keqv / gqa_decode_keqv_paged call with these sizes
 * runs on the current device.  `capacity` is the cache capacity in positions: S
 * for a contiguous cache, 16 * max_pages for a paged one.  The choice depends on
 * the capacity and the device's SM count only (never on the lengths, which stay
 * on the device): a cache of at least 64 tiles of 128 positions per SM takes the
 * tcgen05 kernel (GQA_KERNEL_TCGEN05), a smaller one the split-KV mma.sync kernel
 * (GQA_KERNEL_SPLIT_DECODE).  Returns GQA_KERNEL_NONE for arguments the call would
 * refuse (other geometries, B outside [1, 256], capacity outside [1, 262144]) or
 * when the device cannot be queried.  One CUDA attribute query on first use per
 * device; nothing is enqueued.
 */
typedef enum {
    GQA_KERNEL_NONE = 0,
    GQA_KERNEL_SPLIT_DECODE = 1, /* gqa_decode_kernel: persistent split-KV, warp-level mma */
    GQA_KERNEL_TCGEN05 = 2       /* gqa_mq_kernel: tcgen05 mma with TMEM accumulators */
} gqa_kernel_t;

gqa_kernel_t gqa_decode_keqv_kernel(int B, int capacity, int H, int KVH, int D);

/*
 * Test modes, for the library's own tests (0 in normal use).  The mode is
 * process-wide; every gqa_decode* call reads it once when it is made, so a change
 * affects the calls made after it returns.  gqa_set_test_mode returns the previous
 * mode; bits other than these are ignored.
 *
 *   GQA_TEST_SINGLE_PIECE  every (sequence, KV head) segment is computed in one
 *       piece by one CTA and written straight to the output: no split-KV partials
 *       and no combine.  The result differs from a normal call by rounding only;
 *       the tests check that it agrees within 1e-5.  Slow (one SM does all work).
 *   GQA_TEST_STALL  each CTA's producer, after issuing its first tile, waits on a
 *       barrier that nothing completes.  That wait gives up after 1 ms: the call
 *       takes its timeout exit (every role leaves, copies and tensor-core work in
 *       flight are drained, TMEM is released), raises GQA_DEVICE_WAIT_TIMEOUT and
 *       leaves its outputs invalid.  The workspace is fit for the next call once
 *       gqa_device_status (or gqa_noalloc_status) has read and cleared the word.
 */
#define GQA_TEST_SINGLE_PIECE 1u
#define GQA_TEST_STALL 2u

uint32_t gqa_set_test_mode(uint32_t flags);
uint32_t gqa_get_test_mode(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char *gqa_status_string(gqa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
