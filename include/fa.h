/*
 * fa.h -- C ABI of libfa: exact IO-aware attention (FlashAttention forward, backward and
 * split-KV decode) for NVIDIA GB300 (sm_103a).
 *
 * Pages this interface follows (cited by title and section):
 *   [Lesson4]  "FlashAttention and online softmax", ML Systems lesson 4.
 *   [Scratch]  "FlashAttention from Scratch -- The Paradox of Doing More Math to Go Faster".
 *
 * Conventions shared by every call
 * --------------------------------
 *  Layout     q, k, v, o, dO, dq, dk, dv are dense row-major [B, H, N, d] arrays of bfloat16
 *             (raw 16-bit patterns, type fa_bf16_t), d fastest.  lse is fp32 [B, H, N_q],
 *             natural logarithm.  Shapes (batch, heads, N, d) as in [Lesson4] section 5.
 *  Pointers   All array pointers are DEVICE pointers owned by the caller.  The library never
 *             allocates, frees or keeps a pointer after the call returns.  Every array must be
 *             16-byte aligned (TMA requirement).
 *  Streams    ``stream`` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *             Calls only enqueue work and return; nothing synchronises except fa_sync_status.
 *  Support    d in {64, 128}; 1 <= B*H; N_q, N_kv >= 0 and < 2^31 / d.  ``causal`` means query i
 *             sees keys j <= i ([Lesson4] "Causal masks") and requires N_q == N_kv.
 *  Errors     Argument problems are reported by the return value BEFORE anything is launched;
 *             there is no fallback path (a silent fallback is the failure mode [Scratch] "How
 *             this shows up in practice" warns about).  Device-side bounded waits that run out
 *             are reported later by fa_sync_status.  fa_last_error_message() gives a one-line
 *             description of the last failure on the calling thread.
 *  Empty      N_kv == 0 gives O = 0 and lse = -inf; N_q == 0 does nothing
 *             ([Lesson4] section 3 "Compute it stably": an empty set has lse = -inf).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fa_bf16_t; /* raw bfloat16 bits */
typedef uint8_t fa_e4m3_t;  /* raw 8-bit float code: 1 sign, 4 exponent (bias 7), 3 mantissa bits */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, misaligned pointer, bad scale */
  FA_ERR_UNSUPPORTED = 2,    /* d not in {64,128}; causal with N_q != N_kv; size limits */
  FA_ERR_WORKSPACE = 3,      /* workspace pointer null or smaller than the *_workspace_size */
  FA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed (message has the detail) */
  FA_ERR_DEVICE_TIMEOUT = 5  /* a kernel's bounded wait ran out; its outputs are invalid */
} fa_status_t;

/*
 * fa_fwd -- attention forward pass.  [Lesson4] section 3 "The tiled forward pass" and
 * "The online softmax theorem"; [Scratch] "Online softmax: shrink the running total".
 *
 *   O   = softmax(scale * Q K^T (+ causal mask)) V         bf16 [B, H, N_q, d]
 *   lse = m + log(l) per query row (natural log)           fp32 [B, H, N_q]
 *
 * Tiles of 128 query rows stay on chip while 128-key tiles of K and V stream through shared
 * memory; the N_q x N_kv score matrix is never written to memory.
 * q: [B,H,N_q,d]; k, v: [B,H,N_kv,d]; o: [B,H,N_q,d] (written); lse: [B,H,N_q] (written).
 * scale must be finite and > 0 (normally 1/sqrt(d)).
 */
fa_status_t fa_fwd(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v, fa_bf16_t* o,
                   float* lse, int B, int H, int N_q, int N_kv, int d, float scale, int causal,
                   void* stream);

/*
 * fa_fwd_window / fa_bwd_window -- attention under a sliding window, forward and backward
 * ([Lesson4] section 6 "Where it shows up": long-context training uses causal and
 * sliding-window masks, both with tile skipping; section "Causal masks" for the skipping).
 *
 * Query i sees key j iff  i - window_left <= j <= i + window_right  over one sequence
 * (N_q = N_kv = N); a negative bound is unbounded on that side, so (-1, 0) is causal and
 * (-1, -1) is no mask.  Key tiles outside every row of a query tile's windows are never
 * loaded; tiles cut by a window edge are masked element by element.  Otherwise exactly
 * fa_fwd / fa_bwd (same layouts, workspace, errors).
 */
fa_status_t fa_fwd_window(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          fa_bf16_t* o, float* lse, int B, int H, int N, int d, float scale,
                          int window_left, int window_right, void* stream);
fa_status_t fa_bwd_window(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO,
                          fa_bf16_t* dq, fa_bf16_t* dk, fa_bf16_t* dv, void* ws, size_t ws_bytes,
                          int B, int H, int N, int d, float scale, int window_left,
                          int window_right, void* stream);

/*
 * fa_fwd_block_sparse / fa_bwd_block_sparse -- block-sparse attention, forward and backward
 * ([Scratch] "Results": the method's own block-sparse variant, the same IO-aware tiling applied
 * to a sparse pattern; the pages fix no pattern, so the pattern is the caller's).
 *
 * Blocks are 128 queries x 128 keys.  block_mask is a DEVICE array of bytes, nonzero = the
 * block is computed: [ceil(N_q/128)][ceil(N_kv/128)] shared by every head (mask_per_head = 0)
 * or [B*H][ceil(N_q/128)][ceil(N_kv/128)] (mask_per_head = 1), row-major, read during the
 * call in stream order; the caller owns it.  Query i sees key j iff the block (i/128, j/128)
 * is set and, with causal (N_q == N_kv), j <= i.  A row that sees no key gets O = 0 and
 * lse = -inf, and its gradients are 0.  Key blocks no row of a query tile pair sees are never
 * loaded; the backward visits, for each key block, only the query blocks set with it.
 * ceil(N_kv/128) <= 1024, else FA_ERR_UNSUPPORTED; mask_per_head not 0/1 or a null mask
 * (with N_q, N_kv > 0): FA_ERR_INVALID_ARG.  Otherwise exactly fa_fwd / fa_bwd (same layouts,
 * workspace, errors).
 */
fa_status_t fa_fwd_block_sparse(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                                fa_bf16_t* o, float* lse, int B, int H, int N_q, int N_kv, int d,
                                float scale, int causal, const unsigned char* block_mask,
                                int mask_per_head, void* stream);
fa_status_t fa_bwd_block_sparse(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                                const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO,
                                fa_bf16_t* dq, fa_bf16_t* dk, fa_bf16_t* dv, void* ws,
                                size_t ws_bytes, int B, int H, int N_q, int N_kv, int d,
                                float scale, int causal, const unsigned char* block_mask,
                                int mask_per_head, void* stream);

/*
 * fa_fwd_fp8 -- attention forward from 8-bit inputs (the low-precision FP8 path [Lesson4]
 * "Causal masks and FlashAttention-3" and [Scratch] "Later versions" name; the pages give no
 * formula, so this follows the plainest reading: one scale per tensor).
 *
 *   Q = descale_q * Q8, K = descale_k * K8, V = descale_v * V8   (Q8, K8, V8: e4m3 codes)
 *   O, lse = fa_fwd(Q, K, V) with the given scale                bf16 O, fp32 lse
 *
 * q, k, v: [B,H,N,d] e4m3 codes; o, lse as for fa_fwd.  d must be 128.  Scores accumulate in
 * fp32 from exact code products; the attention weights are rounded to e4m3 for the P V product
 * (the tensor core's 8-bit kind takes both operands in 8 bits), so O differs from the exact
 * result by at most 2^-4 * sum_j P_ij |V_j| (plus bf16 output rounding), and by much less on
 * average (the roundings are to nearest and independent); lse uses the unrounded weights.
 * scale, descale_* must be finite and > 0; other rules as for fa_fwd.
 */
fa_status_t fa_fwd_fp8(const fa_e4m3_t* q, const fa_e4m3_t* k, const fa_e4m3_t* v, fa_bf16_t* o,
                       float* lse, int B, int H, int N_q, int N_kv, int d, float scale,
                       float descale_q, float descale_k, float descale_v, int causal,
                       void* stream);

/*
 * fa_fwd_varlen -- attention forward over a batch of sequences of different lengths, packed
 * without padding (variable-length batches with cu_seqlens boundaries, as [Scratch] "How this
 * shows up in practice" describes; padding every sequence to the longest would pay for the
 * padded work).  Same computation as fa_fwd, per sequence.
 *
 *  q, o : [total_q, H, d] bf16, token-major (token t of all heads, then token t+1, ...)
 *  k, v : [total_k, H, d] bf16
 *  lse  : [H, total_q] fp32, natural log
 *  cu_seqlens_q, cu_seqlens_k : DEVICE int arrays of n_seqs + 1 entries; sequence s owns query
 *         rows [cu_q[s], cu_q[s+1]) and key rows [cu_k[s], cu_k[s+1]); non-decreasing, starting
 *         at 0 and ending at total_q / total_k.
 *  max_seqlen_q, max_seqlen_k : upper bounds on the per-sequence lengths (size the launch).
 *  causal : query i of a sequence sees that sequence's keys j <= i (positions within the
 *         sequence; meant for self-attention, where each sequence's two lengths are equal).
 * The kernels check every boundary they read; a boundary outside [0, total] or a length above
 * max_seqlen_q makes the affected work item write nothing and fa_sync_status report
 * FA_ERR_INVALID_ARG.  A sequence with no keys gets O = 0 and lse = -inf.
 */
fa_status_t fa_fwd_varlen(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          fa_bf16_t* o, float* lse, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, int n_seqs, int H, int total_q, int total_k,
                          int max_seqlen_q, int max_seqlen_k, int d, float scale, int causal,
                          void* stream);

/*
 * Workspace bytes fa_bwd needs: an fp32 dQ accumulator [B,H,N_q,d] plus fp32 D [B,H,N_q]
 * plus alignment padding.  Returns 0 for unsupported arguments.  Both arrays come from
 * [Lesson4] section 3 "Backward pass: recompute instead of store": step 3 forms
 * D_i = dO_i . O_i once per query row, and step 4's dQ_i += scale dS K_j adds one term per key
 * tile, which this library sums in fp32 across the CTAs of different key tiles.  N_kv does not
 * change the size; it is taken so the signature matches fa_bwd's.
 */
size_t fa_bwd_workspace_size(int B, int H, int N_q, int N_kv, int d);

/*
 * fa_bwd -- recompute-based backward pass.  [Lesson4] section 3 "Backward pass: recompute
 * instead of store", steps 1-4; [Scratch] "Recomputing on purpose in the backward pass".
 *
 *   D  = rowsum(dO o O)                     (pre-kernel, fp32, into the workspace)
 *   P  = exp(scale * Q K^T - lse)           (recomputed tile by tile, never stored)
 *   dV = P^T dO;  dP = dO V^T;  dS = P o (dP - D)
 *   dQ = scale * dS K;  dK = scale * dS^T Q
 *
 * o and lse must be the outputs of fa_fwd for the same q, k, v, scale and causal.
 * dq [B,H,N_q,d], dk and dv [B,H,N_kv,d] are written (not accumulated).  ``ws`` is a device
 * buffer of at least fa_bwd_workspace_size(...) bytes, 256-byte aligned; its contents on entry
 * are ignored and on exit are unspecified.  dQ is accumulated with fp32 atomics, so dq can
 * differ between runs in the last bits; dk and dv are deterministic.
 */
fa_status_t fa_bwd(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                   const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO, fa_bf16_t* dq,
                   fa_bf16_t* dk, fa_bf16_t* dv, void* ws, size_t ws_bytes, int B, int H,
                   int N_q, int N_kv, int d, float scale, int causal, void* stream);

/*
 * The three steps fa_bwd runs, in this order on one stream, exposed so a caller can schedule
 * or time them separately.  Arguments mean the same as in fa_bwd; the same ``ws`` must be
 * passed to all three, and only the arrays each step reads or writes are needed (others may
 * be NULL):
 *   fa_bwd_prep    D_i = sum_k dO_ik O_ik (fp32, into ws) and clears the fp32 dQ accumulator
 *                  ([Lesson4] "Backward pass", step 3: D_i = dO_i . O_i).  Reads o, dO.
 *   fa_bwd_main    recomputes S and P = exp(scale QK^T - lse) per 128-key tile, writes dK and
 *                  dV, and adds the tile's dS K (not yet multiplied by scale) into the fp32 dQ
 *                  accumulator (steps 1-4).
 *                  Reads q, k, v, lse, dO and D; writes dk, dv.
 *   fa_bwd_finish  dq = bf16(scale * accumulator).  Writes dq.
 */
fa_status_t fa_bwd_prep(const fa_bf16_t* o, const fa_bf16_t* dO, void* ws, size_t ws_bytes,
                        int B, int H, int N_q, int N_kv, int d, void* stream);
fa_status_t fa_bwd_main(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                        const float* lse, const fa_bf16_t* dO, fa_bf16_t* dk, fa_bf16_t* dv,
                        void* ws, size_t ws_bytes, int B, int H, int N_q, int N_kv, int d,
                        float scale, int causal, void* stream);
fa_status_t fa_bwd_finish(fa_bf16_t* dq, const void* ws, size_t ws_bytes, int B, int H, int N_q,
                          int N_kv, int d, float scale, void* stream);

/*
 * fa_bwd_varlen -- backward pass for fa_fwd_varlen: same computation as fa_bwd, per sequence,
 * on packed token-major tensors (q, o, dO, dq: [total_q, H, d]; k, v, dk, dv: [total_k, H, d];
 * lse: [H, total_q]) with the same device cu_seqlens arrays and bounds as the forward.  ``ws``
 * holds at least fa_bwd_workspace_size(1, H, total_q, total_k, d) bytes, 256-byte aligned.
 * Invalid boundaries are checked in the kernel and reported by fa_sync_status as for the
 * forward.  dq is accumulated with fp32 atomics (last-bit run-to-run differences).
 */
fa_status_t fa_bwd_varlen(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                          const fa_bf16_t* o, const float* lse, const fa_bf16_t* dO,
                          fa_bf16_t* dq, fa_bf16_t* dk, fa_bf16_t* dv, void* ws, size_t ws_bytes,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int n_seqs, int H,
                          int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                          float scale, int causal, void* stream);

/*
 * Workspace bytes fa_decode_splitkv needs for n_splits partial states per (b, h):
 * fp32 (m, l, o~[d]), the per-chunk state of [Lesson4] section 3 "Split-KV for decoding
 * (flash-decoding)" that the merge step combines.  n_splits <= 0 means "automatic" (as
 * fa_decode_splitkv chooses).  The call takes N_kv because the automatic split count depends on
 * it (at least ~256 keys per chunk); with an explicit n_splits N_kv does not change the size.
 * Returns 0 for unsupported arguments (including B*H*n_splits >= 2^31).
 */
size_t fa_decode_workspace_size(int B, int H, int N_kv, int d, int n_splits);

/*
 * fa_decode_splitkv -- single-query decode with the KV axis split into chunks
 * ([Lesson4] section 3 "Split-KV for decoding (flash-decoding)").
 *
 * Each (b, h, chunk) computes its online state (m, l, o~) over c consecutive keys, where
 * c = ceil(N_kv / n_splits) rounded up to a multiple of 64 (trailing chunks may be empty);
 * a second kernel merges the states of a row with
 *   m = max m_c,  l = sum e^{m_c - m} l_c,  O = sum e^{m_c - m} o~_c / l,  lse = m + log l
 * ([Lesson4] section 3 "Merging two partial results"; empty chunks weigh 0).
 *
 * q: [B,H,1,d]; k, v: [B,H,N_kv,d]; o: [B,H,1,d]; lse: [B,H,1].  n_splits in [1, 1024], or
 * <= 0 for automatic; B*H*n_splits < 2^31 (else FA_ERR_UNSUPPORTED).  ``ws`` holds at least
 * fa_decode_workspace_size(...) bytes, 16-byte aligned; contents on entry ignored.
 */
fa_status_t fa_decode_splitkv(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                              fa_bf16_t* o, float* lse, int B, int H, int N_kv, int d,
                              float scale, int n_splits, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * fa_decode_paged -- fa_decode_splitkv over a paged KV cache
 * ([Lesson4] section 3 "Split-KV for decoding (flash-decoding)"; the cache paging itself is a
 * serving-side layout the pages do not describe: the arithmetic is exactly that of
 * fa_decode_splitkv on each row's first seqlens_k[b] keys).
 *
 * Layout: k_cache, v_cache [num_blocks, block_size, H, d] bf16 (token-major inside a block);
 * block_table [B, max_blocks_per_seq] int32 on the device; seqlens_k [B] int32 on the device.
 * Logical key j (0 <= j < seqlens_k[b]) of batch b lives in cache block
 * block_table[b * max_blocks_per_seq + j / block_size] at row j % block_size.  Rows of a block
 * past a sequence's end are never read into the result (they may hold anything).
 * q: [B,H,1,d]; o: [B,H,1,d]; lse: [B,H,1].  A row with seqlens_k[b] == 0 gets O = 0 and
 * lse = -inf.
 *
 *  - block_size must be a positive multiple of 64; num_blocks * block_size < 2^31;
 *    max_seqlen_k <= max_blocks_per_seq * block_size (else FA_ERR_INVALID_ARG / UNSUPPORTED).
 *  - The chunks of the split are sized from max_seqlen_k, which must bound every seqlens_k[b].
 *  - Device-side checks: seqlens_k[b] outside [0, max_seqlen_k], or a block id outside
 *    [0, num_blocks) in the part of the table a row uses, is recorded (the kernel stays in
 *    bounds) and fa_sync_status then returns FA_ERR_INVALID_ARG; the outputs are undefined.
 *  - ws: at least fa_decode_workspace_size(B, H, max_seqlen_k, d, n_splits) bytes, 16-byte
 *    aligned.  n_splits as for fa_decode_splitkv.
 */
fa_status_t fa_decode_paged(const fa_bf16_t* q, const fa_bf16_t* k_cache,
                            const fa_bf16_t* v_cache, fa_bf16_t* o, float* lse,
                            const int* block_table, const int* seqlens_k, int B, int H,
                            int max_blocks_per_seq, int block_size, int num_blocks,
                            int max_seqlen_k, int d, float scale, int n_splits, void* ws,
                            size_t ws_bytes, void* stream);

/*
 * fa_decode_splitkv_noalloc -- fa_decode_splitkv for callers that cannot allocate device
 * memory (no counterpart in the pages; an interface convenience).
 *
 * Some callers have no way to hand the decode a workspace: a plugin inside a host process
 * whose memory manager owns all device memory, or a latency-critical serving loop that must
 * not call cudaMalloc (which can synchronise the device).  This entry point computes exactly
 * what fa_decode_splitkv computes, with the same kernels, but keeps the per-chunk states in a
 * fixed scratch array compiled into the library (FA_DECODE_NOALLOC_SCRATCH_BYTES of device
 * memory, held on every GPU that loads the library until the process exits).  It never calls
 * cudaMalloc, cudaFree or any allocating routine.
 *
 *  - Arguments are those of fa_decode_splitkv without ws/ws_bytes.
 *  - Limit: B * H * n_splits * (d + 2) * 4 bytes must not exceed the scratch size (for the
 *    automatic n_splits the library's choice is checked); larger calls return
 *    FA_ERR_UNSUPPORTED before anything is launched.
 *  - The first call on a device looks up the scratch's device address (cudaGetSymbolAddress)
 *    with that device current; make that first call before any stream capture.
 *    The address stays cached for the life of the process: after cudaDeviceReset the
 *    library's device image may be reloaded elsewhere, so do not use this entry point after
 *    resetting a device in the same process.
 *  - Every call shares the one array and leaves its contents behind.  Nothing in it needs to
 *    start at zero (each call writes every state it reads), but two calls whose kernels overlap
 *    on the GPU (different streams, or different host threads) race on it: serialise them.
 */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
fa_status_t fa_decode_splitkv_noalloc(const fa_bf16_t* q, const fa_bf16_t* k, const fa_bf16_t* v,
                                      fa_bf16_t* o, float* lse, int B, int H, int N_kv, int d,
                                      float scale, int n_splits, void* stream);

/*
 * fa_sync_status -- synchronise ``stream`` and report device-side failures recorded by any
 * kernel of this library since the last call (a bounded pipeline wait that ran out,
 * FA_ERR_DEVICE_TIMEOUT; a bad varlen boundary or paged-cache entry, FA_ERR_INVALID_ARG).
 * Clears the recorded state.  Also returns FA_ERR_CUDA if the stream reports an asynchronous
 * CUDA error.  This is how the library fails loudly rather than handing back wrong results
 * ([Scratch] "How this shows up in practice": a kernel that cannot do the job must say so,
 * never fall back silently); the pages define no such call, only the behaviour.
 */
fa_status_t fa_sync_status(void* stream);

/*
 * fa_selftest_wait_timeout -- diagnostic for the library's failure detection.  Enqueues one
 * tiny kernel that waits, with the bounded wait every pipeline here uses, on an mbarrier that
 * nothing ever arrives at; after ``limit_us`` microseconds it records a timeout and returns.
 * The following fa_sync_status(stream) then reports FA_ERR_DEVICE_TIMEOUT (and clears it), and
 * the CUDA context stays usable.  Failing loudly instead of hanging or silently producing
 * garbage is the behaviour [Scratch] "How this shows up in practice" asks for.  limit_us must
 * be in [1, 10^7]; otherwise FA_ERR_INVALID_ARG.
 */
fa_status_t fa_selftest_wait_timeout(unsigned int limit_us, void* stream);

/*
 * fa_debug_counters -- diagnostic counters of the tile skipping ([Lesson4] "Causal masks": the
 * kernel skips tiles above the diagonal and computes T(T+1)/2 of the T^2 tiles; the same
 * skipping serves sliding windows and block masks).
 *
 * device_counters: a DEVICE array of at least 2 unsigned 64-bit counters owned by the caller,
 * or NULL to turn counting off (the default).  While set (process-wide, for launches issued
 * after the call), every forward kernel adds to [0] the number of S = Q K^T tile products
 * (128-query tile x 128-key tile) it computed, and every backward main kernel adds to [1] the
 * number of (128-key tile, query step) pairs it visited (a query step is 64 queries at d = 128,
 * 128 at d = 64).  The caller zeroes the counters and reads them after synchronising.
 * Always FA_OK.
 */
fa_status_t fa_debug_counters(unsigned long long* device_counters);

/*
 * Static, human-readable name of a status code.  The pages have no counterpart; like
 * fa_last_error_message it serves the loud failure [Scratch] "How this shows up in practice"
 * asks for (an error the caller can print, not a silent fallback).
 */
const char* fa_status_string(fa_status_t status);

/* One-line description of the last non-OK status returned on the calling thread. */
const char* fa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
