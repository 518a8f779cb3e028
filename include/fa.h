/*
 * fa.h -- C ABI of the exact IO-aware attention library (libfa.so).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T  [+ causal mask]) V
 *
 * on one GB300 GPU (sm_103a) without ever writing the N x N scores S or the
 * probabilities P to device memory: query tiles stay on chip while key/value
 * tiles stream past, and an online softmax carries a running maximum m, a
 * denominator l and an unnormalised numerator per query row. Sources:
 *   "Flash Attention: IO-Aware Exact Attention", sections "Why intermediate
 *   matrices cost memory traffic" (the problem: Q, K, V in, O out),
 *   "Online softmax makes tiling exact" (the recurrence) and "Loop order
 *   changes which data is reloaded" (queries resident, keys/values
 *   streamed); "FlashAttention -- the same attention, made memory-aware",
 *   section 00 (scale 1/sqrt(d), causal mask, [B, heads, T, head size]
 *   layout); "FlashAttention" (Road to Intelligence), section "The
 *   solution" (the backward recomputes scores instead of storing them).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers owned by the caller. The
 *    library keeps no allocation of its own between calls.
 *  - q, k, v, o, dO, dq, dk, dv: bfloat16, shape [B, H, N, d], contiguous
 *    row-major (d fastest). lse and the backward's D: float32 [B, H, N].
 *  - d must be 64 or 128; the forward forms (fa_fwd, fa_fwd_ex,
 *    fa_decode_splitkv) also take d = 256 (with d_v = 256). N may be any
 *    length (ragged tail tiles are masked). Keys and queries have the same length N, except in
 *    fa_fwd_ex and fa_decode_splitkv, which take Nq queries over Nk keys.
 *  - causal != 0 masks key j for query i when j > i (the diagonal is
 *    visible). scale multiplies Q K^T before masking and softmax; it must be
 *    finite and >= 0 (0 gives uniform weights over the visible keys).
 *  - lse[b,h,i] = m_i + ln(l_i): the natural-log log-sum-exp of row i of the
 *    scaled, masked scores (the normalisation statistic the backward needs).
 *  - B, H or N equal to 0 is an empty problem: the call returns FA_OK and
 *    touches nothing (pointers may then be NULL). Negative sizes, NULL
 *    pointers or pointers that are not 16-byte aligned return
 *    FA_ERR_INVALID before anything is launched.
 *  - Calls are asynchronous on the given stream (stream 0 for the forms
 *    without a stream argument); argument checks are synchronous. Outputs
 *    must not alias inputs.
 *  - Each wait inside the kernels is bounded (about one second). A wait that
 *    runs out makes the kernel wind down and raise a device status word that
 *    fa_get_last_device_status() reads (FA_ERR_TIMEOUT); no kernel traps.
 *  - Thread safety: calls from several host threads are safe; the device
 *    status word is shared by all calls on a device.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define FA_OK 0
#define FA_ERR_INVALID -1      /* bad pointer, size, alignment or scale      */
#define FA_ERR_UNSUPPORTED -2  /* head size not supported by the call, or not a CC 10.3 device */
#define FA_ERR_LAUNCH -3       /* a CUDA call failed (launch, attribute, map) */
#define FA_ERR_TIMEOUT -4      /* a bounded wait in a kernel ran out          */
#define FA_ERR_WORKSPACE -5    /* workspace missing or too small              */

/*
 * Forward pass.
 *   q, k, v : in,  bf16 [B,H,N,d]
 *   o       : out, bf16 [B,H,N,d]   O = softmax(scale*QK^T [+mask]) V
 *   lse     : out, fp32 [B,H,N]     per-row log-sum-exp (natural log)
 * Sources: "Flash Attention: IO-Aware Exact Attention", sections "Online
 * softmax makes tiling exact" and "Check the recurrence on CPU" (the
 * recurrence and its final division, one per row); "Storage, arithmetic and
 * IO are separate quantities" (only the output and per-row statistics are
 * kept for the backward).
 * Runs on stream 0.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, int causal, float scale);

/* fa_fwd on `cuda_stream` (a cudaStream_t; NULL is the legacy stream). */
int fa_fwd_stream(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int N, int d, int causal, float scale, void* cuda_stream);

/*
 * Backward pass by recomputation.
 *   q, k, v, o : in,  bf16 [B,H,N,d]  (o: the forward's output)
 *   lse        : in,  fp32 [B,H,N]    (the forward's log-sum-exp)
 *   dO         : in,  bf16 [B,H,N,d]  gradient of the loss w.r.t. O
 *   dq, dk, dv : out, bf16 [B,H,N,d]  gradients w.r.t. Q, K, V
 * Computes, with P = exp(scale*QK^T [masked] - lse) recomputed tile by tile:
 *   dV = P^T dO, dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D),
 *   dQ = scale * dS K, dK = scale * dS^T Q.
 * Source: "FlashAttention" (Road to Intelligence), sections "The solution"
 * and "What to remember" (scores recomputed from Q, K, V rather than
 * stored); the gradient formulas follow from the forward's definition.
 * d must be 64 or 128 (d = 256, which the forward takes, returns
 * FA_ERR_UNSUPPORTED here and in every backward form: its five tensor-memory
 * accumulators would not fit).
 * This form allocates its float32 workspace (fa_bwd_workspace_bytes) with
 * cudaMallocAsync on stream 0 and frees it stream-ordered after the call.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
           float scale);

/*
 * fa_bwd on `cuda_stream` with a caller-provided device workspace of at
 * least fa_bwd_workspace_bytes(B,H,N,d) bytes, 256-byte aligned. The
 * workspace holds D = rowsum(dO * O) and the LSE in log2 units (fp32, each
 * over N rounded up to 128 per head) and the fp32 dQ accumulator (the same
 * padded rows x d, in a blocked layout of the library's choosing); its
 * contents on entry do not matter and on return are unspecified. Two calls
 * in flight at once need two workspaces.
 */
int fa_bwd_stream(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, float scale, void* workspace, size_t ws_bytes, void* cuda_stream);

/*
 * The backward's three stages, for callers that schedule or time them one
 * by one. fa_bwd_stream is exactly these three calls, in this order, on one
 * stream with one workspace; each checks its arguments like fa_bwd_stream.
 *   preprocess: D = rowsum(dO * O) and LSE in log2 units into the
 *               workspace; zeroes the workspace's fp32 dQ accumulator.
 *   main:       per block of 128 keys, recomputes the score and probability
 *               tiles of every query block and accumulates dK, dV (written
 *               to dk, dv) and dQ (added into the workspace).
 *   finish:     dq = bf16(workspace dQ accumulator).
 */
int fa_bwd_preprocess_stream(const void* o, const float* lse, const void* dO, int B, int H,
                             int N, int d, void* workspace, size_t ws_bytes, void* cuda_stream);
int fa_bwd_main_stream(const void* q, const void* k, const void* v, const void* dO, void* dk,
                       void* dv, int B, int H, int N, int d, int causal, float scale,
                       void* workspace, size_t ws_bytes, void* cuda_stream);
int fa_bwd_finish_stream(void* dq, int B, int H, int N, int d, const void* workspace,
                         size_t ws_bytes, void* cuda_stream);

/*
 * fa_bwd_noalloc: fa_bwd_stream without a caller workspace and without
 * allocating anything. The pages have no counterpart to this entry point; it
 * exists for callers that cannot allocate device memory: a host framework
 * that owns every device allocation and forbids libraries to allocate, or a
 * serving loop with a fixed memory budget that must not call cudaMalloc on
 * its hot path (the call can synchronise the device and can fail once memory
 * is fragmented).
 * The workspace is a file-scope device array of
 * FA_BWD_NOALLOC_MAX_SCRATCH_BYTES bytes inside the library. Problems whose
 * fa_bwd_workspace_bytes exceed it return FA_ERR_WORKSPACE and launch
 * nothing. The first call on a device looks up the array's device address;
 * with lazy module loading (the CUDA default) that lookup is also what loads
 * the library's device code holding the array onto that device and reserves
 * the 64 MiB there, until the process exits. That first call can therefore
 * fail with FA_ERR_LAUNCH when the device is out of memory, and must not run
 * inside a stream capture: make it during set-up, on every device the caller
 * will use. Later calls on the device allocate and load nothing. All calls
 * share the array: calls whose kernels overlap on the GPU (other streams,
 * other host threads) race and corrupt each other's results, so serialise
 * them on one stream. Arguments and results are those of fa_bwd_stream.
 */
#define FA_BWD_NOALLOC_MAX_SCRATCH_BYTES ((size_t)64 << 20)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, void* cuda_stream);

/* Workspace bytes fa_bwd_stream needs for these sizes (0 when empty). */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Extended forward: Nq queries over Nk keys, head sizes d (queries, keys)
 * and dv (values, output), optional sliding window.
 *   q       : in,  bf16 [B,H,Nq,d]
 *   k       : in,  bf16 [B,H,Nk,d]   (e.g. a key/value cache)
 *   v       : in,  bf16 [B,H,Nk,dv]
 *   o       : out, bf16 [B,H,Nq,dv]
 *   lse     : out, fp32 [B,H,Nq]     natural-log log-sum-exp of each row
 * d and dv are each 64 or 128, or both 256 (FA_ERR_UNSUPPORTED otherwise);
 * the pages count the forward's work as O(N^2 (d + d_v)) ("Flash Attention:
 * IO-Aware Exact Attention", section "Storage, arithmetic and IO are
 * separate quantities"), with d_v = d as the square special case.
 * With causal != 0 the queries are the last Nq positions of the Nk keys:
 * query i sits at position p = i + Nk - Nq and sees keys j <= p (Nq <= Nk
 * required). window = W >= 1 (causal only) further keeps only the keys
 * p - W < j <= p; window = 0 means no window. Key tiles wholly outside a
 * query tile's range are neither loaded nor multiplied.
 * Sources: "Flash Attention: IO-Aware Exact Attention", section "What
 * changes in FlashAttention-2" (KV caching for decode-time history;
 * sliding-window attention changes which historical keys participate);
 * "FlashAttention -- the same attention, made memory-aware", section 00
 * (the causal mask).
 * Errors as fa_fwd; additionally FA_ERR_INVALID for window < 0, a window
 * without causal, Nk = 0 with Nq > 0, or causal with Nq > Nk.
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, int dv, int causal, int window, float scale,
              void* cuda_stream);

/*
 * Backward of fa_fwd_ex for training (Nq = Nk = N) with head sizes d (q, k,
 * dq, dk: [B,H,N,d]) and d_v (v, o, dO, dv: [B,H,N,d_v]), each 64 or 128,
 * and an optional causal sliding window of `window` keys (0 = none);
 * workspace (fa_bwd_workspace_bytes(B,H,N,d)) and results as
 * fa_bwd_stream. Key/value blocks skip the query blocks that see none of
 * their keys, and the boundary blocks are masked per element.
 * FA_ERR_INVALID for window < 0 or a window without causal.
 */
int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
              int d_v, int causal, int window, float scale, void* workspace, size_t ws_bytes,
              void* cuda_stream);

/*
 * Split-key-range forward for decode (few queries over a long key/value
 * cache): the keys are cut into n_splits contiguous ranges of whole 128-key
 * tiles, each (range, batch-head) is reduced by its own CTA to a partial
 * state (fp32 output normalised within the range, and its LSE), and a second
 * kernel merges the parts with the rule of "FlashAttention -- the same
 * attention, made memory-aware", section 03 (rescale each part by
 * exp(m_part - m_new) and sum): LSE = log sum_s exp(LSE_s),
 * O = sum_s exp(LSE_s - LSE) O_s. Arguments and masks as fa_fwd_ex.
 *   n_splits  : requested number of ranges; <= 0 chooses one from the
 *               problem size and the device's SM count; clamped to the
 *               number of key tiles (fa_decode_num_splits gives the count
 *               actually used).
 *   workspace : device memory of at least fa_decode_workspace_bytes(...)
 *               bytes, 256-byte aligned, owned by the caller (partial
 *               outputs [splits,B,H,Nq,dv] fp32 then partial LSE
 *               [splits,B,H,Nq] fp32); FA_ERR_WORKSPACE otherwise.
 */
int fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, int dv, int causal, int window, float scale,
                      int n_splits, void* workspace, size_t ws_bytes, void* cuda_stream);
int fa_decode_num_splits(int B, int H, int Nq, int Nk, int n_splits);
size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int dv, int n_splits);

/*
 * Forward and backward with dropout on the attention probabilities. The
 * pages name dropout only as a setting to hold equal between implementations
 * ("Flash Attention: IO-Aware Exact Attention", section "What changes in
 * FlashAttention-2"); the form here is inverted dropout on P:
 *     O = (P * M) V / keep,   LSE as without dropout (the softmax statistic)
 * and the backward is the exact gradient of that O for the same mask M:
 *     dV = (P*M/keep)^T dO, dP = (dO V^T) * M / keep, dS = P * (dP - D),
 *     D = rowsum(dO * O), dQ = scale dS K, dK = scale dS^T Q.
 *   dropout_p : 0 <= p < 1 (else FA_ERR_INVALID), applied as the byte
 *               threshold t = round(256 p) (at most 255): an element is kept
 *               when its generator byte is >= t, so keep = (256 - t) / 256
 *               and p = 0 is exactly attention without dropout.
 *   seed, offset : the mask of batch-head bh, query i, key j is byte (j & 3)
 *               of word (i & 3) of Philox4x32-10 (Salmon, Moraes, Dror and
 *               Shaw, SC 2011) with counter (j >> 2, i >> 2, bh,
 *               offset mod 2^32) and key (seed mod 2^32, seed >> 32). The
 *               backward must get the forward's seed and offset; a new
 *               offset per call gives a new mask.
 * d must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise); other arguments,
 * layouts, the workspace and errors as fa_fwd_stream and fa_bwd_stream.
 */
int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, int causal, float scale, float dropout_p, unsigned long long seed,
                   unsigned long long offset, void* cuda_stream);
int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, float dropout_p, unsigned long long seed,
                   unsigned long long offset, void* workspace, size_t ws_bytes,
                   void* cuda_stream);

/* Static description of a return code. Never NULL. */
const char* fa_strerror(int code);

/*
 * Device status word of the current device: FA_OK, or FA_ERR_TIMEOUT when a
 * kernel launched since the last read gave up on a bounded wait. Reading
 * synchronises the device and clears the word. Returns FA_ERR_LAUNCH if the
 * word cannot be read.
 */
int fa_get_last_device_status(void);

/* Library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
