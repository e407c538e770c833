/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward library
 * (libattn_gb300.so).
 *
 * The operation is the fused scaled-dot-product attention forward pass,
 * "Fused attention kernel" (wikillm concept card), Overview and
 * Implementation sketch:
 *
 *     S = scale * Q K^T            (per batch entry / sequence and head)
 *     P = softmax(S) row by row    (causal: query i sees keys j <= i)
 *     O = P V,   lse_i = log sum_j exp(S_ij)   (natural log)
 *
 * computed tile by tile with a running row maximum and row sum so that S and
 * P never leave the chip.  The 8-bit variant and its pre-step follow the same
 * card's section "8-bit forward pass (FP8, Hopper)": e4m3 operands, one scale
 * per block of Q, K and V, and Q, K rotated by a random-sign diagonal times a
 * Hadamard matrix ("incoherent processing").
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer owned by the caller, except
 *    where stated.  Buffers must not overlap.  Tensor pointers must be 16-byte
 *    aligned (they are read and written by the Tensor Memory Accelerator).
 *  - Layouts are row-major and contiguous:
 *        dense  Q, K, V, O : [B, N, H, d]  (token-major, head dim innermost)
 *        dense  lse        : [B, H, N] float32
 *        varlen Q, K, V, O : [T, H, d]     (sequences packed back to back)
 *        varlen lse        : [H, T] float32
 *  - Supported head dimensions: d = 64 and d = 128 (attn_bwd: d = 128 only;
 *    other values return ATTN_ERR_UNSUPPORTED).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call is asynchronous on that stream; the return value reports
 *    argument validation and launch errors only.  Errors detected on the
 *    device (a pipeline wait that timed out, malformed cu_seqlens) are
 *    recorded in a device status word read by attn_get_status().
 *  - No call throws, prints, or synchronises (except attn_get_status).
 *  - The library keeps a per-device workspace (status word, varlen tile
 *    list, split partials, backward accumulators), allocated on first use,
 *    grown when a larger problem needs it and released by attn_shutdown().
 *    Calls that share a device must be issued from one host thread at a time
 *    or be serialised by the caller, and calls that use the same workspace
 *    must not run at the same time on different streams.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, non-finite scale */
    ATTN_ERR_UNSUPPORTED = 2,   /* head dimension or dtype this build does not provide */
    ATTN_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned */
    ATTN_ERR_LAUNCH = 4,        /* the kernel launch failed */
    ATTN_ERR_TIMEOUT = 5,       /* device: a pipeline wait exceeded its budget */
    ATTN_ERR_BAD_SEQLENS = 6,   /* device: cu_seqlens not non-decreasing from 0 or over total */
    ATTN_ERR_CUDA = 7,          /* a CUDA runtime call failed (no device, out of memory) */
    ATTN_ERR_TOO_LARGE = 8      /* a size exceeds the library's index range */
} attn_status_t;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype_t;

/*
 * Dense attention forward, 16-bit inputs.
 *   q, k, v : [B, N, H, d] in `dtype`;  o : [B, N, H, d] in `dtype`;
 *   lse     : [B, H, N] float32 (may be NULL: not written).
 *   scale   : multiplies Q K^T (normally 1/sqrt(d)); must be finite.
 *   causal  : nonzero = query i attends to keys 0..i of its own sequence.
 * The result matches exact attention; S and P stay on chip.
 * Non-causal shapes whose last wave of 256-row work tiles would fill at most
 * half of the SMs run those last tiles as two key halves, each writing
 * O / l and lse in fp32 to the per-device workspace, and a second kernel
 * merges them (lse = log(e^lse0 + e^lse1), O = sum_i e^(lse_i - lse) O_i).
 * The same holds for attn_fwd_gqa, attn_fwd_bias and attn_fwd_fp8.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int H, int N, int d, float scale, int causal,
                       attn_dtype_t dtype, void *stream);

/*
 * attn_fwd with HOST buffers: the same dense forward for data that lives in
 * host memory (q, k, v, o, lse as in attn_fwd, but host pointers; H_kv = H).
 * The library moves the work in chunks -- whole batch entries, and for the
 * first and the last entry groups of heads (the fewest heads whose work
 * tiles still fill every SM once) -- copying one chunk in while earlier
 * chunks are computed and copied back: three device staging sets in the
 * per-device workspace, internal copy-in, copy-out and second compute
 * streams, and events.  The compute runs on `stream` and the second compute
 * stream in turn, without the split last wave (each tile computed whole),
 * and `stream` waits for the last copy back, so later work on it sees the
 * outputs; the host buffers must stay valid until then.  Use page-locked
 * host memory (cudaHostAlloc or cudaHostRegister): copies from pageable
 * memory are correct but do not overlap.  Errors as attn_fwd, plus
 * ATTN_ERR_CUDA when a copy or event call fails.
 */
attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int N, int d, float scale, int causal,
                            attn_dtype_t dtype, void *stream);


/*
 * Dense attention forward with grouped K/V heads (grouped-query attention;
 * H_kv = 1 is multi-query attention).  The pages name serving LLMs as the
 * open target ("optimizing for LLM inference", FlashAttention-3 summary,
 * arxivlens, Limitations); they do not define the grouping, so this library
 * takes the usual one: query head h attends with K/V head h / (H / H_kv).
 *   q, o : [B, N, H, d];  k, v : [B, N, H_kv, d];  lse : [B, H, N] float32
 *   H_kv : >= 1 and dividing H (else ATTN_ERR_INVALID_ARG).
 * Everything else as attn_fwd, which is this call with H_kv = H.
 */
attn_status_t attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int H_kv, int N, int d, float scale, int causal,
                           attn_dtype_t dtype, void *stream);

/*
 * Dense attention forward with an additive score bias (the "[+mask]" of the
 * problem; "Bias" among the additions of the HippoAttention case study,
 * streamhpc.com, "Our approach"):
 *     S_ij = scale * q_i . k_j + bias[b * sb + h * sh + i * sr + j]
 * in natural-log units, before the softmax; -inf removes a key (a row with
 * every allowed key removed gets O = 0, lse = -inf).
 *   bias : DEVICE float32, keys contiguous; strides sb (batch), sh (head),
 *          sr (query row) in elements, each >= 0 (0 broadcasts: [1, H, N, N],
 *          [B, 1, 1, N] key masks, ...).  The bias pointer must be 16-byte
 *          aligned and every stride a multiple of 4 (ATTN_ERR_MISALIGNED).
 *   Grouped K/V heads as attn_fwd_gqa (H_kv = H for plain attention).
 *   Other arguments and layouts as attn_fwd.  The bias is read once per
 *   (query row, key) pair it applies to, so a full [B, H, N, N] bias makes
 *   the call bound by its bytes.
 */
attn_status_t attn_fwd_bias(const void *q, const void *k, const void *v, const float *bias,
                            long long bias_stride_b, long long bias_stride_h,
                            long long bias_stride_row, void *o, float *lse, int B, int H,
                            int H_kv, int N, int d, float scale, int causal, attn_dtype_t dtype,
                            void *stream);

/*
 * Packed variable-length attention forward ("Varlen", named among the
 * features of the HippoAttention case study, streamhpc.com).
 *   cu_seqlens   : DEVICE int32 [nseq + 1]; sequence s occupies tokens
 *                  cu_seqlens[s] .. cu_seqlens[s+1]-1; cu_seqlens[0] = 0,
 *                  non-decreasing, cu_seqlens[nseq] = total_tokens.
 *   total_tokens : T, the packed length (host value).
 *   max_seqlen   : an upper bound on every sequence length (host value).
 *   q, k, v, o   : [T, H, d];  lse : [H, T] float32 (may be NULL).
 * Attention never crosses a sequence boundary.  A violated cu_seqlens
 * contract is reported as ATTN_ERR_BAD_SEQLENS by attn_get_status() and the
 * outputs are then unspecified.
 */
attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int nseq, int total_tokens,
                              int max_seqlen, int H, int d, float scale, int causal,
                              attn_dtype_t dtype, void *stream);

/*
 * attn_fwd_varlen with grouped K/V heads (see attn_fwd_gqa):
 *   q, o : [T, H, d];  k, v : [T, H_kv, d];  lse : [H, T] float32.
 */
attn_status_t attn_fwd_varlen_gqa(const void *q, const void *k, const void *v, void *o,
                                  float *lse, const int32_t *cu_seqlens, int nseq,
                                  int total_tokens, int max_seqlen, int H, int H_kv, int d,
                                  float scale, int causal, attn_dtype_t dtype, void *stream);

/*
 * attn_fwd_varlen without any device allocation.  (The paper has no
 * counterpart: this is a calling convention of this library, not a step of
 * the method.)
 *
 * Same operation, arguments and result as attn_fwd_varlen, for callers that
 * cannot allocate device memory -- a plugin or custom op whose device memory
 * is planned by a host framework or inference runtime, or a service that
 * forbids allocation after start-up.  attn_fwd_varlen calls cudaMalloc on
 * first use and cudaFree when its tile list must grow; this call never
 * allocates or frees.  Its scratch (status word, tile list) is one
 * file-scope device array of 256 + 8 * 32768 bytes (about 256 KiB) that
 * every GPU loading the library holds until the process exits.
 *   status : DEVICE int32 (may be NULL).  Set to 0 on `stream` at the start
 *            of the call; a device-detected error (ATTN_ERR_BAD_SEQLENS,
 *            ATTN_ERR_TIMEOUT) is then written there.  With NULL such errors
 *            are not reported.  attn_get_status() does not see this call.
 * Limits: total_tokens / 256 + nseq must not exceed 32768 (the tile list's
 * capacity); larger problems are rejected with ATTN_ERR_TOO_LARGE before any
 * device work.
 * Set-up: the first call on each device looks up the device address of the
 * scratch array and the SM count, with that device current (no allocation).
 * Make that first call before any stream capture.
 * Sharing: every call on a device uses the same scratch, which keeps the
 * last call's contents.  Calls that overlap on the GPU (on different streams,
 * or from different host threads) race on it: serialise them.
 */
attn_status_t attn_fwd_varlen_noalloc(const void *q, const void *k, const void *v, void *o,
                                      float *lse, const int32_t *cu_seqlens, int nseq,
                                      int total_tokens, int max_seqlen, int H, int d,
                                      float scale, int causal, attn_dtype_t dtype,
                                      int32_t *status, void *stream);

/*
 * Attention of the newest Nq queries of each sequence against a paged K/V
 * cache, split over key ranges ("Paged Attention", named among the additions
 * of the HippoAttention case study, streamhpc.com, "Our approach"; the
 * FlashAttention-3 summary, arxivlens, Limitations, names LLM inference as
 * the open target).  Exact attention as in attn_fwd, with grouped K/V heads
 * (query head h uses K/V head h / (H / H_kv)).
 *   q            : [B, Nq, H, d];  o : [B, Nq, H, d] (same dtype);
 *   lse          : [B, H, Nq] float32 (may be NULL).
 *   k_cache,
 *   v_cache      : [num_pages, page_size, H_kv, d].  Key position t of
 *                  sequence b is row t % page_size of page
 *                  block_table[b * max_pages + t / page_size].
 *   block_table  : DEVICE int32 [B, max_pages]; entries past a sequence's
 *                  last page are not read.  Every entry that is read must lie
 *                  in [0, num_pages): the library does not check the table.
 *   seqlens_k    : DEVICE int32 [B]; 0 <= seqlens_k[b] <= max_seqlen_k <=
 *                  max_pages * page_size.
 *   causal       : the Nq queries are the last Nq positions of the sequence:
 *                  query i sees keys j <= seqlens_k[b] - Nq + i (a query that
 *                  sees no key gets O = 0 and lse = -inf).
 *   num_splits   : key ranges per (sequence, K/V head) computed by separate
 *                  CTAs and merged (O = sum_s exp(lse_s - lse) O_s); 0 = chosen
 *                  from the problem size.  The partial results live in a
 *                  per-device workspace the library allocates on first use
 *                  and grows when needed.
 * Limits: d = 64 or 128; (H / H_kv) * Nq <= 16 (ATTN_ERR_UNSUPPORTED
 * otherwise); any page_size >= 1.  Page sizes that split into pieces of 16,
 * 32 or 64 rows are loaded by tensor copies whose waits are bounded: a wait
 * past its budget records ATTN_ERR_TIMEOUT in the status word
 * (attn_get_status) and the output is then undefined.
 */
attn_status_t attn_fwd_paged(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_table, const int32_t *seqlens_k, void *o,
                             float *lse, int B, int Nq, int H, int H_kv, int d, int page_size,
                             int max_pages, int num_pages, int max_seqlen_k, float scale,
                             int causal, attn_dtype_t dtype, int num_splits, void *stream);

/*
 * 8-bit attention forward (e4m3 operands, block scales).
 *   q8, k8, v8 : [B, N, H, d] e4m3 codes (uint8 storage), as produced by
 *                qkv_block_quant_hadamard (Q and K possibly rotated: the
 *                rotation cancels in Q K^T).
 *   descale_q/k/v : float32 [B, H, ceil(N/128)]; block j of (b, h) covers
 *                tokens 128j .. 128j+127 and dequantises as code * descale.
 *                Every descale must be finite and positive (the quantiser
 *                below writes 1 for an all-zero block); other values give
 *                undefined output.
 *   o   : [B, N, H, d] bf16;  lse : [B, H, N] float32 (may be NULL).
 *   d   : 128, or 64: a 64-byte row is copied into a 128-byte swizzle row
 *         whose upper half the copy fills with zeros, so d = 64 runs the
 *         d = 128 kernel (twice the tensor work per useful flop).
 * V is consumed in its stored [token, d] layout (no transpose in memory).
 */
attn_status_t attn_fwd_fp8(const void *q8, const void *k8, const void *v8,
                           const float *descale_q, const float *descale_k,
                           const float *descale_v, void *o, float *lse,
                           int B, int H, int N, int d, float scale, int causal,
                           void *stream);

/*
 * fp8 pre-step: incoherent processing and block quantisation.
 *   q, k, v    : [B, N, H, d] bf16 inputs.
 *   signs      : DEVICE int8 [d] of +1/-1 (the random sign diagonal D), or
 *                NULL for no rotation.  Q and K are replaced by
 *                x * D * H_d / sqrt(d) (H_d: Sylvester Hadamard matrix); V is
 *                not rotated.
 *   per_tensor : 0 = one scale per 128-token block of each (b, h);
 *                1 = one scale per tensor (the baseline the block scheme is
 *                compared against).
 *   outputs    : q8, k8, v8 [B, N, H, d] e4m3; descale_q/k/v [B, H, ceil(N/128)]
 *                float32 with scale = amax|x| / 448 (1 for an all-zero block),
 *                codes = round-to-nearest-even(x * (1 / scale)) with x, the
 *                rotation and the product in float32, saturated to +-448.
 *                This can differ by one e4m3 step from RNE(x / scale) where
 *                x / scale lies within a few float32 ulps of a midpoint
 *                between two codes.
 */
attn_status_t qkv_block_quant_hadamard(const void *q, const void *k, const void *v,
                                       void *q8, void *k8, void *v8,
                                       float *descale_q, float *descale_k, float *descale_v,
                                       const int8_t *signs, int per_tensor,
                                       int B, int H, int N, int d, void *stream);

/*
 * The 8-bit path on HOST buffers: qkv_block_quant_hadamard (block scales,
 * per_tensor = 0) and attn_fwd_fp8 for data that lives in host memory.
 *   q, k, v : HOST [B, N, H, d] bf16;  o : HOST [B, N, H, d] bf16;
 *   lse     : HOST [B, H, N] float32 (may be NULL).
 *   signs   : HOST int8 [d] of +1/-1 (the random sign diagonal), or NULL for
 *             no rotation; copied to the device by the call (page-locked, like
 *             the other host buffers, so that the call does not wait for
 *             earlier work on the copy stream).
 * The work moves in the chunks of attn_fwd_host (batch entries, and head
 * groups of the first and last entry): each chunk is copied in, quantised
 * with one scale per 128-token block of each (b, h) -- so the codes and
 * scales equal those of the whole tensor -- computed by the e4m3 kernel
 * with its last wave whole, and copied out, overlapped with the other
 * chunks' copies and compute.  Staging (bf16 inputs, codes, scales,
 * outputs) lives in the per-device workspace.  Stream order, page-locked
 * memory and errors as attn_fwd_host; d = 64 or 128.
 */
attn_status_t attn_fwd_fp8_host(const void *q, const void *k, const void *v,
                                const int8_t *signs, void *o, float *lse, int B, int H, int N,
                                int d, float scale, int causal, void *stream);

/*
 * Backward pass: gradients of the dense forward (attn_fwd / attn_fwd_gqa)
 * with respect to Q, K and V, given the upstream gradient dO (the backward
 * pass of the FlashAttention-3 summary, arxivlens, Key Results; "backward
 * pass needed" in the "Fused attention kernel" card, "When to use which").
 * With P the forward's softmax (recomputed from its lse) and
 * D_i = rowsum(dO_i * O_i):
 *     dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q
 * grouped K/V heads sum dK and dV over their query heads.
 *   q, o, dout, dq : [B, N, H, d];  k, v, dk, dv : [B, N, H_kv, d]
 *   lse            : [B, H, N] float32, as the forward wrote it.
 *   d = 128 only (other values: ATTN_ERR_UNSUPPORTED).
 * The library keeps an fp32 dQ accumulator and the D vector in a per-device
 * workspace it allocates on first use and grows when needed.
 */
attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                       int H, int H_kv, int N, int d, float scale, int causal,
                       attn_dtype_t dtype, void *stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device (ATTN_OK if no device-side error was recorded since the
 * last call).  Returns ATTN_ERR_CUDA if the synchronisation itself failed.
 */
attn_status_t attn_get_status(void *stream);

/* Static, human-readable name of a status code. */
const char *attn_status_string(attn_status_t status);

/* Releases the per-device workspaces.  Safe to call more than once. */
void attn_shutdown(void);

/* Library ABI version: 0x00MMmmpp. */
uint32_t attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
