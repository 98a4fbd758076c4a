/*
 * fa.h -- C ABI of the exact, IO-aware scaled-dot-product attention library
 * for NVIDIA GB300 (sm_103a).
 *
 * What it computes. For every batch b and head h, with q, k, v the [N, d]
 * slices of that head,
 *     O = softmax(scale * q k^T [+ causal mask]) v
 * exactly, not an approximation: the pages this follows state that the tiled
 * method returns softmax(QK^T)V itself, differing from a whole-matrix
 * computation only by floating-point rounding
 * ("FlashAttention does more arithmetic to move less data", section
 * "FlashAttention never writes the full score table to HBM";
 * "FlashAttention and GPU Memory", chapters 01, 08 and 12). The N x N score
 * matrix never reaches device memory: score tiles live in on-chip tensor
 * memory (chapter 07, "Blocks").
 *
 * The forward pass also returns one number per row, the natural-log
 * logsumexp of the scaled, masked scores, which folds the running maximum m
 * and running sum l that the method keeps per row (chapter 08, "A softmax with
 * a running tally"; chapter 09 keeps those two values for each row). The backward
 * pass rebuilds score tiles from q, k, v and that logsumexp instead of
 * reading a stored probability matrix (chapter 09, "Backward: recomputing
 * beats reading").
 *
 * Conventions shared by every call:
 *   - q, k, v, o, dO, dq, dk, dv: bf16, contiguous [B, H, N, d], d innermost.
 *   - lse: fp32, contiguous [B, H, N].
 *   - Self-attention: queries and keys have the same length N, except in
 *     fa_fwd_kv (Nq query rows against Nk keys).
 *   - causal != 0 masks key j for query i when j > i (row 0 sees key 0 only);
 *     with Nq != Nk the queries are the last Nq positions: key j is masked
 *     for query i when j > i + Nk - Nq.
 *   - d must be 64 or 128. B, H, N >= 1, B * H * N * d < 2^31.
 *   - scale must be finite and > 0 (usually 1 / sqrt(d)).
 *   - Every pointer is a DEVICE pointer (the current CUDA device), 16-byte
 *     aligned. The caller owns all memory; the library allocates no device
 *     memory. Buffers must not overlap.
 *   - stream is a cudaStream_t (NULL = the legacy default stream). Calls
 *     enqueue work and return without synchronising.
 *   - Arguments are checked before anything is launched; on any error the
 *     call returns a non-zero fa_status and leaves the outputs untouched.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, B/H/N < 1, size overflow, bad scale */
  FA_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, or no sm_100-family GPU */
  FA_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = 4,   /* workspace pointer null or smaller than required */
  FA_ERR_LAUNCH = 5,      /* the CUDA runtime rejected a launch or a query */
  FA_ERR_TIMEOUT = 6      /* a kernel gave up waiting (reported by fa_device_status) */
} fa_status;

/*
 * Forward pass (the tiled loop of chapter 07 with the running-max softmax of
 * chapter 08, fused into one kernel that writes only o and lse).
 *   q, k, v  [in]  bf16 [B, H, N, d]
 *   o        [out] bf16 [B, H, N, d]
 *   lse      [out] fp32 [B, H, N], lse[i] = ln sum_{j visible to i} exp(scale q_i . k_j)
 * Returns FA_OK or an fa_status error code.
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, void* stream);

/*
 * Bytes of device workspace with which fa_fwd_kv may split the keys of this
 * shape over several CTAs per query block on the current device (0: the
 * shape has enough query blocks to fill the GPU, or too few keys to split;
 * also 0 for an invalid shape or without a usable device). The partial
 * results are fp32 O / l [splits][B, H, Nq, d] and logsumexps
 * [splits][B, H, Nq], each padded to 256 bytes.
 */
FA_API size_t fa_fwd_kv_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/*
 * Forward pass of Nq query rows against Nk keys, e.g. a decoding step (a few
 * new queries against a long cache of keys and values) -- the unequal-length
 * and decode-style attention the pages name as the next steps, computed as
 * in fa_fwd with the query rows aligned to the last Nq keys under the mask.
 *   q        [in]  bf16 [B, H, Nq, d]
 *   k, v     [in]  bf16 [B, H, Nk, d]
 *   o        [out] bf16 [B, H, Nq, d]
 *   lse      [out] fp32 [B, H, Nq], lse[i] = ln sum_{j visible to i} exp(scale q_i . k_j)
 *   causal   key j is visible to query i iff j <= i + Nk - Nq; needs Nq <= Nk
 *            (FA_ERR_INVALID_ARG otherwise, since the first rows would see no key)
 *   seqlens_q, seqlens_k
 *            [in]  optional device int32 [B] (NULL: every sequence has Nq
 *            rows / Nk keys), 4-byte aligned: padding masks for a batch of
 *            sequences of different lengths stored at the full size.
 *            Sequence b has only its first sq = seqlens_q[b] query rows and
 *            sk = seqlens_k[b] keys, with the causal rule above written for
 *            those lengths (j <= i + sk - sq). Rows i >= sq get o = 0 and
 *            lse = -inf; keys j >= sk are seen by no row. The padding
 *            entries of q, k, v are never used for a result but must hold
 *            finite values: the blocks that straddle a length multiply them
 *            by zero weights. Lengths are read on the device: one outside
 *            [1, Nq] / [1, Nk] (or, under causal, sq > sk) is clamped into
 *            range and reported by fa_device_status as FA_ERR_INVALID_ARG.
 *   workspace, workspace_bytes
 *            optional (NULL / 0: one pass over the keys per query block). With
 *            fa_fwd_kv_workspace_bytes bytes (or fewer: then fewer ranges), a
 *            call with few query blocks splits the keys into ranges, computes
 *            each range's O / l and logsumexp, and merges them with the
 *            running-maximum rule of chapter 08 written for logsumexps:
 *            lse = m + ln sum_z e^(lse_z - m), o = sum_z e^(lse_z - lse) o_z.
 * fa_fwd(..., N, ...) is fa_fwd_kv(..., N, N, ..., NULL, NULL, NULL, 0, stream).
 * Returns FA_OK or an fa_status error code.
 */
FA_API int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                     int d, float scale, int causal, const int* seqlens_q, const int* seqlens_k, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * 8-bit forward: the FP8 mode the pages give the third version ("FlashAttention
 * does more arithmetic to move less data", the section on the later versions;
 * "FlashAttention and GPU Memory", chapter 11), with both products on 8-bit
 * tensor-core operands and fp32 accumulation.
 *   q, k, v  [in]  E4M3 codes (OCP 8-bit float, one byte per element) [B, H, N, d], d = 128
 *   descale_q, descale_k, descale_v
 *            [in]  per-tensor dequantisation factors (finite, > 0): the inputs
 *            are descale_q * e4m3(q), descale_k * e4m3(k), descale_v * e4m3(v)
 *   o        [out] bf16 [B, H, N, d]
 *   lse      [out] fp32 [B, H, N], the logsumexp of the scaled scores of the dequantised inputs
 *   scale, causal as in fa_fwd.
 * The probabilities enter the second product as E4M3: each row's P is scaled
 * by a power of two, 2^(6 - m) for an integer reference m at most 2 below the
 * row maximum of scores * log2(e) (so P never exceeds 2^8 < 448), rounded to
 * nearest even, and o divides by the sum of the unrounded values. A power-of-
 * two scale makes the rounded values independent of the reference, hence of
 * the order in which the keys are visited (outside the subnormal range).
 * FA_ERR_UNSUPPORTED for d != 128.
 * Returns FA_OK or an fa_status error code.
 */
FA_API int fa_fwd_fp8(const void* q, const void* k, const void* v, float descale_q, float descale_k, float descale_v,
                      void* o, float* lse, int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Bytes of device workspace fa_bwd needs for this shape: the fp32 row terms
 * D_i = dO_i . o_i [B, H, N], padded to 256 bytes, then 256 bytes of work
 * counters that the backward kernels use to hand out (head, block) tiles to
 * their persistent CTAs. Returns 0 if the shape is invalid.
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass (chapter 09): gradients of a loss L with respect to q, k, v
 * given dO = dL/dO, rebuilding each score tile from q, k and lse.
 *   q, k, v, o, dO [in]  bf16 [B, H, N, d]  (o and lse from fa_fwd on the same q, k, v, scale, causal)
 *   lse            [in]  fp32 [B, H, N]
 *   dq, dk, dv     [out] bf16 [B, H, N, d]
 *   workspace      [scratch] device memory of at least fa_bwd_workspace_bytes(B, H, N, d)
 *                  bytes, 256-byte aligned; its contents on entry do not matter
 *                  and are overwritten. It must not be used by another call
 *                  that may run concurrently.
 * dq, dk and dv are each summed on chip in a fixed order: repeated calls on
 * the same inputs give bit-identical results.
 * Returns FA_OK or an fa_status error code.
 */
FA_API int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* workspace,
           size_t workspace_bytes, void* stream);

/*
 * fa_bwd for Nq query rows against Nk keys (the backward of fa_fwd_kv, with
 * the same causal rule: key j visible to query i iff j <= i + Nk - Nq, which
 * needs Nq <= Nk). q, o, dO, dq are [B, H, Nq, d]; k, v, dk, dv [B, H, Nk, d];
 * lse [B, H, Nq] (the logsumexp fa_fwd_kv returned). The workspace holds D
 * for the Nq rows and the work counters: fa_bwd_kv_workspace_bytes bytes,
 * 256-byte aligned. seqlens_q, seqlens_k are the padding masks of fa_fwd_kv
 * (NULL: none), the same as in the forward call: padding rows get dq = 0,
 * padding keys dk = dv = 0, and the padding entries of q, k, v, o, dO must
 * hold finite values. fa_bwd(..., N, ...) is fa_bwd_kv(..., N, N, ..., NULL,
 * NULL, ...).
 * Returns FA_OK or an fa_status error code.
 */
FA_API size_t fa_bwd_kv_workspace_bytes(int B, int H, int Nq, int Nk, int d);
FA_API int fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                     const int* seqlens_q, const int* seqlens_k, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * Largest scratch, in bytes, that fa_bwd_noalloc holds per device: the
 * shapes it accepts are those with fa_bwd_workspace_bytes(B, H, N, d) <= this
 * (B * H * N up to 8,388,544 rows).
 */
#define FA_BWD_NOALLOC_MAX_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * Backward pass for callers that cannot allocate device memory. The pages
 * have no counterpart to this call; it exists for callers that are given no
 * allocator (a plug-in inside a host framework that owns all device memory) or
 * may not call cudaMalloc (a latency-critical path that cannot afford its
 * implicit synchronisation).
 *
 * Same arguments, results and errors as fa_bwd, without the workspace: the
 * scratch lives in a fixed FA_BWD_NOALLOC_MAX_SCRATCH_BYTES device array
 * inside the library, which every GPU that loads the library holds until the
 * process exits. The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   - Shapes whose scratch need exceeds the maximum are rejected with
 *     FA_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current). Make that first call
 *     on a device before any stream capture begins.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (each call writes every value it later reads). Calls
 *     that may overlap on the GPU, e.g. on two streams of one device, race on
 *     it: order them on one stream or synchronise between them.
 */
FA_API int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                          int causal, void* stream);

/*
 * Forward and backward with dropout of P after the softmax ("FlashAttention
 * and GPU Memory": chapter 07 fuses dropout into the one kernel; chapter 09's
 * backward stores no mask: it regenerates it from the generator's state).
 *   p256     dropout probability p256 / 256, 0 .. 255 (FA_ERR_INVALID_ARG
 *            otherwise; 0 is the plain pass); kept elements are scaled by
 *            256 / (256 - p256)
 *   seed, offset
 *            the mask: element (query i, key j) of head bh = b * H + h is kept
 *            iff byte (j mod 4) of word (i mod 4) of Philox4x32-10 (Salmon,
 *            Moraes, Dror and Shaw, SC 2011) with counter (j / 4, i / 4, bh,
 *            offset) and key (seed mod 2^32, seed / 2^32) is >= p256. The same
 *            (seed, offset) in fa_bwd_dropout gives the same mask.
 * o = (P o Z) v with Z = kept / (1 - p); lse is that of the undropped scores
 * (what the backward needs). Other arguments, layouts and errors as in
 * fa_fwd / fa_bwd (self-attention, N query rows and keys).
 */
FA_API int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                          int d, float scale, int causal, int p256, unsigned long long seed, unsigned int offset,
                          void* stream);
FA_API int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                          int causal, int p256, unsigned long long seed, unsigned int offset, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Static, human-readable name of a status code. Never NULL. */
FA_API const char* fa_status_string(int status);

/*
 * Reads (and, if reset != 0, clears) the device-side error word that kernels
 * set when one of their internal waits exceeds its time limit, or when a
 * per-sequence length was out of range, on the current device. Synchronises
 * the device. Returns FA_OK, FA_ERR_TIMEOUT (a wait gave up), FA_ERR_INVALID_ARG
 * (only lengths were out of range), or FA_ERR_LAUNCH if the word cannot be read.
 */
FA_API int fa_device_status(int reset);

/*
 * Test hook for the failure path; the pages have no counterpart to it. Arms a
 * one-shot fault that the next forward launch (fa_fwd, fa_fwd_kv,
 * fa_fwd_fp8 or fa_fwd_dropout, from any thread) consumes:
 *   kind 1  every CTA's load warp withholds the copy of its first query
 *           tile, so the MMA warp's bounded wait for it runs out after the
 *           kernels' wait limit (one second). Each CTA then lets the copies
 *           it issued land, frees its tensor memory, stores no output and sets
 *           the device error word: fa_device_status returns FA_ERR_TIMEOUT.
 *           The outputs of that call are left as they were; the stream and
 *           the context remain usable.
 *   kind 0  disarms a fault not yet consumed.
 * Returns FA_OK, or FA_ERR_INVALID_ARG for another kind. Not for production
 * use: it exists so that tests can drive the timeout path without a GPU fault.
 */
FA_API int fa_test_arm_fault(int kind);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
