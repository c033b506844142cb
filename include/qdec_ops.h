/*
 * qdec_ops.h — per-kernel entry points of the qdec library, for testing one
 * step of the decoder path in isolation.  All pointers are DEVICE pointers
 * unless stated; work is queued on `stream` (a cudaStream_t, NULL = legacy
 * default stream) and nothing is synchronised.  Return 0 or a QDEC_E_* code
 * (include/qdec.h); a launch failure returns QDEC_E_CUDA.
 */
#ifndef QDEC_OPS_H
#define QDEC_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QDEC_GEMM_STORE_F32   0   /* C[m,n] = acc                               (fp32 C) */
#define QDEC_GEMM_ADD_F32     1   /* C[m,n] += acc   (residual add)             (fp32 C) */
#define QDEC_GEMM_SWIGLU_BF16 2   /* C[m,n] = silu(gate) * up, W = [gate rows; up rows at up_off] (bf16 C) */
#define QDEC_GEMM_STORE_BF16  3   /* C[m,n] = bf16(acc)                         (bf16 C) */
#define QDEC_GEMM_ATOMIC_F32  4   /* C[m,n] += acc with fp32 atomics (TCGEN05 only; fp32 C) */

#define QDEC_IMPL_SIMT     0      /* CUDA-core kernel */
#define QDEC_IMPL_TCGEN05  1      /* tcgen05 / TMEM / TMA kernel */

/* C[M, N] = A[M, K] . W[N, K]^T with bf16 A (row stride lda elements) and W
 * (row-major, K contiguous), fp32 accumulation, and the epilogue `mode`
 * ("Forward map - funasr_nano", LLM decoder table: the block's projections,
 * residual adds and packed gate_up SwiGLU).  ldc is C's row stride in
 * elements.  Shape limits: K % 64 == 0 for TCGEN05, K % 32 == 0 for SIMT;
 * TCGEN05 also needs C 16-byte aligned with ldc >= N and ldc x element size a
 * multiple of 16 bytes (its epilogue writes C by TMA). */
int qdec_op_gemm(const void *A, int32_t lda, const void *W, int32_t M, int32_t N, int32_t K, int32_t mode,
                 int32_t up_off, void *C, int32_t ldc, int32_t impl, void *stream);

/* C[M, N] += A[M, K] . W[N, K]^T on the tcgen05 tensor cores with K split over
 * `splits` CTAs per output tile whose fp32 partials are added with atomics
 * (summation order, hence the last bits, may vary between runs).  Used by the
 * few-row GEMMs of the lockstep batch decode.  Shape limits as TCGEN05 above;
 * C fp32 with row stride ldc (16-byte aligned rows). */
int qdec_op_gemm_splitk(const void *A, int32_t lda, const void *W, int32_t M, int32_t N, int32_t K, int32_t splits,
                        float *C, int32_t ldc, void *stream);

/* Tile width of the tcgen05 GEMMs (qdec_op_gemm and the context's prefill):
 * 0 lets the library choose per shape (128 x 256 tiles when the problem has
 * enough tiles to fill the SMs, else 128 x 128), 128 or 256 forces one (a
 * shape that a 256-wide tile does not divide still uses 128).  Process-wide
 * and not thread-safe: meant for tuning and tests.  Returns the previous
 * setting, or QDEC_E_INVALID_ARG for any other value. */
int qdec_op_gemm_tile_width(int32_t bn);

/* Tile height of the 256-wide tcgen05 GEMM tiles: 128 runs each tile on one CTA, 256 runs
 * 256 x 256 tiles on a pair of CTAs (a cluster of two SMs, tcgen05 cta_group::2, each CTA
 * loading its own 128 rows of A and of B), 0 (the default) lets the library choose, which
 * is one CTA: the pair measured slower on every prefill shape.
 * Process-wide and not thread-safe: for tuning and tests.  Returns the previous setting, or
 * QDEC_E_INVALID_ARG for any other value. */
int qdec_op_gemm_tile_rows(int32_t bm);

/* Programmatic dependent launch of the prefill chain (the GEMMs, attention, norms and
 * the other kernels between the embedding and the head): 1 (the default) launches each
 * with programmatic stream serialisation, so its CTAs start their prologue and request
 * their first weight tiles while the preceding kernel finishes, and wait for that kernel
 * before touching what it writes; 0 launches them plainly.  Results are identical either
 * way.  Process-wide and not thread-safe: for measurements and tests.  Returns the previous
 * setting, or QDEC_E_INVALID_ARG for a value other than 0 or 1. */
int qdec_op_programmatic_launch(int32_t on);

/* The token choice of qdec_set_sampling (include/qdec.h) on one logits vector: logits
 * fp32 [V] (device), history int32 [n_history] (device ids; ids outside [0, V) are
 * ignored), the draw at position `pos` under `seed`; *token (device int32) receives the
 * chosen id.  V <= 262,144.  Errors: INVALID_ARG for null pointers, negative sizes or
 * parameters outside the ranges of qdec_set_sampling. */
int qdec_op_sample(const float *logits, int32_t V, const int32_t *history, int32_t n_history, float temperature,
                   int32_t top_k, float top_p, float repetition_penalty, uint64_t seed, int32_t pos, int32_t *token,
                   void *stream);

/* Block quantization of W bf16 [N, K] (K % 32 == 0) into the library's formats
 * (QDEC_WEIGHTS_Q8B32 / QDEC_WEIGHTS_Q4B32 of include/qdec.h; "Fun-ASR-Nano Native Runtime
 * Implementation Plan", Task 8, names quantized decoders without defining the formats):
 * codes int8 [N, K] (q8b32) or packed nibbles uint8 [N, K / 2] (q4b32), scales fp16
 * [N, K / 32].  Deterministic and exact: the scale and the quotients are evaluated in double. */
int qdec_op_quantize(const void *W, int32_t N, int32_t K, int32_t fmt, void *codes, void *scales, void *stream);

/* y = W' . xhat on quantized weights (the decode GEMV): xhat = x * rsqrt(mean x^2 + eps) *
 * norm_g when norm_g is given, else x (fp32 [K]); mode 0 stores y (fp32 [rows]), 1 adds into
 * y, 2 stores silu(gate) * up with the up rows at row offset up_off.  K % 256 == 0. */
int qdec_op_gemv_q(const void *codes, const void *scales, int32_t fmt, int32_t rows, int32_t K, const float *x,
                   const void *norm_g, float eps, int32_t mode, int32_t up_off, float *y, void *stream);

/* Synchronises the device and reports whether a tensor-core kernel launched
 * through these entry points gave up on a bounded wait since the last call:
 * QDEC_OK, or QDEC_E_TIMEOUT (the flag is then cleared). */
int qdec_op_device_error(void);

/* Causal GQA attention for T query rows at positions pos0..pos0+T-1 over
 * cache keys [0, pos0 + T): Q bf16 [T, HQ, D]; k_cache / v_cache bf16
 * [HKV][max_seq][D]; O bf16 [T, HQ * D] ("Qwen3ASR ncnn多平台移植" §5, the
 * prefill's upper-triangular causal mask; GQA 16/8 in the forward map). */
int qdec_op_attention_prefill(const void *Q, int32_t T, int32_t HQ, int32_t HKV, int32_t D, int32_t max_seq,
                              int32_t pos0, const void *k_cache, const void *v_cache, void *O, int32_t impl,
                              void *stream);

/* Bytes of scratch qdec_op_lm_head_argmax needs for a vocabulary of V rows. */
size_t qdec_op_lm_head_scratch_bytes(int32_t V);

/* Tied lm_head with the final RMSNorm fused in front ("Forward map -
 * funasr_nano": `rms_norm * w` then `mul_mat(token_w, last_x)`):
 * h = x * rsqrt(mean x^2 + eps) * g_final, logits[v] = E[v] . h (fp32 [V]),
 * *argmax = lowest index among the maximal logits (device int32).
 * x fp32 [H]; E bf16 [V, H]; g_final bf16 [H].  `scratch` (caller-owned,
 * >= qdec_op_lm_head_scratch_bytes(V)) holds per-block partial maxima and a
 * ticket counter whose first 4 bytes must be zero before the first call;
 * every call leaves them zero again.  Calls sharing a scratch must not
 * overlap on the GPU. */
int qdec_op_lm_head_argmax(const void *E, int32_t V, int32_t H, const float *x, const void *g_final, float eps,
                           float *logits, int32_t *argmax, void *scratch, size_t scratch_bytes, void *stream);

/* Largest vocabulary qdec_op_lm_head_argmax_static accepts. */
#define QDEC_LM_HEAD_STATIC_MAX_VOCAB 262144

/* The same tied lm_head + argmax as qdec_op_lm_head_argmax, for callers that
 * cannot let a library allocate device memory: hosts that own all GPU memory
 * through their own pooling allocator, or real-time threads where cudaMalloc's
 * implicit device synchronisation and latency are not acceptable.  This call
 * allocates nothing: the per-block partial maxima and the ticket counter live
 * in one library-owned static device array of about 64 KB (enough for
 * QDEC_LM_HEAD_STATIC_MAX_VOCAB rows), which every GPU that loads the library
 * holds until the process exits.  The paper has no counterpart of this call.
 * The caller still passes inputs and outputs (as for qdec_op_lm_head_argmax).
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  The
 * address is kept for the life of the process: after cudaDeviceReset on a
 * device, this call is no longer valid there.  Each call
 * clears the ticket counter on `stream` before its kernel.  All calls share
 * the one array, so calls that overlap on the GPU (different streams, or other
 * host threads) race and give wrong results: serialise them.  Errors:
 * INVALID_ARG for a null pointer, H % 8 != 0, or V > the maximum. */
int qdec_op_lm_head_argmax_static(const void *E, int32_t V, int32_t H, const float *x, const void *g_final, float eps,
                                  float *logits, int32_t *argmax, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* QDEC_OPS_H */
