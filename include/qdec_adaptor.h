/*
 * qdec_adaptor.h — the projector and bidirectional adaptor that turn audio-encoder frames
 * into the audio rows spliced into the decoder's prompt ("Forward map - funasr_nano", the
 * Adaptor table: linear1 enc -> proj with bias + ReLU, linear2 proj -> hidden with bias,
 * then n_blocks pre-norm blocks of LayerNorm + multi-head self-attention (q/k/v/out
 * projections with biases, no rotary embedding, no mask within a clip) + residual and
 * LayerNorm + a ReLU feed-forward hidden -> ffn -> hidden with biases + residual; the host
 * keeps the first fake_token_len(T) rows; "Fun-ASR-Nano Native Runtime Implementation Plan",
 * Task 5: eight heads, bidirectional).
 *
 * Readings where the pages are silent: attention over every frame of the clip, scaled by
 * 1/sqrt(head_dim), heads contiguous in the projection rows; no norm after the last block;
 * LayerNorm with the population variance.  Precision on the GPU: bf16 weights and GEMM
 * operands (frames, normalised rows, hidden activations, attention q/k/v and probabilities),
 * fp32 accumulation, residual stream, LayerNorm and softmax; the output rows are bf16 (what
 * qdec_prefill splices).
 *
 * All calls return 0 or a negative QDEC_E_* code (include/qdec.h); messages through
 * qdec_last_error().  Weights are BORROWED device pointers that must outlive the adaptor.
 */
#ifndef QDEC_ADAPTOR_H
#define QDEC_ADAPTOR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shape.  Fun-ASR-Nano: enc_dim 512, proj_dim 2048, hidden 1024, n_heads 8, ffn 256,
 * n_blocks 2, ln_eps 1e-12.  Supported: hidden / n_heads = 128; enc_dim, proj_dim, hidden
 * and ffn multiples of 128. */
typedef struct {
    int32_t enc_dim, proj_dim, hidden, n_heads, ffn, n_blocks;
    float ln_eps;
} qdec_adaptor_config;

/* Device weights.  Matrices bf16 row-major [out, in]; biases and LayerNorm parameters fp32.
 * Per-block entries are HOST arrays of n_blocks device pointers (read during create only).
 *   w1 [proj_dim, enc_dim], b1 [proj_dim];  w2 [hidden, proj_dim], b2 [hidden]
 *   ln1_g, ln1_b, ln2_g, ln2_b [hidden]
 *   wqkv [3 hidden, hidden] (rows: q, then k, then v), bqkv [3 hidden]
 *   wo [hidden, hidden], bo [hidden];  fc1 [ffn, hidden], fc1_b [ffn];  fc2 [hidden, ffn], fc2_b [hidden]
 * Every pointer must be 16-byte aligned. */
typedef struct {
    const void *w1, *w2;
    const float *b1, *b2;
    const float *const *ln1_g, *const *ln1_b, *const *ln2_g, *const *ln2_b;
    const void *const *wqkv, *const *wo, *const *fc1, *const *fc2;
    const float *const *bqkv, *const *bo, *const *fc1_b, *const *fc2_b;
} qdec_adaptor_weights;

typedef struct qdec_adaptor qdec_adaptor;

/* Rows the adaptor keeps for T encoder frames: three applications of (n - 1) / 2 + 1
 * ("Forward map - funasr_nano": the frontend's three stride-2 stages; 183 -> 23). */
int32_t qdec_fake_token_len(int32_t n_frames);

/* Creates an adaptor on the given stream (a cudaStream_t that outlives it; NULL = one the
 * adaptor creates).  Errors: INVALID_ARG (null or misaligned pointer, non-positive size),
 * UNSUPPORTED (shape outside the list above). */
int qdec_adaptor_create(const qdec_adaptor_config *cfg, const qdec_adaptor_weights *w, void *cuda_stream,
                        qdec_adaptor **out);

/* Runs the adaptor on `frames` (bf16 [n_frames, enc_dim], host or device) and writes the first
 * qdec_fake_token_len(n_frames) output rows to `rows_out` (bf16 [that many, hidden], host or
 * device; device rows can be passed straight to qdec_prefill).  *n_rows_out (HOST, may be
 * NULL) receives the row count.  Synchronises the stream when rows_out is host memory.
 * Errors: INVALID_ARG (null pointer, n_frames <= 0). */
int qdec_adaptor_run(qdec_adaptor *a, const void *frames, int32_t n_frames, void *rows_out, int32_t *n_rows_out);

/* Frees the adaptor's scratch (waits for its queued work).  NULL is a no-op. */
void qdec_adaptor_destroy(qdec_adaptor *a);

#ifdef __cplusplus
}
#endif
#endif /* QDEC_ADAPTOR_H */
