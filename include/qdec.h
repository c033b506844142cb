/*
 * qdec.h — C ABI of a GB300 (sm_103a) library for the Qwen3-0.6B-shape causal
 * decoder behind the speech-LLM ASR pipelines described in "Forward map -
 * funasr_nano" (transcribe.cpp), "Qwen3ASR ncnn多平台移植" (ncnn discussion) and
 * "Fun-ASR-Nano Native Runtime Implementation Plan" (audio.cpp).
 *
 * The path: multimodal prefill (token-embedding gather with audio rows spliced
 * in at an offset), then single-token incremental decode over a per-layer KV
 * cache, then the tied lm_head with greedy argmax; contexts can be cloned to
 * branch from one prefill state and stepped together in a batch.
 *
 * Conventions shared by every call:
 *  - All calls return 0 (QDEC_OK) or a negative QDEC_E_* code; nothing throws
 *    across the ABI.  On an error other than QDEC_E_CUDA the context is left
 *    unchanged.  qdec_last_error() gives a message for the calling thread.
 *  - Weights are BORROWED device pointers (bf16, row-major [out, in]) that
 *    must stay valid for the life of every context created from them,
 *    clones included.  A context OWNS its KV cache and scratch.
 *  - Work is queued on the stream given to qdec_create (NULL = a stream the
 *    context creates).  Calls that return an argmax to the host synchronise
 *    that stream; calls without host outputs only queue work.
 *  - Pointers documented as "host or device" are classified with
 *    cudaPointerGetAttributes: device and managed memory are used in place,
 *    anything else is copied through a staging buffer.
 *  - A context is not thread-safe; distinct contexts may be used from
 *    distinct threads if they use distinct streams.
 */
#ifndef QDEC_H
#define QDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QDEC_OK              0
#define QDEC_E_INVALID_ARG  (-1)  /* null pointer, id outside [0, vocab), bad sizes/offsets */
#define QDEC_E_CAPACITY     (-2)  /* the step would write a KV slot >= max_seq */
#define QDEC_E_STATE        (-3)  /* decode before prefill, mixed contexts in a batch */
#define QDEC_E_CUDA         (-4)  /* a CUDA runtime/driver call failed (context may be unusable) */
#define QDEC_E_OOM          (-5)  /* device or pinned allocation failed */
#define QDEC_E_TIMEOUT      (-6)  /* a bounded device-side wait gave up (error flag set by a kernel);
                                       the step's outputs are invalid; see qdec_decode_step */
#define QDEC_E_UNSUPPORTED  (-7)  /* model shape outside what the kernels implement */

/* Model shape.  Qwen3-0.6B: hidden 1024, 28 layers, 16 q heads, 8 kv heads,
 * head_dim 128, ffn 3072, vocab 151936, rope_theta 1e6, rms_eps 1e-6
 * ("Fun-ASR-Nano Native Runtime Implementation Plan", Task 1 Step 1; "Forward
 * map - funasr_nano", LLM decoder table).  max_seq is the KV-cache capacity
 * in positions (prompt + generated tokens).
 * Supported by the kernels: head_dim in {32, 64, 128}; n_q_heads a multiple of
 * n_kv_heads with at most 8 q heads per kv head; hidden and ffn multiples of
 * 128; (n_q_heads + 2 n_kv_heads) * head_dim a multiple of 128. */
typedef struct {
    int32_t hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    float   rope_theta, rms_eps;
    int32_t max_seq;
} qdec_config;

/* Device pointers to bf16 weights.  Per-layer entries are HOST arrays of
 * n_layers device pointers (read during qdec_create only).
 *   embed      [vocab, hidden]   token embedding, also the tied lm_head
 *   final_norm [hidden]
 *   wqkv[l]    [(Hq + 2 Hkv) D, hidden]  rows: q heads, then k heads, then v heads
 *   wo[l]      [hidden, Hq D]
 *   wgu[l]     [2 ffn, hidden]   rows [0, ffn) gate, [ffn, 2 ffn) up ("packed gate_up")
 *   wd[l]      [hidden, ffn]
 *   g_in[l], g_post[l] [hidden];  g_q[l], g_k[l] [head_dim]  RMSNorm gains
 * Every pointer must be 16-byte aligned. */
typedef struct {
    const void *embed;
    const void *final_norm;
    const void *const *wqkv, *const *wo, *const *wgu, *const *wd;
    const void *const *g_in, *const *g_post, *const *g_q, *const *g_k;
} qdec_weights;

typedef struct qdec_ctx qdec_ctx;

/* Creates a context ("Fun-ASR-Nano Native Runtime Implementation Plan",
 * Task 1 Step 1 fixes the shape tuple; Task 3 keeps the weights as
 * non-owning tensors; "Qwen3ASR ncnn多平台移植" §5 holds a generation's state in
 * a context object): validates the shape, records the weight pointers,
 * allocates the KV cache [n_layers][2][n_kv_heads][max_seq][head_dim] bf16,
 * the decode scratch and a RoPE cos/sin table [max_seq][head_dim/2] (angles
 * p * theta^(-2i/D) evaluated in double on the host, stored as fp32).
 * `cuda_stream` is a cudaStream_t that must outlive this context and its
 * clones, or NULL: the library then creates a stream, shares it with the
 * context's clones and destroys it with the last of them.  *out receives the
 * context. */
int qdec_create(const qdec_config *cfg, const qdec_weights *w, void *cuda_stream, qdec_ctx **out);

/* Prefill ("Forward map - funasr_nano", Generation / KV Path, "Prefill, all
 * positions"; "Qwen3ASR ncnn多平台移植" §4-§5).  Resets the context to position
 * 0, embeds ids[0..n_ids) (HOST int32), overrides rows [audio_offset,
 * audio_offset + n_audio) with audio_rows (bf16 [n_audio, hidden], host or
 * device; the ids under them are range-checked and otherwise ignored), runs
 * all layers writing KV slots [0, n_ids), and evaluates the tied lm_head on
 * the LAST position only.
 *   logits_out: NULL or fp32 [vocab], host or device.
 *   argmax_out: NULL or HOST int32; lowest index among equal maxima.
 * Synchronises the stream only when argmax_out is given.
 * Errors: INVALID_ARG (n_ids <= 0, id out of range, audio range outside the
 * prompt, n_audio > 0 with NULL rows), CAPACITY (n_ids > max_seq). */
int qdec_prefill(qdec_ctx *ctx, const int32_t *ids, int32_t n_ids,
                 const void *audio_rows, int32_t n_audio, int32_t audio_offset,
                 float *logits_out, int32_t *argmax_out);

/* One incremental decode step at position n = qdec_position(ctx)
 * ("Qwen3ASR ncnn多平台移植" §5 steps 1-6; "Forward map - funasr_nano",
 * "Single-step decode @ n_past >= T_prompt").  token >= 0 is embedded; token
 * == -1 feeds back the previous step's argmax without a host round trip.
 * Writes KV slot n, advances the position by one, evaluates the lm_head.
 * logits_out / argmax_out as in qdec_prefill.  Errors: STATE (no prefill),
 * CAPACITY (n >= max_seq), INVALID_ARG (token < -1 or >= vocab), TIMEOUT (a
 * wait of the persistent step gave up, QDEC_OPT_SPIN_LIMIT).  A TIMEOUT
 * reported by this call (argmax_out given) leaves the position, the device
 * argmax and slots [0, n) as they were, so the step can be run again with the
 * same token (pass it explicitly when the context samples); a TIMEOUT that
 * surfaces later through qdec_sync needs a new prefill. */
int qdec_decode_step(qdec_ctx *ctx, int32_t token, float *logits_out, int32_t *argmax_out);

/* One lockstep decode step for n contexts (clones of one prefill or
 * independent prompts) sharing weights and shape.  The pages run one
 * context at a time ("Qwen3ASR ncnn多平台移植" §1 lists no batch inference);
 * this call is each context's step of §5 taken together for the branching
 * workload (one 415-position prefill cloned into 64 streams), so each stream
 * computes exactly its own single-context step.  tokens: HOST int32 [n]
 * (-1 = previous argmax of that context).  logits_out: NULL or fp32
 * [n, vocab] (host or device); argmax_out: NULL or HOST int32 [n].  Each
 * context advances by one.  Errors as qdec_decode_step, plus STATE when the
 * contexts were not created from the same weights and shape. */
int qdec_decode_step_batch(qdec_ctx *const *ctxs, int32_t n, const int32_t *tokens,
                           float *logits_out, int32_t *argmax_out);

/* Deep copy of a context ("Qwen3ASR ncnn多平台移植" §5: generation clones its
 * input context so several branches can start from one prefill state): KV
 * slots [0, position), token history, position and last argmax.  Weights are
 * shared; the clone gets its own scratch and uses the source's stream. */
int qdec_clone(const qdec_ctx *src, qdec_ctx **out);

/* Number of positions written (prompt + decoded tokens); 0 before prefill;
 * a negative code for a NULL context.  This is n_past of "Forward map -
 * funasr_nano", Generation / KV Path (decode runs at n_past >= T_prompt), the
 * position counter of the context in "Qwen3ASR ncnn多平台移植" §5. */
int qdec_position(const qdec_ctx *ctx);

/* Copies KV slots [pos0, pos0 + n_pos) of one layer to HOST memory as bf16
 * [n_kv_heads][n_pos][head_dim].  kind 0 = K (after Q/K-norm and RoPE),
 * 1 = V.  Synchronises the stream. */
int qdec_read_kv(const qdec_ctx *ctx, int32_t layer, int32_t kind, int32_t pos0, int32_t n_pos,
                 void *host_dst);

/* Copies the token history [0, position) (prompt ids, then each decode
 * step's input token) to HOST int32.  Synchronises the stream. */
int qdec_read_history(const qdec_ctx *ctx, int32_t *host_dst, int32_t n);

/* Waits for all work queued by this context.  Returns QDEC_E_TIMEOUT if a
 * queued persistent decode step gave up on a bounded device-side wait. */
int qdec_sync(const qdec_ctx *ctx);

/* Per-context options. */
#define QDEC_OPT_DECODE_KERNEL   1   /* which kernels run a decode step: */
#define QDEC_DECODE_PERSISTENT   0   /*   one persistent kernel per step (default when supported) */
#define QDEC_DECODE_GRAPH        1   /*   one kernel per operation, replayed as a CUDA graph */
#define QDEC_OPT_TRACE           2   /* 1: the persistent decode step records a phase trace */
#define QDEC_OPT_PREFILL_IMPL    3   /* prefill projections and attention on: */
#define QDEC_PREFILL_TCGEN05     0   /*   tcgen05 tensor cores, TMA-fed (default, where the shape
                                            allows: attention needs head_dim 128) */
#define QDEC_PREFILL_SIMT        1   /*   CUDA cores */
#define QDEC_OPT_ATTN_UNIT_KEYS  4   /* keys per attention unit of the persistent decode step
                                        (the KV history is split into units of about this many
                                        positions, at most one unit per SM; the last unit of a
                                        kv head merges them): 0 = the library default (one unit
                                        up to 160 keys, else about 64 keys per unit), or
                                        8 .. 4096 in multiples of 8 */
#define QDEC_OPT_SPIN_LIMIT      5   /* how long each wait of the persistent decode step polls
                                        (ring-stage barriers, tagged hand-off vectors) before it
                                        gives up and the step reports QDEC_E_TIMEOUT: 0 = the
                                        library default (2^21 polls, about a second), or a
                                        positive count.  Small values make waits that are not
                                        satisfied almost at once give up: a way to exercise the
                                        timeout path without any fault.  The kernel's final wait
                                        for its own copies in flight keeps the default. */

#define QDEC_OPT_SHARED_PREFIX   7   /* 1 (default): in qdec_decode_step_batch, contexts cloned
                                        from one prefill attend the prompt positions they hold
                                        in common once for all of them (read from one member's
                                        cache), and only their own positions past it per
                                        context; 0: every context attends over its own copy.
                                        Read from the batch's first context. */

#define QDEC_OPT_WEIGHTS         8   /* weights of the decode steps' layer projections: */
#define QDEC_WEIGHTS_BF16        0   /*   the borrowed bf16 matrices (default) */
#define QDEC_WEIGHTS_Q8B32       1   /*   the library's q8b32 copy: per 32 weights along K one fp16
                                            scale d = max|w| / 127 and int8 codes
                                            round_half_even(w / d) (1.0625 bytes a weight) */
#define QDEC_WEIGHTS_Q4B32       2   /*   q4b32: d = max|w| / 7, 4-bit codes (code + 8 in a nibble,
                                            lower nibble first; 0.5625 bytes a weight)
                                        ("Fun-ASR-Nano Native Runtime Implementation Plan", Task 8,
                                        ships Q8_0 / Q4_K_M decoders without defining the formats;
                                        these are the library's own).  Setting a quantized format
                                        quantizes the layer matrices on the device into a copy the
                                        context and its clones share, and selects
                                        QDEC_DECODE_GRAPH (the persistent kernel reads bf16).  The
                                        prefill, the embedding and the tied lm_head keep bf16; a
                                        lockstep batch returns UNSUPPORTED for quantized contexts.
                                        Needs hidden, n_q_heads * head_dim and ffn multiples of
                                        256. */

/* Sets an option.  QDEC_OPT_DECODE_KERNEL = QDEC_DECODE_PERSISTENT returns
 * UNSUPPORTED when the persistent kernel does not cover the shape (head_dim /
 * GQA group / ffn combination) or the device (cooperative launch with one
 * CTA per SM).  Clones inherit the setting. */
int qdec_set_option(qdec_ctx *ctx, int32_t option, int32_t value);

/* Current value of an option, or a negative code. */
int qdec_get_option(const qdec_ctx *ctx, int32_t option);

/* Token choice of qdec_prefill and qdec_decode_step ("Qwen3ASR ncnn多平台移植" §1: greedy,
 * temperature, top-k, top-p and repetition penalty; §6: greedy by default).  The page
 * names the options without defining them; this library applies, in order:
 *   1. repetition_penalty r over the distinct ids of the context's history (prompt ids
 *      and the tokens fed so far, the current one included): a positive logit is divided
 *      by r, a non-positive one multiplied by r (r = 1: no penalty);
 *   2. temperature T (T = 0: the lowest-index argmax of the penalised logits);
 *   3. top_k (0: off): keep the logits >= the k-th largest, ties kept;
 *   4. top_p (1: off): keep a token while the probability of the kept tokens strictly
 *      more probable than it sums to < top_p, ties kept;
 *   5. the draw: u = top 24 bits of output pos + 1 of splitmix64 started at state `seed`,
 *      pos = the position of the logits row (the last prompt position after a prefill,
 *      the fed token's position after a step); the token is the smallest kept id whose
 *      cumulative kept probability in id order exceeds u times the kept total.
 * The choice is deterministic for given logits, history and (seed, pos).  It replaces the
 * argmax: argmax_out returns it and token = -1 feeds it to the next step.  The returned
 * logits stay the raw lm_head logits.  Defaults (greedy): T = 0, top_k = 0, top_p = 1,
 * r = 1.  Clones inherit the setting; qdec_decode_step_batch with n > 1 returns
 * QDEC_E_UNSUPPORTED for a sampling context (the lockstep batch is greedy).  Errors:
 * INVALID_ARG for T < 0, top_k < 0, top_p outside (0, 1], r <= 0 or a vocabulary over
 * 262,144. */
int qdec_set_sampling(qdec_ctx *ctx, float temperature, int32_t top_k, float top_p, float repetition_penalty,
                      uint64_t seed);

/* Phase trace of the last persistent decode step (QDEC_OPT_TRACE = 1): one
 * row of 11 * n_layers + 8 entries per CTA of the grid (globaltimer ns).
 * Row layout: [10 l + 2 ph] input ready and [10 l + 2 ph + 1] phase done for
 * phases ph = 0 QKV, 1 attention, 2 o_proj, 3 gate_up, 4 down_proj of layer
 * l (0 where the CTA had no work in that phase); [10 NL] start, [10 NL + 1]
 * lm_head input ready, [10 NL + 2] lm_head done, [10 NL + 3] CTA done;
 * [10 NL + 4 + l] the producer issued its last copy of layer l;
 * [11 NL + 5] and [11 NL + 6]: SM clock cycles consumer thread 0 spent
 * waiting for ring stages and for tagged input vectors.  With
 * host_dst NULL returns the number of entries; otherwise copies them (HOST,
 * capacity >= that number), synchronises and returns the number. */
int qdec_read_trace(const qdec_ctx *ctx, uint64_t *host_dst, int32_t capacity);

/* Frees the context (KV cache, scratch, graphs) — the end of a context's
 * life in "Qwen3ASR ncnn多平台移植" §5.  Waits for the context's queued work
 * first.  NULL is a no-op. */
void qdec_destroy(qdec_ctx *ctx);

/* Static description of a status code.  The pages give their C/C++ calls no
 * error convention ("Qwen3ASR ncnn多平台移植" §5 names the steps only); the
 * codes above are this library's. */
const char *qdec_strerror(int status);

/* Message of the most recent failure on the calling thread ("" if none). */
const char *qdec_last_error(void);

/* Number of kernels this library has launched in the process so far (a CUDA
 * graph replay counts its kernel nodes).  A diagnostic for benchmarks. */
uint64_t qdec_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* QDEC_H */
