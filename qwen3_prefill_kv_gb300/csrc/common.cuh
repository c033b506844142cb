// Internal helpers and kernel launchers shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace qdec {

typedef uint16_t bf16_t;   // raw bf16 bits

// bf16 -> fp32 widening is exact: the bf16 bits are the high half of the fp32 word.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf1(bf16_t h) { return __uint_as_float(((uint32_t)h) << 16); }
__device__ __forceinline__ bf16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- programmatic dependent launch.  The kernels of the prefill chain call pdl_trigger() on
// entry, which lets the stream's next kernel place its CTAs (prologue, weight prefetch)
// while this grid finishes, and pdl_wait() before their first access to anything an earlier
// kernel of the stream writes: it returns once the preceding grid has completed and its
// writes are visible (at once for a kernel launched without the attribute).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Process-wide switch of the launch attribute (on unless switched off); returns the previous value.
int set_programmatic_launch(int on);
bool programmatic_launch();

// kern<<<grid, block, smem, s>>>(args...) with programmatic stream serialisation when the
// switch is on (the kernel must then call pdl_wait() as described above).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = programmatic_launch() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// silu(z) = z / (1 + e^-z), with CUDA's fast exponential and division: every use rounds the
// result (or its product with the up projection) to bf16, far coarser than their error of
// a few ulp; for z below about -87 the quotient is 0, as silu's value there is below fp32's.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// (value, index) with "greater value wins, lower index wins a tie"; NaN never wins.
struct ArgMax { float v; int i; };
__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// Token choice after the lm_head (k_sample.cu): greedy when temperature is 0, else the
// repetition penalty, temperature, top-k, top-p and a splitmix64 counter draw at `pos`;
// one CTA, writes *token (device).  The history bitmap limits V to kSampleMaxVocab.
constexpr int kSampleMaxVocab = 262144;
bool sample_params_valid(int V, float temperature, int top_k, float top_p, float penalty);
cudaError_t launch_sample(const float* logits, int V, const int* hist, int n_hist, float temperature, int top_k,
                          float top_p, float penalty, unsigned long long seed, int pos, int* token, cudaStream_t s);

// Device-side model shape (mirrors qdec_config).
struct Shape {
    int H, NL, HQ, HKV, D, F, V, max_seq;
    float theta, eps;
    int qkv_rows() const { return (HQ + 2 * HKV) * D; }
};

// ---------------------------------------------------------------- launchers
// Embedding gather + audio splice into the fp32 residual X [T, H].
cudaError_t launch_embed_splice(const bf16_t* E, const int* ids_dev, int T, int H,
                                const bf16_t* audio, int n_audio, int off, float* X,
                                int* history, cudaStream_t s);
// Decode: id = token >= 0 ? token : *prev_argmax; x = E[id]; history[*pos] = id.
cudaError_t launch_embed_token(const bf16_t* E, int token, const int* prev_argmax,
                               const int* pos, int H, float* x, int* history, cudaStream_t s);
// *pos += n (keeps the device-side position of a captured decode step current).
cudaError_t launch_advance_position(int* pos, int n, cudaStream_t s);
// *p = v, queued on the stream (no host memory involved).
cudaError_t launch_set_int(int* p, int v, cudaStream_t s);

// Count of kernel launches issued by the library (graph replays add their kernel nodes).
void count_launches(uint64_t n);
// Records a message for qdec_last_error() and returns `code`.
int set_error(int code, const char* fmt, ...);
// out[t] = bf16(X[t] * rsqrt(mean X[t]^2 + eps) * g)
cudaError_t launch_rmsnorm_bf16(const float* X, int T, int H, const bf16_t* g, float eps,
                                bf16_t* out, cudaStream_t s);
// The same after X[t] += sum_z part[z * pstride + t * H] (z = 0 .. splits-1 in order; X is
// updated in place): the residual add of a split-K projection folded into the next norm.
cudaError_t launch_rmsnorm_fold_bf16(float* X, const float* part, int splits, size_t pstride, int T, int H,
                                     const bf16_t* g, float eps, bf16_t* out, cudaStream_t s);
// X[i] += sum_z part[z * pstride + i] for i < n (fixed order).
cudaError_t launch_fold_partials(float* X, const float* part, int splits, size_t pstride, size_t n, cudaStream_t s);

enum GemmMode { GEMM_STORE_F32 = 0, GEMM_ADD_F32 = 1, GEMM_SWIGLU_BF16 = 2, GEMM_STORE_BF16 = 3, GEMM_ATOMIC_F32 = 4,
                GEMM_QKV_ROPE = 5, GEMM_PARTIAL_F32 = 6 };
// GEMM_PARTIAL_F32 splits K over `splits` CTAs per tile; split z stores its fp32 partial to
// C + z * M * ldc (plain stores, no atomics): the consumer adds the slabs in a fixed order.
// C[M, N] (op) A[M, K] . W[N, K]^T.  SWIGLU: W is [2N, K] (gate rows, then up rows at
// offset `up_off` rows) and C_bf16[m, n] = silu(gate) * up.
cudaError_t launch_gemm_simt(const bf16_t* A, int lda, const bf16_t* W, int M, int N, int K, int mode,
                             int up_off, float* Cf, bf16_t* Cb, int ldc, cudaStream_t s);

// The same GEMM on the tcgen05 tensor cores (TMA-fed, TMEM accumulator).  Needs K % 64 == 0,
// lda % 8 == 0, N % 128 == 0 (SwiGLU: N % 64 == 0) and 16-byte aligned A, W.
bool gemm_tc_supported(int N, int K, int mode, int lda);
// GEMM_ATOMIC_F32 (C += acc with fp32 vector atomics) and GEMM_PARTIAL_F32 may split K over
// `splits` CTAs per tile.  gemm_tc_splits() gives the count the launcher actually uses (every
// split gets at least one 64-wide k-block).
int gemm_tc_splits(int K, int splits);
// Forces the tcgen05 GEMM's tile width (128 or 256; 0 = chosen per shape); returns the previous
// setting.  Process-wide, not thread-safe: for tuning and tests.
int set_gemm_tile_width(int bn);
int gemm_tile_width();   // the current setting (0, 128 or 256)
// The same for the tile height of the 256-wide tiles (128 or 256 rows; 0 = chosen per shape).
int set_gemm_tile_rows(int bm);
int gemm_tile_rows();
// bias (fp32 [N], optional) is added to every row and relu (0/1) clamps at zero, after the
// accumulation, in the STORE_F32, ADD_F32 (C += acc + bias) and STORE_BF16 modes.
cudaError_t launch_gemm_tc(const bf16_t* A, int lda, const bf16_t* W, int M, int N, int K, int mode, int up_off,
                           float* Cf, bf16_t* Cb, int ldc, cudaStream_t s, int splits = 1,
                           const float* bias = nullptr, int relu = 0);
// The packed QKV projection with the per-head epilogue fused (head_dim 128, one head per
// 128-column tile): q heads -> RMSNorm(g_q) + NeoX RoPE at pos0 + row -> bf16 q [M][HQ][128];
// k heads -> RMSNorm(g_k) + RoPE -> bf16 K cache slot pos0 + row; v heads -> bf16 V cache.
struct QkvRopeEpi {
    const float2* rope;        // [max_seq][64] (cos, sin)
    const float2* rope_t;      // the same values as [64][max_seq]
    const bf16_t *g_q, *g_k;   // [128]
    bf16_t *q, *kc, *vc;       // q [M][HQ][128]; this layer's K and V cache [HKV][max_seq][128]
    int pos0, HQ, HKV, max_seq;
    float eps;
};
bool gemm_tc_qkv_rope_supported(const Shape& sh, int lda);
cudaError_t launch_gemm_tc_qkv_rope(const bf16_t* A, int lda, const bf16_t* W, int M, int K, const QkvRopeEpi& epi,
                                    cudaStream_t s);
// First timeout code recorded by a tensor-core kernel since the last call (0 = none);
// synchronous, clears the flag.
int tc_error_read_and_clear();

// Per-head RMSNorm + NeoX RoPE on q and k, V copy, KV append at slots pos0 + t.
// qkv fp32 [T, (HQ+2HKV) D]; q_out: bf16 [T, HQ, D] (q_bf16) or fp32 (q_f32).
// qkv may be the first of `splits` split-K partial slabs pstride floats apart (summed in order).
cudaError_t launch_qk_norm_rope_append(const float* qkv, int T, const Shape& sh, const int* pos0,
                                       const bf16_t* g_q, const bf16_t* g_k, const float2* rope_cs,
                                       bf16_t* q_bf16, float* q_f32, bf16_t* k_cache, bf16_t* v_cache,
                                       cudaStream_t s, int splits = 1, size_t pstride = 0);

// Bidirectional multi-head attention (the audio adaptor, head_dim 128, one kv head per q head):
// every query row attends every key row of the clip.  Q, K, V bf16 views [T][heads][128] with
// rows row_stride elements apart; O bf16 [T][heads * 128].
cudaError_t launch_attention_bidir_tc(const bf16_t* Q, const bf16_t* K, const bf16_t* V, int row_stride, int T,
                                      int heads, bf16_t* O, cudaStream_t s);
// Prefill attention: Q bf16 [T, HQ, D] at positions pos0..pos0+T-1 over cache keys [0, pos0+T).
cudaError_t launch_attention_prefill_simt(const bf16_t* Q, int T, const Shape& sh, int pos0,
                                          const bf16_t* k_cache, const bf16_t* v_cache,
                                          bf16_t* O, cudaStream_t s);

// The same prefill attention on the tcgen05 tensor cores (head_dim 128 only).
bool attention_tc_supported(const Shape& sh);
int fa_error_read_and_clear();   // as tc_error_read_and_clear, for the attention kernel
cudaError_t launch_attention_prefill_tc(const bf16_t* Q, int T, const Shape& sh, int pos0, const bf16_t* k_cache,
                                        const bf16_t* v_cache, bf16_t* O, cudaStream_t s);

// Decode attention, split over the KV length L = *pos + 1.
// q fp32 [HQ, D]; partials sized [HQ][n_split] (+ D for o); out fp32 [HQ, D].
int attention_decode_splits(const Shape& sh);
cudaError_t launch_attention_decode(const float* q, const Shape& sh, const int* pos,
                                    const bf16_t* k_cache, const bf16_t* v_cache, int n_split,
                                    float* part_ml, float* part_o, float* out, cudaStream_t s);

// Decode GEMV y = W . xhat with fp32 activations.
enum GemvMode { GEMV_STORE = 0, GEMV_ADD = 1, GEMV_SWIGLU = 2 };
// norm_g != nullptr: xhat = x * rsqrt(mean x^2 + eps) * norm_g, else xhat = x.
cudaError_t launch_gemv(const bf16_t* W, int rows, int K, const float* x, const bf16_t* norm_g,
                        float eps, int mode, int up_off, float* y, cudaStream_t s);

// Block-quantized layer weights (k_quant.cu): QUANT_Q8B32 int8 codes [N, K], QUANT_Q4B32
// nibbles [N, K / 2] (lower nibble first, code + 8); fp16 scales [N, K / 32] for both.
enum QuantFormat { QUANT_NONE = 0, QUANT_Q8B32 = 1, QUANT_Q4B32 = 2 };
size_t quant_code_bytes(int fmt, size_t N, size_t K);
size_t quant_scale_bytes(size_t N, size_t K);
cudaError_t launch_quantize(const bf16_t* W, int N, int K, int fmt, void* codes, void* scales, cudaStream_t s);
// launch_gemv on quantized weights (K a multiple of 256).
cudaError_t launch_gemv_q(const void* codes, const void* scales, int fmt, int rows, int K, const float* x,
                          const bf16_t* norm_g, float eps, int mode, int up_off, float* y, cudaStream_t s);

// Tied lm_head on one row with fused final RMSNorm and a deterministic grid argmax.
// scratch: >= lm_head_scratch_bytes(V); its first 4 bytes (ticket counter) must be zero
// before the first launch and are returned to zero by every launch.
size_t lm_head_scratch_bytes(int V);
cudaError_t launch_lm_head_argmax(const bf16_t* E, int V, int H, const float* x, const bf16_t* g_final,
                                  float eps, float* logits, int* argmax, void* scratch, cudaStream_t s);

// ---------------------------------------------------------------- batched (lockstep) decode
struct BatchStream {        // one context of a lockstep batch
    bf16_t* kv;             // its KV cache [NL][2][HKV][max_seq][D]
    int* pos;               // its device position (advanced by the step)
    int* argmax;            // its previous / new argmax
    int* hist;              // its token history
    const float2* rope;     // its RoPE table
    int max_seq;
    int shared;             // keys [0, shared) are attended by the shared-prefix kernel (0 = none)
};
// A block of streams whose caches hold the same keys and values at [0, P) (clones of one
// prefill): members[first .. first + count) are their indices in the batch; kv is one member's
// cache, from which the prefix is read once for all of them.
struct PrefixItem {
    const bf16_t* kv;
    int P, first, count;
};
cudaError_t launch_batch_embed(const bf16_t* E, int H, const int* tokens, const BatchStream* bs, int n, float* X,
                               cudaStream_t st);
cudaError_t launch_batch_qk_rope(const float* qkv, const Shape& sh, int layer, const bf16_t* g_q, const bf16_t* g_k,
                                 const BatchStream* bs, int n, float* q_out, cudaStream_t st);
// Attention of every stream over its keys [shared, L) in n_split splits, plus (n_items > 0) the
// shared prefixes in max_chunks further splits, all merged into bf16 out [n, HQ * D].
cudaError_t launch_batch_attention(const float* q, const Shape& sh, int layer, const BatchStream* bs, int n, int n_split,
                                   const PrefixItem* items, int n_items, const int* members, int max_chunks,
                                   float* part_ml, float* part_o, bf16_t* out, cudaStream_t st);
// Shared-prefix attention (k_batch_prefix.cu): head_dim 128 and a GQA group of 1, 2, 4 or 8.
bool prefix_attention_supported(const Shape& sh);
int prefix_item_streams(const Shape& sh);   // streams one PrefixItem may hold
int prefix_chunks(int P);                   // key chunks of a prefix of P positions
cudaError_t launch_prefix_attention(const float* q, const Shape& sh, int layer, const PrefixItem* items, int n_items,
                                    const int* members, int max_chunks, int n_split_total, int split0, float* part_ml,
                                    float* part_o, cudaStream_t st);
// h = silu(g) * u from gu [n, 2F] (gate, then up), or from the sum of `splits` partial slabs of
// it pstride floats apart.
cudaError_t launch_batch_swiglu(const float* gu, int F, int n, bf16_t* h, cudaStream_t st, int splits = 1,
                                size_t pstride = 0);
cudaError_t launch_batch_argmax(const float* logits, int V, int ld, const BatchStream* bs, int n, int* out,
                                cudaStream_t st);

// ---------------------------------------------------------------- persistent decode
struct DecodeLayer {
    const bf16_t *wqkv, *wo, *wgu, *wd, *g_in, *g_post, *g_q, *g_k;
    bf16_t *kc, *vc;   // this layer's K and V cache [HKV][max_seq][D]
};

struct DecodeParams {
    const DecodeLayer* layers;          // device [NL]
    const bf16_t* embed;
    const bf16_t* final_norm;
    const float2* rope;                 // [max_seq][D/2] (cos, sin)
    int H, NL, HQ, HKV, D, F, V, max_seq;
    float eps;
    int pos;                            // position of the new token
    int token;                          // >= 0, or -1 for *argmax
    uint32_t epoch;                     // distinct per launch for one context's buffers
    int n_chunks, chunk;                // attention split of [0, pos + 1)
    int nslot;                          // filled by the launcher
    int* argmax;                        // in: previous argmax; out: this step's
    int* pos_out;                       // set to pos + 1 at the end of the step
    int* history;                       // [max_seq]
    float* logits;                      // [V]
    unsigned long long *ll_x, *ll_qkv, *ll_o, *ll_h;   // tagged vectors {tag, fp32}
    float* attn_part;                   // [HQ][max_chunks][D + 2]
    unsigned int* attn_count;           // [NL * HKV], zero between steps
    ArgMax* am_part;                    // [grid]
    unsigned int* am_count;             // zero between steps
    int* err;                           // 0, or the first error code of the step
    uint32_t spin_limit;                // polls / barrier tests before a wait gives up
    unsigned long long* trace;          // optional [grid][11 NL + 4] globaltimer stamps, or null
};

// Default of DecodeParams::spin_limit: about a second of polls before a wait gives up.
constexpr uint32_t kDecodeSpinDefault = 1u << 21;

struct DecodeLaunch {
    const void* fn = nullptr;
    int grid = 0, threads = 0, smem = 0, nslot = 0, max_chunks = 1;
};

// Chooses the instantiation, ring depth and grid for `sh` on `device`; cudaErrorNotSupported
// when the persistent kernel does not cover the shape or the device.
cudaError_t decode_persistent_plan(const Shape& sh, int device, DecodeLaunch* out);
// keys: positions per attention unit (0 = 256).
void decode_persistent_chunks(const DecodeLaunch& cfg, int L, int keys, int* n_chunks, int* chunk);
cudaError_t launch_decode_persistent(const DecodeParams& p, const DecodeLaunch& cfg, cudaStream_t s);

}  // namespace qdec
