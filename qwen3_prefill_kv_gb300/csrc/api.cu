// C ABI (include/qdec.h): context lifetime, argument validation, host/device buffer
// handling, and the prefill / decode / clone orchestration of the kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "../../include/qdec.h"
#include "common.cuh"

using namespace qdec;

namespace {

thread_local std::string g_last_error;
std::atomic<unsigned long long> g_prefix_ids{0};

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

#define CK(call)                                                                                   \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess)                                                                     \
            return fail(e_ == cudaErrorMemoryAllocation ? QDEC_E_OOM : QDEC_E_CUDA, "%s: %s (%s:%d)", \
                        #call, cudaGetErrorString(e_), __FILE__, __LINE__);                        \
    } while (0)

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct LayerW {
    const bf16_t *wqkv, *wo, *wgu, *wd, *g_in, *g_post, *g_q, *g_k;
};

// Block-quantized copies of the layer matrices (QDEC_OPT_WEIGHTS), made once from the
// borrowed bf16 weights and shared by a context and its clones.
struct QuantWeights {
    int fmt = 0;
    std::vector<void*> bufs;   // every allocation, freed with the last user
    struct Layer { const void *c[4], *sc[4]; };   // codes / scales of wqkv, wo, wgu, wd
    std::vector<Layer> layers;
    ~QuantWeights() {
        for (void* p : bufs)
            if (p) cudaFree(p);
    }
};

// A stream the library created; shared by a context and its clones and destroyed with
// the last of them.
struct OwnedStream {
    cudaStream_t s = nullptr;
    ~OwnedStream() {
        if (s) cudaStreamDestroy(s);
    }
};

}  // namespace

namespace qdec {
int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}
static unsigned long long g_launches = 0;
void count_launches(uint64_t n) { __atomic_fetch_add(&g_launches, (unsigned long long)n, __ATOMIC_RELAXED); }
}  // namespace qdec

// Workspace of a lockstep batch step (owned by the batch's first context).
struct BatchWork {
    int cap = 0;                         // streams the buffers hold
    std::vector<const qdec_ctx*> members;   // composition the stream table was built for
    BatchStream* d_streams = nullptr;
    int* d_tokens = nullptr;
    int* d_am = nullptr;
    int* h_am = nullptr;                 // pinned
    float *X = nullptr, *qkv = nullptr, *q = nullptr, *part_ml = nullptr, *part_o = nullptr, *gu = nullptr,
          *logits = nullptr;
    bf16_t *Xn = nullptr, *attn = nullptr, *h = nullptr;
    int* h_tokens = nullptr;             // pinned staging of the step's tokens, two buffers of cap
    // shared prefixes of the composition: blocks of member streams that attend a common
    // [0, P) once (PrefixItem), and the prefix ids / setting the table was built for
    PrefixItem* d_items = nullptr;
    int* d_members = nullptr;
    int n_items = 0, max_chunks = 0, split_cap = 0;
    std::vector<unsigned long long> member_prefix;
    int shared_setting = -1;
    cudaEvent_t tok_ev[2] = {nullptr, nullptr};   // each buffer's upload
    int tok_slot = 0;
    int n_split = 1;
    // The step's kernels as a CUDA graph for the current composition: the first step of a
    // composition runs eagerly, the second is captured, later ones replay it.
    cudaGraphExec_t exec = nullptr;
    uint64_t graph_kernels = 0;
    int steps_same = 0;                  // steps run since the composition last changed
    int graph_impl = -1;                 // GEMM implementation the graph was captured with
    void drop_graph() {
        if (exec) cudaGraphExecDestroy(exec);
        exec = nullptr;
        graph_kernels = 0;
        steps_same = 0;
    }
    void release() {
        drop_graph();
        void* ps[] = {d_streams, d_tokens, d_am, X, qkv, q, part_ml, part_o, gu, logits, Xn, attn, h, d_items,
                      d_members};
        for (void* p : ps)
            if (p) cudaFree(p);
        if (h_am) cudaFreeHost(h_am);
        if (h_tokens) cudaFreeHost(h_tokens);
        for (cudaEvent_t e : tok_ev)
            if (e) cudaEventDestroy(e);
        *this = BatchWork();
    }
};

struct qdec_ctx {
    qdec_config cfg;
    Shape sh;
    const bf16_t* embed = nullptr;
    const bf16_t* final_norm = nullptr;
    std::vector<LayerW> layers;
    cudaStream_t stream = nullptr;
    std::shared_ptr<OwnedStream> stream_owner;   // set when the library created `stream`
    cudaStream_t cap_stream = nullptr;   // internal stream used only for graph capture
    int device = 0;

    int position = 0;
    bool prefilled = false;

    // persistent device state
    bf16_t* kv = nullptr;        // [NL][2][HKV][max_seq][D]
    float2* rope = nullptr;      // [max_seq][D/2] (cos, sin), then the same values as [D/2][max_seq]
    int* d_hist = nullptr;       // [max_seq]
    int* d_pos = nullptr;        // position of the next token
    int* d_zero = nullptr;       // constant 0 (prefill start position)
    int* d_argmax = nullptr;

    // decode scratch
    float *d_x = nullptr, *d_qkv = nullptr, *d_q = nullptr, *d_attn = nullptr, *d_h = nullptr;
    float *d_logits = nullptr, *d_part_ml = nullptr, *d_part_o = nullptr;
    void* d_lm_scratch = nullptr;
    int n_split = 1;

    // prefill scratch (grown on demand)
    int pf_cap = 0;
    float *p_X = nullptr, *p_qkv = nullptr;
    float* p_part = nullptr;     // split-K partial slabs of the short-prompt prefill GEMMs
    size_t part_cap = 0;         // floats
    bf16_t *p_Xn = nullptr, *p_Q = nullptr, *p_O = nullptr, *p_H = nullptr;
    int* p_ids = nullptr;
    int audio_cap = 0;
    bf16_t* p_audio = nullptr;

    int* h_pinned = nullptr;     // pinned host staging (argmax values)
    int h_pinned_cap = 0;

    cudaGraphExec_t decode_exec = nullptr;
    uint64_t decode_graph_kernels = 0;   // kernel nodes in decode_exec
    // Prefill bodies (layers, head, position) as CUDA graphs, one per (prompt length,
    // implementation, GEMM tile width); a length is captured on its second prefill.
    struct PrefillGraph {
        int T, impl, tile;
        int uses;                        // eager prefills of this key before capture
        cudaGraphExec_t exec;
        uint64_t kernels;
    };
    std::vector<PrefillGraph> pf_graphs;
    void drop_prefill_graphs() {
        for (auto& g : pf_graphs)
            if (g.exec) cudaGraphExecDestroy(g.exec);
        pf_graphs.clear();
    }

    // persistent single-kernel decode step
    int decode_kernel = QDEC_DECODE_PERSISTENT;
    bool persistent_ok = false;
    DecodeLaunch dp;
    DecodeLayer* d_layers = nullptr;
    unsigned long long *ll_x = nullptr, *ll_qkv = nullptr, *ll_o = nullptr, *ll_h = nullptr;
    float* attn_part = nullptr;
    unsigned int* attn_count = nullptr;
    ArgMax* am_part = nullptr;
    unsigned int* am_count = nullptr;
    uint32_t epoch = 0;
    int* d_err = nullptr;                // d_argmax + 1
    unsigned long long* d_trace = nullptr;   // phase trace of the persistent step (QDEC_OPT_TRACE)
    int prefill_gemm = QDEC_PREFILL_TCGEN05;
    int attn_unit_keys = 0;      // QDEC_OPT_ATTN_UNIT_KEYS (0 = default)
    int spin_limit = 0;          // QDEC_OPT_SPIN_LIMIT (0 = default)
    int shared_prefix = 1;       // QDEC_OPT_SHARED_PREFIX
    std::shared_ptr<QuantWeights> quant;   // QDEC_OPT_WEIGHTS other than bf16
    // Which prefill this context's KV prefix comes from, and how many of its positions came from
    // it: a prefill takes a new id and inherits its prompt; a clone keeps both.  Positions below
    // `inherited` are never rewritten, so contexts with one id hold the same [0, inherited).
    unsigned long long prefix_id = 0;
    int inherited = 0;
    // token choice (qdec_set_sampling); greedy while temperature is 0 and penalty 1
    float samp_t = 0.f, samp_p = 1.f, samp_r = 1.f;
    int samp_k = 0;
    unsigned long long samp_seed = 0ull;
    bool sampling() const { return samp_t != 0.f || samp_r != 1.f; }
    BatchWork* batch = nullptr;          // lockstep-batch workspace when this context led a batch
    int sms = 0;

    size_t kv_layer_stride() const { return (size_t)2 * sh.HKV * sh.max_seq * sh.D; }
    bf16_t* k_cache(int l) { return kv + (size_t)l * kv_layer_stride(); }
    bf16_t* v_cache(int l) { return kv + (size_t)l * kv_layer_stride() + (size_t)sh.HKV * sh.max_seq * sh.D; }
};

namespace {

template <typename T>
cudaError_t dalloc(T** p, size_t n) {
    return cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T) > 0 ? n * sizeof(T) : 16);
}

void free_all(qdec_ctx* c) {
    if (c->batch) {
        c->batch->release();
        delete c->batch;
        c->batch = nullptr;
    }
    if (c->decode_exec) cudaGraphExecDestroy(c->decode_exec);
    c->drop_prefill_graphs();
    void* ptrs[] = {c->kv, c->rope, c->d_hist, c->d_pos, c->d_zero, c->d_argmax, c->d_x, c->d_qkv, c->d_q,
                    c->d_attn, c->d_h, c->d_logits, c->d_part_ml, c->d_part_o, c->d_lm_scratch, c->p_X,
                    c->p_qkv, c->p_Xn, c->p_Q, c->p_O, c->p_H, c->p_ids, c->p_audio, c->p_part, c->d_layers, c->ll_x,
                    c->ll_qkv, c->ll_o, c->ll_h, c->attn_part, c->attn_count, c->am_part, c->am_count,
                    c->d_trace};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    if (c->h_pinned) cudaFreeHost(c->h_pinned);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    c->stream_owner.reset();
}

int validate_config(const qdec_config* c) {
    if (c->hidden <= 0 || c->n_layers <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->ffn <= 0 || c->vocab <= 0 || c->max_seq <= 0)
        return fail(QDEC_E_INVALID_ARG, "non-positive dimension in qdec_config");
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f))
        return fail(QDEC_E_INVALID_ARG, "rms_eps and rope_theta must be positive");
    if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
        return fail(QDEC_E_UNSUPPORTED, "head_dim %d not in {32, 64, 128}", c->head_dim);
    if (c->n_q_heads % c->n_kv_heads != 0)
        return fail(QDEC_E_UNSUPPORTED, "n_q_heads must be a multiple of n_kv_heads");
    const int g = c->n_q_heads / c->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return fail(QDEC_E_UNSUPPORTED, "q heads per kv head (%d) not in {1, 2, 4, 8}", g);
    if (c->hidden % 128 != 0 || c->ffn % 128 != 0)
        return fail(QDEC_E_UNSUPPORTED, "hidden and ffn must be multiples of 128");
    if (((c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim) % 128 != 0)
        return fail(QDEC_E_UNSUPPORTED, "(n_q_heads + 2 n_kv_heads) * head_dim must be a multiple of 128");
    if ((c->n_q_heads * c->head_dim) % 128 != 0)
        return fail(QDEC_E_UNSUPPORTED, "n_q_heads * head_dim must be a multiple of 128");
    return QDEC_OK;
}

int alloc_persistent(qdec_ctx* c);

int alloc_state(qdec_ctx* c) {
    const Shape& sh = c->sh;
    CK(cudaGetDevice(&c->device));
    CK(cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->device));
    CK(cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));
    CK(dalloc(&c->kv, (size_t)sh.NL * c->kv_layer_stride()));
    CK(cudaMemset(c->kv, 0, (size_t)sh.NL * c->kv_layer_stride() * sizeof(bf16_t)));
    CK(dalloc(&c->rope, 2 * (size_t)sh.max_seq * (sh.D / 2)));
    CK(dalloc(&c->d_hist, (size_t)sh.max_seq));
    CK(dalloc(&c->d_pos, 1));
    CK(dalloc(&c->d_zero, 1));
    CK(dalloc(&c->d_argmax, 4));   // [0] argmax, [1] error word of the persistent step
    c->d_err = c->d_argmax + 1;
    CK(cudaMemset(c->d_pos, 0, sizeof(int)));
    CK(cudaMemset(c->d_zero, 0, sizeof(int)));
    CK(cudaMemset(c->d_argmax, 0, 4 * sizeof(int)));
    CK(dalloc(&c->d_x, sh.H));
    CK(dalloc(&c->d_qkv, sh.qkv_rows()));
    CK(dalloc(&c->d_q, (size_t)sh.HQ * sh.D));
    CK(dalloc(&c->d_attn, (size_t)sh.HQ * sh.D));
    CK(dalloc(&c->d_h, sh.F));
    CK(dalloc(&c->d_logits, sh.V));
    c->n_split = attention_decode_splits(sh);
    CK(dalloc(&c->d_part_ml, (size_t)sh.HQ * c->n_split * 2));
    CK(dalloc(&c->d_part_o, (size_t)sh.HQ * c->n_split * sh.D));
    const size_t lm = lm_head_scratch_bytes(sh.V);
    CK(cudaMalloc(&c->d_lm_scratch, lm));
    CK(cudaMemset(c->d_lm_scratch, 0, lm));
    CK(cudaMallocHost(reinterpret_cast<void**>(&c->h_pinned), 64 * sizeof(int)));
    c->h_pinned_cap = 64;
    return alloc_persistent(c);
}

// Buffers of the persistent decode kernel; leaves persistent_ok false (and the graph
// path selected) when the kernel does not cover the shape or the device.
int alloc_persistent(qdec_ctx* c) {
    const Shape& sh = c->sh;
    cudaError_t e = decode_persistent_plan(sh, c->device, &c->dp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        c->persistent_ok = false;
        c->decode_kernel = QDEC_DECODE_GRAPH;
        return QDEC_OK;
    }
    CK(dalloc(&c->d_layers, (size_t)sh.NL));
    std::vector<DecodeLayer> hl(sh.NL);
    for (int l = 0; l < sh.NL; ++l) {
        const LayerW& w = c->layers[l];
        hl[l] = DecodeLayer{w.wqkv, w.wo, w.wgu, w.wd, w.g_in, w.g_post, w.g_q, w.g_k, c->k_cache(l), c->v_cache(l)};
    }
    CK(cudaMemcpy(c->d_layers, hl.data(), hl.size() * sizeof(DecodeLayer), cudaMemcpyHostToDevice));
    CK(dalloc(&c->ll_x, (size_t)sh.H));
    CK(dalloc(&c->ll_qkv, (size_t)sh.qkv_rows()));
    CK(dalloc(&c->ll_o, (size_t)sh.HQ * sh.D));
    CK(dalloc(&c->ll_h, (size_t)sh.F));
    CK(cudaMemset(c->ll_x, 0, (size_t)sh.H * 8));
    CK(cudaMemset(c->ll_qkv, 0, (size_t)sh.qkv_rows() * 8));
    CK(cudaMemset(c->ll_o, 0, (size_t)sh.HQ * sh.D * 8));
    CK(cudaMemset(c->ll_h, 0, (size_t)sh.F * 8));
    CK(dalloc(&c->attn_part, (size_t)sh.HQ * c->dp.max_chunks * (sh.D + 2)));
    CK(dalloc(&c->attn_count, (size_t)sh.NL * sh.HKV));
    CK(cudaMemset(c->attn_count, 0, (size_t)sh.NL * sh.HKV * sizeof(unsigned int)));
    CK(dalloc(&c->am_part, (size_t)c->dp.grid));
    CK(dalloc(&c->am_count, 1));
    CK(cudaMemset(c->am_count, 0, sizeof(unsigned int)));
    c->persistent_ok = true;
    c->decode_kernel = QDEC_DECODE_PERSISTENT;
    return QDEC_OK;
}

// QDEC_OPT_WEIGHTS: quantizes the layer matrices on the device into a shared copy (the
// decode step then runs its projections on it with the per-operation kernels), or drops it.
int set_weight_format(qdec_ctx* c, int fmt) {
    if (fmt != QDEC_WEIGHTS_BF16 && fmt != QDEC_WEIGHTS_Q8B32 && fmt != QDEC_WEIGHTS_Q4B32)
        return fail(QDEC_E_INVALID_ARG, "QDEC_OPT_WEIGHTS takes 0 (bf16), 1 (q8b32) or 2 (q4b32)");
    const Shape& sh = c->sh;
    if (fmt != QDEC_WEIGHTS_BF16 && (sh.H % 256 || (sh.HQ * sh.D) % 256 || sh.F % 256))
        return fail(QDEC_E_UNSUPPORTED, "quantized decode needs hidden, q width and ffn multiples of 256");
    if ((c->quant ? c->quant->fmt : 0) == fmt) return QDEC_OK;
    CK(cudaStreamSynchronize(c->stream));
    if (c->decode_exec) {   // the captured step reads the old weights
        cudaGraphExecDestroy(c->decode_exec);
        c->decode_exec = nullptr;
    }
    if (fmt == QDEC_WEIGHTS_BF16) {
        c->quant.reset();
        if (c->persistent_ok) c->decode_kernel = QDEC_DECODE_PERSISTENT;
        return QDEC_OK;
    }
    auto q = std::make_shared<QuantWeights>();
    q->fmt = fmt;
    q->layers.resize(sh.NL);
    const int qf = fmt == QDEC_WEIGHTS_Q8B32 ? QUANT_Q8B32 : QUANT_Q4B32;
    for (int l = 0; l < sh.NL; ++l) {
        const LayerW& w = c->layers[l];
        const bf16_t* mats[4] = {w.wqkv, w.wo, w.wgu, w.wd};
        const int rows[4] = {sh.qkv_rows(), sh.H, 2 * sh.F, sh.H};
        const int ks[4] = {sh.H, sh.HQ * sh.D, sh.H, sh.F};
        for (int m = 0; m < 4; ++m) {
            void *codes = nullptr, *scales = nullptr;
            CK(cudaMalloc(&codes, quant_code_bytes(qf, rows[m], ks[m])));
            q->bufs.push_back(codes);
            CK(cudaMalloc(&scales, quant_scale_bytes(rows[m], ks[m])));
            q->bufs.push_back(scales);
            CK(launch_quantize(mats[m], rows[m], ks[m], qf, codes, scales, c->stream));
            q->layers[l].c[m] = codes;
            q->layers[l].sc[m] = scales;
        }
    }
    CK(cudaStreamSynchronize(c->stream));
    c->quant = q;
    c->decode_kernel = QDEC_DECODE_GRAPH;
    return QDEC_OK;
}

// (cos, sin) of position p and NeoX pair i, by position ([max_seq][D/2]: the pairs of one
// position contiguous) and then by pair ([D/2][max_seq]: consecutive positions contiguous, for
// the prefill epilogue whose threads own consecutive positions).
int build_rope_table(qdec_ctx* c) {
    const int half = c->sh.D / 2, S = c->sh.max_seq;
    std::vector<float2> t(2 * (size_t)S * half);
    for (int p = 0; p < S; ++p)
        for (int i = 0; i < half; ++i) {
            const double inv = std::pow((double)c->cfg.rope_theta, -2.0 * i / (double)c->sh.D);
            const double a = (double)p * inv;
            const float2 v = make_float2((float)std::cos(a), (float)std::sin(a));
            t[(size_t)p * half + i] = v;
            t[(size_t)S * half + (size_t)i * S + p] = v;
        }
    CK(cudaMemcpy(c->rope, t.data(), t.size() * sizeof(float2), cudaMemcpyHostToDevice));
    return QDEC_OK;
}

int ensure_prefill_scratch(qdec_ctx* c, int T) {
    if (!c->p_part && c->prefill_gemm == QDEC_PREFILL_TCGEN05) {
        // partial slabs of a split GEMM: splits * M * N <= (SMs + tiles) * 128 * 128 with
        // tiles <= SMs / 2 (prefill_splits)
        const size_t cap = (size_t)2 * c->sms * 128 * 128;
        CK(dalloc(&c->p_part, cap));
        c->part_cap = cap;
    }
    if (T <= c->pf_cap) return QDEC_OK;
    c->drop_prefill_graphs();   // they hold the buffers about to be replaced
    const Shape& sh = c->sh;
    void* old[] = {c->p_X, c->p_qkv, c->p_Xn, c->p_Q, c->p_O, c->p_H, c->p_ids};
    CK(cudaStreamSynchronize(c->stream));
    for (void* p : old)
        if (p) cudaFree(p);
    c->p_X = c->p_qkv = nullptr;
    c->p_Xn = c->p_Q = c->p_O = c->p_H = nullptr;
    c->p_ids = nullptr;
    c->pf_cap = 0;
    CK(dalloc(&c->p_X, (size_t)T * sh.H));
    CK(dalloc(&c->p_qkv, (size_t)T * sh.qkv_rows()));
    CK(dalloc(&c->p_Xn, (size_t)T * sh.H));
    CK(dalloc(&c->p_Q, (size_t)T * sh.HQ * sh.D));
    CK(dalloc(&c->p_O, (size_t)T * sh.HQ * sh.D));
    CK(dalloc(&c->p_H, (size_t)T * sh.F));
    CK(dalloc(&c->p_ids, (size_t)T));
    c->pf_cap = T;
    return QDEC_OK;
}

int ensure_audio_staging(qdec_ctx* c, int n) {
    if (n <= c->audio_cap) return QDEC_OK;
    CK(cudaStreamSynchronize(c->stream));
    if (c->p_audio) cudaFree(c->p_audio);
    c->p_audio = nullptr;
    c->audio_cap = 0;
    CK(dalloc(&c->p_audio, (size_t)n * c->sh.H));
    c->audio_cap = n;
    return QDEC_OK;
}

// Copies the step's logits to the caller (host or device) on the context's stream.
int copy_logits_out(qdec_ctx* c, float* dst) {
    if (!dst) return QDEC_OK;
    CK(cudaMemcpyAsync(dst, c->d_logits, (size_t)c->sh.V * sizeof(float), cudaMemcpyDefault, c->stream));
    return QDEC_OK;
}

// Prefill GEMM: tcgen05 kernel where the shape allows it (and it is selected), else CUDA cores.
cudaError_t prefill_gemm(const qdec_ctx* c, const bf16_t* A, int lda, const bf16_t* W, int M, int N, int K, int mode,
                         int up_off, float* Cf, bf16_t* Cb, int ldc, cudaStream_t s) {
    if (c->prefill_gemm == QDEC_PREFILL_TCGEN05 && gemm_tc_supported(N, K, mode, lda))
        return launch_gemm_tc(A, lda, W, M, N, K, mode, up_off, Cf, Cb, ldc, s);
    return launch_gemm_simt(A, lda, W, M, N, K, mode, up_off, Cf, Cb, ldc, s);
}

// Split-K factor of a prefill GEMM on the tensor cores.  A short prompt has few 128 x 128
// output tiles (64 rows and o_proj's 1024 columns: 8 tiles for 152 SMs), so each tile's K is
// split over enough CTAs to fill the SMs once; split z stores an fp32 partial slab and the
// kernel that consumes the product adds the slabs in order (deterministic).  1 = no split.
int prefill_splits(const qdec_ctx* c, int M, int N, int K, int lda) {
    if (c->prefill_gemm != QDEC_PREFILL_TCGEN05 || !gemm_tc_supported(N, K, GEMM_PARTIAL_F32, lda)) return 1;
    const int tiles = ((M + 127) / 128) * (N / 128);
    if (2 * tiles > c->sms) return 1;
    const int sp = gemm_tc_splits(K, (c->sms + tiles - 1) / tiles);
    if ((size_t)sp * M * N > c->part_cap) return 1;
    return sp;
}

// One layer of the prefill over T rows starting at position 0.  *fold carries split-K
// partials of the previous down projection still to be added into the residual (0 = none);
// *kernels counts the launches.
int prefill_layer(qdec_ctx* c, int l, int T, int* fold, uint64_t* kernels, cudaStream_t s) {
    const Shape& sh = c->sh;
    const LayerW& w = c->layers[l];
    const int qd = sh.HQ * sh.D, nq = sh.qkv_rows();
    uint64_t k = 0;
    if (*fold > 1)
        CK(launch_rmsnorm_fold_bf16(c->p_X, c->p_part, *fold, (size_t)T * sh.H, T, sh.H, w.g_in, sh.eps, c->p_Xn, s));
    else
        CK(launch_rmsnorm_bf16(c->p_X, T, sh.H, w.g_in, sh.eps, c->p_Xn, s));
    *fold = 0;
    ++k;
    const int sq = prefill_splits(c, T, nq, sh.H, sh.H);
    if (sq > 1) {
        CK(launch_gemm_tc(c->p_Xn, sh.H, w.wqkv, T, nq, sh.H, GEMM_PARTIAL_F32, 0, c->p_part, nullptr, nq, s, sq));
        CK(launch_qk_norm_rope_append(c->p_part, T, sh, c->d_zero, w.g_q, w.g_k, c->rope, c->p_Q, nullptr,
                                      c->k_cache(l), c->v_cache(l), s, sq, (size_t)T * nq));
        k += 2;
    } else if (c->prefill_gemm == QDEC_PREFILL_TCGEN05 && gemm_tc_qkv_rope_supported(sh, sh.H)) {
        // QKV projection with the per-head norm, RoPE and KV append in its epilogue
        QkvRopeEpi e{c->rope, c->rope + (size_t)sh.max_seq * (sh.D / 2), w.g_q, w.g_k, c->p_Q, c->k_cache(l),
                     c->v_cache(l), 0, sh.HQ, sh.HKV, sh.max_seq, sh.eps};
        CK(launch_gemm_tc_qkv_rope(c->p_Xn, sh.H, w.wqkv, T, sh.H, e, s));
        k += 1;
    } else {
        CK(prefill_gemm(c, c->p_Xn, sh.H, w.wqkv, T, nq, sh.H, GEMM_STORE_F32, 0, c->p_qkv, nullptr, nq, s));
        CK(launch_qk_norm_rope_append(c->p_qkv, T, sh, c->d_zero, w.g_q, w.g_k, c->rope, c->p_Q, nullptr,
                                      c->k_cache(l), c->v_cache(l), s));
        k += 2;
    }
    if (c->prefill_gemm == QDEC_PREFILL_TCGEN05 && attention_tc_supported(sh))
        CK(launch_attention_prefill_tc(c->p_Q, T, sh, 0, c->k_cache(l), c->v_cache(l), c->p_O, s));
    else
        CK(launch_attention_prefill_simt(c->p_Q, T, sh, 0, c->k_cache(l), c->v_cache(l), c->p_O, s));
    ++k;
    const int so = prefill_splits(c, T, sh.H, qd, qd);
    if (so > 1) {   // o_proj partials, added into the residual by the post-attention norm
        CK(launch_gemm_tc(c->p_O, qd, w.wo, T, sh.H, qd, GEMM_PARTIAL_F32, 0, c->p_part, nullptr, sh.H, s, so));
        CK(launch_rmsnorm_fold_bf16(c->p_X, c->p_part, so, (size_t)T * sh.H, T, sh.H, w.g_post, sh.eps, c->p_Xn, s));
    } else {
        CK(prefill_gemm(c, c->p_O, qd, w.wo, T, sh.H, qd, GEMM_ADD_F32, 0, c->p_X, nullptr, sh.H, s));
        CK(launch_rmsnorm_bf16(c->p_X, T, sh.H, w.g_post, sh.eps, c->p_Xn, s));
    }
    k += 2;
    const int sg = prefill_splits(c, T, 2 * sh.F, sh.H, sh.H);
    if (sg > 1) {   // gate and up partials, summed by the SwiGLU kernel
        CK(launch_gemm_tc(c->p_Xn, sh.H, w.wgu, T, 2 * sh.F, sh.H, GEMM_PARTIAL_F32, 0, c->p_part, nullptr, 2 * sh.F,
                          s, sg));
        CK(launch_batch_swiglu(c->p_part, sh.F, T, c->p_H, s, sg, (size_t)T * 2 * sh.F));
        k += 2;
    } else {
        CK(prefill_gemm(c, c->p_Xn, sh.H, w.wgu, T, sh.F, sh.H, GEMM_SWIGLU_BF16, sh.F, nullptr, c->p_H, sh.F, s));
        k += 1;
    }
    const int sd = prefill_splits(c, T, sh.H, sh.F, sh.F);
    if (sd > 1) {   // down partials: added by the next layer's norm (or after the last layer)
        CK(launch_gemm_tc(c->p_H, sh.F, w.wd, T, sh.H, sh.F, GEMM_PARTIAL_F32, 0, c->p_part, nullptr, sh.H, s, sd));
        *fold = sd;
    } else {
        CK(prefill_gemm(c, c->p_H, sh.F, w.wd, T, sh.H, sh.F, GEMM_ADD_F32, 0, c->p_X, nullptr, sh.H, s));
    }
    k += 1;
    *kernels += k;
    return QDEC_OK;
}

// Queues the decode step body (everything after the token embedding) on stream s.
int enqueue_decode_body(qdec_ctx* c, cudaStream_t s) {
    const Shape& sh = c->sh;
    for (int l = 0; l < sh.NL; ++l) {
        const LayerW& w = c->layers[l];
        const QuantWeights::Layer* ql = c->quant ? &c->quant->layers[l] : nullptr;
        const int qf = c->quant ? c->quant->fmt : 0;
        if (ql)
            CK(launch_gemv_q(ql->c[0], ql->sc[0], qf, sh.qkv_rows(), sh.H, c->d_x, w.g_in, sh.eps, GEMV_STORE, 0,
                             c->d_qkv, s));
        else
            CK(launch_gemv(w.wqkv, sh.qkv_rows(), sh.H, c->d_x, w.g_in, sh.eps, GEMV_STORE, 0, c->d_qkv, s));
        CK(launch_qk_norm_rope_append(c->d_qkv, 1, sh, c->d_pos, w.g_q, w.g_k, c->rope, nullptr, c->d_q,
                                      c->k_cache(l), c->v_cache(l), s));
        CK(launch_attention_decode(c->d_q, sh, c->d_pos, c->k_cache(l), c->v_cache(l), c->n_split, c->d_part_ml,
                                   c->d_part_o, c->d_attn, s));
        if (ql) {
            CK(launch_gemv_q(ql->c[1], ql->sc[1], qf, sh.H, sh.HQ * sh.D, c->d_attn, nullptr, sh.eps, GEMV_ADD, 0,
                             c->d_x, s));
            CK(launch_gemv_q(ql->c[2], ql->sc[2], qf, sh.F, sh.H, c->d_x, w.g_post, sh.eps, GEMV_SWIGLU, sh.F, c->d_h,
                             s));
            CK(launch_gemv_q(ql->c[3], ql->sc[3], qf, sh.H, sh.F, c->d_h, nullptr, sh.eps, GEMV_ADD, 0, c->d_x, s));
        } else {
            CK(launch_gemv(w.wo, sh.H, sh.HQ * sh.D, c->d_attn, nullptr, sh.eps, GEMV_ADD, 0, c->d_x, s));
            CK(launch_gemv(w.wgu, sh.F, sh.H, c->d_x, w.g_post, sh.eps, GEMV_SWIGLU, sh.F, c->d_h, s));
            CK(launch_gemv(w.wd, sh.H, sh.F, c->d_h, nullptr, sh.eps, GEMV_ADD, 0, c->d_x, s));
        }
    }
    CK(launch_lm_head_argmax(c->embed, sh.V, sh.H, c->d_x, c->final_norm, sh.eps, c->d_logits, c->d_argmax,
                             c->d_lm_scratch, s));
    CK(launch_advance_position(c->d_pos, 1, s));
    return QDEC_OK;
}

int ensure_decode_graph(qdec_ctx* c) {
    if (c->decode_exec) return QDEC_OK;
    cudaGraph_t g = nullptr;
    CK(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    int rc = enqueue_decode_body(c, c->cap_stream);
    cudaError_t e = cudaStreamEndCapture(c->cap_stream, &g);
    if (rc != QDEC_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    CK(e);
    size_t n_nodes = 0;
    e = cudaGraphGetNodes(g, nullptr, &n_nodes);
    if (e == cudaSuccess) {
        std::vector<cudaGraphNode_t> nodes(n_nodes);
        e = cudaGraphGetNodes(g, nodes.data(), &n_nodes);
        c->decode_graph_kernels = 0;
        for (size_t i = 0; e == cudaSuccess && i < n_nodes; ++i) {
            cudaGraphNodeType t;
            e = cudaGraphNodeGetType(nodes[i], &t);
            if (t == cudaGraphNodeTypeKernel) ++c->decode_graph_kernels;
        }
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&c->decode_exec, g, 0);
    cudaGraphDestroy(g);
    CK(e);
    return QDEC_OK;
}

// Queues one decode step (no host synchronisation).
int enqueue_decode_step(qdec_ctx* c, int token) {
    if (c->decode_kernel == QDEC_DECODE_PERSISTENT) {
        const Shape& sh = c->sh;
        DecodeParams p{};
        p.layers = c->d_layers;
        p.embed = c->embed;
        p.final_norm = c->final_norm;
        p.rope = c->rope;
        p.H = sh.H; p.NL = sh.NL; p.HQ = sh.HQ; p.HKV = sh.HKV; p.D = sh.D; p.F = sh.F; p.V = sh.V;
        p.max_seq = sh.max_seq;
        p.eps = sh.eps;
        p.pos = c->position;
        p.token = token;
        p.epoch = ++c->epoch;
        decode_persistent_chunks(c->dp, c->position + 1, c->attn_unit_keys, &p.n_chunks, &p.chunk);
        p.argmax = c->d_argmax;
        p.pos_out = c->d_pos;
        p.history = c->d_hist;
        p.logits = c->d_logits;
        p.ll_x = c->ll_x; p.ll_qkv = c->ll_qkv; p.ll_o = c->ll_o; p.ll_h = c->ll_h;
        p.attn_part = c->attn_part;
        p.attn_count = c->attn_count;
        p.am_part = c->am_part;
        p.am_count = c->am_count;
        p.err = c->d_err;
        p.spin_limit = c->spin_limit > 0 ? (uint32_t)c->spin_limit : kDecodeSpinDefault;
        p.trace = c->d_trace;
        if (p.trace)
            CK(cudaMemsetAsync(p.trace, 0, (size_t)c->dp.grid * (11 * sh.NL + 8) * sizeof(unsigned long long),
                               c->stream));
        CK(launch_decode_persistent(p, c->dp, c->stream));
        count_launches(1);
        return QDEC_OK;
    }
    int rc = ensure_decode_graph(c);
    if (rc != QDEC_OK) return rc;
    CK(launch_embed_token(c->embed, token, c->d_argmax, c->d_pos, c->sh.H, c->d_x, c->d_hist, c->stream));
    CK(cudaGraphLaunch(c->decode_exec, c->stream));
    count_launches(1 + c->decode_graph_kernels);
    return QDEC_OK;
}

// Reads the step's argmax and the persistent kernel's error word into the pinned staging
// (slots [s], [s+1]) and waits.  A device-side timeout is reported as QDEC_E_TIMEOUT and
// the error word is cleared.
int sync_status(qdec_ctx* c, int s, int* argmax) {
    CK(cudaMemcpyAsync(&c->h_pinned[s], c->d_argmax, 2 * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    if (c->h_pinned[s + 1] != 0) {
        const int code = c->h_pinned[s + 1];
        CK(cudaMemsetAsync(c->d_err, 0, sizeof(int), c->stream));
        CK(cudaStreamSynchronize(c->stream));
        return fail(QDEC_E_TIMEOUT, "decode kernel gave up waiting (device error code %d)", code);
    }
    const int tc = tc_error_read_and_clear(), fa = fa_error_read_and_clear();
    if (tc > 0 || fa > 0)
        return fail(QDEC_E_TIMEOUT, "a tensor-core prefill kernel gave up waiting (codes %d, %d)", tc, fa);
    if (argmax) *argmax = c->h_pinned[s];
    return QDEC_OK;
}

int check_decode_args(const qdec_ctx* c, int token) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    if (!c->prefilled) return fail(QDEC_E_STATE, "decode before prefill");
    if (c->position >= c->sh.max_seq)
        return fail(QDEC_E_CAPACITY, "position %d reached max_seq %d", c->position, c->sh.max_seq);
    if (token < -1 || token >= c->sh.V) return fail(QDEC_E_INVALID_ARG, "token %d out of range", token);
    return QDEC_OK;
}

// ---------------------------------------------------------------- lockstep batch
int ensure_batch_work(qdec_ctx* const* ctxs, int n) {
    qdec_ctx* c0 = ctxs[0];
    const Shape& sh = c0->sh;
    if (!c0->batch) c0->batch = new (std::nothrow) BatchWork();
    if (!c0->batch) return fail(QDEC_E_OOM, "host allocation failed");
    BatchWork& b = *c0->batch;
    if (n > b.cap) {
        CK(cudaStreamSynchronize(c0->stream));
        b.release();
        const int target = 4 * c0->sms;
        int ns = (target + sh.HKV * n - 1) / (sh.HKV * n);
        b.n_split = ns < 1 ? 1 : (ns > 32 ? 32 : ns);
        const size_t qd = (size_t)sh.HQ * sh.D;
        CK(dalloc(&b.d_streams, (size_t)n));
        CK(dalloc(&b.d_tokens, (size_t)n));
        CK(dalloc(&b.d_am, (size_t)n));
        CK(cudaMallocHost(reinterpret_cast<void**>(&b.h_am), (size_t)n * sizeof(int)));
        CK(cudaMallocHost(reinterpret_cast<void**>(&b.h_tokens), (size_t)2 * n * sizeof(int)));
        for (cudaEvent_t& e : b.tok_ev) CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        CK(dalloc(&b.X, (size_t)n * sh.H));
        CK(dalloc(&b.Xn, (size_t)n * sh.H));
        CK(dalloc(&b.qkv, (size_t)n * sh.qkv_rows()));
        CK(dalloc(&b.q, (size_t)n * qd));
        b.split_cap = b.n_split + (prefix_attention_supported(sh) ? prefix_chunks(sh.max_seq) : 0);
        CK(dalloc(&b.part_ml, (size_t)n * sh.HQ * b.split_cap * 2));
        CK(dalloc(&b.part_o, (size_t)n * sh.HQ * b.split_cap * sh.D));
        CK(dalloc(&b.d_members, (size_t)n));
        CK(dalloc(&b.d_items, (size_t)n));
        CK(dalloc(&b.attn, (size_t)n * qd));
        CK(dalloc(&b.gu, (size_t)n * 2 * sh.F));
        CK(dalloc(&b.h, (size_t)n * sh.F));
        CK(dalloc(&b.logits, (size_t)n * sh.V));
        b.cap = n;
    }
    const int want_shared = (c0->shared_prefix && prefix_attention_supported(sh)) ? 1 : 0;
    bool same = (int)b.members.size() == n && b.shared_setting == want_shared;
    for (int i = 0; same && i < n; ++i) same = b.members[i] == ctxs[i] && b.member_prefix[i] == ctxs[i]->prefix_id;
    if (!same) {
        b.drop_graph();
        b.members.assign(ctxs, ctxs + n);
        b.member_prefix.resize(n);
        for (int i = 0; i < n; ++i) b.member_prefix[i] = ctxs[i]->prefix_id;
        b.shared_setting = want_shared;
        // streams grouped by the prefill their prefix comes from; a group of two or more shares
        // [0, P) with P the smallest inherited length among its members
        std::vector<int> shared(n, 0), members;
        std::vector<PrefixItem> items;
        int max_chunks = 0;
        if (want_shared) {
            std::map<unsigned long long, std::vector<int>> groups;
            for (int i = 0; i < n; ++i)
                if (ctxs[i]->prefix_id != 0 && ctxs[i]->inherited > 0) groups[ctxs[i]->prefix_id].push_back(i);
            const int per_item = prefix_item_streams(sh);
            for (auto& kv : groups) {
                const std::vector<int>& g = kv.second;
                if (g.size() < 2) continue;
                int P = ctxs[g[0]]->inherited;
                for (int i : g) P = ctxs[i]->inherited < P ? ctxs[i]->inherited : P;
                for (size_t a = 0; a < g.size(); a += per_item) {
                    const int cnt = (int)(g.size() - a) < per_item ? (int)(g.size() - a) : per_item;
                    items.push_back(PrefixItem{ctxs[g[0]]->kv, P, (int)members.size(), cnt});
                    for (int k = 0; k < cnt; ++k) members.push_back(g[a + k]);
                }
                for (int i : g) shared[i] = P;
                max_chunks = prefix_chunks(P) > max_chunks ? prefix_chunks(P) : max_chunks;
            }
        }
        if (b.n_split + max_chunks > b.split_cap) return fail(QDEC_E_UNSUPPORTED, "shared prefix longer than max_seq");
        b.n_items = (int)items.size();
        b.max_chunks = max_chunks;
        std::vector<BatchStream> hs(n);
        for (int i = 0; i < n; ++i)
            hs[i] = BatchStream{ctxs[i]->kv, ctxs[i]->d_pos, ctxs[i]->d_argmax, ctxs[i]->d_hist, ctxs[i]->rope,
                                ctxs[i]->sh.max_seq, shared[i]};
        CK(cudaMemcpyAsync(b.d_streams, hs.data(), n * sizeof(BatchStream), cudaMemcpyHostToDevice, c0->stream));
        if (!items.empty()) {
            CK(cudaMemcpyAsync(b.d_items, items.data(), items.size() * sizeof(PrefixItem), cudaMemcpyHostToDevice,
                               c0->stream));
            CK(cudaMemcpyAsync(b.d_members, members.data(), members.size() * sizeof(int), cudaMemcpyHostToDevice,
                               c0->stream));
        }
        CK(cudaStreamSynchronize(c0->stream));   // host vectors go out of scope
    }
    return QDEC_OK;
}

// C[n, N] = A . W^T, stored (accumulate = false) or added into C: tcgen05 with split-K fp32
// atomics where the shape allows it (the few-row batch GEMM needs the extra CTAs), CUDA cores
// otherwise.
int batch_gemm(qdec_ctx* c, const bf16_t* A, int lda, const bf16_t* W, int M, int N, int K, bool accumulate,
               float* C, int ldc, cudaStream_t s) {
    if (c->prefill_gemm == QDEC_PREFILL_TCGEN05 && gemm_tc_supported(N, K, GEMM_ATOMIC_F32, lda)) {
        if (!accumulate) CK(cudaMemsetAsync(C, 0, (size_t)M * ldc * sizeof(float), s));
        const int tiles = (N / 128) * ((M + 127) / 128);
        const int splits = (2 * c->sms + tiles - 1) / tiles;
        CK(launch_gemm_tc(A, lda, W, M, N, K, GEMM_ATOMIC_F32, 0, C, nullptr, ldc, s, splits));
        return QDEC_OK;
    }
    CK(launch_gemm_simt(A, lda, W, M, N, K, accumulate ? GEMM_ADD_F32 : GEMM_STORE_F32, 0, C, nullptr, ldc, s));
    return QDEC_OK;
}

// The kernels of one lockstep step, reading d_tokens and writing b.logits and d_am; returns
// the number of kernels launched through *kernels.
int batch_body(qdec_ctx* c0, int n, cudaStream_t s, uint64_t* kernels) {
    const Shape& sh = c0->sh;
    BatchWork& b = *c0->batch;
    int rc;
    CK(launch_batch_embed(c0->embed, sh.H, b.d_tokens, b.d_streams, n, b.X, s));
    const int qd = sh.HQ * sh.D;
    uint64_t k = 1;
    for (int l = 0; l < sh.NL; ++l) {
        const LayerW& w = c0->layers[l];
        CK(launch_rmsnorm_bf16(b.X, n, sh.H, w.g_in, sh.eps, b.Xn, s));
        if ((rc = batch_gemm(c0, b.Xn, sh.H, w.wqkv, n, sh.qkv_rows(), sh.H, false, b.qkv, sh.qkv_rows(), s))) return rc;
        CK(launch_batch_qk_rope(b.qkv, sh, l, w.g_q, w.g_k, b.d_streams, n, b.q, s));
        CK(launch_batch_attention(b.q, sh, l, b.d_streams, n, b.n_split, b.d_items, b.n_items, b.d_members,
                                  b.max_chunks, b.part_ml, b.part_o, b.attn, s));
        if ((rc = batch_gemm(c0, b.attn, qd, w.wo, n, sh.H, qd, true, b.X, sh.H, s))) return rc;
        CK(launch_rmsnorm_bf16(b.X, n, sh.H, w.g_post, sh.eps, b.Xn, s));
        if ((rc = batch_gemm(c0, b.Xn, sh.H, w.wgu, n, 2 * sh.F, sh.H, false, b.gu, 2 * sh.F, s))) return rc;
        CK(launch_batch_swiglu(b.gu, sh.F, n, b.h, s));
        if ((rc = batch_gemm(c0, b.h, sh.F, w.wd, n, sh.H, sh.F, true, b.X, sh.H, s))) return rc;
        k += 10;
    }
    CK(launch_rmsnorm_bf16(b.X, n, sh.H, c0->final_norm, sh.eps, b.Xn, s));
    if ((rc = batch_gemm(c0, b.Xn, sh.H, c0->embed, n, sh.V, sh.H, false, b.logits, sh.V, s))) return rc;
    CK(launch_batch_argmax(b.logits, sh.V, sh.V, b.d_streams, n, b.d_am, s));
    *kernels = k + 3;
    return QDEC_OK;
}

// Captures batch_body into b.exec on the context's capture stream.
int capture_batch(qdec_ctx* c0, int n) {
    BatchWork& b = *c0->batch;
    cudaGraph_t g = nullptr;
    uint64_t kernels = 0;
    CK(cudaStreamBeginCapture(c0->cap_stream, cudaStreamCaptureModeThreadLocal));
    int rc = batch_body(c0, n, c0->cap_stream, &kernels);
    cudaError_t e = cudaStreamEndCapture(c0->cap_stream, &g);
    if (rc != QDEC_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    CK(e);
    e = cudaGraphInstantiate(&b.exec, g, 0);
    cudaGraphDestroy(g);
    CK(e);
    b.graph_kernels = kernels;
    b.graph_impl = c0->prefill_gemm;
    return QDEC_OK;
}

int batch_step(qdec_ctx* const* ctxs, int n, const int32_t* tokens, float* logits_out, int32_t* argmax_out) {
    qdec_ctx* c0 = ctxs[0];
    const Shape& sh = c0->sh;
    cudaStream_t s = c0->stream;
    // order against work queued on the other contexts' streams
    std::vector<cudaEvent_t> evs;
    for (int i = 1; i < n; ++i) {
        if (ctxs[i]->stream == s) continue;
        cudaEvent_t e;
        CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        evs.push_back(e);
        CK(cudaEventRecord(e, ctxs[i]->stream));
        CK(cudaStreamWaitEvent(s, e, 0));
    }
    int rc = ensure_batch_work(ctxs, n);
    if (rc != QDEC_OK) return rc;
    BatchWork& b = *c0->batch;
    if (b.exec && b.graph_impl != c0->prefill_gemm) b.drop_graph();
    // two pinned staging buffers: wait only for the upload that last used this one
    int* ht = b.h_tokens + (size_t)b.tok_slot * b.cap;
    CK(cudaEventSynchronize(b.tok_ev[b.tok_slot]));
    memcpy(ht, tokens, (size_t)n * sizeof(int));
    CK(cudaMemcpyAsync(b.d_tokens, ht, (size_t)n * sizeof(int), cudaMemcpyHostToDevice, s));
    CK(cudaEventRecord(b.tok_ev[b.tok_slot], s));
    b.tok_slot ^= 1;
    if (!b.exec && b.steps_same >= 1) {
        rc = capture_batch(c0, n);
        if (rc != QDEC_OK) return rc;
    }
    if (b.exec) {
        CK(cudaGraphLaunch(b.exec, s));
        count_launches(b.graph_kernels);
    } else {
        uint64_t kernels = 0;
        if ((rc = batch_body(c0, n, s, &kernels))) return rc;
        count_launches(kernels);
    }
    ++b.steps_same;
    for (int i = 0; i < n; ++i) ctxs[i]->position += 1;
    if (logits_out)
        CK(cudaMemcpyAsync(logits_out, b.logits, (size_t)n * sh.V * sizeof(float), cudaMemcpyDefault, s));
    for (cudaEvent_t e : evs) {   // the other streams wait for the batch before their next work
        CK(cudaEventRecord(e, s));
    }
    int k = 0;
    for (int i = 1; i < n; ++i) {
        if (ctxs[i]->stream == s) continue;
        CK(cudaStreamWaitEvent(ctxs[i]->stream, evs[k++], 0));
    }
    for (cudaEvent_t e : evs) cudaEventDestroy(e);
    if (argmax_out) {
        CK(cudaMemcpyAsync(b.h_am, b.d_am, (size_t)n * sizeof(int), cudaMemcpyDeviceToHost, s));
        rc = sync_status(c0, 6, nullptr);
        if (rc != QDEC_OK) return rc;
        for (int i = 0; i < n; ++i) argmax_out[i] = b.h_am[i];
    }
    return QDEC_OK;
}

}  // namespace

extern "C" {

int qdec_create(const qdec_config* cfg, const qdec_weights* w, void* cuda_stream, qdec_ctx** out) {
    if (!cfg || !w || !out) return fail(QDEC_E_INVALID_ARG, "null argument");
    *out = nullptr;
    int rc = validate_config(cfg);
    if (rc != QDEC_OK) return rc;
    if (!w->embed || !w->final_norm || !w->wqkv || !w->wo || !w->wgu || !w->wd || !w->g_in || !w->g_post ||
        !w->g_q || !w->g_k)
        return fail(QDEC_E_INVALID_ARG, "null weight pointer");
    for (int l = 0; l < cfg->n_layers; ++l) {
        const void* ps[] = {w->wqkv[l], w->wo[l], w->wgu[l], w->wd[l], w->g_in[l], w->g_post[l], w->g_q[l], w->g_k[l]};
        for (const void* p : ps) {
            if (!p) return fail(QDEC_E_INVALID_ARG, "null weight pointer in layer %d", l);
            if (!aligned16(p)) return fail(QDEC_E_INVALID_ARG, "weight pointer of layer %d not 16-byte aligned", l);
        }
    }
    if (!aligned16(w->embed) || !aligned16(w->final_norm))
        return fail(QDEC_E_INVALID_ARG, "embed / final_norm not 16-byte aligned");
    qdec_ctx* c = new (std::nothrow) qdec_ctx();
    if (!c) return fail(QDEC_E_OOM, "host allocation failed");
    c->cfg = *cfg;
    c->sh = Shape{cfg->hidden, cfg->n_layers, cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim, cfg->ffn,
                  cfg->vocab, cfg->max_seq, cfg->rope_theta, cfg->rms_eps};
    c->embed = static_cast<const bf16_t*>(w->embed);
    c->final_norm = static_cast<const bf16_t*>(w->final_norm);
    c->layers.resize(cfg->n_layers);
    for (int l = 0; l < cfg->n_layers; ++l)
        c->layers[l] = LayerW{static_cast<const bf16_t*>(w->wqkv[l]), static_cast<const bf16_t*>(w->wo[l]),
                              static_cast<const bf16_t*>(w->wgu[l]), static_cast<const bf16_t*>(w->wd[l]),
                              static_cast<const bf16_t*>(w->g_in[l]), static_cast<const bf16_t*>(w->g_post[l]),
                              static_cast<const bf16_t*>(w->g_q[l]), static_cast<const bf16_t*>(w->g_k[l])};
    if (cuda_stream) {
        c->stream = static_cast<cudaStream_t>(cuda_stream);
    } else {
        auto owner = std::make_shared<OwnedStream>();
        cudaError_t e = cudaStreamCreateWithFlags(&owner->s, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            owner->s = nullptr;
            delete c;
            return fail(QDEC_E_CUDA, "cudaStreamCreate: %s", cudaGetErrorString(e));
        }
        c->stream = owner->s;
        c->stream_owner = owner;
    }
    rc = alloc_state(c);
    if (rc == QDEC_OK) rc = build_rope_table(c);
    if (rc != QDEC_OK) {
        free_all(c);
        delete c;
        return rc;
    }
    *out = c;
    return QDEC_OK;
}

}  // extern "C"

namespace {

// The prefill after the embedding: the layers, the fold of the last split-K partials, the
// tied head on the last row and the device position, queued on s.
int prefill_body(qdec_ctx* c, int T, cudaStream_t s, uint64_t* kernels) {
    const Shape& sh = c->sh;
    uint64_t k = 2;   // lm_head, position
    int fold = 0;
    for (int l = 0; l < sh.NL; ++l) {
        const int rc = prefill_layer(c, l, T, &fold, &k, s);
        if (rc != QDEC_OK) return rc;
    }
    if (fold > 1) {   // the last down projection's partials, for the row the head reads
        const size_t last = (size_t)(T - 1) * sh.H;
        CK(launch_fold_partials(c->p_X + last, c->p_part + last, fold, (size_t)T * sh.H, (size_t)sh.H, s));
        ++k;
    }
    CK(launch_lm_head_argmax(c->embed, sh.V, sh.H, c->p_X + (size_t)(T - 1) * sh.H, c->final_norm, sh.eps,
                             c->d_logits, c->d_argmax, c->d_lm_scratch, s));
    CK(launch_set_int(c->d_pos, T, s));
    *kernels += k;
    return QDEC_OK;
}

// Runs the prefill body on the context's stream: eagerly the first time a (length,
// implementation, tile width) key is seen, from a CUDA graph captured on the second and
// replayed after that (about 250 launches for a short prompt become one).
int prefill_run_body(qdec_ctx* c, int T, uint64_t* kernels) {
    // the forced tile settings and the launch attribute key the graph
    const int tile = gemm_tile_width() + 1000 * gemm_tile_rows() + 1000000 * (programmatic_launch() ? 1 : 0);
    qdec_ctx::PrefillGraph* g = nullptr;
    for (auto& e : c->pf_graphs)
        if (e.T == T && e.impl == c->prefill_gemm && e.tile == tile) g = &e;
    if (g && g->exec) {
        CK(cudaGraphLaunch(g->exec, c->stream));
        *kernels += g->kernels;
        return QDEC_OK;
    }
    if (!g) {
        if (c->pf_graphs.size() >= 8) {   // keep a few keys; forget the oldest
            if (c->pf_graphs.front().exec) cudaGraphExecDestroy(c->pf_graphs.front().exec);
            c->pf_graphs.erase(c->pf_graphs.begin());
        }
        c->pf_graphs.push_back(qdec_ctx::PrefillGraph{T, c->prefill_gemm, tile, 0, nullptr, 0});
        g = &c->pf_graphs.back();
    }
    if (g->uses++ == 0) return prefill_body(c, T, c->stream, kernels);   // first use: eager
    cudaGraph_t graph = nullptr;
    uint64_t k = 0;
    CK(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    int rc = prefill_body(c, T, c->cap_stream, &k);
    cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
    if (rc != QDEC_OK) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&g->exec, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        g->exec = nullptr;
        cudaGetLastError();
        return prefill_body(c, T, c->stream, kernels);   // could not capture: run eagerly
    }
    g->kernels = k;
    CK(cudaGraphLaunch(g->exec, c->stream));
    *kernels += k;
    return QDEC_OK;
}

}  // namespace

extern "C" {

int qdec_prefill(qdec_ctx* c, const int32_t* ids, int32_t n_ids, const void* audio_rows, int32_t n_audio,
                 int32_t audio_offset, float* logits_out, int32_t* argmax_out) {
    if (!c || !ids) return fail(QDEC_E_INVALID_ARG, "null context or ids");
    if (n_ids <= 0) return fail(QDEC_E_INVALID_ARG, "n_ids must be positive");
    if (n_ids > c->sh.max_seq) return fail(QDEC_E_CAPACITY, "prompt of %d exceeds max_seq %d", n_ids, c->sh.max_seq);
    if (n_audio < 0 || audio_offset < 0 || (int64_t)audio_offset + n_audio > n_ids)
        return fail(QDEC_E_INVALID_ARG, "audio rows [%d, %d) outside the prompt of %d", audio_offset,
                    audio_offset + n_audio, n_ids);
    if (n_audio > 0 && !audio_rows) return fail(QDEC_E_INVALID_ARG, "null audio rows");
    for (int i = 0; i < n_ids; ++i)
        if (ids[i] < 0 || ids[i] >= c->sh.V) return fail(QDEC_E_INVALID_ARG, "id %d at %d out of range", ids[i], i);
    const Shape& sh = c->sh;
    const int T = n_ids;
    int rc = ensure_prefill_scratch(c, T);
    if (rc != QDEC_OK) return rc;
    cudaStream_t s = c->stream;
    CK(cudaMemcpyAsync(c->p_ids, ids, (size_t)T * sizeof(int), cudaMemcpyHostToDevice, s));
    const bf16_t* audio = nullptr;
    if (n_audio > 0) {
        if (is_device_ptr(audio_rows) && aligned16(audio_rows)) {
            audio = static_cast<const bf16_t*>(audio_rows);
        } else {
            rc = ensure_audio_staging(c, n_audio);
            if (rc != QDEC_OK) return rc;
            CK(cudaMemcpyAsync(c->p_audio, audio_rows, (size_t)n_audio * sh.H * sizeof(bf16_t), cudaMemcpyDefault, s));
            audio = c->p_audio;
        }
    }
    c->prefilled = false;
    c->position = 0;
    CK(launch_embed_splice(c->embed, c->p_ids, T, sh.H, audio, n_audio, audio_offset, c->p_X, c->d_hist, s));
    uint64_t kernels = 1;
    rc = prefill_run_body(c, T, &kernels);
    if (rc != QDEC_OK) return rc;
    if (c->sampling()) {   // the first generated token is drawn at the last prompt position
        CK(launch_sample(c->d_logits, sh.V, c->d_hist, T, c->samp_t, c->samp_k, c->samp_p, c->samp_r, c->samp_seed,
                         T - 1, c->d_argmax, s));
        ++kernels;
    }
    count_launches(kernels);
    c->position = T;
    c->prefilled = true;
    c->prefix_id = ++g_prefix_ids;
    c->inherited = T;
    rc = copy_logits_out(c, logits_out);
    if (rc != QDEC_OK) return rc;
    if (argmax_out) return sync_status(c, 0, argmax_out);
    return QDEC_OK;
}

int qdec_decode_step(qdec_ctx* c, int32_t token, float* logits_out, int32_t* argmax_out) {
    int rc = check_decode_args(c, token);
    if (rc != QDEC_OK) return rc;
    rc = enqueue_decode_step(c, token);
    if (rc != QDEC_OK) return rc;
    if (c->sampling()) {   // replaces the step's argmax; the history holds positions 0 .. position
        CK(launch_sample(c->d_logits, c->sh.V, c->d_hist, c->position + 1, c->samp_t, c->samp_k, c->samp_p,
                         c->samp_r, c->samp_seed, c->position, c->d_argmax, c->stream));
        count_launches(1);
    }
    c->position += 1;
    rc = copy_logits_out(c, logits_out);
    if (rc != QDEC_OK) return rc;
    if (!argmax_out) return QDEC_OK;
    rc = sync_status(c, 0, argmax_out);
    // A step that gave up on a wait advanced nothing on the device (position, argmax); the
    // host position follows, so the same step can be run again and rewrites its KV slot.
    if (rc == QDEC_E_TIMEOUT) c->position -= 1;
    return rc;
}

int qdec_decode_step_batch(qdec_ctx* const* ctxs, int32_t n, const int32_t* tokens, float* logits_out,
                           int32_t* argmax_out) {
    if (!ctxs || !tokens || n <= 0) return fail(QDEC_E_INVALID_ARG, "null contexts/tokens or n <= 0");
    for (int i = 0; i < n; ++i) {
        int rc = check_decode_args(ctxs[i], tokens[i]);
        if (rc != QDEC_OK) return rc;
        if (ctxs[i]->embed != ctxs[0]->embed || memcmp(&ctxs[i]->cfg, &ctxs[0]->cfg, sizeof(qdec_config)) != 0 ||
            ctxs[i]->device != ctxs[0]->device)
            return fail(QDEC_E_STATE, "batch contexts differ in weights, shape or device");
        for (int j = 0; j < i; ++j)
            if (ctxs[j] == ctxs[i]) return fail(QDEC_E_INVALID_ARG, "context %d repeated in the batch", i);
        if (n > 1 && ctxs[i]->sampling())
            return fail(QDEC_E_UNSUPPORTED, "the lockstep batch step is greedy: context %d samples", i);
        if (n > 1 && ctxs[i]->quant)
            return fail(QDEC_E_UNSUPPORTED, "the lockstep batch step reads bf16 weights: context %d is quantized", i);
    }
    if (n == 1) return qdec_decode_step(ctxs[0], tokens[0], logits_out, argmax_out);
    return batch_step(ctxs, n, tokens, logits_out, argmax_out);
}

int qdec_clone(const qdec_ctx* src, qdec_ctx** out) {
    if (!src || !out) return fail(QDEC_E_INVALID_ARG, "null argument");
    *out = nullptr;
    qdec_ctx* c = new (std::nothrow) qdec_ctx();
    if (!c) return fail(QDEC_E_OOM, "host allocation failed");
    c->cfg = src->cfg;
    c->sh = src->sh;
    c->embed = src->embed;
    c->final_norm = src->final_norm;
    c->layers = src->layers;
    c->stream = src->stream;
    c->stream_owner = src->stream_owner;   // keeps a library-created stream alive while any clone uses it
    int rc = alloc_state(c);
    if (rc == QDEC_OK) {
        const Shape& sh = c->sh;
        const size_t L = (size_t)src->position;
        cudaError_t e = cudaSuccess;
        if (L > 0) {
            const size_t row = (size_t)sh.max_seq * sh.D * sizeof(bf16_t);   // one (layer, kind, head) block
            e = cudaMemcpy2DAsync(c->kv, row, src->kv, row, L * sh.D * sizeof(bf16_t), (size_t)sh.NL * 2 * sh.HKV,
                                  cudaMemcpyDeviceToDevice, c->stream);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(c->d_hist, src->d_hist, L * sizeof(int), cudaMemcpyDeviceToDevice, c->stream);
        }
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(c->rope, src->rope, 2 * (size_t)sh.max_seq * (sh.D / 2) * sizeof(float2),
                                cudaMemcpyDeviceToDevice, c->stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync(c->d_pos, src->d_pos, sizeof(int), cudaMemcpyDeviceToDevice, c->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(c->d_argmax, src->d_argmax, sizeof(int), cudaMemcpyDeviceToDevice, c->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
        if (e != cudaSuccess) rc = fail(QDEC_E_CUDA, "clone copy: %s", cudaGetErrorString(e));
    }
    if (rc != QDEC_OK) {
        free_all(c);
        delete c;
        return rc;
    }
    c->position = src->position;
    c->prefilled = src->prefilled;
    if (c->persistent_ok) c->decode_kernel = src->decode_kernel;
    c->prefill_gemm = src->prefill_gemm;
    c->attn_unit_keys = src->attn_unit_keys;
    c->spin_limit = src->spin_limit;
    c->shared_prefix = src->shared_prefix;
    c->quant = src->quant;
    c->prefix_id = src->prefix_id;
    c->inherited = src->inherited < src->position ? src->inherited : src->position;
    c->samp_t = src->samp_t; c->samp_p = src->samp_p; c->samp_r = src->samp_r; c->samp_k = src->samp_k;
    c->samp_seed = src->samp_seed;
    *out = c;
    return QDEC_OK;
}

int qdec_position(const qdec_ctx* c) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    return c->position;
}

int qdec_read_kv(const qdec_ctx* c, int32_t layer, int32_t kind, int32_t pos0, int32_t n_pos, void* host_dst) {
    if (!c || !host_dst) return fail(QDEC_E_INVALID_ARG, "null argument");
    const Shape& sh = c->sh;
    if (layer < 0 || layer >= sh.NL || (kind != 0 && kind != 1) || pos0 < 0 || n_pos <= 0 ||
        (int64_t)pos0 + n_pos > sh.max_seq)
        return fail(QDEC_E_INVALID_ARG, "bad layer/kind/range");
    qdec_ctx* m = const_cast<qdec_ctx*>(c);
    const bf16_t* base = (kind == 0 ? m->k_cache(layer) : m->v_cache(layer)) + (size_t)pos0 * sh.D;
    const size_t spitch = (size_t)sh.max_seq * sh.D * sizeof(bf16_t);
    const size_t width = (size_t)n_pos * sh.D * sizeof(bf16_t);
    CK(cudaMemcpy2DAsync(host_dst, width, base, spitch, width, sh.HKV, cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    return QDEC_OK;
}

int qdec_read_history(const qdec_ctx* c, int32_t* host_dst, int32_t n) {
    if (!c || !host_dst || n < 0 || n > c->position) return fail(QDEC_E_INVALID_ARG, "bad history request");
    if (n == 0) return QDEC_OK;
    CK(cudaMemcpyAsync(host_dst, c->d_hist, (size_t)n * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    return QDEC_OK;
}

int qdec_sync(const qdec_ctx* c) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    return sync_status(const_cast<qdec_ctx*>(c), 4, nullptr);
}

int qdec_set_option(qdec_ctx* c, int32_t option, int32_t value) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    if (option == QDEC_OPT_PREFILL_IMPL) {
        if (value != QDEC_PREFILL_TCGEN05 && value != QDEC_PREFILL_SIMT)
            return fail(QDEC_E_INVALID_ARG, "bad value %d for QDEC_OPT_PREFILL_IMPL", value);
        c->prefill_gemm = value;
        return QDEC_OK;
    }
    if (option == QDEC_OPT_ATTN_UNIT_KEYS) {
        if (value != 0 && (value < 8 || value > 4096 || value % 8 != 0))
            return fail(QDEC_E_INVALID_ARG, "QDEC_OPT_ATTN_UNIT_KEYS takes 0 or 8..4096 in multiples of 8");
        c->attn_unit_keys = value;
        return QDEC_OK;
    }
    if (option == QDEC_OPT_WEIGHTS) return set_weight_format(c, value);
    if (option == QDEC_OPT_SHARED_PREFIX) {
        if (value != 0 && value != 1) return fail(QDEC_E_INVALID_ARG, "QDEC_OPT_SHARED_PREFIX takes 0 or 1");
        c->shared_prefix = value;
        return QDEC_OK;
    }
    if (option == QDEC_OPT_SPIN_LIMIT) {
        if (value < 0) return fail(QDEC_E_INVALID_ARG, "QDEC_OPT_SPIN_LIMIT takes 0 (default) or a positive count");
        c->spin_limit = value;
        return QDEC_OK;
    }
    if (option == QDEC_OPT_TRACE) {
        if (value != 0 && value != 1) return fail(QDEC_E_INVALID_ARG, "QDEC_OPT_TRACE takes 0 or 1");
        if (value == 1 && !c->persistent_ok) return fail(QDEC_E_UNSUPPORTED, "no persistent decode kernel to trace");
        if (value == 1 && !c->d_trace) {
            const size_t n = (size_t)c->dp.grid * (11 * c->sh.NL + 8);
            CK(dalloc(&c->d_trace, n));
            CK(cudaMemset(c->d_trace, 0, n * sizeof(unsigned long long)));
        } else if (value == 0 && c->d_trace) {
            CK(cudaStreamSynchronize(c->stream));
            cudaFree(c->d_trace);
            c->d_trace = nullptr;
        }
        return QDEC_OK;
    }
    if (option != QDEC_OPT_DECODE_KERNEL) return fail(QDEC_E_INVALID_ARG, "unknown option %d", option);
    if (value != QDEC_DECODE_PERSISTENT && value != QDEC_DECODE_GRAPH)
        return fail(QDEC_E_INVALID_ARG, "bad value %d for QDEC_OPT_DECODE_KERNEL", value);
    if (value == QDEC_DECODE_PERSISTENT && !c->persistent_ok)
        return fail(QDEC_E_UNSUPPORTED, "the persistent decode kernel does not cover this shape or device");
    if (value == QDEC_DECODE_PERSISTENT && c->quant)
        return fail(QDEC_E_UNSUPPORTED, "quantized weights decode with the per-operation kernels");
    c->decode_kernel = value;
    return QDEC_OK;
}

int qdec_set_sampling(qdec_ctx* c, float temperature, int32_t top_k, float top_p, float repetition_penalty,
                      uint64_t seed) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    if (!sample_params_valid(c->sh.V, temperature, top_k, top_p, repetition_penalty))
        return fail(QDEC_E_INVALID_ARG, "sampling needs temperature >= 0, top_k >= 0, 0 < top_p <= 1, penalty > 0 "
                                        "and a vocabulary of at most %d", kSampleMaxVocab);
    c->samp_t = temperature;
    c->samp_k = top_k;
    c->samp_p = top_p;
    c->samp_r = repetition_penalty;
    c->samp_seed = (unsigned long long)seed;
    return QDEC_OK;
}

int qdec_get_option(const qdec_ctx* c, int32_t option) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    if (option == QDEC_OPT_TRACE) return c->d_trace ? 1 : 0;
    if (option == QDEC_OPT_PREFILL_IMPL) return c->prefill_gemm;
    if (option == QDEC_OPT_ATTN_UNIT_KEYS) return c->attn_unit_keys;
    if (option == QDEC_OPT_SPIN_LIMIT) return c->spin_limit;
    if (option == QDEC_OPT_SHARED_PREFIX) return c->shared_prefix;
    if (option == QDEC_OPT_WEIGHTS) return c->quant ? c->quant->fmt : QDEC_WEIGHTS_BF16;
    if (option != QDEC_OPT_DECODE_KERNEL) return fail(QDEC_E_INVALID_ARG, "unknown option %d", option);
    return c->decode_kernel;
}

void qdec_destroy(qdec_ctx* c) {
    if (!c) return;
    if (c->stream) cudaStreamSynchronize(c->stream);
    free_all(c);
    delete c;
}

int qdec_read_trace(const qdec_ctx* c, uint64_t* host_dst, int32_t capacity) {
    if (!c) return fail(QDEC_E_INVALID_ARG, "null context");
    if (!c->d_trace) return fail(QDEC_E_STATE, "tracing is off (QDEC_OPT_TRACE)");
    const int n = c->dp.grid * (11 * c->sh.NL + 8);
    if (!host_dst) return n;
    if (capacity < n) return fail(QDEC_E_INVALID_ARG, "trace needs %d entries", n);
    CK(cudaMemcpyAsync(host_dst, c->d_trace, (size_t)n * sizeof(uint64_t), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    return n;
}

const char* qdec_strerror(int status) {
    switch (status) {
        case QDEC_OK: return "ok";
        case QDEC_E_INVALID_ARG: return "invalid argument";
        case QDEC_E_CAPACITY: return "KV-cache capacity exceeded";
        case QDEC_E_STATE: return "invalid state";
        case QDEC_E_CUDA: return "CUDA error";
        case QDEC_E_OOM: return "out of memory";
        case QDEC_E_TIMEOUT: return "device wait timed out";
        case QDEC_E_UNSUPPORTED: return "unsupported model shape";
        default: return "unknown status";
    }
}

const char* qdec_last_error(void) { return g_last_error.c_str(); }

uint64_t qdec_kernel_launches(void) { return __atomic_load_n(&qdec::g_launches, __ATOMIC_RELAXED); }

}  // extern "C"
