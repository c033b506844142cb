// The audio adaptor (include/qdec_adaptor.h): projector + bidirectional transformer blocks
// that produce the audio rows spliced into the decoder's prompt.  Every projection is the
// tcgen05 GEMM with its bias (and ReLU) in the epilogue; attention is the tcgen05 flash
// kernel without the causal mask, reading q/k/v straight out of the fused projection's
// output; LayerNorm runs on CUDA cores between them.
#include <cstdarg>
#include <cstdio>
#include <vector>

#include "../../include/qdec.h"
#include "../../include/qdec_adaptor.h"
#include "common.cuh"

using namespace qdec;

namespace {

// (x - mean) * rsqrt(var + eps) * g + b over each row of X fp32 [T, H], population variance,
// into bf16.  One 256-thread block per row; two passes over the row (mean, then variance of
// the centred values) so a large mean does not cancel.
__global__ void layer_norm_bf16_kernel(const float* __restrict__ X, int H, const float* __restrict__ g,
                                       const float* __restrict__ b, float eps, bf16_t* __restrict__ out) {
    __shared__ float red[8];
    const float* x = X + (size_t)blockIdx.x * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto block_sum = [&](float v) {
        v = warp_sum(v);
        __syncthreads();
        if (lane == 0) red[warp] = v;
        __syncthreads();
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += red[w];
        return t;
    };
    float s = 0.f;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(x + i);
        s += v.x + v.y + v.z + v.w;
    }
    const float mu = block_sum(s) / (float)H;
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(x + i);
        const float a = v.x - mu, c = v.y - mu, d = v.z - mu, e = v.w - mu;
        ss += a * a + c * c + d * d + e * e;
    }
    const float r = rsqrtf(block_sum(ss) / (float)H + eps);
    bf16_t* o = out + (size_t)blockIdx.x * H;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        const float4 v = *reinterpret_cast<const float4*>(x + i);
        const float4 gg = *reinterpret_cast<const float4*>(g + i);
        const float4 bb = *reinterpret_cast<const float4*>(b + i);
        uint2 w;
        w.x = pack_bf2((v.x - mu) * r * gg.x + bb.x, (v.y - mu) * r * gg.y + bb.y);
        w.y = pack_bf2((v.z - mu) * r * gg.z + bb.z, (v.w - mu) * r * gg.w + bb.w);
        *reinterpret_cast<uint2*>(o + i) = w;
    }
}

// out[i] = bf16(X[i]) for i < n (n a multiple of 4).
__global__ void to_bf16_kernel(const float* __restrict__ X, size_t n, bf16_t* __restrict__ out) {
    const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= n) return;
    const float4 v = *reinterpret_cast<const float4*>(X + i);
    *reinterpret_cast<uint2*>(out + i) = make_uint2(pack_bf2(v.x, v.y), pack_bf2(v.z, v.w));
}

struct Block {
    const float *ln1_g, *ln1_b, *ln2_g, *ln2_b, *bqkv, *bo, *fc1_b, *fc2_b;
    const bf16_t *wqkv, *wo, *fc1, *fc2;
};

bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_device(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

struct qdec_adaptor {
    qdec_adaptor_config cfg;
    const bf16_t *w1 = nullptr, *w2 = nullptr;
    const float *b1 = nullptr, *b2 = nullptr;
    std::vector<Block> blocks;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    int cap = 0;   // frames the scratch holds
    bf16_t *frames = nullptr, *h1 = nullptr, *xn = nullptr, *qkv = nullptr, *o = nullptr, *hf = nullptr, *rows = nullptr;
    float* X = nullptr;
    void release() {
        void* ps[] = {frames, h1, xn, qkv, o, hf, rows, X};
        for (void* p : ps)
            if (p) cudaFree(p);
        frames = h1 = xn = qkv = o = hf = rows = nullptr;
        X = nullptr;
        cap = 0;
    }
};

namespace {

#define ACK(call)                                                                                      \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess)                                                                         \
            return set_error(e_ == cudaErrorMemoryAllocation ? QDEC_E_OOM : QDEC_E_CUDA, "%s: %s (%s:%d)", \
                             #call, cudaGetErrorString(e_), __FILE__, __LINE__);                       \
    } while (0)

int ensure(qdec_adaptor* a, int T) {
    if (T <= a->cap) return QDEC_OK;
    ACK(cudaStreamSynchronize(a->stream));
    a->release();
    const qdec_adaptor_config& c = a->cfg;
    const size_t t = (size_t)T;
    ACK(cudaMalloc(&a->frames, t * c.enc_dim * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->h1, t * c.proj_dim * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->xn, t * c.hidden * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->qkv, t * 3 * c.hidden * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->o, t * c.hidden * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->hf, t * c.ffn * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->rows, t * c.hidden * sizeof(bf16_t)));
    ACK(cudaMalloc(&a->X, t * c.hidden * sizeof(float)));
    a->cap = T;
    return QDEC_OK;
}

}  // namespace

extern "C" {

int32_t qdec_fake_token_len(int32_t n) {
    if (n <= 0) return 0;
    for (int i = 0; i < 3; ++i) n = (n - 1) / 2 + 1;
    return n;
}

int qdec_adaptor_create(const qdec_adaptor_config* cfg, const qdec_adaptor_weights* w, void* cuda_stream,
                        qdec_adaptor** out) {
    if (!cfg || !w || !out) return set_error(QDEC_E_INVALID_ARG, "null argument");
    *out = nullptr;
    const qdec_adaptor_config& c = *cfg;
    if (c.enc_dim <= 0 || c.proj_dim <= 0 || c.hidden <= 0 || c.n_heads <= 0 || c.ffn <= 0 || c.n_blocks < 0 ||
        !(c.ln_eps > 0.f))
        return set_error(QDEC_E_INVALID_ARG, "non-positive size in qdec_adaptor_config");
    if (c.hidden != 128 * c.n_heads || c.enc_dim % 128 || c.proj_dim % 128 || c.hidden % 128 || c.ffn % 128)
        return set_error(QDEC_E_UNSUPPORTED, "adaptor needs head_dim 128 and dimensions that are multiples of 128");
    if (!al16(w->w1) || !al16(w->w2) || !al16(w->b1) || !al16(w->b2))
        return set_error(QDEC_E_INVALID_ARG, "projector weight pointer null or not 16-byte aligned");
    if (c.n_blocks > 0 && (!w->ln1_g || !w->ln1_b || !w->ln2_g || !w->ln2_b || !w->wqkv || !w->wo || !w->fc1 ||
                           !w->fc2 || !w->bqkv || !w->bo || !w->fc1_b || !w->fc2_b))
        return set_error(QDEC_E_INVALID_ARG, "null per-block weight array");
    qdec_adaptor* a = new (std::nothrow) qdec_adaptor();
    if (!a) return set_error(QDEC_E_OOM, "host allocation failed");
    a->cfg = c;
    a->w1 = static_cast<const bf16_t*>(w->w1);
    a->w2 = static_cast<const bf16_t*>(w->w2);
    a->b1 = w->b1;
    a->b2 = w->b2;
    for (int l = 0; l < c.n_blocks; ++l) {
        Block b{w->ln1_g[l], w->ln1_b[l], w->ln2_g[l], w->ln2_b[l], w->bqkv[l], w->bo[l], w->fc1_b[l], w->fc2_b[l],
                static_cast<const bf16_t*>(w->wqkv[l]), static_cast<const bf16_t*>(w->wo[l]),
                static_cast<const bf16_t*>(w->fc1[l]), static_cast<const bf16_t*>(w->fc2[l])};
        const void* ps[] = {b.ln1_g, b.ln1_b, b.ln2_g, b.ln2_b, b.bqkv, b.bo, b.fc1_b, b.fc2_b, b.wqkv, b.wo, b.fc1, b.fc2};
        for (const void* p : ps)
            if (!al16(p)) {
                delete a;
                return set_error(QDEC_E_INVALID_ARG, "block %d weight pointer null or not 16-byte aligned", l);
            }
        a->blocks.push_back(b);
    }
    if (cuda_stream) {
        a->stream = static_cast<cudaStream_t>(cuda_stream);
    } else {
        cudaError_t e = cudaStreamCreateWithFlags(&a->stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            delete a;
            return set_error(QDEC_E_CUDA, "cudaStreamCreate: %s", cudaGetErrorString(e));
        }
        a->own_stream = true;
    }
    *out = a;
    return QDEC_OK;
}

int qdec_adaptor_run(qdec_adaptor* a, const void* frames, int32_t n_frames, void* rows_out, int32_t* n_rows_out) {
    if (!a || !frames || !rows_out) return set_error(QDEC_E_INVALID_ARG, "null argument");
    if (n_frames <= 0) return set_error(QDEC_E_INVALID_ARG, "n_frames must be positive");
    const qdec_adaptor_config& c = a->cfg;
    const int T = n_frames, H = c.hidden;
    int rc = ensure(a, T);
    if (rc != QDEC_OK) return rc;
    cudaStream_t s = a->stream;
    const bf16_t* fr = static_cast<const bf16_t*>(frames);
    if (!(is_device(frames) && al16(frames))) {
        ACK(cudaMemcpyAsync(a->frames, frames, (size_t)T * c.enc_dim * sizeof(bf16_t), cudaMemcpyDefault, s));
        fr = a->frames;
    }
    uint64_t k = 0;
    // projector: ReLU(frames W1^T + b1) W2^T + b2
    ACK(launch_gemm_tc(fr, c.enc_dim, a->w1, T, c.proj_dim, c.enc_dim, GEMM_STORE_BF16, 0, nullptr, a->h1, c.proj_dim,
                       s, 1, a->b1, 1));
    ACK(launch_gemm_tc(a->h1, c.proj_dim, a->w2, T, H, c.proj_dim, GEMM_STORE_F32, 0, a->X, nullptr, H, s, 1, a->b2, 0));
    k += 2;
    for (const Block& b : a->blocks) {
        layer_norm_bf16_kernel<<<T, 256, 0, s>>>(a->X, H, b.ln1_g, b.ln1_b, c.ln_eps, a->xn);
        ACK(cudaGetLastError());
        ACK(launch_gemm_tc(a->xn, H, b.wqkv, T, 3 * H, H, GEMM_STORE_BF16, 0, nullptr, a->qkv, 3 * H, s, 1, b.bqkv, 0));
        ACK(launch_attention_bidir_tc(a->qkv, a->qkv + H, a->qkv + 2 * H, 3 * H, T, c.n_heads, a->o, s));
        ACK(launch_gemm_tc(a->o, H, b.wo, T, H, H, GEMM_ADD_F32, 0, a->X, nullptr, H, s, 1, b.bo, 0));
        layer_norm_bf16_kernel<<<T, 256, 0, s>>>(a->X, H, b.ln2_g, b.ln2_b, c.ln_eps, a->xn);
        ACK(cudaGetLastError());
        ACK(launch_gemm_tc(a->xn, H, b.fc1, T, c.ffn, H, GEMM_STORE_BF16, 0, nullptr, a->hf, c.ffn, s, 1, b.fc1_b, 1));
        ACK(launch_gemm_tc(a->hf, c.ffn, b.fc2, T, H, c.ffn, GEMM_ADD_F32, 0, a->X, nullptr, H, s, 1, b.fc2_b, 0));
        k += 7;
    }
    const int n_out = qdec_fake_token_len(T);
    const size_t n = (size_t)n_out * H;
    const bool dev_out = is_device(rows_out) && al16(rows_out);
    bf16_t* dst = dev_out ? static_cast<bf16_t*>(rows_out) : a->rows;
    to_bf16_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(a->X, n, dst);
    ACK(cudaGetLastError());
    count_launches(k + 1);
    if (!dev_out) {
        ACK(cudaMemcpyAsync(rows_out, a->rows, n * sizeof(bf16_t), cudaMemcpyDefault, s));
        ACK(cudaStreamSynchronize(s));
    }
    if (n_rows_out) *n_rows_out = n_out;
    if (!dev_out) {   // synchronised already: report a tensor-core kernel that gave up on a wait
        const int tc = tc_error_read_and_clear(), fa = fa_error_read_and_clear();
        if (tc > 0 || fa > 0)
            return set_error(QDEC_E_TIMEOUT, "a tensor-core kernel gave up waiting (codes %d, %d)", tc, fa);
    }
    return QDEC_OK;
}

void qdec_adaptor_destroy(qdec_adaptor* a) {
    if (!a) return;
    if (a->stream) cudaStreamSynchronize(a->stream);
    a->release();
    if (a->own_stream) cudaStreamDestroy(a->stream);
    delete a;
}

}  // extern "C"
