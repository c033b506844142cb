// Row-wise kernels: embedding gather + audio splice, RMSNorm, per-head Q/K RMSNorm +
// NeoX RoPE + KV-cache append.
//
// "Forward map - funasr_nano", LLM decoder table: token embed (row gather), the audio-row
// override of inputs_embeds at [fbank_beg, fbank_beg + fake_token_len), rms_norm, and the
// per-head Q/K-RMSNorm + NeoX RoPE @ 1e6; Generation / KV Path: KV cache write.
// "Qwen3ASR ncnn多平台移植" §5: each step builds RoPE for its absolute position and appends
// its key/value to the cache.
#include "common.cuh"

namespace qdec {

namespace {
int g_programmatic = 1;
}
int set_programmatic_launch(int on) {
    const int prev = g_programmatic;
    g_programmatic = on ? 1 : 0;
    return prev;
}
bool programmatic_launch() { return g_programmatic != 0; }

// One block per row; 8-byte loads of 4 bf16, 16-byte stores of 4 fp32.
__global__ void embed_splice_kernel(const bf16_t* __restrict__ E, const int* __restrict__ ids, int H,
                                    const bf16_t* __restrict__ audio, int n_audio, int off,
                                    float* __restrict__ X, int* __restrict__ history) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const bool is_audio = (t >= off) && (t < off + n_audio);
    const int id = ids[t];
    const bf16_t* src = is_audio ? audio + (size_t)(t - off) * H : E + (size_t)id * H;
    float* dst = X + (size_t)t * H;
    for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
        uint2 w = *reinterpret_cast<const uint2*>(src + i);
        *reinterpret_cast<float4*>(dst + i) = make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
    }
    if (threadIdx.x == 0 && history) history[t] = id;
}

cudaError_t launch_embed_splice(const bf16_t* E, const int* ids_dev, int T, int H, const bf16_t* audio,
                                int n_audio, int off, float* X, int* history, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    return launch_pdl(embed_splice_kernel, dim3(T), dim3(128), 0, s, E, ids_dev, H, audio, n_audio, off, X, history);
}

// Decode embedding: token >= 0 is embedded; -1 embeds the previous step's argmax (greedy
// feedback kept on the device).  The token also goes into the history at slot *pos.
__global__ void embed_token_kernel(const bf16_t* __restrict__ E, int token, const int* __restrict__ prev_argmax,
                                   const int* __restrict__ pos, int H, float* __restrict__ x,
                                   int* __restrict__ history) {
    const int id = token >= 0 ? token : *prev_argmax;
    const bf16_t* src = E + (size_t)id * H;
    for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
        uint2 w = *reinterpret_cast<const uint2*>(src + i);
        *reinterpret_cast<float4*>(x + i) = make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
    }
    if (threadIdx.x == 0) history[*pos] = id;
}

cudaError_t launch_embed_token(const bf16_t* E, int token, const int* prev_argmax, const int* pos, int H, float* x,
                               int* history, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    embed_token_kernel<<<1, 256, 0, s>>>(E, token, prev_argmax, pos, H, x, history);
    return cudaGetLastError();
}

__global__ void advance_position_kernel(int* pos, int n) { *pos += n; }
__global__ void set_int_kernel(int* p, int v) {
    pdl_trigger();
    pdl_wait();
    *p = v;
}

cudaError_t launch_set_int(int* p, int v, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    return launch_pdl(set_int_kernel, dim3(1), dim3(1), 0, s, p, v);
}

cudaError_t launch_advance_position(int* pos, int n, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    advance_position_kernel<<<1, 1, 0, s>>>(pos, n);
    return cudaGetLastError();
}

// Block-wide sum over 256 threads.
__device__ __forceinline__ float block_sum_256(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = (l < 8) ? red[l] : 0.f;
    return warp_sum(r);
}

__global__ void rmsnorm_bf16_kernel(const float* __restrict__ X, int H, const bf16_t* __restrict__ g,
                                    float eps, bf16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[8];
    const float* x = X + (size_t)blockIdx.x * H;
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        float4 v = *reinterpret_cast<const float4*>(x + i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum_256(ss, red);
    const float r = rsqrtf(ss / (float)H + eps);
    bf16_t* o = out + (size_t)blockIdx.x * H;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        float4 v = *reinterpret_cast<const float4*>(x + i);
        uint2 gw = *reinterpret_cast<const uint2*>(g + i);
        uint2 ow;
        ow.x = pack_bf2(v.x * r * bf_lo(gw.x), v.y * r * bf_hi(gw.x));
        ow.y = pack_bf2(v.z * r * bf_lo(gw.y), v.w * r * bf_hi(gw.y));
        *reinterpret_cast<uint2*>(o + i) = ow;
    }
}

// H = 1024 (the 0.6B shape): 128 threads per row, each holding 8 values in registers (two
// 16-byte loads in flight), so a row is read once and twice as many rows are in flight per
// SM as with 256 threads.
__global__ void __launch_bounds__(128) rmsnorm1024_bf16_kernel(const float* __restrict__ X,
                                                               const bf16_t* __restrict__ g, float eps,
                                                               bf16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[4];
    const float4* x = reinterpret_cast<const float4*>(X + (size_t)blockIdx.x * 1024);
    const int t = threadIdx.x;
    const float4 a = x[t], b = x[t + 128];
    float ss = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
    ss = warp_sum(ss);
    if ((t & 31) == 0) red[t >> 5] = ss;
    __syncthreads();
    const float r = rsqrtf((red[0] + red[1] + red[2] + red[3]) / 1024.f + eps);
    const uint2 ga = reinterpret_cast<const uint2*>(g)[t], gb = reinterpret_cast<const uint2*>(g)[t + 128];
    uint2* o = reinterpret_cast<uint2*>(out + (size_t)blockIdx.x * 1024);
    o[t] = make_uint2(pack_bf2(a.x * r * bf_lo(ga.x), a.y * r * bf_hi(ga.x)),
                      pack_bf2(a.z * r * bf_lo(ga.y), a.w * r * bf_hi(ga.y)));
    o[t + 128] = make_uint2(pack_bf2(b.x * r * bf_lo(gb.x), b.y * r * bf_hi(gb.x)),
                            pack_bf2(b.z * r * bf_lo(gb.y), b.w * r * bf_hi(gb.y)));
}

// H = 1024, many rows (a long prompt): one warp per row, 8 rows per block, each lane holding
// 32 values (eight 16-byte loads in flight); the row's sum of squares is a warp reduction,
// with no block barrier.
__global__ void __launch_bounds__(256) rmsnorm1024_rows_kernel(const float* __restrict__ X, int T,
                                                               const bf16_t* __restrict__ g, float eps,
                                                               bf16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= T) return;
    const float4* x = reinterpret_cast<const float4*>(X + (size_t)row * 1024);
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = x[lane + 32 * k];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    const float r = rsqrtf(warp_sum(ss) / 1024.f + eps);
    const uint2* g2 = reinterpret_cast<const uint2*>(g);
    uint2* o = reinterpret_cast<uint2*>(out + (size_t)row * 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint2 gw = g2[lane + 32 * k];
        o[lane + 32 * k] = make_uint2(pack_bf2(v[k].x * r * bf_lo(gw.x), v[k].y * r * bf_hi(gw.x)),
                                      pack_bf2(v[k].z * r * bf_lo(gw.y), v[k].w * r * bf_hi(gw.y)));
    }
}

cudaError_t launch_rmsnorm_bf16(const float* X, int T, int H, const bf16_t* g, float eps, bf16_t* out,
                                cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (H == 1024 && T >= 1024)
        return launch_pdl(rmsnorm1024_rows_kernel, dim3((T + 7) / 8), dim3(256), 0, s, X, T, g, eps, out);
    if (H == 1024) return launch_pdl(rmsnorm1024_bf16_kernel, dim3(T), dim3(128), 0, s, X, g, eps, out);
    return launch_pdl(rmsnorm_bf16_kernel, dim3(T), dim3(256), 0, s, X, H, g, eps, out);
}

// rmsnorm_bf16_kernel after folding split-K partials into the residual row: each thread
// updates the elements it later normalises, so its own writes are what it reads back.
__global__ void rmsnorm_fold_bf16_kernel(float* __restrict__ X, const float* __restrict__ part, int splits,
                                         size_t pstride, int H, const bf16_t* __restrict__ g, float eps,
                                         bf16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[8];
    float* x = X + (size_t)blockIdx.x * H;
    const float* pr = part + (size_t)blockIdx.x * H;
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        float4 v = *reinterpret_cast<const float4*>(x + i);
        for (int z = 0; z < splits; ++z) {
            const float4 d = *reinterpret_cast<const float4*>(pr + z * pstride + i);
            v.x += d.x; v.y += d.y; v.z += d.z; v.w += d.w;
        }
        *reinterpret_cast<float4*>(x + i) = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum_256(ss, red);
    const float r = rsqrtf(ss / (float)H + eps);
    bf16_t* o = out + (size_t)blockIdx.x * H;
    for (int i = threadIdx.x * 4; i < H; i += 1024) {
        float4 v = *reinterpret_cast<const float4*>(x + i);
        uint2 gw = *reinterpret_cast<const uint2*>(g + i);
        uint2 ow;
        ow.x = pack_bf2(v.x * r * bf_lo(gw.x), v.y * r * bf_hi(gw.x));
        ow.y = pack_bf2(v.z * r * bf_lo(gw.y), v.w * r * bf_hi(gw.y));
        *reinterpret_cast<uint2*>(o + i) = ow;
    }
}

cudaError_t launch_rmsnorm_fold_bf16(float* X, const float* part, int splits, size_t pstride, int T, int H,
                                     const bf16_t* g, float eps, bf16_t* out, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (H % 4 != 0 || pstride % 4 != 0 || splits < 1) return cudaErrorInvalidValue;
    return launch_pdl(rmsnorm_fold_bf16_kernel, dim3(T), dim3(256), 0, s, X, part, splits, pstride, H, g, eps, out);
}

__global__ void fold_partials_kernel(float* __restrict__ X, const float* __restrict__ part, int splits,
                                     size_t pstride, size_t n) {
    pdl_trigger();
    pdl_wait();
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = X[i];
    for (int z = 0; z < splits; ++z) v += part[z * pstride + i];
    X[i] = v;
}

cudaError_t launch_fold_partials(float* X, const float* part, int splits, size_t pstride, size_t n, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    return launch_pdl(fold_partials_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, X, part, splits, pstride,
                      n);
}

// grid (T, HQ + 2 HKV), block max(32, D/2): thread i < D/2 owns the NeoX pair (i, i + D/2) of one head.
__global__ void qk_norm_rope_append_kernel(const float* __restrict__ qkv, int HQ, int HKV, int D, int max_seq,
                                           float eps, const int* __restrict__ pos0,
                                           const bf16_t* __restrict__ g_q, const bf16_t* __restrict__ g_k,
                                           const float2* __restrict__ rope_cs,
                                           bf16_t* __restrict__ q_bf16, float* __restrict__ q_f32,
                                           bf16_t* __restrict__ k_cache, bf16_t* __restrict__ v_cache,
                                           int splits, size_t pstride) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[4];
    const int t = blockIdx.x, hh = blockIdx.y, i = threadIdx.x, half = D >> 1;
    const int rows = (HQ + 2 * HKV) * D;
    const int p = *pos0 + t;
    const bool act = i < half;   // the block is padded to a whole warp when D/2 < 32
    const float* src = qkv + (size_t)t * rows + (size_t)hh * D;
    float a = act ? src[i] : 0.f, b = act ? src[i + half] : 0.f;
    for (int z = 1; z < splits; ++z)   // split-K partial slabs, added in order
        if (act) {
            a += src[z * pstride + i];
            b += src[z * pstride + i + half];
        }
    if (hh >= HQ + HKV) {  // value head: plain copy into the cache
        const int g = hh - HQ - HKV;
        bf16_t* dst = v_cache + ((size_t)g * max_seq + p) * D;
        if (act) {
            dst[i] = f2bf(a);
            dst[i + half] = f2bf(b);
        }
        return;
    }
    float ss = warp_sum(a * a + b * b);
    if (half > 32) {
        if ((i & 31) == 0) red[i >> 5] = ss;
        __syncthreads();
        ss = 0.f;
        for (int w = 0; w < (half >> 5); ++w) ss += red[w];
    }
    const float r = rsqrtf(ss / (float)D + eps);
    if (!act) return;
    const bf16_t* g = hh < HQ ? g_q : g_k;
    a *= r * bf1(g[i]);
    b *= r * bf1(g[i + half]);
    const float2 cs = rope_cs[(size_t)p * half + i];
    const float ra = a * cs.x - b * cs.y;
    const float rb = b * cs.x + a * cs.y;
    if (hh < HQ) {
        if (q_bf16) {
            bf16_t* dst = q_bf16 + ((size_t)t * HQ + hh) * D;
            dst[i] = f2bf(ra);
            dst[i + half] = f2bf(rb);
        } else {
            float* dst = q_f32 + ((size_t)t * HQ + hh) * D;
            dst[i] = ra;
            dst[i + half] = rb;
        }
    } else {
        const int g2 = hh - HQ;
        bf16_t* dst = k_cache + ((size_t)g2 * max_seq + p) * D;
        dst[i] = f2bf(ra);
        dst[i + half] = f2bf(rb);
    }
}

cudaError_t launch_qk_norm_rope_append(const float* qkv, int T, const Shape& sh, const int* pos0,
                                       const bf16_t* g_q, const bf16_t* g_k, const float2* rope_cs,
                                       bf16_t* q_bf16, float* q_f32, bf16_t* k_cache, bf16_t* v_cache,
                                       cudaStream_t s, int splits, size_t pstride) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (splits < 1) return cudaErrorInvalidValue;
    dim3 grid(T, sh.HQ + 2 * sh.HKV);
    return launch_pdl(qk_norm_rope_append_kernel, grid, dim3(sh.D / 2 < 32 ? 32 : sh.D / 2), 0, s, qkv, sh.HQ, sh.HKV,
                      sh.D, sh.max_seq, sh.eps, pos0, g_q, g_k, rope_cs, q_bf16, q_f32, k_cache, v_cache, splits,
                      pstride);
}

}  // namespace qdec
