// Batch-1 decode GEMVs (bf16 weights, fp32 activations and accumulation) and the tied
// lm_head with a fused final RMSNorm and a deterministic grid-wide argmax.
//
// "Forward map - funasr_nano", LLM decoder table (projections, packed gate_up SwiGLU,
// final rms_norm, tied lm_head `mul_mat(token_w, last_x)`); Generation / KV Path (one
// token per step).  "Qwen3ASR ncnn多平台移植" §5 step 5-6 (LM head over the full vocabulary,
// greedy pick).
#include "common.cuh"

namespace qdec {

namespace {
constexpr int GEMV_THREADS = 256;

// Loads x [K] into shared memory, optionally replaced by rmsnorm(x) * g.
__device__ __forceinline__ void load_x(float* xs, const float* __restrict__ x, int K,
                                       const bf16_t* __restrict__ norm_g, float eps, float* red) {
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < K; i += GEMV_THREADS * 4) {
        float4 v = *reinterpret_cast<const float4*>(x + i);
        *reinterpret_cast<float4*>(xs + i) = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (norm_g) {
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < GEMV_THREADS / 32; ++w) tot += red[w];
        const float r = rsqrtf(tot / (float)K + eps);
        for (int i = threadIdx.x; i < K; i += GEMV_THREADS) xs[i] = xs[i] * r * bf1(norm_g[i]);
    }
    __syncthreads();
}

__device__ __forceinline__ float dot8(const uint4 w, const float* xv) {
    float a = bf_lo(w.x) * xv[0];
    a = fmaf(bf_hi(w.x), xv[1], a);
    a = fmaf(bf_lo(w.y), xv[2], a);
    a = fmaf(bf_hi(w.y), xv[3], a);
    a = fmaf(bf_lo(w.z), xv[4], a);
    a = fmaf(bf_hi(w.z), xv[5], a);
    a = fmaf(bf_lo(w.w), xv[6], a);
    a = fmaf(bf_hi(w.w), xv[7], a);
    return a;
}

// Each warp owns R consecutive rows (and, for SWIGLU, the matching up rows).
template <int MODE, int R>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_kernel(const bf16_t* __restrict__ W, int rows, int K,
                                                            const float* __restrict__ x,
                                                            const bf16_t* __restrict__ norm_g, float eps,
                                                            int up_off, float* __restrict__ y) {
    extern __shared__ float xs[];
    __shared__ float red[GEMV_THREADS / 32];
    load_x(xs, x, K, norm_g, eps, red);
    constexpr int NA = (MODE == GEMV_SWIGLU) ? 2 : 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * (GEMV_THREADS / 32) + warp) * R;
    float acc[NA][R];
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[a][r] = 0.f;
    for (int k = lane * 8; k < K; k += 256) {
        float xv[8];
        *reinterpret_cast<float4*>(xv) = *reinterpret_cast<const float4*>(xs + k);
        *reinterpret_cast<float4*>(xv + 4) = *reinterpret_cast<const float4*>(xs + k + 4);
        uint4 w[NA][R];
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = row0 + r;
                w[a][r] = row < rows ? __ldcs(reinterpret_cast<const uint4*>(W + (size_t)(row + a * up_off) * K + k))
                                     : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[a][r] += dot8(w[a][r], xv);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = row0 + r;
        float v0 = warp_sum(acc[0][r]);
        float v1 = NA > 1 ? warp_sum(acc[NA - 1][r]) : 0.f;
        if (lane == 0 && row < rows) {
            if (MODE == GEMV_STORE) y[row] = v0;
            else if (MODE == GEMV_ADD) y[row] += v0;
            else y[row] = silu(v0) * v1;
        }
    }
}

constexpr int LM_R = 4;                                  // rows per warp
constexpr int LM_ROWS_PER_BLOCK = (GEMV_THREADS / 32) * LM_R;

__global__ void __launch_bounds__(GEMV_THREADS) lm_head_argmax_kernel(const bf16_t* __restrict__ E, int V, int H,
                                                                      const float* __restrict__ x,
                                                                      const bf16_t* __restrict__ g, float eps,
                                                                      float* __restrict__ logits,
                                                                      int* __restrict__ argmax, void* scratch) {
    extern __shared__ float xs[];
    __shared__ float red[GEMV_THREADS / 32];
    __shared__ float bv[GEMV_THREADS / 32];
    __shared__ int bi[GEMV_THREADS / 32];
    __shared__ bool last;
    pdl_trigger();
    pdl_wait();
    load_x(xs, x, H, g, eps, red);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * (GEMV_THREADS / 32) + warp) * LM_R;
    float acc[LM_R];
#pragma unroll
    for (int r = 0; r < LM_R; ++r) acc[r] = 0.f;
    for (int k = lane * 8; k < H; k += 256) {
        float xv[8];
        *reinterpret_cast<float4*>(xv) = *reinterpret_cast<const float4*>(xs + k);
        *reinterpret_cast<float4*>(xv + 4) = *reinterpret_cast<const float4*>(xs + k + 4);
        uint4 w[LM_R];
#pragma unroll
        for (int r = 0; r < LM_R; ++r)
            w[r] = (row0 + r) < V ? __ldcs(reinterpret_cast<const uint4*>(E + (size_t)(row0 + r) * H + k))
                                  : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < LM_R; ++r) acc[r] += dot8(w[r], xv);
    }
    float best = -INFINITY;
    int besti = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < LM_R; ++r) {
        const float v = warp_sum(acc[r]);
        const int row = row0 + r;
        if (row < V) {
            if (lane == 0) logits[row] = v;
            if (am_better(v, row, best, besti)) { best = v; besti = row; }
        }
    }
    if (lane == 0) { bv[warp] = best; bi[warp] = besti; }
    __syncthreads();
    unsigned int* counter = reinterpret_cast<unsigned int*>(scratch);
    ArgMax* part = reinterpret_cast<ArgMax*>(reinterpret_cast<char*>(scratch) + 16);
    if (threadIdx.x == 0) {
        float b = bv[0];
        int ib = bi[0];
        for (int w = 1; w < GEMV_THREADS / 32; ++w)
            if (am_better(bv[w], bi[w], b, ib)) { b = bv[w]; ib = bi[w]; }
        part[blockIdx.x].v = b;
        part[blockIdx.x].i = ib;
        __threadfence();
        const unsigned int ticket = atomicAdd(counter, 1u);
        last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    float b = -INFINITY;
    int ib = 0x7fffffff;
    for (int j = threadIdx.x; j < (int)gridDim.x; j += GEMV_THREADS) {
        const float v = __ldcg(&part[j].v);
        const int i = __ldcg(&part[j].i);
        if (am_better(v, i, b, ib)) { b = v; ib = i; }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, b, o);
        const int i = __shfl_xor_sync(0xffffffffu, ib, o);
        if (am_better(v, i, b, ib)) { b = v; ib = i; }
    }
    if (lane == 0) { bv[warp] = b; bi[warp] = ib; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < GEMV_THREADS / 32; ++w)
            if (am_better(bv[w], bi[w], b, ib)) { b = bv[w]; ib = bi[w]; }
        // All logits NaN: report index 0 rather than an out-of-range value.
        *argmax = (ib == 0x7fffffff) ? 0 : ib;
        *counter = 0u;
    }
}
}  // namespace

cudaError_t launch_gemv(const bf16_t* W, int rows, int K, const float* x, const bf16_t* norm_g, float eps,
                        int mode, int up_off, float* y, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (K % 8 != 0) return cudaErrorInvalidValue;
    constexpr int R = 2;
    const int grid = (rows + (GEMV_THREADS / 32) * R - 1) / ((GEMV_THREADS / 32) * R);
    const size_t smem = (size_t)K * sizeof(float);
    switch (mode) {
        case GEMV_STORE: gemv_kernel<GEMV_STORE, R><<<grid, GEMV_THREADS, smem, s>>>(W, rows, K, x, norm_g, eps, up_off, y); break;
        case GEMV_ADD: gemv_kernel<GEMV_ADD, R><<<grid, GEMV_THREADS, smem, s>>>(W, rows, K, x, norm_g, eps, up_off, y); break;
        case GEMV_SWIGLU: gemv_kernel<GEMV_SWIGLU, R><<<grid, GEMV_THREADS, smem, s>>>(W, rows, K, x, norm_g, eps, up_off, y); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

size_t lm_head_scratch_bytes(int V) {
    const size_t blocks = (size_t)(V + LM_ROWS_PER_BLOCK - 1) / LM_ROWS_PER_BLOCK;
    return 16 + blocks * sizeof(ArgMax);
}

cudaError_t launch_lm_head_argmax(const bf16_t* E, int V, int H, const float* x, const bf16_t* g_final, float eps,
                                  float* logits, int* argmax, void* scratch, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (H % 8 != 0) return cudaErrorInvalidValue;
    const int grid = (V + LM_ROWS_PER_BLOCK - 1) / LM_ROWS_PER_BLOCK;
    return launch_pdl(lm_head_argmax_kernel, dim3(grid), dim3(GEMV_THREADS), (size_t)H * sizeof(float), s, E, V, H, x,
                      g_final, eps, logits, argmax, scratch);
}

}  // namespace qdec
