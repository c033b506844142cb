// Block-quantized layer weights for decode: the library's q8b32 and q4b32 formats (blocks of
// 32 weights along K, one fp16 scale per block; "Fun-ASR-Nano Native Runtime Implementation
// Plan", Task 8 packages Q8_0 / Q4_K_M decoders without defining the formats, so the library
// defines its own):
//   q8b32: d = fp16(max|w| / 127), q = clamp(round_half_even(w / d), -127, 127) as int8;
//   q4b32: d = fp16(max|w| / 7),   q = clamp(round_half_even(w / d), -7, 7) stored as q + 8
//          in a nibble, the lower nibble first;
// w' = q * d, an all-zero block has d = 0 and codes 0.  The quantizer computes the scale
// and the quotients in double (the same roundings as the definition), so its codes and
// scales are exact.  The decode GEMV streams the codes and scales and dequantizes in
// registers: every product is q * x in fp32, and a lane's 16 columns share one block scale.
#include <cuda_fp16.h>

#include "common.cuh"

namespace qdec {

namespace {

constexpr int QT_THREADS = 256;

// One thread per block of 32 weights (row, block) of W [N, K].
__global__ void quantize_kernel(const bf16_t* __restrict__ W, int N, int K, int qmax, int8_t* __restrict__ codes8,
                                uint8_t* __restrict__ codes4, __half* __restrict__ scales) {
    const int nb = K / 32;
    const long long gb = (long long)blockIdx.x * QT_THREADS + threadIdx.x;   // global block index
    if (gb >= (long long)N * nb) return;
    const int row = (int)(gb / nb), b = (int)(gb % nb);
    const bf16_t* w = W + (size_t)row * K + (size_t)b * 32;
    float v[32];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(w + i);
        v[i] = bf_lo(u.x); v[i + 1] = bf_hi(u.x); v[i + 2] = bf_lo(u.y); v[i + 3] = bf_hi(u.y);
        v[i + 4] = bf_lo(u.z); v[i + 5] = bf_hi(u.z); v[i + 6] = bf_lo(u.w); v[i + 7] = bf_hi(u.w);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const __half dh = __double2half((double)amax / (double)qmax);
    const double d = (double)__half2float(dh);
    scales[gb] = dh;
    int q[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        double t = d > 0.0 ? rint((double)v[i] / d) : 0.0;
        t = fmin(fmax(t, (double)-qmax), (double)qmax);
        q[i] = (int)t;
    }
    if (codes8) {
        int8_t* c = codes8 + (size_t)row * K + (size_t)b * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<uint32_t*>(c + i) = (uint32_t)(q[i] & 255) | ((uint32_t)(q[i + 1] & 255) << 8) |
                                                  ((uint32_t)(q[i + 2] & 255) << 16) | ((uint32_t)(q[i + 3] & 255) << 24);
    } else {
        uint8_t* c = codes4 + (size_t)row * (K / 2) + (size_t)b * 16;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) word |= (uint32_t)(q[i + j] + 8) << (4 * j);
            *reinterpret_cast<uint32_t*>(c + i / 2) = word;
        }
    }
}

constexpr int GQ_THREADS = 128;   // 4 warps, each R rows: many small CTAs keep every SM streaming
constexpr int GQ_R = 2;
constexpr int GQ_MAXC = 6;         // 16-code chunks a lane loads per row (K <= 32 * 16 * 6 = 3072)

// 16 codes of one row (columns k .. k + 15, half a block) times x, unscaled.
template <int BITS>
__device__ __forceinline__ float qdot16(const uint4 c, const float* xv) {
    float a = 0.f;
    if constexpr (BITS == 8) {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) a = fmaf((float)(int8_t)(w[i] >> (8 * j)), xv[4 * i + j], a);
    } else {   // 16 nibbles in the low 8 bytes (c.x, c.y)
        const uint32_t w[2] = {c.x, c.y};
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) a = fmaf((float)((int)((w[i] >> (4 * j)) & 15u) - 8), xv[8 * i + j], a);
    }
    return a;
}

// y = W' . xhat for quantized W'.  Each warp owns GQ_R consecutive rows (SWIGLU: and the up
// rows at up_off); lane l takes the 16-column chunks l, l + 32, ... of every row.  All of a
// lane's code and scale loads are issued before any arithmetic (up to GQ_MAXC chunks per
// row in flight), which is what keeps HBM busy for a small matrix.
template <int MODE, int BITS>
__global__ void __launch_bounds__(GQ_THREADS) gemv_q_kernel(const void* __restrict__ codes,
                                                           const __half* __restrict__ scales, int rows, int K,
                                                           const float* __restrict__ x,
                                                           const bf16_t* __restrict__ norm_g, float eps, int up_off,
                                                           float* __restrict__ y) {
    extern __shared__ float xs[];
    __shared__ float red[GQ_THREADS / 32];
    constexpr int NA = (MODE == GEMV_SWIGLU) ? 2 : 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * (GQ_THREADS / 32) + warp) * GQ_R;
    const int nchunk = K / 16, nc = (nchunk - lane + 31) / 32;   // chunks of this lane per row
    const size_t row_bytes = BITS == 8 ? (size_t)K : (size_t)K / 2;
    const int nb = K / 32;
    // issue the weight loads first: they do not depend on x
    uint4 cw[NA][GQ_R][GQ_MAXC];
    float sc[NA][GQ_R][GQ_MAXC];
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int r = 0; r < GQ_R; ++r) {
            const int row = min(row0 + r, rows - 1);
            const size_t rr = (size_t)(row + a * up_off);
            const uint8_t* cb = static_cast<const uint8_t*>(codes) + rr * row_bytes;
#pragma unroll
            for (int i = 0; i < GQ_MAXC; ++i) {
                if (i < nc) {
                    const int ch = lane + 32 * i;
                    if (BITS == 8) {
                        cw[a][r][i] = __ldcs(reinterpret_cast<const uint4*>(cb + (size_t)ch * 16));
                    } else {
                        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(cb + (size_t)ch * 8));
                        cw[a][r][i] = make_uint4(v.x, v.y, 0u, 0u);
                    }
                    sc[a][r][i] = __half2float(scales[rr * nb + (ch >> 1)]);
                }
            }
        }
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < K; i += GQ_THREADS * 4) {
        const float4 v = *reinterpret_cast<const float4*>(x + i);
        *reinterpret_cast<float4*>(xs + i) = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (norm_g) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < GQ_THREADS / 32; ++w) tot += red[w];
        const float r = rsqrtf(tot / (float)K + eps);
        for (int i = threadIdx.x; i < K; i += GQ_THREADS) xs[i] = xs[i] * r * bf1(norm_g[i]);
    }
    __syncthreads();
    float acc[NA][GQ_R];
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int r = 0; r < GQ_R; ++r) acc[a][r] = 0.f;
#pragma unroll
    for (int i = 0; i < GQ_MAXC; ++i) {
        if (i < nc) {
            float xv[16];
            const float4* xp = reinterpret_cast<const float4*>(xs + (lane + 32 * i) * 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) *reinterpret_cast<float4*>(xv + 4 * j) = xp[j];
#pragma unroll
            for (int a = 0; a < NA; ++a)
#pragma unroll
                for (int r = 0; r < GQ_R; ++r) acc[a][r] = fmaf(sc[a][r][i], qdot16<BITS>(cw[a][r][i], xv), acc[a][r]);
        }
    }
#pragma unroll
    for (int r = 0; r < GQ_R; ++r) {
        const int row = row0 + r;
        const float v0 = warp_sum(acc[0][r]);
        const float v1 = NA > 1 ? warp_sum(acc[NA - 1][r]) : 0.f;
        if (lane == 0 && row < rows) {
            if (MODE == GEMV_STORE) y[row] = v0;
            else if (MODE == GEMV_ADD) y[row] += v0;
            else y[row] = silu(v0) * v1;
        }
    }
}

template <int BITS>
cudaError_t launch_gemv_q_bits(const void* codes, const __half* scales, int rows, int K, const float* x,
                               const bf16_t* norm_g, float eps, int mode, int up_off, float* y, cudaStream_t s) {
    const int grid = (rows + (GQ_THREADS / 32) * GQ_R - 1) / ((GQ_THREADS / 32) * GQ_R);
    const size_t smem = (size_t)K * sizeof(float);
    switch (mode) {
        case GEMV_STORE:
            gemv_q_kernel<GEMV_STORE, BITS><<<grid, GQ_THREADS, smem, s>>>(codes, scales, rows, K, x, norm_g, eps, up_off, y);
            break;
        case GEMV_ADD:
            gemv_q_kernel<GEMV_ADD, BITS><<<grid, GQ_THREADS, smem, s>>>(codes, scales, rows, K, x, norm_g, eps, up_off, y);
            break;
        case GEMV_SWIGLU:
            gemv_q_kernel<GEMV_SWIGLU, BITS><<<grid, GQ_THREADS, smem, s>>>(codes, scales, rows, K, x, norm_g, eps, up_off, y);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

size_t quant_code_bytes(int fmt, size_t N, size_t K) { return fmt == QUANT_Q8B32 ? N * K : N * K / 2; }
size_t quant_scale_bytes(size_t N, size_t K) { return N * (K / 32) * 2; }

cudaError_t launch_quantize(const bf16_t* W, int N, int K, int fmt, void* codes, void* scales, cudaStream_t s) {
    (void)cudaGetLastError();
    if (!W || !codes || !scales || N <= 0 || K <= 0 || K % 32 != 0 || (fmt != QUANT_Q8B32 && fmt != QUANT_Q4B32))
        return cudaErrorInvalidValue;
    const long long blocks = (long long)N * (K / 32);
    const int grid = (int)((blocks + QT_THREADS - 1) / QT_THREADS);
    quantize_kernel<<<grid, QT_THREADS, 0, s>>>(W, N, K, fmt == QUANT_Q8B32 ? 127 : 7,
                                                fmt == QUANT_Q8B32 ? static_cast<int8_t*>(codes) : nullptr,
                                                fmt == QUANT_Q4B32 ? static_cast<uint8_t*>(codes) : nullptr,
                                                static_cast<__half*>(scales));
    return cudaGetLastError();
}

cudaError_t launch_gemv_q(const void* codes, const void* scales, int fmt, int rows, int K, const float* x,
                          const bf16_t* norm_g, float eps, int mode, int up_off, float* y, cudaStream_t s) {
    (void)cudaGetLastError();
    if (K % 256 != 0 || K > 32 * 16 * GQ_MAXC) return cudaErrorInvalidValue;   // whole 16-column chunks per lane
    const __half* sc = static_cast<const __half*>(scales);
    if (fmt == QUANT_Q8B32) return launch_gemv_q_bits<8>(codes, sc, rows, K, x, norm_g, eps, mode, up_off, y, s);
    if (fmt == QUANT_Q4B32) return launch_gemv_q_bits<4>(codes, sc, rows, K, x, norm_g, eps, mode, up_off, y, s);
    return cudaErrorInvalidValue;
}

}  // namespace qdec
