// CUDA-core GEMM C = A . W^T (bf16 operands, fp32 accumulation) with the decoder's epilogues.
// It is the correctness baseline that the tcgen05 GEMM is tested against, and the fallback
// for shapes the tensor-core kernel does not tile.
//
// Epilogues ("Forward map - funasr_nano", LLM decoder table): plain store (QKV projection),
// residual add (o_proj and down_proj add into the fp32 residual stream), and SwiGLU on the
// packed gate_up projection (silu(gate) * up, stored bf16 as the down projection's operand).
#include "common.cuh"

namespace qdec {

namespace {
constexpr int BM = 64, BN = 64, BK = 32, NT = 256;

template <int MODE>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const bf16_t* __restrict__ A, int lda,
                                                       const bf16_t* __restrict__ W, int M, int N, int K,
                                                       int up_off, float* __restrict__ Cf,
                                                       bf16_t* __restrict__ Cb, int ldc) {
    constexpr int NW = (MODE == GEMM_SWIGLU_BF16) ? 2 : 1;   // weight tiles per block (gate, up)
    __shared__ float As[BK][BM + 4];
    __shared__ float Ws[NW][BK][BN + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    float acc[NW][4][4];
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[w][i][j] = 0.f;

    // loader mapping: 64 rows x 32 k = 256 x 8 elements (one 16-byte load per thread)
    const int lr = tid >> 2, lk = (tid & 3) * 8;
    for (int k0 = 0; k0 < K; k0 += BK) {
        {
            const int m = m0 + lr;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m < M) v = *reinterpret_cast<const uint4*>(A + (size_t)m * lda + k0 + lk);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                As[lk + 2 * q][lr] = bf_lo(u[q]);
                As[lk + 2 * q + 1][lr] = bf_hi(u[q]);
            }
        }
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int n = n0 + lr;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (n < N) v = *reinterpret_cast<const uint4*>(W + (size_t)(n + w * up_off) * K + k0 + lk);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                Ws[w][lk + 2 * q][lr] = bf_lo(u[q]);
                Ws[w][lk + 2 * q + 1][lr] = bf_hi(u[q]);
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < BK; ++k) {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                float b[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Ws[w][k][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[w][i][j] = fmaf(a[i], b[j], acc[w][i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            const size_t o = (size_t)m * ldc + n;
            if (MODE == GEMM_STORE_F32) Cf[o] = acc[0][i][j];
            else if (MODE == GEMM_ADD_F32) Cf[o] += acc[0][i][j];
            else if (MODE == GEMM_STORE_BF16) Cb[o] = f2bf(acc[0][i][j]);
            else Cb[o] = f2bf(silu(acc[0][i][j]) * acc[NW - 1][i][j]);
        }
    }
}
}  // namespace

cudaError_t launch_gemm_simt(const bf16_t* A, int lda, const bf16_t* W, int M, int N, int K, int mode, int up_off,
                             float* Cf, bf16_t* Cb, int ldc, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (K % BK != 0 || lda % 8 != 0) return cudaErrorInvalidValue;
    dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
    switch (mode) {
        case GEMM_STORE_F32: gemm_simt_kernel<GEMM_STORE_F32><<<grid, NT, 0, s>>>(A, lda, W, M, N, K, up_off, Cf, Cb, ldc); break;
        case GEMM_ADD_F32: gemm_simt_kernel<GEMM_ADD_F32><<<grid, NT, 0, s>>>(A, lda, W, M, N, K, up_off, Cf, Cb, ldc); break;
        case GEMM_SWIGLU_BF16: gemm_simt_kernel<GEMM_SWIGLU_BF16><<<grid, NT, 0, s>>>(A, lda, W, M, N, K, up_off, Cf, Cb, ldc); break;
        case GEMM_STORE_BF16: gemm_simt_kernel<GEMM_STORE_BF16><<<grid, NT, 0, s>>>(A, lda, W, M, N, K, up_off, Cf, Cb, ldc); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qdec
