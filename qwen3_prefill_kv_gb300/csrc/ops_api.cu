// Per-kernel C entry points (include/qdec_ops.h).
#include "../../include/qdec.h"
#include "../../include/qdec_ops.h"
#include "common.cuh"

using namespace qdec;

namespace {
int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return QDEC_OK;
    return set_error(QDEC_E_CUDA, "kernel launch: %s", cudaGetErrorString(e));
}
}

extern "C" {

int qdec_op_gemm(const void* A, int32_t lda, const void* W, int32_t M, int32_t N, int32_t K, int32_t mode,
                 int32_t up_off, void* C, int32_t ldc, int32_t impl, void* stream) {
    if (!A || !W || !C || M <= 0 || N <= 0 || K <= 0 || mode < 0 || mode > 4)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_gemm: null pointer or bad size/mode");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool f32 = (mode == QDEC_GEMM_STORE_F32 || mode == QDEC_GEMM_ADD_F32 || mode == QDEC_GEMM_ATOMIC_F32);
    float* Cf = f32 ? static_cast<float*>(C) : nullptr;
    bf16_t* Cb = f32 ? nullptr : static_cast<bf16_t*>(C);
    if (impl == QDEC_IMPL_SIMT) {
        if (mode == QDEC_GEMM_ATOMIC_F32) return set_error(QDEC_E_UNSUPPORTED, "the atomic mode is tcgen05-only");
        if (K % 32 != 0 || lda % 8 != 0) return set_error(QDEC_E_UNSUPPORTED, "SIMT GEMM needs K %% 32 == 0, lda %% 8 == 0");
        return cuda_status(launch_gemm_simt(static_cast<const bf16_t*>(A), lda, static_cast<const bf16_t*>(W), M, N,
                                            K, mode, up_off, Cf, Cb, ldc, s));
    }
    if (impl == QDEC_IMPL_TCGEN05) {
        if (!gemm_tc_supported(N, K, mode, lda))
            return set_error(QDEC_E_UNSUPPORTED, "tcgen05 GEMM needs K %% 64 == 0, N %% 128 == 0 (SwiGLU: %% 64)");
        if (reinterpret_cast<uintptr_t>(C) % 16 != 0 || ((size_t)ldc * (f32 ? 4 : 2)) % 16 != 0 || ldc < N)
            return set_error(QDEC_E_UNSUPPORTED, "tcgen05 GEMM needs C 16-byte aligned, ldc >= N, rows 16-byte multiples");
        return cuda_status(launch_gemm_tc(static_cast<const bf16_t*>(A), lda, static_cast<const bf16_t*>(W), M, N, K,
                                          mode, up_off, Cf, Cb, ldc, s));
    }
    return set_error(QDEC_E_INVALID_ARG, "unknown impl %d", impl);
}

int qdec_op_gemm_splitk(const void* A, int32_t lda, const void* W, int32_t M, int32_t N, int32_t K, int32_t splits,
                        float* C, int32_t ldc, void* stream) {
    if (!A || !W || !C || M <= 0 || N <= 0 || K <= 0 || splits < 1)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_gemm_splitk: null pointer or bad size");
    if (!gemm_tc_supported(N, K, GEMM_ATOMIC_F32, lda))
        return set_error(QDEC_E_UNSUPPORTED, "tcgen05 GEMM needs K %% 64 == 0, N %% 128 == 0");
    return cuda_status(launch_gemm_tc(static_cast<const bf16_t*>(A), lda, static_cast<const bf16_t*>(W), M, N, K,
                                      GEMM_ATOMIC_F32, 0, C, nullptr, ldc, static_cast<cudaStream_t>(stream), splits));
}

int qdec_op_programmatic_launch(int32_t on) {
    if (on != 0 && on != 1) return set_error(QDEC_E_INVALID_ARG, "qdec_op_programmatic_launch: %d is not 0 or 1", on);
    return set_programmatic_launch(on);
}

int qdec_op_gemm_tile_rows(int32_t bm) {
    if (bm != 0 && bm != 128 && bm != 256)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_gemm_tile_rows: %d is not 0, 128 or 256", bm);
    return set_gemm_tile_rows(bm);
}

int qdec_op_gemm_tile_width(int32_t bn) {
    if (bn != 0 && bn != 128 && bn != 256)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_gemm_tile_width: %d is not 0, 128 or 256", bn);
    return set_gemm_tile_width(bn);
}

int qdec_op_sample(const float* logits, int32_t V, const int32_t* history, int32_t n_history, float temperature,
                   int32_t top_k, float top_p, float repetition_penalty, uint64_t seed, int32_t pos, int32_t* token,
                   void* stream) {
    if (!logits || !token || n_history < 0 || (n_history > 0 && !history) || pos < 0)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_sample: null pointer or negative size/position");
    if (!sample_params_valid(V, temperature, top_k, top_p, repetition_penalty))
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_sample: temperature >= 0, top_k >= 0, 0 < top_p <= 1, "
                                             "penalty > 0, 0 < V <= %d", kSampleMaxVocab);
    return cuda_status(launch_sample(logits, V, history, n_history, temperature, top_k, top_p, repetition_penalty,
                                     (unsigned long long)seed, pos, token, static_cast<cudaStream_t>(stream)));
}

int qdec_op_quantize(const void* W, int32_t N, int32_t K, int32_t fmt, void* codes, void* scales, void* stream) {
    if (!W || !codes || !scales || N <= 0 || K <= 0 || K % 32 != 0 || (fmt != 1 && fmt != 2))
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_quantize: null pointer, bad size or format");
    cudaError_t e = launch_quantize(static_cast<const bf16_t*>(W), N, K, fmt == 1 ? QUANT_Q8B32 : QUANT_Q4B32, codes,
                                    scales, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QDEC_OK : set_error(QDEC_E_CUDA, "qdec_op_quantize: %s", cudaGetErrorString(e));
}

int qdec_op_gemv_q(const void* codes, const void* scales, int32_t fmt, int32_t rows, int32_t K, const float* x,
                   const void* norm_g, float eps, int32_t mode, int32_t up_off, float* y, void* stream) {
    if (!codes || !scales || !x || !y || rows <= 0 || K <= 0 || K % 256 != 0 || (fmt != 1 && fmt != 2) || mode < 0 ||
        mode > 2)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_gemv_q: null pointer, bad size, format or mode");
    cudaError_t e = launch_gemv_q(codes, scales, fmt == 1 ? QUANT_Q8B32 : QUANT_Q4B32, rows, K, x,
                                  static_cast<const bf16_t*>(norm_g), eps, mode, up_off, y,
                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QDEC_OK : set_error(QDEC_E_CUDA, "qdec_op_gemv_q: %s", cudaGetErrorString(e));
}

int qdec_op_device_error(void) {
    const int v1 = tc_error_read_and_clear(), v2 = fa_error_read_and_clear();
    if (v1 < 0 || v2 < 0) return set_error(QDEC_E_CUDA, "reading the device error word failed");
    const int v = v1 ? v1 : v2;
    return v ? set_error(QDEC_E_TIMEOUT, "a tensor-core kernel gave up waiting (code %d)", v) : QDEC_OK;
}

int qdec_op_attention_prefill(const void* Q, int32_t T, int32_t HQ, int32_t HKV, int32_t D, int32_t max_seq,
                              int32_t pos0, const void* k_cache, const void* v_cache, void* O, int32_t impl,
                              void* stream) {
    if (!Q || !k_cache || !v_cache || !O || T <= 0 || HQ <= 0 || HKV <= 0 || HQ % HKV != 0 || pos0 < 0 ||
        pos0 + T > max_seq)
        return QDEC_E_INVALID_ARG;
    Shape sh{};
    sh.HQ = HQ;
    sh.HKV = HKV;
    sh.D = D;
    sh.max_seq = max_seq;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (impl == QDEC_IMPL_SIMT)
        return cuda_status(launch_attention_prefill_simt(static_cast<const bf16_t*>(Q), T, sh, pos0,
                                                         static_cast<const bf16_t*>(k_cache),
                                                         static_cast<const bf16_t*>(v_cache), static_cast<bf16_t*>(O), s));
    if (impl == QDEC_IMPL_TCGEN05) {
        if (!attention_tc_supported(sh)) return set_error(QDEC_E_UNSUPPORTED, "tcgen05 attention needs head_dim 128");
        return cuda_status(launch_attention_prefill_tc(static_cast<const bf16_t*>(Q), T, sh, pos0,
                                                       static_cast<const bf16_t*>(k_cache),
                                                       static_cast<const bf16_t*>(v_cache), static_cast<bf16_t*>(O), s));
    }
    return set_error(QDEC_E_INVALID_ARG, "unknown impl %d", impl);
}

size_t qdec_op_lm_head_scratch_bytes(int32_t V) { return V > 0 ? lm_head_scratch_bytes(V) : 0; }

int qdec_op_lm_head_argmax(const void* E, int32_t V, int32_t H, const float* x, const void* g_final, float eps,
                           float* logits, int32_t* argmax, void* scratch, size_t scratch_bytes, void* stream) {
    if (!E || !x || !g_final || !logits || !argmax || !scratch || V <= 0 || H <= 0 || H % 8 != 0)
        return QDEC_E_INVALID_ARG;
    if (scratch_bytes < lm_head_scratch_bytes(V)) return QDEC_E_INVALID_ARG;
    return cuda_status(launch_lm_head_argmax(static_cast<const bf16_t*>(E), V, H, x,
                                             static_cast<const bf16_t*>(g_final), eps, logits, argmax, scratch,
                                             static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
