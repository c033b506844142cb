// Causal GQA attention over the bf16 KV cache.
//
// "Forward map - funasr_nano", LLM decoder table: GQA 16/8 (q head h reads kv head
// h / (HQ/HKV)); "Qwen3ASR ncnn多平台移植" §5: the prefill uses an upper-triangular causal
// mask, each decode step a single-row mask covering the history and itself.
// Scores are q.k / sqrt(D); the softmax is computed online (running max and sum), which
// is the max-subtracted softmax rearranged over key tiles.
#include "common.cuh"

namespace qdec {

namespace {

// ------------------------------------------------------------------ prefill (CUDA cores)
constexpr int PBQ = 32, PBK = 16, PNT = 128, KPT = PBK / 4;   // KPT keys per thread per tile

template <int D>
__global__ void __launch_bounds__(PNT) attn_prefill_simt_kernel(const bf16_t* __restrict__ Q, int T, int HQ, int HKV,
                                                               int max_seq, int pos0,
                                                               const bf16_t* __restrict__ kc,
                                                               const bf16_t* __restrict__ vc,
                                                               bf16_t* __restrict__ O) {
    __shared__ float Qs[PBQ][D];
    __shared__ float Ks[PBK][D + 1];
    __shared__ float Vs[PBK][D];
    __shared__ float Ps[PBQ][PBK + 1];
    const int tid = threadIdx.x, h = blockIdx.y, g = h / (HQ / HKV);
    const int q0 = blockIdx.x * PBQ;
    const int r = tid >> 2, part = tid & 3;          // row of this thread, quarter of the row
    const float scale = rsqrtf((float)D);
    for (int e = tid; e < PBQ * D; e += PNT) {
        const int rr = e / D, d = e % D;
        const int t = q0 + rr;
        Qs[rr][d] = t < T ? bf1(Q[((size_t)t * HQ + h) * D + d]) : 0.f;
    }
    constexpr int DP = D / 4;                          // output dims per thread
    float o[DP];
#pragma unroll
    for (int i = 0; i < DP; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int t_last = min(T, q0 + PBQ) - 1;
    const int key_end = pos0 + t_last + 1;             // keys [0, key_end) can be visible
    const int my_pos = pos0 + q0 + r;
    const bf16_t* kb = kc + (size_t)g * max_seq * D;
    const bf16_t* vb = vc + (size_t)g * max_seq * D;
    for (int j0 = 0; j0 < key_end; j0 += PBK) {
        __syncthreads();
        for (int e = tid; e < PBK * D; e += PNT) {
            const int jj = e / D, d = e % D;
            const int j = j0 + jj;
            Ks[jj][d] = j < key_end ? bf1(kb[(size_t)j * D + d]) : 0.f;
            Vs[jj][d] = j < key_end ? bf1(vb[(size_t)j * D + d]) : 0.f;
        }
        __syncthreads();
        float s[KPT];
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < KPT; ++c) {
            const int jj = part * KPT + c;
            float acc = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) acc = fmaf(Qs[r][d], Ks[jj][d], acc);
            const int j = j0 + jj;
            s[c] = (j <= my_pos && j < key_end) ? acc * scale : -INFINITY;
            tmax = fmaxf(tmax, s[c]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m, tmax);
        const float corr = (m_new == -INFINITY) ? 1.f : expf(m - m_new);
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < KPT; ++c) {
            const float p = (s[c] == -INFINITY) ? 0.f : expf(s[c] - m_new);
            Ps[r][part * KPT + c] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        l = l * corr + psum;
        m = m_new;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < DP; ++i) o[i] *= corr;
        for (int jj = 0; jj < PBK; ++jj) {
            const float p = Ps[r][jj];
#pragma unroll
            for (int i = 0; i < DP; ++i) o[i] = fmaf(p, Vs[jj][part * DP + i], o[i]);
        }
    }
    const int t = q0 + r;
    if (t < T) {
        const float inv = 1.f / l;
        bf16_t* dst = O + (size_t)t * HQ * D + (size_t)h * D + part * DP;
#pragma unroll
        for (int i = 0; i < DP; ++i) dst[i] = f2bf(o[i] * inv);
    }
}

// ------------------------------------------------------------------ decode (split over KV)
constexpr int DNT = 128, DWARPS = DNT / 32;

template <int D, int G>
__global__ void __launch_bounds__(DNT) attn_decode_kernel(const float* __restrict__ q, int max_seq,
                                                          const int* __restrict__ pos,
                                                          const bf16_t* __restrict__ kc,
                                                          const bf16_t* __restrict__ vc, int n_split,
                                                          float* __restrict__ part_ml, float* __restrict__ part_o) {
    constexpr int EPL = D / 32;                       // elements per lane
    __shared__ float sm[DWARPS][G];
    __shared__ float sl[DWARPS][G];
    __shared__ float so[DWARPS][G][D];
    const int gk = blockIdx.x, split = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = *pos + 1;
    const int chunk = (L + n_split - 1) / n_split;
    const int j0 = split * chunk, j1 = min(L, j0 + chunk);
    const float scale = rsqrtf((float)D);
    float qv[G][EPL];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
        for (int e = 0; e < EPL; ++e) qv[gi][e] = q[(gk * G + gi) * D + lane * EPL + e] * scale;
    float m[G], l[G], o[G][EPL];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        m[gi] = -INFINITY;
        l[gi] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[gi][e] = 0.f;
    }
    const bf16_t* kb = kc + (size_t)gk * max_seq * D;
    const bf16_t* vb = vc + (size_t)gk * max_seq * D;
    for (int j = j0 + warp; j < j1; j += DWARPS) {
        float kf[EPL], vf[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            kf[e] = bf1(kb[(size_t)j * D + lane * EPL + e]);
            vf[e] = bf1(vb[(size_t)j * D + lane * EPL + e]);
        }
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) s = fmaf(qv[gi][e], kf[e], s);
            s = warp_sum(s);
            const float m_new = fmaxf(m[gi], s);
            const float corr = expf(m[gi] - m_new);   // m = -inf on the first key gives 0
            const float p = expf(s - m_new);
            l[gi] = l[gi] * corr + p;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[gi][e] = fmaf(p, vf[e], o[gi][e] * corr);
            m[gi] = m_new;
        }
    }
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        if (lane == 0) { sm[warp][gi] = m[gi]; sl[warp][gi] = l[gi]; }
#pragma unroll
        for (int e = 0; e < EPL; ++e) so[warp][gi][lane * EPL + e] = o[gi][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += DNT) {
        const int gi = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < DWARPS; ++w) M = fmaxf(M, sm[w][gi]);
        float lt = 0.f, ot = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < DWARPS; ++w) {
                const float f = expf(sm[w][gi] - M);
                lt += f * sl[w][gi];
                ot += f * so[w][gi][d];
            }
        }
        const int h = gk * G + gi;
        part_o[((size_t)h * n_split + split) * D + d] = ot;
        if (d == 0) {
            part_ml[((size_t)h * n_split + split) * 2 + 0] = M;
            part_ml[((size_t)h * n_split + split) * 2 + 1] = lt;
        }
    }
}

__global__ void attn_decode_merge_kernel(int D, int n_split, const float* __restrict__ part_ml,
                                         const float* __restrict__ part_o, float* __restrict__ out) {
    const int h = blockIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, part_ml[((size_t)h * n_split + s) * 2]);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float lt = 0.f, ot = 0.f;
        for (int s = 0; s < n_split; ++s) {
            const float ms = part_ml[((size_t)h * n_split + s) * 2];
            if (ms == -INFINITY) continue;
            const float f = expf(ms - M);
            lt += f * part_ml[((size_t)h * n_split + s) * 2 + 1];
            ot += f * part_o[((size_t)h * n_split + s) * D + d];
        }
        out[(size_t)h * D + d] = ot / lt;
    }
}

template <int D>
cudaError_t launch_decode_d(const float* q, const Shape& sh, const int* pos, const bf16_t* kc, const bf16_t* vc,
                            int n_split, float* part_ml, float* part_o, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    dim3 grid(sh.HKV, n_split);
    switch (sh.HQ / sh.HKV) {
        case 1: attn_decode_kernel<D, 1><<<grid, DNT, 0, s>>>(q, sh.max_seq, pos, kc, vc, n_split, part_ml, part_o); break;
        case 2: attn_decode_kernel<D, 2><<<grid, DNT, 0, s>>>(q, sh.max_seq, pos, kc, vc, n_split, part_ml, part_o); break;
        case 4: attn_decode_kernel<D, 4><<<grid, DNT, 0, s>>>(q, sh.max_seq, pos, kc, vc, n_split, part_ml, part_o); break;
        case 8: attn_decode_kernel<D, 8><<<grid, DNT, 0, s>>>(q, sh.max_seq, pos, kc, vc, n_split, part_ml, part_o); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_prefill_simt(const bf16_t* Q, int T, const Shape& sh, int pos0, const bf16_t* k_cache,
                                          const bf16_t* v_cache, bf16_t* O, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    dim3 grid((T + PBQ - 1) / PBQ, sh.HQ);
    switch (sh.D) {
        case 32: attn_prefill_simt_kernel<32><<<grid, PNT, 0, s>>>(Q, T, sh.HQ, sh.HKV, sh.max_seq, pos0, k_cache, v_cache, O); break;
        case 64: attn_prefill_simt_kernel<64><<<grid, PNT, 0, s>>>(Q, T, sh.HQ, sh.HKV, sh.max_seq, pos0, k_cache, v_cache, O); break;
        case 128: attn_prefill_simt_kernel<128><<<grid, PNT, 0, s>>>(Q, T, sh.HQ, sh.HKV, sh.max_seq, pos0, k_cache, v_cache, O); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

int attention_decode_splits(const Shape& sh) {
    int s = 256 / sh.HKV;
    return s < 1 ? 1 : (s > 128 ? 128 : s);
}

cudaError_t launch_attention_decode(const float* q, const Shape& sh, const int* pos, const bf16_t* k_cache,
                                    const bf16_t* v_cache, int n_split, float* part_ml, float* part_o, float* out,
                                    cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    cudaError_t e;
    switch (sh.D) {
        case 32: e = launch_decode_d<32>(q, sh, pos, k_cache, v_cache, n_split, part_ml, part_o, s); break;
        case 64: e = launch_decode_d<64>(q, sh, pos, k_cache, v_cache, n_split, part_ml, part_o, s); break;
        case 128: e = launch_decode_d<128>(q, sh, pos, k_cache, v_cache, n_split, part_ml, part_o, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    attn_decode_merge_kernel<<<sh.HQ, 128, 0, s>>>(sh.D, n_split, part_ml, part_o, out);
    return cudaGetLastError();
}

}  // namespace qdec
