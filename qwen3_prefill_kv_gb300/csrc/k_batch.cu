// Lockstep decode of n contexts (one token each): the per-stream pieces of the step.  The
// projections run as one tcgen05 GEMM over all n rows (weights read once per step); these
// kernels handle what is per stream: its token, its position, its KV cache.
//
// "Qwen3ASR ncnn多平台移植" §5: contexts can be cloned so several branches start from one
// prefill state; each step embeds the token, rotates q/k at the stream's own absolute
// position, appends K/V to the stream's cache, attends over that stream's history and picks
// the next token greedily.
#include "common.cuh"

namespace qdec {

namespace {

// Token of stream i: the forced token, or the stream's previous argmax when it is -1.
__global__ void batch_embed_kernel(const bf16_t* __restrict__ E, int H, const int* __restrict__ tokens,
                                   const BatchStream* __restrict__ bs, float* __restrict__ X) {
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x;
    const int t0 = tokens[i];
    const int id = t0 >= 0 ? t0 : *bs[i].argmax;
    const bf16_t* src = E + (size_t)id * H;
    float* dst = X + (size_t)i * H;
    for (int k = threadIdx.x * 4; k < H; k += blockDim.x * 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(src + k);
        *reinterpret_cast<float4*>(dst + k) = make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
    }
    if (threadIdx.x == 0) bs[i].hist[*bs[i].pos] = id;
}

// Per-head RMSNorm + NeoX RoPE of stream s at its position; K/V into its cache of layer l.
// grid (n, HQ + 2 HKV), block max(32, D/2).
__global__ void batch_qk_rope_kernel(const float* __restrict__ qkv, int HQ, int HKV, int D, float eps, int layer,
                                     const bf16_t* __restrict__ g_q, const bf16_t* __restrict__ g_k,
                                     const BatchStream* __restrict__ bs, float* __restrict__ q_out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[4];
    const int s = blockIdx.x, hh = blockIdx.y, i = threadIdx.x, half = D >> 1;
    const int rows = (HQ + 2 * HKV) * D;
    const BatchStream st = bs[s];
    const int p = *st.pos;
    const size_t layer_stride = (size_t)2 * HKV * st.max_seq * D;
    bf16_t* kc = st.kv + (size_t)layer * layer_stride;
    bf16_t* vc = kc + (size_t)HKV * st.max_seq * D;
    const bool act = i < half;
    const float* src = qkv + (size_t)s * rows + (size_t)hh * D;
    float a = act ? src[i] : 0.f, b = act ? src[i + half] : 0.f;
    if (hh >= HQ + HKV) {
        if (act) {
            bf16_t* dst = vc + ((size_t)(hh - HQ - HKV) * st.max_seq + p) * D;
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
    const float2 cs = st.rope[(size_t)p * half + i];
    const float ra = a * cs.x - b * cs.y, rb = b * cs.x + a * cs.y;
    if (hh < HQ) {
        float* dst = q_out + ((size_t)s * HQ + hh) * D;
        dst[i] = ra;
        dst[i + half] = rb;
    } else {
        bf16_t* dst = kc + ((size_t)(hh - HQ) * st.max_seq + p) * D;
        dst[i] = f2bf(ra);
        dst[i + half] = f2bf(rb);
    }
}

constexpr int BNT = 128, BWARPS = BNT / 32;
constexpr int BP = 8;   // key positions a warp loads and scores together

// 2^x with the MUFU instruction (relative error about 2^-22); -inf gives +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The EPL bf16 values of lane `lane` in a D-wide row, widened to fp32.
template <int EPL>
__device__ __forceinline__ void row_lane(const bf16_t* row, int lane, float (&out)[EPL]) {
    if constexpr (EPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 4);
        out[0] = bf_lo(w.x); out[1] = bf_hi(w.x); out[2] = bf_lo(w.y); out[3] = bf_hi(w.y);
    } else if constexpr (EPL == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 2);
        out[0] = bf_lo(w); out[1] = bf_hi(w);
    } else {
        out[0] = bf1(row[lane]);
    }
}

// Split-KV attention of one stream's kv head over its keys [shared, pos + 1).
// grid (HKV, n_split, n); partials [n][HQ][n_split_total] (m, l) and (o[D]), m in log2 units:
// splits [0, n_split) here, the rest written by the shared-prefix kernel.
// Each warp takes groups of BP positions: their K/V loads are all in flight together, the
// BP x G scores are reduced across the warp together, then one online-softmax update
// (exp2 of scores pre-scaled by log2(e)/sqrt(D)) folds the group in.
template <int D, int G>
__global__ void __launch_bounds__(BNT) batch_attn_kernel(const float* __restrict__ q, int HQ, int HKV, int layer,
                                                         const BatchStream* __restrict__ bs, int n_split,
                                                         int n_split_total, float* __restrict__ part_ml,
                                                         float* __restrict__ part_o) {
    pdl_trigger();
    pdl_wait();
    constexpr int EPL = D / 32;
    __shared__ float sm[BWARPS][G];
    __shared__ float sl[BWARPS][G];
    __shared__ float so[BWARPS][G][D];
    const int gk = blockIdx.x, split = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const BatchStream st = bs[s];
    const int L = *st.pos + 1;
    const int chunk = (L - st.shared + n_split - 1) / n_split;   // this stream's own keys [shared, L)
    const int j0 = st.shared + split * chunk, j1 = min(L, j0 + chunk);
    const size_t layer_stride = (size_t)2 * HKV * st.max_seq * D;
    const bf16_t* kb = st.kv + (size_t)layer * layer_stride + (size_t)gk * st.max_seq * D;
    const bf16_t* vb = kb + (size_t)HKV * st.max_seq * D;
    const float scale = rsqrtf((float)D) * 1.4426950408889634f;   // scores in log2 units
    float qv[G][EPL], m[G], l[G], o[G][EPL];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qv[gi][e] = q[((size_t)s * HQ + gk * G + gi) * D + lane * EPL + e] * scale;
            o[gi][e] = 0.f;
        }
        m[gi] = -INFINITY;
        l[gi] = 0.f;
    }
    for (int jb = j0 + warp * BP; jb < j1; jb += BWARPS * BP) {
        float kf[BP][EPL], vf[BP][EPL];
#pragma unroll
        for (int p = 0; p < BP; ++p) {
            const int jj = min(jb + p, j1 - 1);   // past the end: a valid row, weighted 0 below
            row_lane<EPL>(kb + (size_t)jj * D, lane, kf[p]);
            row_lane<EPL>(vb + (size_t)jj * D, lane, vf[p]);
        }
        float sc[BP][G];
#pragma unroll
        for (int p = 0; p < BP; ++p)
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                float d0 = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d0 = fmaf(qv[gi][e], kf[p][e], d0);
                sc[p][gi] = d0;
            }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
            for (int p = 0; p < BP; ++p)
#pragma unroll
                for (int gi = 0; gi < G; ++gi) sc[p][gi] += __shfl_xor_sync(0xffffffffu, sc[p][gi], sh);
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float mx = -INFINITY;
#pragma unroll
            for (int p = 0; p < BP; ++p)
                if (jb + p < j1) mx = fmaxf(mx, sc[p][gi]);
            const float mn = fmaxf(m[gi], mx);   // finite: position jb is always valid
            const float corr = ex2(m[gi] - mn);  // 0 while m is -inf
            float psum = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[gi][e] *= corr;
#pragma unroll
            for (int p = 0; p < BP; ++p) {
                const float pr = (jb + p < j1) ? ex2(sc[p][gi] - mn) : 0.f;
                psum += pr;
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[gi][e] = fmaf(pr, vf[p][e], o[gi][e]);
            }
            l[gi] = l[gi] * corr + psum;
            m[gi] = mn;
        }
    }
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        if (lane == 0) {
            sm[warp][gi] = m[gi];
            sl[warp][gi] = l[gi];
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) so[warp][gi][lane * EPL + e] = o[gi][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += BNT) {
        const int gi = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < BWARPS; ++w) M = fmaxf(M, sm[w][gi]);
        float lt = 0.f, ot = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < BWARPS; ++w) {
                const float f = ex2(sm[w][gi] - M);
                lt += f * sl[w][gi];
                ot += f * so[w][gi][d];
            }
        }
        const size_t base = ((size_t)s * HQ + gk * G + gi) * n_split_total + split;
        part_o[base * D + d] = ot;
        if (d == 0) {
            part_ml[base * 2 + 0] = M;
            part_ml[base * 2 + 1] = lt;
        }
    }
}

// Merge of the splits; writes the attention output bf16 [n, HQ * D] (the o_proj GEMM operand).
// A stream without a shared prefix has only its own n_split splits; one with a shared prefix
// also has the prefix kernel's splits [n_split, n_split_total).
__global__ void batch_attn_merge_kernel(int HQ, int D, int n_split_own, int n_split_total,
                                        const BatchStream* __restrict__ bs, const float* __restrict__ part_ml,
                                        const float* __restrict__ part_o, bf16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int h = blockIdx.x, s = blockIdx.y;
    const size_t base = ((size_t)s * HQ + h) * n_split_total;
    const int n_split = bs[s].shared > 0 ? n_split_total : n_split_own;
    float M = -INFINITY;
    for (int k = 0; k < n_split; ++k) M = fmaxf(M, part_ml[(base + k) * 2]);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float lt = 0.f, ot = 0.f;
        for (int k = 0; k < n_split; ++k) {
            const float mk = part_ml[(base + k) * 2];
            if (mk == -INFINITY) continue;
            const float f = ex2(mk - M);
            lt += f * part_ml[(base + k) * 2 + 1];
            ot += f * part_o[(base + k) * D + d];
        }
        out[((size_t)s * HQ + h) * D + d] = f2bf(ot / lt);
    }
}

// h = silu(gate) * up from the fp32 [n, 2F] projection (gate columns first), bf16 [n, F].
// One thread per pair of columns (F even) over all n rows.
__global__ void batch_swiglu_kernel(const float* __restrict__ gu, int F, int n, bf16_t* __restrict__ h, int splits,
                                    size_t pstride) {
    pdl_trigger();
    pdl_wait();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;   // pair index
    const int half = F >> 1;
    if (idx >= n * half) return;
    const int s = idx / half, j = 2 * (idx - s * half);
    float2 g = *reinterpret_cast<const float2*>(gu + (size_t)s * 2 * F + j);
    float2 u = *reinterpret_cast<const float2*>(gu + (size_t)s * 2 * F + F + j);
    for (int z = 1; z < splits; ++z) {   // split-K partial slabs, added in order
        const float2 g2 = *reinterpret_cast<const float2*>(gu + z * pstride + (size_t)s * 2 * F + j);
        const float2 u2 = *reinterpret_cast<const float2*>(gu + z * pstride + (size_t)s * 2 * F + F + j);
        g.x += g2.x; g.y += g2.y; u.x += u2.x; u.y += u2.y;
    }
    *reinterpret_cast<uint32_t*>(h + (size_t)s * F + j) = pack_bf2(silu(g.x) * u.x, silu(g.y) * u.y);
}

// Argmax of each logits row (lowest index on ties), into the stream's argmax and out[s];
// then the stream's position advances.
__global__ void batch_argmax_kernel(const float* __restrict__ logits, int V, int ld, const BatchStream* __restrict__ bs,
                                    int* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float bv[32];
    __shared__ int bi[32];
    const int s = blockIdx.x;
    const float* z = logits + (size_t)s * ld;
    float b = -INFINITY;
    int ib = 0x7fffffff;
    for (int j = threadIdx.x; j < V; j += blockDim.x) {
        const float v = z[j];
        if (am_better(v, j, b, ib)) {
            b = v;
            ib = j;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, b, o);
        const int i = __shfl_xor_sync(0xffffffffu, ib, o);
        if (am_better(v, i, b, ib)) {
            b = v;
            ib = i;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        bv[warp] = b;
        bi[warp] = ib;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (am_better(bv[w], bi[w], b, ib)) {
                b = bv[w];
                ib = bi[w];
            }
        const int a = (ib == 0x7fffffff) ? 0 : ib;
        *bs[s].argmax = a;
        out[s] = a;
        *bs[s].pos += 1;
    }
}

template <int D>
cudaError_t launch_attn_d(const float* q, int HQ, int HKV, int layer, const BatchStream* bs, int n, int n_split,
                          int nst, float* part_ml, float* part_o, cudaStream_t st) {
    dim3 grid(HKV, n_split, n);
    switch (HQ / HKV) {
        case 1: return launch_pdl(batch_attn_kernel<D, 1>, grid, dim3(BNT), 0, st, q, HQ, HKV, layer, bs, n_split, nst, part_ml, part_o);
        case 2: return launch_pdl(batch_attn_kernel<D, 2>, grid, dim3(BNT), 0, st, q, HQ, HKV, layer, bs, n_split, nst, part_ml, part_o);
        case 4: return launch_pdl(batch_attn_kernel<D, 4>, grid, dim3(BNT), 0, st, q, HQ, HKV, layer, bs, n_split, nst, part_ml, part_o);
        case 8: return launch_pdl(batch_attn_kernel<D, 8>, grid, dim3(BNT), 0, st, q, HQ, HKV, layer, bs, n_split, nst, part_ml, part_o);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_batch_embed(const bf16_t* E, int H, const int* tokens, const BatchStream* bs, int n, float* X,
                               cudaStream_t st) {
    (void)cudaGetLastError();
    return launch_pdl(batch_embed_kernel, dim3(n), dim3(128), 0, st, E, H, tokens, bs, X);
}

cudaError_t launch_batch_qk_rope(const float* qkv, const Shape& sh, int layer, const bf16_t* g_q, const bf16_t* g_k,
                                 const BatchStream* bs, int n, float* q_out, cudaStream_t st) {
    (void)cudaGetLastError();
    dim3 grid(n, sh.HQ + 2 * sh.HKV);
    return launch_pdl(batch_qk_rope_kernel, grid, dim3(sh.D / 2 < 32 ? 32 : sh.D / 2), 0, st, qkv, sh.HQ, sh.HKV, sh.D,
                      sh.eps, layer, g_q, g_k, bs, q_out);
}

cudaError_t launch_batch_attention(const float* q, const Shape& sh, int layer, const BatchStream* bs, int n, int n_split,
                                   const PrefixItem* items, int n_items, const int* members, int max_chunks,
                                   float* part_ml, float* part_o, bf16_t* out, cudaStream_t st) {
    (void)cudaGetLastError();
    const int nst = n_split + (n_items > 0 ? max_chunks : 0);
    cudaError_t e;
    switch (sh.D) {
        case 32: e = launch_attn_d<32>(q, sh.HQ, sh.HKV, layer, bs, n, n_split, nst, part_ml, part_o, st); break;
        case 64: e = launch_attn_d<64>(q, sh.HQ, sh.HKV, layer, bs, n, n_split, nst, part_ml, part_o, st); break;
        case 128: e = launch_attn_d<128>(q, sh.HQ, sh.HKV, layer, bs, n, n_split, nst, part_ml, part_o, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    if (n_items > 0) {
        e = launch_prefix_attention(q, sh, layer, items, n_items, members, max_chunks, nst, n_split, part_ml, part_o, st);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(batch_attn_merge_kernel, dim3(sh.HQ, n), dim3(128), 0, st, sh.HQ, sh.D, n_split, nst, bs, part_ml,
                      part_o, out);
}

cudaError_t launch_batch_swiglu(const float* gu, int F, int n, bf16_t* h, cudaStream_t st, int splits, size_t pstride) {
    (void)cudaGetLastError();
    if (F % 2 != 0 || splits < 1 || pstride % 2 != 0) return cudaErrorInvalidValue;
    const int pairs = n * (F / 2);
    return launch_pdl(batch_swiglu_kernel, dim3((pairs + 255) / 256), dim3(256), 0, st, gu, F, n, h, splits, pstride);
}

cudaError_t launch_batch_argmax(const float* logits, int V, int ld, const BatchStream* bs, int n, int* out,
                                cudaStream_t st) {
    (void)cudaGetLastError();
    return launch_pdl(batch_argmax_kernel, dim3(n), dim3(1024), 0, st, logits, V, ld, bs, out);
}

}  // namespace qdec
