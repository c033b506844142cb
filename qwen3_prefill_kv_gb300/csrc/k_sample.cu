// The token choice after the tied lm_head: greedy, or sampling with repetition penalty,
// temperature, top-k and top-p and a counter-based draw ("Qwen3ASR ncnn多平台移植" §1: the
// context supports greedy, temperature, top-k, top-p and repetition penalty; §6: greedy is
// the default, the others serve non-deterministic generation).  The page names the options
// without defining them; the definitions taken, in order:
//   1. repetition penalty r over the distinct ids of the history: a positive logit / r,
//      a non-positive one * r;
//   2. temperature T (T = 0: greedy argmax, lowest index on ties);
//   3. top-k: keep the logits >= the k-th largest (ties kept);
//   4. top-p: keep a token while the probability mass of the kept tokens strictly more
//      probable than it is < p (ties kept);
//   5. u = top 24 bits of splitmix64 output pos + 1 from state `seed`; the token is the
//      smallest kept id whose cumulative kept probability (in id order) exceeds u * total.
//
// One CTA of 1024 threads per choice.  Logits are re-read from global memory (L2) on each
// pass and transformed the same way every time.  Top-k and top-p thresholds are found by
// radix selection over an order-preserving 32-bit key of the transformed logit (four passes
// of 8 bits); probabilities enter the top-p search and the draw as 32.32 fixed-point
// integers, so every sum is exact and the choice is deterministic.
#include "common.cuh"

namespace qdec {

namespace {

constexpr int ST = 1024;   // threads
constexpr int SW = ST / 32;

struct SampleArgs {
    const float* logits;
    int V;
    const int* hist;
    int n_hist;
    float temperature, top_p, penalty;
    int top_k;
    unsigned long long seed;
    int pos;
    int* token;
};

__device__ __forceinline__ unsigned long long splitmix64_mix(unsigned long long z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Order-preserving 32-bit key of a float (larger float -> larger key).
__device__ __forceinline__ uint32_t fkey(float t) {
    const uint32_t u = __float_as_uint(t);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <typename T>
__device__ T block_sum(T v, T* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    T r = 0;
    for (int i = 0; i < SW; ++i) r += red[i];
    return r;
}

__global__ void __launch_bounds__(ST, 1) sample_kernel(const SampleArgs a) {
    extern __shared__ uint32_t seen[];               // history bitmap, (V + 31) / 32 words
    __shared__ unsigned long long red64[SW];
    __shared__ float redf[SW];
    __shared__ int redi[SW];
    __shared__ unsigned int hcnt[256];
    __shared__ unsigned long long hmass[256];
    __shared__ uint32_t sel[2];                      // [0]: chosen byte, [1]: unused
    __shared__ unsigned long long sabove;
    const int tid = threadIdx.x, V = a.V;
    const int words = (V + 31) >> 5;
    for (int i = tid; i < words; i += ST) seen[i] = 0u;
    __syncthreads();
    if (a.penalty != 1.0f)
        for (int i = tid; i < a.n_hist; i += ST) {
            const int id = a.hist[i];
            if (id >= 0 && id < V) atomicOr(&seen[id >> 5], 1u << (id & 31));
        }
    __syncthreads();
    // 1. the penalised logit of id i (the same arithmetic on every pass)
    auto pen = [&](int i) -> float {
        float z = __ldg(a.logits + i);
        if (a.penalty != 1.0f && ((seen[i >> 5] >> (i & 31)) & 1u)) z = z > 0.f ? z / a.penalty : z * a.penalty;
        return z;
    };
    if (a.temperature == 0.0f) {   // 2. greedy: lowest index among the largest (NaN never wins)
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += ST) {
            const float z = pen(i);
            if (am_better(z, i, bv, bi)) { bv = z; bi = i; }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (am_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if ((tid & 31) == 0) { redf[tid >> 5] = bv; redi[tid >> 5] = bi; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < SW; ++w)
                if (am_better(redf[w], redi[w], redf[0], redi[0])) { redf[0] = redf[w]; redi[0] = redi[w]; }
            *a.token = redi[0] == 0x7fffffff ? 0 : redi[0];
        }
        return;
    }
    const float invT = 1.0f / a.temperature;
    auto tkey = [&](int i) -> uint32_t { return fkey(pen(i) * invT); };
    // max of the tempered logits (the softmax reference)
    float mx = -INFINITY;
    for (int i = tid; i < V; i += ST) mx = fmaxf(mx, pen(i) * invT);
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) redf[tid >> 5] = mx;
    __syncthreads();
    mx = redf[0];
    for (int w = 1; w < SW; ++w) mx = fmaxf(mx, redf[w]);
    __syncthreads();
    // 3. top-k: the k-th largest key by radix selection (ties at that key are kept)
    uint32_t kmin = 0u;
    if (a.top_k > 0 && a.top_k < V) {
        uint32_t prefix = 0u;
        unsigned int need = (unsigned int)a.top_k;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int b = tid; b < 256; b += ST) hcnt[b] = 0u;
            __syncthreads();
            const uint32_t hmask = shift == 24 ? 0u : ~((1u << (shift + 8)) - 1u);
            for (int i = tid; i < V; i += ST) {
                const uint32_t k = tkey(i);
                if ((k & hmask) == (prefix & hmask)) atomicAdd(&hcnt[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid == 0) {
                unsigned int cum = 0u;
                int b = 255;
                for (; b > 0; --b) {
                    if (cum + hcnt[b] >= need) break;
                    cum += hcnt[b];
                }
                sel[0] = (uint32_t)b;
                sel[1] = need - cum;
            }
            __syncthreads();
            prefix |= sel[0] << shift;
            need = sel[1];
            __syncthreads();
        }
        kmin = prefix;
    }
    // probabilities exp(t - max) as 32.32 fixed point over the top-k set
    auto mass = [&](int i, uint32_t k) -> unsigned long long {
        if (k < kmin) return 0ull;
        const float w = __expf(pen(i) * invT - mx);
        return __float2ull_rz(w * 4294967296.0f);
    };
    unsigned long long part = 0ull;
    for (int i = tid; i < V; i += ST) part += mass(i, tkey(i));
    const unsigned long long S = block_sum(part, red64);
    // 4. top-p: the smallest kept key K0 (mass of kept keys strictly above it < p * S), by
    // radix selection from the top: a bin holds a kept key when the mass above its largest
    // key is below the bound; the lowest such non-empty bin holds K0
    uint32_t pmin = kmin;
    if (a.top_p < 1.0f) {
        const double P = (double)a.top_p * (double)S;
        uint32_t prefix = 0u;
        if (tid == 0) sabove = 0ull;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int b = tid; b < 256; b += ST) { hcnt[b] = 0u; hmass[b] = 0ull; }
            __syncthreads();
            const uint32_t hmask = shift == 24 ? 0u : ~((1u << (shift + 8)) - 1u);
            for (int i = tid; i < V; i += ST) {
                const uint32_t k = tkey(i);
                if (k >= kmin && (k & hmask) == (prefix & hmask)) {
                    atomicAdd(&hcnt[(k >> shift) & 255u], 1u);
                    atomicAdd(&hmass[(k >> shift) & 255u], mass(i, k));
                }
            }
            __syncthreads();
            if (tid == 0) {
                unsigned long long above = sabove, acc = 0ull;
                int chosen = -1;
                unsigned long long above_chosen = above;
                for (int b = 255; b >= 0; --b) {
                    if (hcnt[b] == 0u) continue;
                    if ((double)(above + acc) < P) {
                        chosen = b;
                        above_chosen = above + acc;
                    } else {
                        break;
                    }
                    acc += hmass[b];
                }
                if (chosen < 0) {   // cannot happen for p > 0 (the largest key is always kept)
                    for (int b = 255; b >= 0; --b)
                        if (hcnt[b]) { chosen = b; break; }
                    above_chosen = above;
                }
                sel[0] = (uint32_t)chosen;
                sabove = above_chosen;
            }
            __syncthreads();
            prefix |= sel[0] << shift;
            __syncthreads();
        }
        pmin = prefix;
    }
    // 5. the draw: smallest kept id whose cumulative fixed-point mass (id order) exceeds u * total
    const int seg = (V + ST - 1) / ST, i0 = min(V, tid * seg), i1 = min(V, i0 + seg);
    unsigned long long loc = 0ull;
    for (int i = i0; i < i1; ++i) {
        const uint32_t k = tkey(i);
        if (k >= pmin) loc += mass(i, k);
    }
    // exclusive scan of the segment sums over the block
    unsigned long long incl = loc;
    const int lane = tid & 31, w = tid >> 5;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) red64[w] = incl;
    __syncthreads();
    unsigned long long wbase = 0ull;
    for (int q = 0; q < w; ++q) wbase += red64[q];
    const unsigned long long base = wbase + incl - loc;
    unsigned long long total = 0ull;
    for (int q = 0; q < SW; ++q) total += red64[q];
    const unsigned long long bits = splitmix64_mix(a.seed + (unsigned long long)(a.pos + 1) * 0x9E3779B97F4A7C15ull);
    const double u = (double)(bits >> 40) * (1.0 / 16777216.0);
    const double target = u * (double)total;
    __shared__ int found;
    if (tid == 0) found = 0x7fffffff;
    __syncthreads();
    if ((double)base <= target && (double)(base + loc) > target) {
        unsigned long long run = base;
        for (int i = i0; i < i1; ++i) {
            const uint32_t k = tkey(i);
            if (k < pmin) continue;
            run += mass(i, k);
            if ((double)run > target) {
                atomicMin(&found, i);
                break;
            }
        }
    }
    // the last kept id, should rounding leave no crossing
    int last = -1;
    for (int i = tid; i < V; i += ST)
        if (tkey(i) >= pmin && mass(i, tkey(i)) > 0ull) last = max(last, i);
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (lane == 0) redi[w] = last;
    __syncthreads();
    if (tid == 0) {
        int l = -1;
        for (int q = 0; q < SW; ++q) l = max(l, redi[q]);
        int t = found != 0x7fffffff ? found : l;
        *a.token = t < 0 ? 0 : t;
    }
}

}  // namespace

bool sample_params_valid(int V, float temperature, int top_k, float top_p, float penalty) {
    return V > 0 && V <= kSampleMaxVocab && temperature >= 0.f && penalty > 0.f && top_p > 0.f && top_p <= 1.f &&
           top_k >= 0 && temperature == temperature && penalty == penalty && top_p == top_p;
}

cudaError_t launch_sample(const float* logits, int V, const int* hist, int n_hist, float temperature, int top_k,
                          float top_p, float penalty, unsigned long long seed, int pos, int* token, cudaStream_t s) {
    (void)cudaGetLastError();   // attribute only this launch's errors
    if (!logits || !token || (n_hist > 0 && !hist) || n_hist < 0 ||
        !sample_params_valid(V, temperature, top_k, top_p, penalty))
        return cudaErrorInvalidValue;
    const SampleArgs args{logits, V, hist, n_hist, temperature, top_p, penalty, top_k, seed, pos, token};
    const size_t smem = (size_t)((V + 31) / 32) * 4;
    sample_kernel<<<1, ST, smem, s>>>(args);
    return cudaGetLastError();
}

}  // namespace qdec
