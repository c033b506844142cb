// Shared-prefix attention of a lockstep batch: the part of every stream's attention that
// covers a KV prefix its clones hold in common.
//
// "Qwen3ASR ncnn多平台移植" §5: generation clones its input context, so several branches start
// from one prefill state.  The clones of one prefill hold the same keys and values at the
// prompt positions [0, P) (a clone is a byte copy, and a decode step only writes at or past
// its own position >= P).  Each stream's attention over [0, P) is therefore the same
// product for every stream except for its query: this kernel reads the prefix keys and values
// of one kv head ONCE, from one member's cache, for the queries of all member streams (up to
// 128 query rows: streams x q heads of the group), and leaves per-stream (max, sum, output)
// partials that the batch merge folds together with the stream's own tail [P, L).
//
// GB300 design: one CTA per (kv head, 32-key chunk of the prefix, block of up to 128 query
// rows); 8 warps, warp w owns 16 query rows.  Scores S = Q K^T and O += P V run on the tensor
// cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation), the operands read from
// XOR-swizzled shared memory with ldmatrix; the softmax is online, in log2 units, with P
// rounded to bf16 for the second product (the same precision reading as the prefill's
// flash attention).
#include "common.cuh"

namespace qdec {

namespace {

constexpr int PX_WARPS = 8, PX_THREADS = 32 * PX_WARPS;
constexpr int PX_ROWS = 16 * PX_WARPS;   // query rows per CTA
constexpr int PX_KEYS = 32;              // keys per CTA
constexpr int PX_D = 128;                // head dim this kernel covers

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of 16-byte chunk `ch` (0..15) of row `r` in a [rows][128] bf16 tile whose
// chunks are XOR-swizzled by the row (conflict-free ldmatrix over 8 consecutive rows).
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 256 + ((ch ^ (r & 7)) << 4)); }

__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// grid (HKV, ceil(P_max / 32), n_items), PX_THREADS threads.
template <int G>
__global__ void __launch_bounds__(PX_THREADS) prefix_attn_kernel(const float* __restrict__ q, int HQ, int HKV,
                                                                  int layer, int max_seq,
                                                                  const PrefixItem* __restrict__ items,
                                                                  const int* __restrict__ members, int n_split_total,
                                                                  int split0, float* __restrict__ part_ml,
                                                                  float* __restrict__ part_o) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(1024) unsigned char px_smem[];
    unsigned char* Qs = px_smem;                              // [128 rows][128] bf16, swizzled
    unsigned char* Ks = px_smem + PX_ROWS * 256;              // [32 keys][128]
    unsigned char* Vs = Ks + PX_KEYS * 256;                   // [32 keys][128]
    const int hk = blockIdx.x, chunk = blockIdx.y;
    const PrefixItem it = items[blockIdx.z];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j0 = chunk * PX_KEYS, j1 = min(it.P, j0 + PX_KEYS);
    const int rows = it.count * G;
    if (j0 >= it.P) {   // this item's prefix is shorter: an empty partial
        for (int r = threadIdx.x; r < rows; r += PX_THREADS) {
            const int s = members[it.first + r / G], h = hk * G + r % G;
            const size_t base = ((size_t)s * HQ + h) * n_split_total + split0 + chunk;
            part_ml[base * 2] = -INFINITY;
            part_ml[base * 2 + 1] = 0.f;
        }
        return;
    }
    // queries, pre-scaled into log2 units, rounded to bf16
    const float scale = rsqrtf((float)PX_D) * 1.4426950408889634f;
    for (int idx = threadIdx.x; idx < PX_ROWS * 16; idx += PX_THREADS) {
        const int r = idx >> 4, ch = idx & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) {
            const int s = members[it.first + r / G], h = hk * G + r % G;
            const float4* src = reinterpret_cast<const float4*>(q + ((size_t)s * HQ + h) * PX_D + ch * 8);
            const float4 a = src[0], b = src[1];
            v = make_uint4(pack_bf2(a.x * scale, a.y * scale), pack_bf2(a.z * scale, a.w * scale),
                           pack_bf2(b.x * scale, b.y * scale), pack_bf2(b.z * scale, b.w * scale));
        }
        *reinterpret_cast<uint4*>(Qs + swz(r, ch)) = v;
    }
    // the chunk's keys and values from the item's cache (rows past the prefix: zeros, masked below)
    const size_t layer_stride = (size_t)2 * HKV * max_seq * PX_D;
    const bf16_t* kb = it.kv + (size_t)layer * layer_stride + (size_t)hk * max_seq * PX_D;
    const bf16_t* vb = kb + (size_t)HKV * max_seq * PX_D;
    for (int idx = threadIdx.x; idx < PX_KEYS * 16; idx += PX_THREADS) {
        const int r = idx >> 4, ch = idx & 15, j = j0 + r;
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (j < j1) {
            kv = *reinterpret_cast<const uint4*>(kb + (size_t)j * PX_D + ch * 8);
            vv = *reinterpret_cast<const uint4*>(vb + (size_t)j * PX_D + ch * 8);
        }
        *reinterpret_cast<uint4*>(Ks + swz(r, ch)) = kv;
        *reinterpret_cast<uint4*>(Vs + swz(r, ch)) = vv;
    }
    __syncthreads();
    if (16 * warp >= rows) return;   // no query rows for this warp (no barrier follows)

    // Q fragments of this warp's 16 rows: 8 k-steps of 16 dims
    uint32_t qa[8][4];
    {
        const int r = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) ldsm4(su32(Qs) + swz(r, 2 * ks + (lane >> 4)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }
    float o[16][4];
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows g and g + 8 of this lane
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int kb16 = 0; kb16 < PX_KEYS; kb16 += 16) {
        // S[16 x 16 keys] = Q K^T: two n-tiles of 8 keys
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int key = kb16 + (lane & 7) + 8 * (lane >> 4);
            const int half = (lane >> 3) & 1;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm4(su32(Ks) + swz(key, 2 * ks + half), b00, b01, b10, b11);
                mma16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
                mma16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
            }
        }
        // mask keys past the prefix; online softmax per row (quad-wide maxima)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (j0 + kb16 + nt * 8 + 2 * t4 + (e & 1) >= j1) sc[nt][e] = -INFINITY;
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);   // finite: key j0 is always in range
        const float c0 = ex2f(m0 - n0), c1 = ex2f(m1 - n1);     // 0 while m was -inf
        m0 = n0;
        m1 = n1;
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            p[nt][0] = ex2f(sc[nt][0] - n0);
            p[nt][1] = ex2f(sc[nt][1] - n0);
            p[nt][2] = ex2f(sc[nt][2] - n1);
            p[nt][3] = ex2f(sc[nt][3] - n1);
        }
        // P in bf16 for the second product; the sums take the same rounded values
        uint32_t pa[4];
        pa[0] = pack_bf2(p[0][0], p[0][1]);
        pa[1] = pack_bf2(p[0][2], p[0][3]);
        pa[2] = pack_bf2(p[1][0], p[1][1]);
        pa[3] = pack_bf2(p[1][2], p[1][3]);
        l0 = l0 * c0 + bf_lo(pa[0]) + bf_hi(pa[0]) + bf_lo(pa[2]) + bf_hi(pa[2]);
        l1 = l1 * c1 + bf_lo(pa[1]) + bf_hi(pa[1]) + bf_lo(pa[3]) + bf_hi(pa[3]);
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            o[nd][0] *= c0;
            o[nd][1] *= c0;
            o[nd][2] *= c1;
            o[nd][3] *= c1;
        }
        // O += P V: V^T fragments with ldmatrix.trans, two 8-dim tiles per load
        {
            const int key = kb16 + (lane & 7) + 8 * ((lane >> 3) & 1);
            const int hi = lane >> 4;
#pragma unroll
            for (int nd = 0; nd < 16; nd += 2) {
                uint32_t v00, v01, v10, v11;
                ldsm4t(su32(Vs) + swz(key, nd + hi), v00, v01, v10, v11);
                mma16816(o[nd], pa[0], pa[1], pa[2], pa[3], v00, v01);
                mma16816(o[nd + 1], pa[0], pa[1], pa[2], pa[3], v10, v11);
            }
        }
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = 16 * warp + g + 8 * hr;
        if (r >= rows) continue;
        const int s = members[it.first + r / G], h = hk * G + r % G;
        const size_t base = ((size_t)s * HQ + h) * n_split_total + split0 + chunk;
        if (t4 == 0) {
            part_ml[base * 2] = hr ? m1 : m0;
            part_ml[base * 2 + 1] = hr ? l1 : l0;
        }
        float* dst = part_o + base * PX_D;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd)
            *reinterpret_cast<float2*>(dst + nd * 8 + 2 * t4) = make_float2(o[nd][2 * hr], o[nd][2 * hr + 1]);
    }
}

}  // namespace

bool prefix_attention_supported(const Shape& sh) {
    const int G = sh.HQ / sh.HKV;
    return sh.D == PX_D && (G == 1 || G == 2 || G == 4 || G == 8);
}

int prefix_item_streams(const Shape& sh) { return PX_ROWS / (sh.HQ / sh.HKV); }

int prefix_chunks(int P) { return (P + PX_KEYS - 1) / PX_KEYS; }

cudaError_t launch_prefix_attention(const float* q, const Shape& sh, int layer, const PrefixItem* items, int n_items,
                                    const int* members, int max_chunks, int n_split_total, int split0, float* part_ml,
                                    float* part_o, cudaStream_t st) {
    (void)cudaGetLastError();
    if (!prefix_attention_supported(sh) || n_items <= 0 || max_chunks <= 0) return cudaErrorInvalidValue;
    const size_t smem = (size_t)(PX_ROWS + 2 * PX_KEYS) * 256;
    dim3 grid(sh.HKV, max_chunks, n_items);
    switch (sh.HQ / sh.HKV) {
#define PX_CASE(GG)                                                                                              \
    case GG: {                                                                                                   \
        static bool attr = false;                                                                                \
        if (!attr) {                                                                                             \
            cudaError_t e = cudaFuncSetAttribute(prefix_attn_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                                 (int)smem);                                                     \
            if (e != cudaSuccess) return e;                                                                      \
            attr = true;                                                                                         \
        }                                                                                                        \
        return launch_pdl(prefix_attn_kernel<GG>, grid, dim3(PX_THREADS), smem, st, q, sh.HQ, sh.HKV, layer,       \
                          sh.max_seq, items, members, n_split_total, split0, part_ml, part_o);                   \
    }
        PX_CASE(1)
        PX_CASE(2)
        PX_CASE(4)
        PX_CASE(8)
#undef PX_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qdec
