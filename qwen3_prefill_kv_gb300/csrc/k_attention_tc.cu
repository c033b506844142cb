// Causal GQA prefill attention on the tcgen05 tensor cores (head_dim 128), flash-style.
//
// Computes, for every query row t (absolute position pos0 + t) and q head h, softmax over the
// keys j <= pos0 + t of q.k_j / sqrt(D), times V, with kv head h / (HQ / HKV) ("Qwen3ASR
// ncnn多平台移植" §5: the prefill's upper-triangular causal mask; "Forward map - funasr_nano":
// GQA 16/8).  The softmax is evaluated online over key tiles (running max and sum), i.e. the
// max-subtracted softmax rearranged tile by tile.
//
// One CTA = one 128-query tile of one q head; six warps:
//   warp 0    TMA: the Q tile once, then K and V tiles of 128 keys into a 2-stage ring
//             (3-D tensor maps over [T][HQ][D] and [HKV][max_seq][D], 128-byte swizzle);
//   warp 1    allocates all 512 TMEM columns and issues S_j = Q K_j^T (TMEM, double
//             buffered) and O_j = P_j V_j (TMEM, double buffered; V is the MN-major operand);
//   warps 2-5 one query row per thread: masked online softmax of S_j (fp32), P_j = exp2(..)
//             as bf16 into swizzled shared memory for the next MMA, and the running output
//             O = O * exp2(m_old - m_new) + O_j kept in registers; final O / l stored bf16.
// All waits are bounded (timeouts set the tensor-core error word).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace qdec {

__device__ int g_fa_error;   // first timeout code of the attention kernel (0 = none)

namespace {

constexpr uint32_t FA_SPIN = 1u << 22;
constexpr int QT = 128, KT = 128, HD = 128;
constexpr int TILE_BYTES = QT * HD * 2;          // 32 KB: two 64-column swizzle blocks
constexpr int BLK = 128 * 64 * 2;                // 16 KB: one [128 rows x 64] block

__device__ __forceinline__ uint32_t s32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t c) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s32(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(s32(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t ph) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(s32(b)), "r"(ph)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t ph, int code) {
    for (uint32_t i = 0; i < FA_SPIN; ++i)
        if (mb_try(b, ph)) return true;
    atomicCAS(&g_fa_error, 0, code);
    return false;
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            s32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(s32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s32(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 2^x with the MUFU instruction (relative error about 2^-22, far below P's bf16 rounding);
// -inf gives +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// K-major operand, 128-byte swizzle: 128-byte rows, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_kmajor(const void* p) {
    uint64_t d = (uint64_t)((s32(p) >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// MN-major operand (V: 128 key rows of 64 contiguous d values per swizzle block, 128-byte
// swizzle): 8-key groups 1024 B apart (stride byte offset), the two 64-wide d blocks 16 KB
// apart (leading byte offset).
__device__ __forceinline__ uint64_t desc_mnmajor(const void* p) {
    uint64_t d = (uint64_t)((s32(p) >> 4) & 0x3FFFu);
    d |= (uint64_t)(BLK >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// D fp32, A/B bf16, M = N = 128; b_mn: B is MN-major.
__host__ __device__ constexpr uint32_t idesc_fa(bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(128 >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

struct FaBars {
    uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full[2], p_free[2], o_full[2], o_free[2];
    uint32_t tmem;
};

__global__ void __launch_bounds__(192, 1) attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                 const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV, int T,
                                                                 int HQ, int HKV, int pos0, bf16_t* __restrict__ O,
                                                                 float scale_log2) {
    extern __shared__ __align__(1024) char smem_raw[];
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    char* sQ = smem;                                  // 32 KB
    char* sKV = smem + TILE_BYTES;                    // 2 stages x (K 32 KB + V 32 KB)
    char* sP = sKV + 4 * TILE_BYTES;                  // 2 x 32 KB
    FaBars* B = reinterpret_cast<FaBars*>(sP + 2 * TILE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntq = (T + QT - 1) / QT;
    const int qtile = ntq - 1 - (int)blockIdx.x;      // longest causal rows first
    const int h = blockIdx.y, g = h / (HQ / HKV);
    const int q0 = qtile * QT;
    const int L = pos0 + T;
    const int kend = min(L, pos0 + q0 + QT);          // keys [0, kend) can be visible to this tile
    const int nt = (kend + KT - 1) / KT;

    if (threadIdx.x == 0) {
        mb_init(&B->q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mb_init(&B->kv_full[i], 1);
            mb_init(&B->kv_empty[i], 1);
            mb_init(&B->s_full[i], 1);
            mb_init(&B->s_free[i], 4);
            mb_init(&B->p_full[i], 4);
            mb_init(&B->p_free[i], 1);
            mb_init(&B->o_full[i], 1);
            mb_init(&B->o_free[i], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(s32(&B->tmem))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem;

    if (warp == 0) {
        if (lane == 0) {   // ---- TMA producer
            mb_expect(&B->q_full, TILE_BYTES);
            tma_3d(sQ, &tmQ, 0, h, q0, &B->q_full);
            tma_3d(sQ + BLK, &tmQ, 64, h, q0, &B->q_full);
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int st = j & 1;
                if (!mb_wait(&B->kv_empty[st], ((j >> 1) & 1) ^ 1, 11)) break;
                char* k = sKV + st * 2 * TILE_BYTES;
                char* v = k + TILE_BYTES;
                mb_expect(&B->kv_full[st], 2 * TILE_BYTES);
                tma_3d(k, &tmK, 0, j * KT, g, &B->kv_full[st]);
                tma_3d(k + BLK, &tmK, 64, j * KT, g, &B->kv_full[st]);
                tma_3d(v, &tmV, 0, j * KT, g, &B->kv_full[st]);
                tma_3d(v + BLK, &tmV, 64, j * KT, g, &B->kv_full[st]);
                issued = j + 1;
            }
            mb_wait(&B->q_full, 0, 12);
            for (int j = issued - 2 > 0 ? issued - 2 : 0; j < issued; ++j) mb_wait(&B->kv_full[j & 1], (j >> 1) & 1, 13);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---- MMA issuer
            constexpr uint32_t id_s = idesc_fa(false), id_o = idesc_fa(true);
            bool ok = mb_wait(&B->q_full, 0, 14);
            auto pv = [&](int i) {   // O_i = P_i V_i into the O buffer of i
                const int st = i & 1;
                if (!mb_wait(&B->p_full[st], (i >> 1) & 1, 15)) return false;
                if (!mb_wait(&B->o_free[st], ((i >> 1) & 1) ^ 1, 16)) return false;
                tc_fence_after();
                const char* v = sKV + st * 2 * TILE_BYTES + TILE_BYTES;
                const char* pp = sP + st * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = desc_kmajor(pp + (kk >> 2) * BLK) + 2 * (kk & 3);
                    const uint64_t bd = desc_mnmajor(v) + (uint64_t)((kk * 16 * 128) >> 4);
                    mma_bf16(tmem + 256 + st * 128, ad, bd, id_o, kk != 0);
                }
                mma_commit(&B->o_full[st]);
                mma_commit(&B->p_free[st]);
                mma_commit(&B->kv_empty[st]);
                return true;
            };
            for (int j = 0; j < nt && ok; ++j) {
                const int st = j & 1;
                ok = mb_wait(&B->kv_full[st], (j >> 1) & 1, 17) && mb_wait(&B->s_free[st], ((j >> 1) & 1) ^ 1, 18);
                if (!ok) break;
                tc_fence_after();
                const char* k = sKV + st * 2 * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = desc_kmajor(sQ + (kk >> 2) * BLK) + 2 * (kk & 3);
                    const uint64_t bd = desc_kmajor(k + (kk >> 2) * BLK) + 2 * (kk & 3);
                    mma_bf16(tmem + st * 128, ad, bd, id_s, kk != 0);
                }
                mma_commit(&B->s_full[st]);
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok && nt >= 1) pv(nt - 1);
        }
    } else {   // ---- softmax + output: warps 2..5 own TMEM lane quarters 2, 3, 0, 1
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int qpos = pos0 + q0 + row;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        float o[HD];
#pragma unroll
        for (int d = 0; d < HD; ++d) o[d] = 0.f;
        float m = -INFINITY, l = 0.f, corr_prev = 0.f;
        auto accumulate = [&](int i, float corr) {   // o = o * corr + O_i
            const int st = i & 1;
            mb_wait(&B->o_full[st], (i >> 1) & 1, 19);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                float t[32];
                tmem_ld32(tmem + lane_off + 256 + st * 128 + 32 * c, t);
#pragma unroll
                for (int k = 0; k < 32; ++k) o[32 * c + k] = fmaf(o[32 * c + k], corr, t[k]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mb_arrive(&B->o_free[st]);
        };
        for (int j = 0; j < nt; ++j) {
            const int st = j & 1;
            // a tile wholly below the diagonal (every key visible to every row) needs no mask
            const bool full = (j * KT + KT - 1 <= pos0 + q0) && (j * KT + KT <= L);
            mb_wait(&B->s_full[st], (j >> 1) & 1, 20);
            tc_fence_after();
            const uint32_t sadr = tmem + lane_off + st * 128;
            float mx = -INFINITY;   // max raw score (scale_log2 > 0 commutes with the max)
#pragma unroll
            for (int c = 0; c < KT / 32; ++c) {
                float sv[32];
                tmem_ld32(sadr + 32 * c, sv);
                if (full) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) mx = fmaxf(mx, sv[k]);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int key = j * KT + 32 * c + k;
                        if (key <= qpos && key < L) mx = fmaxf(mx, sv[k]);
                    }
                }
            }
            const float m_new = fmaxf(m, mx * scale_log2);
            const float corr = (m == -INFINITY) ? 0.f : ex2(m - m_new);
            // P_j into the swizzled K-major block layout the MMA reads (rows 128 B, 16-byte
            // chunk c of row r at chunk position c ^ (r & 7))
            mb_wait(&B->p_free[st], ((j >> 1) & 1) ^ 1, 21);
            char* pst = sP + st * TILE_BYTES;
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < KT / 32; ++c) {
                float sv[32];
                tmem_ld32(sadr + 32 * c, sv);
                float pv[32];
                if (full) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        pv[k] = ex2(fmaf(sv[k], scale_log2, -m_new));
                        lsum += pv[k];
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int key = j * KT + 32 * c + k;
                        const bool vis = key <= qpos && key < L && m_new != -INFINITY;
                        pv[k] = vis ? ex2(fmaf(sv[k], scale_log2, -m_new)) : 0.f;
                        lsum += pv[k];
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {   // four 16-byte chunks of 8 keys
                    const int key0 = 32 * c + 8 * u;   // within the tile
                    const int blk = key0 >> 6, ch = (key0 & 63) >> 3;
                    uint4 w;
                    w.x = pack_bf2(pv[8 * u + 0], pv[8 * u + 1]);
                    w.y = pack_bf2(pv[8 * u + 2], pv[8 * u + 3]);
                    w.z = pack_bf2(pv[8 * u + 4], pv[8 * u + 5]);
                    w.w = pack_bf2(pv[8 * u + 6], pv[8 * u + 7]);
                    *reinterpret_cast<uint4*>(pst + blk * BLK + row * 128 + ((ch ^ (row & 7)) << 4)) = w;
                }
            }
            tc_fence_before();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // P is read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                mb_arrive(&B->s_free[st]);
                mb_arrive(&B->p_full[st]);
            }
            l = l * corr + lsum;
            m = m_new;
            if (j >= 1) accumulate(j - 1, corr_prev);
            corr_prev = corr;
        }
        if (nt >= 1) accumulate(nt - 1, corr_prev);
        const int t = q0 + row;
        if (t < T) {
            const float inv = 1.f / l;
            uint4* dst = reinterpret_cast<uint4*>(O + (size_t)t * HQ * HD + (size_t)h * HD);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c)
                dst[c] = make_uint4(pack_bf2(o[8 * c] * inv, o[8 * c + 1] * inv), pack_bf2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                    pack_bf2(o[8 * c + 4] * inv, o[8 * c + 5] * inv), pack_bf2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn3() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// 3-D bf16 map over [d2][d1][d0] (d0 contiguous), box {64, b1, b2}.
bool make_map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
               uint64_t s2_bytes, uint32_t b1, uint32_t b2) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn3();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {64, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int fa_error_read_and_clear() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fa_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (v) {
        const int z = 0;
        cudaMemcpyToSymbol(g_fa_error, &z, sizeof(int));
    }
    return v;
}

bool attention_tc_supported(const Shape& sh) { return sh.D == 128 && sh.HQ % sh.HKV == 0; }

cudaError_t launch_attention_prefill_tc(const bf16_t* Q, int T, const Shape& sh, int pos0, const bf16_t* k_cache,
                                        const bf16_t* v_cache, bf16_t* O, cudaStream_t s) {
    (void)cudaGetLastError();
    if (!attention_tc_supported(sh) || T <= 0 || pos0 < 0 || pos0 + T > sh.max_seq) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    const uint64_t D = 128;
    if (!make_map3(&mq, Q, D, (uint64_t)sh.HQ, (uint64_t)T, D * 2, (uint64_t)sh.HQ * D * 2, 1, QT)) return cudaErrorInvalidValue;
    if (!make_map3(&mk, k_cache, D, (uint64_t)sh.max_seq, (uint64_t)sh.HKV, D * 2, (uint64_t)sh.max_seq * D * 2, KT, 1))
        return cudaErrorInvalidValue;
    if (!make_map3(&mv, v_cache, D, (uint64_t)sh.max_seq, (uint64_t)sh.HKV, D * 2, (uint64_t)sh.max_seq * D * 2, KT, 1))
        return cudaErrorInvalidValue;
    constexpr int smem = 7 * TILE_BYTES + 1024 + 256;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid((T + QT - 1) / QT, sh.HQ);
    const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    attn_prefill_tc_kernel<<<grid, 192, smem, s>>>(mq, mk, mv, T, sh.HQ, sh.HKV, pos0, O, scale_log2);
    return cudaGetLastError();
}

}  // namespace qdec
