// Causal GQA prefill attention on the tcgen05 tensor cores (head_dim 128), flash-style.
//
// Computes, for every query row t (absolute position pos0 + t) and q head h, softmax over the
// keys j <= pos0 + t of q.k_j / sqrt(D), times V, with kv head h / (HQ / HKV) ("Qwen3ASR
// ncnn多平台移植" §5: the prefill's upper-triangular causal mask; "Forward map - funasr_nano":
// GQA 16/8).  The softmax is evaluated online over key tiles (running max and sum), i.e. the
// max-subtracted softmax rearranged tile by tile.
//
// Two kernels.  When each kv head serves an even number of q heads (GQA 16/8), the paired-head
// kernel below (attn_prefill_tc2_kernel) runs; otherwise this one.
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
                                                                 float scale_log2, int causal) {
    pdl_trigger();
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
    const int kend = causal ? min(L, pos0 + q0 + QT) : L;   // keys [0, kend) can be visible to this tile
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
    pdl_wait();   // Q and the caches are written by the preceding kernels

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
            const bool full = (!causal || j * KT + KT - 1 <= pos0 + q0) && (j * KT + KT <= L);
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
                        if ((!causal || key <= qpos) && key < L) mx = fmaxf(mx, sv[k]);
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
                        const bool vis = (!causal || key <= qpos) && key < L && m_new != -INFINITY;
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

// ---------------------------------------------------------------------------------------------
// Paired-head variant: one CTA = one 128-query tile of the two q heads 2c and 2c + 1, which
// share kv head g (HQ / HKV even), so every K and V tile is fetched once for two heads and the
// two heads' softmax warpgroups overlap each other's tensor-core work.  Ten warps:
//   warp 0    TMA: both Q tiles once, then K_0, K_1, V_0, K_2, V_1, ... (the order the MMAs
//             consume them) into a 3-slot ring of 32 KB tiles;
//   warp 1    allocates 512 TMEM columns (per head: S at 256h, O at 256h + 128) and issues
//             S_j(h) = Q_h K_j^T as soon as head h has read S_{j-1}(h) out of TMEM, and
//             O(h) += P_j(h) V_j once P_j(h) is in shared memory (O accumulates in TMEM);
//   warps 2-5 / 6-9  softmax of head 0 / head 1, one query row per thread: S_j read from TMEM
//             once (128 fp32 values in registers), masked row max, P_j = exp2(s*c - m) as
//             bf16 into swizzled shared memory.  The running max m is raised only when a tile
//             exceeds it by more than 2^8 (P stays <= 256); only then is the row's O in TMEM
//             rescaled, after the previous P.V has completed.  Final O / l stored bf16.
// The result equals the max-subtracted softmax: every P_j and the running sum l use the same
// m as the part of O they are added to.
constexpr int NSLOT = 3;
constexpr float LAZY_RESCALE_LOG2 = 8.f;

// Two fp32 values to one bf16x2 word (lo in the low half), round to nearest even: one
// conversion instruction per pair.
__device__ __forceinline__ uint32_t pack_bf2x(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

struct Fa2Bars {
    uint64_t q_full, ring_full[NSLOT], ring_empty[NSLOT], s_full[2], s_free[2], p_full[2], p_free[2], fin;
    uint32_t tmem;
    int abort;
};

// Non-blocking: has the phase of parity ph completed?
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t ph) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(s32(b)), "r"(ph)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mb_wait_ab(uint64_t* b, uint32_t ph, int code, volatile int* abort) {
    for (uint32_t i = 0; i < FA_SPIN; ++i) {
        if (mb_try(b, ph)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    *abort = 1;
    atomicCAS(&g_fa_error, 0, code);
    return false;
}
// Four 32-column TMEM loads of this warp's lanes issued back to back, then one wait; the
// wait names every destination register so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[4][32]) {
    tmem_ld32_issue(taddr, r[0]);
    tmem_ld32_issue(taddr + 32, r[1]);
    tmem_ld32_issue(taddr + 64, r[2]);
    tmem_ld32_issue(taddr + 96, r[3]);
    tmem_wait_ld(r[0]);
    tmem_wait_ld(r[1]);
    tmem_wait_ld(r[2]);
    tmem_wait_ld(r[3]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 :
                 : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

__global__ void __launch_bounds__(320, 1) attn_prefill_tc2_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                  const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV, int T,
                                                                  int HQ, int HKV, int pos0, bf16_t* __restrict__ O,
                                                                  float scale_log2) {
    pdl_trigger();
    extern __shared__ __align__(1024) char smem_raw[];
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    char* sQ = smem;                                  // 2 heads x 32 KB
    char* sRing = sQ + 2 * TILE_BYTES;                // NSLOT x 32 KB (K or V tiles)
    char* sP = sRing + NSLOT * TILE_BYTES;            // 2 heads x 32 KB
    Fa2Bars* B = reinterpret_cast<Fa2Bars*>(sP + 2 * TILE_BYTES);
    volatile int* abort = &B->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntq = (T + QT - 1) / QT;
    const int qtile = ntq - 1 - (int)blockIdx.y;     // longest causal rows first (y is dispatched last)
    const int h0 = 2 * (int)blockIdx.x, g = h0 / (HQ / HKV);
    const int q0 = qtile * QT;
    const int L = pos0 + T;
    const int kend = min(L, pos0 + q0 + QT);          // keys [0, kend) can be visible to this tile
    const int nt = (kend + KT - 1) / KT;

    if (threadIdx.x == 0) {
        mb_init(&B->q_full, 1);
        for (int i = 0; i < NSLOT; ++i) {
            mb_init(&B->ring_full[i], 1);
            mb_init(&B->ring_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mb_init(&B->s_full[i], 1);
            mb_init(&B->s_free[i], 4);
            mb_init(&B->p_full[i], 4);
            mb_init(&B->p_free[i], 1);
        }
        mb_init(&B->fin, 1);
        B->abort = 0;
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
    pdl_wait();   // Q and the caches are written by the preceding kernels

    if (warp == 0) {
        if (lane == 0) {   // ---- TMA producer: items in consumption order K0, K1, V0, K2, V1, ...
            mb_expect(&B->q_full, 2 * TILE_BYTES);
            for (int hh = 0; hh < 2; ++hh) {
                tma_3d(sQ + hh * TILE_BYTES, &tmQ, 0, h0 + hh, q0, &B->q_full);
                tma_3d(sQ + hh * TILE_BYTES + BLK, &tmQ, 64, h0 + hh, q0, &B->q_full);
            }
            uint32_t n = 0;
            bool ok = true;
            auto put = [&](const CUtensorMap* map, int j) {
                const uint32_t slot = n % NSLOT, r = n / NSLOT;
                if (!mb_wait_ab(&B->ring_empty[slot], (r & 1) ^ 1, 31, abort)) return false;
                char* dst = sRing + slot * TILE_BYTES;
                mb_expect(&B->ring_full[slot], TILE_BYTES);
                tma_3d(dst, map, 0, j * KT, g, &B->ring_full[slot]);
                tma_3d(dst + BLK, map, 64, j * KT, g, &B->ring_full[slot]);
                ++n;
                return true;
            };
            for (int j = 0; j < nt && ok; ++j) {
                ok = put(&tmK, j);
                if (ok && j >= 1) ok = put(&tmV, j - 1);
            }
            if (ok) put(&tmV, nt - 1);
            // every copy issued must land before the CTA exits
            mb_wait(&B->q_full, 0, 32);
            for (uint32_t i = n > (uint32_t)NSLOT ? n - NSLOT : 0; i < n; ++i)
                mb_wait(&B->ring_full[i % NSLOT], (i / NSLOT) & 1, 33);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---- MMA issuer: issues whichever MMA of either head is ready
            constexpr uint32_t id_s = idesc_fa(false), id_o = idesc_fa(true);
            // ring item of K_j / V_j in the producer's order K0, K1, V0, K2, V1, ..., V_{nt-1}
            auto kitem = [&](int j) { return j == 0 ? 0 : 2 * j - 1; };
            auto vitem = [&](int j) { return j + 1 < nt ? 2 * j + 2 : 2 * nt - 1; };
            auto ready = [&](uint64_t* bar, uint32_t ph) { return mbar_test(bar, ph); };
            int js[2] = {0, 0}, jp[2] = {0, 0};   // next S and next P.V tile of each head
            bool ok = mb_wait_ab(&B->q_full, 0, 34, abort);
            uint32_t idle = 0;
            while (ok && (jp[0] < nt || jp[1] < nt)) {
                bool issued = false;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    // S_j(h) = Q_h K_j^T once K_j has landed and head h has read S_{j-1}(h)
                    const int j = js[hh];
                    if (j < nt) {
                        const int it = kitem(j);
                        const uint32_t slot = (uint32_t)it % NSLOT;
                        if (ready(&B->ring_full[slot], ((uint32_t)it / NSLOT) & 1) &&
                            (j == 0 || ready(&B->s_free[hh], (j - 1) & 1))) {
                            tc_fence_after();
                            const char* k = sRing + slot * TILE_BYTES;
                            const char* qq = sQ + hh * TILE_BYTES;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t ad = desc_kmajor(qq + (kk >> 2) * BLK) + 2 * (kk & 3);
                                const uint64_t bd = desc_kmajor(k + (kk >> 2) * BLK) + 2 * (kk & 3);
                                mma_bf16(tmem + 256 * hh, ad, bd, id_s, kk != 0);
                            }
                            mma_commit(&B->s_full[hh]);
                            if (js[hh ^ 1] > j) mma_commit(&B->ring_empty[slot]);   // both heads done with K_j
                            js[hh] = j + 1;
                            issued = true;
                        }
                    }
                    // O(h) += P_i(h) V_i once P_i(h) is in shared memory and V_i has landed
                    const int i = jp[hh];
                    if (i < js[hh]) {
                        const int it = vitem(i);
                        const uint32_t slot = (uint32_t)it % NSLOT;
                        if (ready(&B->ring_full[slot], ((uint32_t)it / NSLOT) & 1) && ready(&B->p_full[hh], i & 1)) {
                            tc_fence_after();
                            const char* v = sRing + slot * TILE_BYTES;
                            const char* pp = sP + hh * TILE_BYTES;
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t ad = desc_kmajor(pp + (kk >> 2) * BLK) + 2 * (kk & 3);
                                const uint64_t bd = desc_mnmajor(v) + (uint64_t)((kk * 16 * 128) >> 4);
                                mma_bf16(tmem + 256 * hh + 128, ad, bd, id_o, (i > 0 || kk != 0) ? 1u : 0u);
                            }
                            mma_commit(&B->p_free[hh]);
                            if (jp[hh ^ 1] > i) mma_commit(&B->ring_empty[slot]);   // both heads done with V_i
                            jp[hh] = i + 1;
                            issued = true;
                        }
                    }
                }
                if (issued) {
                    idle = 0;
                } else if (++idle >= FA_SPIN) {
                    *abort = 1;
                    atomicCAS(&g_fa_error, 0, 35);
                    ok = false;
                } else if ((idle & 255) == 255 && *abort) {
                    ok = false;
                }
            }
            mma_commit(&B->fin);   // TMEM is freed only after every issued MMA has completed
            mb_wait(&B->fin, 0, 39);
        }
    } else {   // ---- softmax: warps 2-5 head 0, warps 6-9 head 1; TMEM lane quarter = warp % 4
        const int hh = (warp - 2) >> 2;
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int qpos = pos0 + q0 + row;
        const uint32_t sadr = tmem + ((uint32_t)(32 * q) << 16) + 256 * hh;
        const uint32_t oadr = sadr + 128;
        char* pst = sP + hh * TILE_BYTES;
        float m_run = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt && ok; ++j) {
            // a tile wholly below the diagonal (every key visible to every row) needs no mask
            const bool full = (j * KT + KT - 1 <= pos0 + q0) && (j * KT + KT <= L);
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mb_wait_ab(&B->s_full[hh], j & 1, 40, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[4][32];
            tmem_ld128(sadr, sr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mb_arrive(&B->s_free[hh]);   // S may be overwritten by S_{j+1}
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) mx4[k & 3] = fmaxf(mx4[k & 3], __uint_as_float(sr[c][k]));
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int key = j * KT + 32 * c + k;
                        if (key <= qpos && key < L) mx4[k & 3] = fmaxf(mx4[k & 3], __uint_as_float(sr[c][k]));
                    }
            }
            const float m_tile = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
            const bool need = m_tile > m_run + LAZY_RESCALE_LOG2;   // false while both are -inf
            const bool any = __any_sync(0xffffffffu, need) && j > 0;
            float corr = 1.f;
            if (need) {
                corr = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_tile);
                m_run = m_tile;
            }
            // P_j = exp2(s * c - m) (0 where masked), in two halves of 64 keys: the arguments,
            // then the exponentials, then the row sum and the bf16 pairs, each in bulk over
            // independent values (a half's packed words free half of its registers)
            const bool live = m_run != -INFINITY;
            const float nm = -m_run;
            float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                if (full) {
#pragma unroll
                    for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            sr[c][k] = __float_as_uint(fmaf(__uint_as_float(sr[c][k]), scale_log2, nm));
                } else {
#pragma unroll
                    for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int key = j * KT + 32 * c + k;
                            const bool vis = live && key <= qpos && key < L;
                            sr[c][k] = __float_as_uint(vis ? fmaf(__uint_as_float(sr[c][k]), scale_log2, nm) : -INFINITY);
                        }
                }
#pragma unroll
                for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) sr[c][k] = __float_as_uint(ex2(__uint_as_float(sr[c][k])));
#pragma unroll
                for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        ls4[0] += __uint_as_float(sr[c][k]);
                        ls4[1] += __uint_as_float(sr[c][k + 1]);
                        ls4[2] += __uint_as_float(sr[c][k + 2]);
                        ls4[3] += __uint_as_float(sr[c][k + 3]);
                    }
                // pairs packed in place: word k/2 of chunk c holds keys 32c + k, 32c + k + 1
#pragma unroll
                for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; k += 2)
                        sr[c][k >> 1] = pack_bf2x(__uint_as_float(sr[c][k]), __uint_as_float(sr[c][k + 1]));
            }
            l = l * corr + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
            if (j >= 1) {   // P(h) and O(h) are free once P_{j-1}(h) V_{j-1} has completed
                if (!__all_sync(0xffffffffu, mb_wait_ab(&B->p_free[hh], (j - 1) & 1, 41, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (any) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32_issue(oadr + 32 * c, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
                        tmem_st32(oadr + 32 * c, o);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
            }
            // P_j into the swizzled K-major layout the MMA reads (rows 128 B, 16-byte chunk c
            // of row r at chunk position c ^ (r & 7)); chunk u of column block c holds keys
            // 32c + 8u .. 32c + 8u + 7, i.e. packed words sr[c][4u .. 4u + 3]
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int key0 = 32 * c + 8 * u;
                    const int blk = key0 >> 6, ch = (key0 & 63) >> 3;
                    *reinterpret_cast<uint4*>(pst + blk * BLK + row * 128 + ((ch ^ (row & 7)) << 4)) =
                        make_uint4(sr[c][4 * u], sr[c][4 * u + 1], sr[c][4 * u + 2], sr[c][4 * u + 3]);
                }
            tc_fence_before();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // P is read by the tensor cores
            __syncwarp();
            if (lane == 0) mb_arrive(&B->p_full[hh]);
        }
        if (ok && nt >= 1 && __all_sync(0xffffffffu, mb_wait_ab(&B->p_free[hh], (nt - 1) & 1, 42, abort))) {
            tc_fence_after();
            uint32_t orr[4][32];
            tmem_ld128(oadr, orr);
            const int t = q0 + row;
            if (t < T) {
                const float inv = 1.f / l;
                uint4* dst = reinterpret_cast<uint4*>(O + (size_t)t * HQ * HD + (size_t)(h0 + hh) * HD);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t* w = &orr[c][8 * u];
                        dst[4 * c + u] = make_uint4(pack_bf2(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv),
                                                    pack_bf2(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv),
                                                    pack_bf2(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv),
                                                    pack_bf2(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv));
                    }
            }
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
    static_assert(sizeof(FaBars) <= 256 && sizeof(Fa2Bars) <= 256, "barrier block");
    const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    const int ntq = (T + QT - 1) / QT;
    if ((sh.HQ / sh.HKV) % 2 == 0) {   // two q heads of one kv group per CTA
        static bool attr2 = false;
        if (!attr2) {
            cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr2 = true;
        }
        // x = head pair, y = query tile rank: CTAs are dispatched longest causal rows first
        return launch_pdl(attn_prefill_tc2_kernel, dim3(sh.HQ / 2, ntq), dim3(320), smem, s, mq, mk, mv, T, sh.HQ,
                          sh.HKV, pos0, O, scale_log2);
    }
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch_pdl(attn_prefill_tc_kernel, dim3(ntq, sh.HQ), dim3(192), smem, s, mq, mk, mv, T, sh.HQ, sh.HKV, pos0,
                      O, scale_log2, 1);
}

cudaError_t launch_attention_bidir_tc(const bf16_t* Q, const bf16_t* K, const bf16_t* V, int row_stride, int T,
                                      int heads, bf16_t* O, cudaStream_t s) {
    (void)cudaGetLastError();
    if (T <= 0 || heads <= 0 || row_stride % 8 != 0 || row_stride < heads * 128) return cudaErrorInvalidValue;
    // Q, K and V are views [T][heads][128] with rows row_stride elements apart (the three column
    // blocks of one fused projection); K and V are read as [heads][T][128] through the strides
    CUtensorMap mq, mk, mv;
    const uint64_t D = 128, rs = (uint64_t)row_stride * 2;
    if (!make_map3(&mq, Q, D, (uint64_t)heads, (uint64_t)T, D * 2, rs, 1, QT)) return cudaErrorInvalidValue;
    if (!make_map3(&mk, K, D, (uint64_t)T, (uint64_t)heads, rs, D * 2, KT, 1)) return cudaErrorInvalidValue;
    if (!make_map3(&mv, V, D, (uint64_t)T, (uint64_t)heads, rs, D * 2, KT, 1)) return cudaErrorInvalidValue;
    constexpr int smem = 7 * TILE_BYTES + 1024 + 256;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    const int ntq = (T + QT - 1) / QT;
    return launch_pdl(attn_prefill_tc_kernel, dim3(ntq, heads), dim3(192), smem, s, mq, mk, mv, T, heads, heads, 0, O,
                      scale_log2, 0);
}

}  // namespace qdec
