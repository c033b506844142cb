// Prefill GEMM on the 5th-generation tensor cores: C[M, N] (op)= A[M, K] . W[N, K]^T with bf16
// operands (both K-major), fp32 accumulation in TMEM, and the decoder's epilogues ("Forward
// map - funasr_nano", LLM decoder table: packed QKV projection, o_proj / down_proj with the
// residual add, packed gate_up with SwiGLU).
//
// Persistent: one CTA per resident slot walks work units (128 x BN tile, BN = 128 or 256, K-slice) with a
// stride of the grid size; the accumulator is double-buffered in TMEM so the epilogue of
// one unit overlaps the MMAs of the next.  Six warps:
//   warp 0   TMA producer: 2-D tensor-map loads (128-byte swizzle) of the A tile (128 rows x
//            64 k) and the B tile (BN rows x 64 k; SwiGLU: BN/2 gate rows + the BN/2 matching
//            up rows) into a ring of STAGES shared-memory stages;
//   warp 1   allocates 2 BN TMEM columns and issues tcgen05.mma (M = 128, N = BN, K = 16) from
//            one thread, committing each stage back to its empty barrier;
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (one TMEM lane = one output row),
//            then store / residual add / SwiGLU / split-K atomics to global memory, or for
//            the packed QKV projection the per-head Q/K RMSNorm + NeoX RoPE + KV append
//            ("per-head Q/K-RMSNorm + NeoX RoPE @ 1e6" in the decoder table; every 128
//            columns of a tile are one head).
// Rows past M are zero-filled by TMA and never stored.  Every wait is bounded; a timeout sets
// the error word and the CTA finishes without waiting further (TMEM is freed only after the
// accumulator barrier).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace qdec {

__device__ int g_tc_error;   // first timeout code of a tensor-core kernel (0 = none)

namespace {

constexpr int BM = 128, BK = 64;
constexpr uint32_t TC_SPIN = 1u << 22;

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
    for (uint32_t i = 0; i < TC_SPIN; ++i)
        if (mb_try(b, ph)) return true;
    atomicCAS(&g_tc_error, 0, code);
    return false;
}
// As mb_wait, but gives up at once when another role of the CTA has failed (*abort set),
// and sets *abort itself on a timeout.
__device__ __forceinline__ bool mb_wait_ab(uint64_t* b, uint32_t ph, int code, volatile int* abort) {
    for (uint32_t i = 0; i < TC_SPIN; ++i) {
        if (mb_try(b, ph)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    *abort = 1;
    atomicCAS(&g_tc_error, 0, code);
    return false;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            s32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(s32(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s32(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
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

// Shared-memory matrix descriptor of a K-major tile written by TMA with 128-byte swizzle:
// rows of 64 bf16 (128 B), 8-row groups 1024 B apart (stride byte offset), version 1.
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
    uint64_t d = (uint64_t)((s32(p) >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}
// Instruction descriptor: D fp32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The per-head epilogue of the QKV projection on one 128-wide head row v (one thread owns
// row `row` of the tile; head hd = the tile's column index).
__device__ __forceinline__ void qkv_rope_row(float (&v)[128], int row, int hd, const QkvRopeEpi& e) {
    const int p = e.pos0 + row;
    bf16_t* dst;
    if (hd >= e.HQ + e.HKV) {   // value head: stored as computed
        dst = e.vc + ((size_t)(hd - e.HQ - e.HKV) * e.max_seq + p) * 128;
    } else {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 128; ++i) ss = fmaf(v[i], v[i], ss);
        const float r = rsqrtf(ss / 128.f + e.eps);
        const bf16_t* g = hd < e.HQ ? e.g_q : e.g_k;
        const float2* cs = e.rope + (size_t)p * 64;
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
            const uint32_t ga = *reinterpret_cast<const uint32_t*>(g + i);
            const uint32_t gb = *reinterpret_cast<const uint32_t*>(g + 64 + i);
            const float4 c2 = *reinterpret_cast<const float4*>(cs + i);   // (cos, sin) of pairs i, i + 1
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float a = v[i + u] * (r * (u ? bf_hi(ga) : bf_lo(ga)));
                const float b = v[64 + i + u] * (r * (u ? bf_hi(gb) : bf_lo(gb)));
                const float c = u ? c2.z : c2.x, sn = u ? c2.w : c2.y;
                v[i + u] = a * c - b * sn;
                v[64 + i + u] = b * c + a * sn;
            }
        }
        dst = hd < e.HQ ? e.q + ((size_t)row * e.HQ + hd) * 128
                        : e.kc + ((size_t)(hd - e.HQ) * e.max_seq + p) * 128;
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int j = 0; j < 16; ++j)
        d4[j] = make_uint4(pack_bf2(v[8 * j], v[8 * j + 1]), pack_bf2(v[8 * j + 2], v[8 * j + 3]),
                           pack_bf2(v[8 * j + 4], v[8 * j + 5]), pack_bf2(v[8 * j + 6], v[8 * j + 7]));
}

// Rows of one TMA box of the B (weight) tile: a SwiGLU tile is BN/2 gate rows + BN/2 up rows;
// otherwise boxes of 128 rows.
__host__ __device__ constexpr int b_box_rows(int BN, int MODE) { return MODE == GEMM_SWIGLU_BF16 ? BN / 2 : 128; }

template <int BN, int MODE, int STAGES>
__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                         const __grid_constant__ CUtensorMap tmB, int M, int K,
                                                         int up_off, float* __restrict__ Cf,
                                                         bf16_t* __restrict__ Cb, int ldc, const QkvRopeEpi epi,
                                                         int tiles_m, int tiles_n, int splits,
                                                         const float* __restrict__ bias, int relu) {
    extern __shared__ __align__(1024) char smem_raw[];
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int A_BYTES = BM * BK * 2;
    constexpr int B_BYTES = BN * BK * 2;
    constexpr bool GLU = (MODE == GEMM_SWIGLU_BF16);
    constexpr int B_BOX = b_box_rows(BN, MODE), B_LOADS = BN / B_BOX;
    static_assert(BN == 128 || BN == 256, "tile width");
    constexpr uint32_t ACC_COLS = 2 * BN;   // double-buffered accumulator (512 columns at most)
    char* sA = smem;
    char* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;    // [2]: the MMAs of a unit have completed
    uint64_t* acc_empty = acc_full + 2;     // [2]: the epilogue has read the buffer (4 warps)
    uint64_t* fin = acc_empty + 2;          // every MMA issued by this CTA has completed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // work unit u = (split z, tile t): t walks the M tiles fastest, so CTAs running at the
    // same time share the weight (B) tile through L2; split z covers k-blocks [kb0, kb0 + nk)
    const int nkb = K / BK, per = (nkb + splits - 1) / splits;
    const int tiles = tiles_m * tiles_n, units = tiles * splits;
    auto unit = [&](int u, int& m0, int& nt, int& kb0, int& nk, int& z) {
        z = u / tiles;
        const int t = u - z * tiles;
        m0 = (t % tiles_m) * BM;
        nt = t / tiles_m;
        kb0 = z * per;
        nk = max(0, min(nkb, kb0 + per) - kb0);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mb_init(&full[i], 1);
            mb_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mb_init(&acc_full[i], 1);
            mb_init(&acc_empty[i], 4);
        }
        mb_init(fin, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tslot, ACC_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {   // ---- TMA producer: one stage ring across all of this CTA's units
            uint32_t g = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int m0, nt, kb0, nk, z;
                unit(u, m0, nt, kb0, nk, z);
                const int n0 = nt * (GLU ? BN / 2 : BN);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const uint32_t s = g % STAGES, r = g / STAGES;
                    if (!mb_wait_ab(&empty[s], (r & 1) ^ 1, 1, abort)) {
                        ok = false;
                        break;
                    }
                    mb_expect(&full[s], A_BYTES + B_BYTES);
                    tma_2d(sA + s * A_BYTES, &tmA, (kb0 + kb) * BK, m0, &full[s]);
                    // B: BN rows in boxes of B_BOX rows stacked in shared memory (SwiGLU: the
                    // gate rows, then the matching up rows)
#pragma unroll
                    for (int b = 0; b < B_LOADS; ++b)
                        tma_2d(sB + s * B_BYTES + b * B_BOX * 128, &tmB, (kb0 + kb) * BK,
                               GLU ? (b ? up_off + n0 : n0) : n0 + b * B_BOX, &full[s]);
                }
            }
            // the last copies issued must land before the CTA exits (after an error they may not
            // have been consumed)
            for (uint32_t q = g > (uint32_t)STAGES ? g - STAGES : 0; q < g; ++q)
                mb_wait(&full[q % STAGES], (q / STAGES) & 1, 4);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---- MMA issuer
            constexpr uint32_t idesc = idesc_bf16(BM, BN);
            uint32_t g = 0;
            bool ok = true;
            int j = 0;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
                int m0, nt, kb0, nk, z;
                unit(u, m0, nt, kb0, nk, z);
                const int buf = j & 1;
                if (!mb_wait_ab(&acc_empty[buf], ((j >> 1) & 1) ^ 1, 5, abort)) break;
                tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const uint32_t s = g % STAGES, r = g / STAGES;
                    if (!mb_wait_ab(&full[s], r & 1, 2, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(sA + s * A_BYTES), bd = sw128_desc(sB + s * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)   // 16 bf16 = 32 B per MMA: +2 in the address field
                        mma_bf16(dacc, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(&acc_full[buf]);   // arrives when this unit's MMAs have completed
            }
            mma_commit(fin);   // TMEM is freed only after every issued MMA has completed
            mb_wait(fin, 0, 6);
        }
    } else {   // ---- epilogue: warps 2..5 cover TMEM lane quarters 2, 3, 0, 1
        const int q = warp & 3;
        int j = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            int m0, nt, kb0, nk, z;
            unit(u, m0, nt, kb0, nk, z);
            const int buf = j & 1;
            if (!mb_wait_ab(&acc_full[buf], (j >> 1) & 1, 3, abort)) break;
            tc_fence_after();
            const int row = m0 + 32 * q + lane;
            const int n0 = nt * (GLU ? BN / 2 : BN);
            const uint32_t taddr = tmem + (uint32_t)(buf * BN) + ((uint32_t)(32 * q) << 16);
            if (nk == 0) {
                // an empty K-slice (never produced by the launcher) contributes nothing
            } else if constexpr (MODE == GEMM_QKV_ROPE) {   // one head per 128 columns
#pragma unroll 1
                for (int hb = 0; hb < BN / 128; ++hb) {
                    float v[128];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float t[32];
                        tmem_ld32(taddr + 128 * hb + 32 * c, t);
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[32 * c + k] = t[k];
                    }
                    if (row < M) qkv_rope_row(v, row, nt * (BN / 128) + hb, epi);
                }
            } else if constexpr (GLU) {
#pragma unroll 1
                for (int c0 = 0; c0 < BN / 2; c0 += 32) {
                    float gv[32], uv[32];
                    tmem_ld32(taddr + c0, gv);
                    tmem_ld32(taddr + BN / 2 + c0, uv);
                    if (row < M) {
                        uint4* dst = reinterpret_cast<uint4*>(Cb + (size_t)row * ldc + n0 + c0);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            uint4 w;
                            w.x = pack_bf2(silu(gv[8 * jj + 0]) * uv[8 * jj + 0], silu(gv[8 * jj + 1]) * uv[8 * jj + 1]);
                            w.y = pack_bf2(silu(gv[8 * jj + 2]) * uv[8 * jj + 2], silu(gv[8 * jj + 3]) * uv[8 * jj + 3]);
                            w.z = pack_bf2(silu(gv[8 * jj + 4]) * uv[8 * jj + 4], silu(gv[8 * jj + 5]) * uv[8 * jj + 5]);
                            w.w = pack_bf2(silu(gv[8 * jj + 6]) * uv[8 * jj + 6], silu(gv[8 * jj + 7]) * uv[8 * jj + 7]);
                            dst[jj] = w;
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    float v[32];
                    tmem_ld32(taddr + c0, v);
                    if (bias) {   // per-column bias (the adaptor's linear layers), then ReLU
                        const float4* b4 = reinterpret_cast<const float4*>(bias + n0 + c0);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const float4 b = __ldg(b4 + jj);
                            v[4 * jj] += b.x; v[4 * jj + 1] += b.y; v[4 * jj + 2] += b.z; v[4 * jj + 3] += b.w;
                        }
                    }
                    if (relu) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = fmaxf(v[k], 0.f);
                    }
                    if (row < M) {
                        if (MODE == GEMM_STORE_BF16) {
                            uint4* dst = reinterpret_cast<uint4*>(Cb + (size_t)row * ldc + n0 + c0);
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                dst[jj] = make_uint4(pack_bf2(v[8 * jj], v[8 * jj + 1]), pack_bf2(v[8 * jj + 2], v[8 * jj + 3]),
                                                     pack_bf2(v[8 * jj + 4], v[8 * jj + 5]), pack_bf2(v[8 * jj + 6], v[8 * jj + 7]));
                        } else {
                            // split-K partials go to slab z of M rows
                            float* cbase = MODE == GEMM_PARTIAL_F32 ? Cf + (size_t)z * M * ldc : Cf;
                            float4* dst = reinterpret_cast<float4*>(cbase + (size_t)row * ldc + n0 + c0);
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) {
                                float4 o = make_float4(v[4 * jj], v[4 * jj + 1], v[4 * jj + 2], v[4 * jj + 3]);
                                if (MODE == GEMM_ATOMIC_F32) {   // split-K partials: vector fp32 reductions
                                    atomicAdd(dst + jj, o);
                                    continue;
                                }
                                if (MODE == GEMM_ADD_F32) {
                                    const float4 c = dst[jj];
                                    o.x += c.x; o.y += c.y; o.z += c.z; o.w += c.w;
                                }
                                dst[jj] = o;
                            }
                        }
                    }
                }
            }
            tc_fence_before();   // this warp's accumulator reads are complete
            __syncwarp();
            if (lane == 0) mb_arrive(&acc_empty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ACC_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D bf16 map of a row-major [rows, cols] matrix (row stride in elements), box 64 x box_rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t stride_elems,
              uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {stride_elems * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, int STAGES>
cudaError_t launch_bn(const CUtensorMap& ma, const CUtensorMap& mb, int M, int N, int K, int up_off, float* Cf,
                      bf16_t* Cb, int ldc, int splits, cudaStream_t s, const QkvRopeEpi& epi = QkvRopeEpi{},
                      const float* bias = nullptr, int relu = 0) {
    constexpr int smem = STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 + 256;
    auto kern = gemm_tc_kernel<BN, MODE, STAGES>;
    static int resident = 0;   // CTAs of this instantiation that fit on the device at once
    if (!resident) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int dev = 0, sms = 0, per_sm = 0;
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 192, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        resident = sms * per_sm;
    }
    const int tile_n = (MODE == GEMM_SWIGLU_BF16) ? BN / 2 : BN;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = N / tile_n;
    const long long units = (long long)tiles_m * tiles_n * splits;
    const int grid = (int)(units < resident ? units : resident);   // persistent: each CTA walks units
    kern<<<grid, 192, smem, s>>>(ma, mb, M, K, up_off, Cf, Cb, ldc, epi, tiles_m, tiles_n, splits, bias, relu);
    return cudaGetLastError();
}

// Tile width.  A 128 x 256 tile moves 1.33x fewer operand bytes per FLOP than a 128 x 128 one,
// but has half as many tiles to spread over the SMs (one CTA per SM either way); the wider
// tile is taken when its rounds of tiles, weighted by WIDE_COST (time of a 256-wide tile
// relative to two 128-wide ones), cost less.  set_gemm_tile_width() forces a width.
constexpr double WIDE_COST = 0.75;
int g_tile_width = 0;   // 0 = chosen per shape; 128 or 256 = forced
int gemm_bn_override() { return g_tile_width; }
int device_sms() {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            sms = 148;
        }
    }
    return sms;
}
bool use_wide_tiles(int M, int N, int mode) {
    const bool glu = mode == GEMM_SWIGLU_BF16;
    const int tn128 = glu ? 64 : 128, tn256 = glu ? 128 : 256;
    if (N % tn256 != 0) return false;
    const int ov = gemm_bn_override();
    if (ov == 128 || ov == 256) return ov == 256;
    const long long tiles_m = (M + BM - 1) / BM, sms = device_sms();
    const long long r128 = (tiles_m * (N / tn128) + sms - 1) / sms, r256 = (tiles_m * (N / tn256) + sms - 1) / sms;
    return 2.0 * WIDE_COST * (double)r256 < (double)r128;
}

}  // namespace

int gemm_tc_splits(int K, int splits) {
    const int nkb = K / BK;
    if (splits > nkb) splits = nkb;
    if (splits < 1) splits = 1;
    const int per = (nkb + splits - 1) / splits;
    return (nkb + per - 1) / per;
}

int set_gemm_tile_width(int bn) {
    const int prev = g_tile_width;
    g_tile_width = bn;
    return prev;
}

int gemm_tile_width() { return g_tile_width; }

bool gemm_tc_supported(int N, int K, int mode, int lda) {
    if (K % BK != 0 || lda % 8 != 0) return false;
    if (mode == GEMM_SWIGLU_BF16) return N % 64 == 0;
    return N % 128 == 0;
}

cudaError_t launch_gemm_tc(const bf16_t* A, int lda, const bf16_t* W, int M, int N, int K, int mode, int up_off,
                           float* Cf, bf16_t* Cb, int ldc, cudaStream_t s, int splits, const float* bias, int relu) {
    (void)cudaGetLastError();
    if (!gemm_tc_supported(N, K, mode, lda) || M <= 0) return cudaErrorInvalidValue;
    // a bias or ReLU applies to the plain store / add epilogues only
    if ((bias || relu) && mode != GEMM_STORE_F32 && mode != GEMM_ADD_F32 && mode != GEMM_STORE_BF16)
        return cudaErrorInvalidValue;
    // each split needs at least one k-block; only the atomic and partial modes may be split
    if (splits < 1 || (splits > 1 && mode != GEMM_ATOMIC_F32 && mode != GEMM_PARTIAL_F32)) return cudaErrorInvalidValue;
    splits = gemm_tc_splits(K, splits);
    CUtensorMap ma, mb;
    const int w_rows = (mode == GEMM_SWIGLU_BF16) ? up_off + N : N;
    const bool wide = mode != GEMM_ATOMIC_F32 && mode != GEMM_PARTIAL_F32 && use_wide_tiles(M, N, mode);
    if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, BM)) return cudaErrorInvalidValue;
    if (!make_map(&mb, W, (uint64_t)w_rows, (uint64_t)K, (uint64_t)K, (uint32_t)b_box_rows(wide ? 256 : 128, mode)))
        return cudaErrorInvalidValue;
    if (wide) switch (mode) {
        case GEMM_STORE_F32: return launch_bn<256, GEMM_STORE_F32, 4>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_ADD_F32: return launch_bn<256, GEMM_ADD_F32, 4>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_SWIGLU_BF16: return launch_bn<256, GEMM_SWIGLU_BF16, 4>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        case GEMM_STORE_BF16: return launch_bn<256, GEMM_STORE_BF16, 4>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        default: return cudaErrorInvalidValue;
    }
    switch (mode) {
        case GEMM_STORE_F32: return launch_bn<128, GEMM_STORE_F32, 6>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_ADD_F32: return launch_bn<128, GEMM_ADD_F32, 6>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_SWIGLU_BF16: return launch_bn<128, GEMM_SWIGLU_BF16, 6>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        case GEMM_STORE_BF16: return launch_bn<128, GEMM_STORE_BF16, 6>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        // split-K CTAs run few k-blocks each: a 3-stage ring (97 KB) lets two share an SM
        case GEMM_ATOMIC_F32: return launch_bn<128, GEMM_ATOMIC_F32, 3>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        case GEMM_PARTIAL_F32: return launch_bn<128, GEMM_PARTIAL_F32, 3>(ma, mb, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        default: return cudaErrorInvalidValue;
    }
}

bool gemm_tc_qkv_rope_supported(const Shape& sh, int lda) {
    return sh.D == 128 && gemm_tc_supported(sh.qkv_rows(), sh.H, GEMM_STORE_F32, lda);
}

cudaError_t launch_gemm_tc_qkv_rope(const bf16_t* A, int lda, const bf16_t* W, int M, int K, const QkvRopeEpi& epi,
                                    cudaStream_t s) {
    (void)cudaGetLastError();
    const int N = (epi.HQ + 2 * epi.HKV) * 128;
    if (M <= 0 || K % BK != 0 || lda % 8 != 0 || !epi.q || !epi.kc || !epi.vc || !epi.rope || epi.pos0 < 0 ||
        epi.pos0 + M > epi.max_seq)
        return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, BM)) return cudaErrorInvalidValue;
    if (!make_map(&mb, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    if (use_wide_tiles(M, N, GEMM_QKV_ROPE))   // two heads per 256-column tile
        return launch_bn<256, GEMM_QKV_ROPE, 4>(ma, mb, M, N, K, 0, nullptr, nullptr, 0, 1, s, epi);
    return launch_bn<128, GEMM_QKV_ROPE, 6>(ma, mb, M, N, K, 0, nullptr, nullptr, 0, 1, s, epi);
}

int tc_error_read_and_clear() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (v) {
        const int z = 0;
        cudaMemcpyToSymbol(g_tc_error, &z, sizeof(int));
    }
    return v;
}

}  // namespace qdec
