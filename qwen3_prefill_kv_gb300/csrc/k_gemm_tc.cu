// Prefill GEMM on the 5th-generation tensor cores: C[M, N] (op)= A[M, K] . W[N, K]^T with bf16
// operands (both K-major), fp32 accumulation in TMEM, and the decoder's epilogues ("Forward
// map - funasr_nano", LLM decoder table: packed QKV projection, o_proj / down_proj with the
// residual add, packed gate_up with SwiGLU).
//
// Persistent: one CTA per resident slot walks work units (128 x BN tile, BN = 128 or 256, K-slice) with a
// stride of the grid size; the accumulator is double-buffered in TMEM so the epilogue of
// one unit overlaps the MMAs of the next.  Ten warps:
//   warp 0   TMA producer: 2-D tensor-map loads (128-byte swizzle) of the A tile (128 rows x
//            64 k) and the B tile (BN rows x 64 k; SwiGLU: BN/2 gate rows + the BN/2 matching
//            up rows) into a ring of STAGES shared-memory stages;
//   warp 1   allocates 2 BN TMEM columns and issues tcgen05.mma (M = 128, N = BN, K = 16) from
//            one thread, committing each stage back to its empty barrier;
//   warps 2-9 epilogue, two per TMEM lane quarter, each on half of the tile's columns:
//            tcgen05.ld of the accumulator (one TMEM lane = one output row), then
//            - fp32 store, residual add and bf16 store: through a per-warp shared-memory box
//              written out by TMA (a bulk store, or a bulk add into the residual in L2);
//            - SwiGLU, split-K atomics and partial slabs: direct stores;
//            - the packed QKV projection: the per-head Q/K RMSNorm + NeoX RoPE + KV append
//              ("per-head Q/K-RMSNorm + NeoX RoPE @ 1e6" in the decoder table; every 128
//              columns of a tile are one head).
// A second kernel runs 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2); it is selected
// only on request.  Rows past M are zero-filled by TMA and never stored.  Every wait is
// bounded; a timeout sets the error word and the CTA finishes without waiting further (TMEM
// is freed only after the accumulator barrier).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace qdec {

__device__ int g_tc_error;   // first timeout code of a tensor-core kernel (0 = none)

namespace {

constexpr int BM = 128, BK = 64;
constexpr int EPI_WARPS = 8;                     // two per TMEM lane quarter
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;   // + the TMA and MMA warps
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
// Weight tiles are loaded with an evict-first L2 policy: a prefill streams every layer's
// weights through L2 once, and they should not push out the activations the next kernels read.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
            s32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(s32(bar)), "l"(pol)
        : "memory");
}
// L2 prefetch of one box of a tensor map (no shared memory, no completion to wait for)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
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

// ---- CTA-pair forms (a cluster of two CTAs on two SMs; every tcgen05 instruction of the
// pair kernel uses cta_group::2)
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {   // every thread of both CTAs, warps converged
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared-memory object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(s32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void mb_arrive_cluster(uint32_t caddr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
__device__ __forceinline__ bool mb_try_cluster(uint64_t* b, uint32_t ph) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(s32(b)), "r"(ph)
        : "memory");
    return ok != 0;
}
// As mb_wait_ab, for a barrier that the peer CTA arrives on
__device__ __forceinline__ bool mb_wait_cluster_ab(uint64_t* b, uint32_t ph, int code, volatile int* abort) {
    for (uint32_t i = 0; i < TC_SPIN; ++i) {
        if (mb_try_cluster(b, ph)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    *abort = 1;
    atomicCAS(&g_tc_error, 0, code);
    return false;
}
// A tile load into this CTA's shared memory whose completion is counted on an mbarrier of
// either CTA of the pair (caddr: a shared::cluster address)
__device__ __forceinline__ void tma_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t caddr) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            s32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(caddr)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s32(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
// arrives on the mbarrier at shared::cluster address caddr once the pair's MMAs issued so far complete
__device__ __forceinline__ void mma_commit_pair(uint32_t caddr) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(caddr)
                 : "memory");
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

// Sum of squares of one head's 128 accumulator columns (TMEM lane = tile row), in column order.
__device__ __forceinline__ float head_sumsq(uint32_t taddr) {
    float ss = 0.f;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
        float t[32];
        tmem_ld32(taddr + c, t);
#pragma unroll
        for (int k = 0; k < 32; ++k) ss = fmaf(t[k], t[k], ss);
    }
    return ss;
}

// The per-head epilogue of the QKV projection on the rotation pairs (i, i + 64), i in
// [c, c + 32), of one head row (the calling thread owns tile row `row`; hd = head index):
// query and key heads are RMS-normalised (1 / r = the row's RMS) with their gain, rotated
// (NeoX), and stored to q or the key cache; value heads are stored as computed.  Every lane
// reads TMEM; only lanes with `store` write.
__device__ __forceinline__ void qkv_rope_block(uint32_t taddr, int c, float r, int row, int hd, bool store,
                                               const QkvRopeEpi& e) {
    float x[32], y[32];
    tmem_ld32(taddr + c, x);
    tmem_ld32(taddr + 64 + c, y);
    if (!store) return;
    const int p = e.pos0 + row;
    bf16_t* dst;
    if (hd >= e.HQ + e.HKV) {   // value head: stored as computed
        dst = e.vc + ((size_t)(hd - e.HQ - e.HKV) * e.max_seq + p) * 128;
    } else {
        const bf16_t* g = hd < e.HQ ? e.g_q : e.g_k;
        // (cos, sin) of pair c + i at this row's position from the pair-major table: the lanes
        // own consecutive positions, so each load is contiguous across the warp
        const float2* cs = e.rope_t + (size_t)c * e.max_seq + p;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint32_t ga = *reinterpret_cast<const uint32_t*>(g + c + i);
            const uint32_t gb = *reinterpret_cast<const uint32_t*>(g + 64 + c + i);
            const float2 cs0 = cs[(size_t)i * e.max_seq], cs1 = cs[(size_t)(i + 1) * e.max_seq];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float a = x[i + u] * (r * (u ? bf_hi(ga) : bf_lo(ga)));
                const float b = y[i + u] * (r * (u ? bf_hi(gb) : bf_lo(gb)));
                const float cn = u ? cs1.x : cs0.x, sn = u ? cs1.y : cs0.y;
                x[i + u] = a * cn - b * sn;
                y[i + u] = b * cn + a * sn;
            }
        }
        dst = hd < e.HQ ? e.q + ((size_t)row * e.HQ + hd) * 128
                        : e.kc + ((size_t)(hd - e.HQ) * e.max_seq + p) * 128;
    }
    uint4* dx = reinterpret_cast<uint4*>(dst + c);
    uint4* dy = reinterpret_cast<uint4*>(dst + 64 + c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        dx[j] = make_uint4(pack_bf2(x[8 * j], x[8 * j + 1]), pack_bf2(x[8 * j + 2], x[8 * j + 3]),
                           pack_bf2(x[8 * j + 4], x[8 * j + 5]), pack_bf2(x[8 * j + 6], x[8 * j + 7]));
        dy[j] = make_uint4(pack_bf2(y[8 * j], y[8 * j + 1]), pack_bf2(y[8 * j + 2], y[8 * j + 3]),
                           pack_bf2(y[8 * j + 4], y[8 * j + 5]), pack_bf2(y[8 * j + 6], y[8 * j + 7]));
    }
}

// ---- bulk (TMA) output of the epilogue: each epilogue warp stages a box of 32 rows x 128
// bytes in its own 4 KB of shared memory (128-byte swizzle: 16-byte chunk j of row r at chunk
// position j ^ (r % 8), so the 32 lanes' row writes are free of bank conflicts) and one lane
// hands it to the TMA, which stores it, or adds it into the fp32 residual in L2
// (cp.reduce.async.bulk .add): the SMs never read the residual and write whole lines.
// (The SwiGLU epilogue keeps its direct stores: with bulk output it measured ~8 us slower per
// launch at 415 and 1100 rows, for reasons not found.)
constexpr int EPI_BOX = 32 * 128;   // bytes of one staging box
__host__ __device__ constexpr bool tma_epilogue(int BN, int MODE) {
    return (MODE == GEMM_STORE_F32 || MODE == GEMM_ADD_F32 || MODE == GEMM_STORE_BF16) && (BN == 128 || BN == 256);
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(x), "r"(y), "r"(s32(src))
                 : "memory");
}
__device__ __forceinline__ void tma_add_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     map),
                 "r"(x), "r"(y), "r"(s32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// the warp's staging box may be rewritten: lane 0's earlier bulk copies have read it
__device__ __forceinline__ void box_ready(int lane) {
    if (lane == 0) bulk_wait_read();
    __syncwarp();
}
__device__ __forceinline__ void stage_row(char* box, int lane, const uint4 (&c)[8]) {
    char* r = box + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(r + ((j ^ (lane & 7)) << 4)) = c[j];
}
// the box (rows y .. y + 31 of the output, columns from x) to global memory; rows past the
// map's last row are dropped by the TMA
template <bool ADD>
__device__ __forceinline__ void flush_box(const CUtensorMap* map, char* box, int x, int y, int lane) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the generic-proxy writes, to the TMA
    __syncwarp();
    if (lane == 0) {
        if (ADD) tma_add_2d(map, x, y, box);
        else tma_store_2d(map, x, y, box);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}
// per-column bias (the adaptor's linear layers), then ReLU, on 32 columns from col
__device__ __forceinline__ void bias_relu(float (&v)[32], const float* __restrict__ bias, int relu, int col) {
    if (bias) {
        const float4* b4 = reinterpret_cast<const float4*>(bias + col);
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
}
__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
    return make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
}
__device__ __forceinline__ uint4 swiglu8_bf16(const float* g, const float* u) {
    return make_uint4(pack_bf2(silu(g[0]) * u[0], silu(g[1]) * u[1]), pack_bf2(silu(g[2]) * u[2], silu(g[3]) * u[3]),
                      pack_bf2(silu(g[4]) * u[4], silu(g[5]) * u[5]), pack_bf2(silu(g[6]) * u[6], silu(g[7]) * u[7]));
}

// Rows of one TMA box of the B (weight) tile: a SwiGLU tile is BN/2 gate rows + BN/2 up rows;
// otherwise boxes of 128 rows.
__host__ __device__ constexpr int b_box_rows(int BN, int MODE) { return MODE == GEMM_SWIGLU_BF16 ? BN / 2 : 128; }

// Epilogue of one accumulator row, half h of its columns: the calling thread owns TMEM lane
// `taddr`, tile row row0 + lane of the output (row0: the warp's first row); two warps share
// each lane quarter, one per half; nt is the tile's column index, z its K-split; tmC and box
// (the warp's staging box) serve the bulk-output modes.
template <int BN, int MODE>
__device__ __forceinline__ void epilogue_row(uint32_t taddr, int row0, int lane, int M, int nt, int z, int ldc,
                                             float* __restrict__ Cf, bf16_t* __restrict__ Cb,
                                             const QkvRopeEpi& epi, const float* __restrict__ bias, int relu,
                                             int h, const CUtensorMap* tmC, char* box) {
    constexpr bool GLU = (MODE == GEMM_SWIGLU_BF16);
    const int n0 = nt * (GLU ? BN / 2 : BN);
    const int row = row0 + lane;
    if constexpr (tma_epilogue(BN, MODE)) {
        const bool live = row0 < M;   // warp-uniform: a box that would start past the last row is not issued
        if constexpr (MODE == GEMM_STORE_F32 || MODE == GEMM_ADD_F32) {
#pragma unroll 1
            for (int c0 = h * (BN / 2); c0 < (h + 1) * (BN / 2); c0 += 32) {
                float v[32];
                tmem_ld32(taddr + c0, v);
                bias_relu(v, bias, relu, n0 + c0);
                uint4 c[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    c[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                      __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                box_ready(lane);
                stage_row(box, lane, c);
                if (live) flush_box<MODE == GEMM_ADD_F32>(tmC, box, n0 + c0, row0, lane);
            }
        } else if constexpr (MODE == GEMM_STORE_BF16) {
#pragma unroll 1
            for (int c0 = h * (BN / 2); c0 < (h + 1) * (BN / 2); c0 += 64) {
                uint4 c[8];
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    float v[32];
                    tmem_ld32(taddr + c0 + 32 * sub, v);
                    bias_relu(v, bias, relu, n0 + c0 + 32 * sub);
#pragma unroll
                    for (int j = 0; j < 4; ++j) c[4 * sub + j] = pack8_bf16(v + 8 * j);
                }
                box_ready(lane);
                stage_row(box, lane, c);
                if (live) flush_box<false>(tmC, box, n0 + c0, row0, lane);
            }
        }
    } else if constexpr (MODE == GEMM_QKV_ROPE) {   // one head per 128 columns
        // rotation-pair blocks pb = 2 head + (c / 32): half h takes NH of the tile's 2 NH
        constexpr int NH = BN / 128;
        int cur = -1;
        float r = 0.f;
#pragma unroll 1
        for (int pb = h * NH; pb < (h + 1) * NH; ++pb) {
            const int hb = pb >> 1, hd = nt * NH + hb;
            const uint32_t th = taddr + 128 * hb;
            if (hb != cur) {
                cur = hb;
                if (hd < epi.HQ + epi.HKV) r = rsqrtf(head_sumsq(th) / 128.f + epi.eps);
            }
            qkv_rope_block(th, (pb & 1) * 32, r, row, hd, row < M, epi);
        }
    } else if constexpr (GLU) {
#pragma unroll 1
        for (int c0 = h * (BN / 4); c0 < (h + 1) * (BN / 4); c0 += 32) {
            float gv[32], uv[32];
            tmem_ld32(taddr + c0, gv);
            tmem_ld32(taddr + BN / 2 + c0, uv);
            if (row < M) {
                uint4* dst = reinterpret_cast<uint4*>(Cb + (size_t)row * ldc + n0 + c0);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) dst[jj] = swiglu8_bf16(gv + 8 * jj, uv + 8 * jj);
            }
        }
    } else {
#pragma unroll 1
        for (int c0 = h * (BN / 2); c0 < (h + 1) * (BN / 2); c0 += 32) {
            float v[32];
            tmem_ld32(taddr + c0, v);
            bias_relu(v, bias, relu, n0 + c0);
            if (row < M) {
                if (MODE == GEMM_STORE_BF16) {
                    uint4* dst = reinterpret_cast<uint4*>(Cb + (size_t)row * ldc + n0 + c0);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) dst[jj] = pack8_bf16(v + 8 * jj);
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
}

template <int BN, int MODE, int STAGES>
__global__ void __launch_bounds__(GEMM_THREADS, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                         const __grid_constant__ CUtensorMap tmB,
                                                         const __grid_constant__ CUtensorMap tmC, int M, int K,
                                                         int up_off, float* __restrict__ Cf,
                                                         bf16_t* __restrict__ Cb, int ldc, const QkvRopeEpi epi,
                                                         int tiles_m, int tiles_n, int splits,
                                                         const float* __restrict__ bias, int relu) {
    pdl_trigger();
    extern __shared__ __align__(1024) char smem_raw[];
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int A_BYTES = BM * BK * 2;
    constexpr int B_BYTES = BN * BK * 2;
    constexpr bool GLU = (MODE == GEMM_SWIGLU_BF16);
    constexpr int B_BOX = b_box_rows(BN, MODE), B_LOADS = BN / B_BOX;
    static_assert(BN == 128 || BN == 256, "tile width");
    constexpr uint32_t ACC_COLS = 2 * BN;   // double-buffered accumulator (512 columns at most)
    constexpr bool TE = tma_epilogue(BN, MODE);
    char* sA = smem;
    char* sB = smem + STAGES * A_BYTES;
    char* sE = sB + STAGES * B_BYTES;       // bulk-output modes: one staging box per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(sE + (TE ? EPI_WARPS * EPI_BOX : 0));
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;    // [2]: the MMAs of a unit have completed
    uint64_t* acc_empty = acc_full + 2;     // [2]: the epilogue has read the buffer (8 warps)
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
            mb_init(&acc_empty[i], EPI_WARPS);
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
    if (warp != 0) pdl_wait();   // the producer waits after requesting its first weight tiles

    if (warp == 0) {
        if (lane == 0) {   // ---- TMA producer: one stage ring across all of this CTA's units
            // B: BN rows in boxes of B_BOX rows stacked in shared memory (SwiGLU: the gate
            // rows, then the matching up rows)
            const uint64_t wpol = policy_evict_first();
            auto load_b = [&](uint32_t s, int n0, int kb) {
#pragma unroll
                for (int b = 0; b < B_LOADS; ++b)
                    tma_2d_hint(sB + s * B_BYTES + b * B_BOX * 128, &tmB, kb * BK,
                                GLU ? (b ? up_off + n0 : n0) : n0 + b * B_BOX, &full[s], wpol);
            };
            // The weights do not depend on the preceding kernel: the whole weight matrix is
            // prefetched into L2 (boxes dealt over the CTAs; a prefill streams each layer's
            // weights from HBM once, and without it the first touch of a tile waits for HBM), and
            // the B tiles of the first stages are requested, before waiting for it; their A tiles
            // after.
            {
                const int wrows = GLU ? up_off + tiles_n * (BN / 2) : tiles_n * BN;
                const int nb = ((wrows + B_BOX - 1) / B_BOX) * nkb;
                for (int b = blockIdx.x; b < nb; b += gridDim.x) tma_prefetch_2d(&tmB, (b % nkb) * BK, (b / nkb) * B_BOX);
            }
            uint32_t npre = 0;
            for (int u = blockIdx.x; u < units && npre < (uint32_t)STAGES; u += gridDim.x) {
                int m0, nt, kb0, nk, z;
                unit(u, m0, nt, kb0, nk, z);
                for (int kb = 0; kb < nk && npre < (uint32_t)STAGES; ++kb, ++npre) {
                    mb_expect(&full[npre], A_BYTES + B_BYTES);
                    load_b(npre, nt * (GLU ? BN / 2 : BN), kb0 + kb);
                }
            }
            pdl_wait();
            uint32_t g = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int m0, nt, kb0, nk, z;
                unit(u, m0, nt, kb0, nk, z);
                const int n0 = nt * (GLU ? BN / 2 : BN);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const uint32_t s = g % STAGES, r = g / STAGES;
                    if (g >= npre) {
                        if (!mb_wait_ab(&empty[s], (r & 1) ^ 1, 1, abort)) {
                            ok = false;
                            break;
                        }
                        mb_expect(&full[s], A_BYTES + B_BYTES);
                        load_b(s, n0, kb0 + kb);
                    }
                    tma_2d(sA + s * A_BYTES, &tmA, (kb0 + kb) * BK, m0, &full[s]);
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
    } else {   // ---- epilogue: warps 2..9 cover TMEM lane quarters 2, 3, 0, 1 twice (column halves 0, 1)
        const int q = warp & 3;
        int j = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            int m0, nt, kb0, nk, z;
            unit(u, m0, nt, kb0, nk, z);
            const int buf = j & 1;
            if (!mb_wait_ab(&acc_full[buf], (j >> 1) & 1, 3, abort)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (uint32_t)(buf * BN) + ((uint32_t)(32 * q) << 16);
            if (nk > 0)   // an empty K-slice (never produced by the launcher) contributes nothing
                epilogue_row<BN, MODE>(taddr, m0 + 32 * q, lane, M, nt, z, ldc, Cf, Cb, epi, bias, relu,
                                       (warp - 2) >> 2, &tmC, sE + (warp - 2) * EPI_BOX);
            tc_fence_before();   // this warp's accumulator reads are complete
            __syncwarp();
            if (lane == 0) mb_arrive(&acc_empty[buf]);
        }
        if (TE && lane == 0) bulk_wait_all();   // the staged boxes are written out before the CTA ends
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ACC_COLS);
    }
}

// Pair tiles: a cluster of two CTAs on two SMs computes a 256 x 256 tile with tcgen05.mma
// cta_group::2 (M = 256, N = 256).  CTA r of the pair TMA-loads rows [128 r, 128 r + 128) of
// the A tile and its own 128 rows of the B tile (128 r of the 256 output columns; SwiGLU:
// CTA 0 the 128 gate rows, CTA 1 the matching up rows) into its ring; the stage barrier that
// counts both CTAs' bytes lives in CTA 0, whose MMA thread reads the A and B halves of both
// CTAs and accumulates CTA r's 128 rows x 256 columns in CTA r's TMEM (two 256-column
// buffers).  Against the 128 x 256 tile of one CTA, a k-block moves 32 KB of operands into
// each SM instead of 48 KB for the same MMA work, and the ring holds STAGES of them.  The
// epilogue of each CTA is the 256-column one; CTA 1's epilogue warps arrive on CTA 0's
// accumulator-empty barrier, CTA 0's MMA thread commits to the barriers of both CTAs.  Used
// only when forced (set_gemm_tile_rows(256)): see use_pair_tiles for the measurements.
template <int MODE, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, int M, int K,
                    int up_off, float* __restrict__ Cf, bf16_t* __restrict__ Cb, int ldc, const QkvRopeEpi epi,
                    int tiles_m, int tiles_n, const float* __restrict__ bias, int relu) {
    pdl_trigger();
    extern __shared__ __align__(1024) char smem_raw[];
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int BN = 256;
    constexpr int A_BYTES = BM * BK * 2;    // this CTA's 128 rows of A
    constexpr int B_BYTES = 128 * BK * 2;   // this CTA's 128 rows of B
    constexpr bool GLU = (MODE == GEMM_SWIGLU_BF16);
    constexpr uint32_t ACC_COLS = 2 * BN;
    constexpr bool TE = tma_epilogue(BN, MODE);
    char* sA = smem;
    char* sB = smem + STAGES * A_BYTES;
    char* sE = sB + STAGES * B_BYTES;       // bulk-output modes: one staging box per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(sE + (TE ? EPI_WARPS * EPI_BOX : 0));   // CTA 0's count both CTAs' bytes
    uint64_t* empty = full + STAGES;        // each CTA's: the pair's MMAs have read stage s
    uint64_t* acc_full = empty + STAGES;    // each CTA's [2]: the unit's MMAs have completed
    uint64_t* acc_empty = acc_full + 2;     // CTA 0's [2]: both CTAs' epilogues have read the buffer
    uint64_t* fin = acc_empty + 2;          // each CTA's: every MMA of the pair has completed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int nkb = K / BK, units = tiles_m * tiles_n;   // t walks the 256-row M tiles fastest

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mb_init(&full[i], 1);
            mb_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mb_init(&acc_full[i], 1);
            mb_init(&acc_empty[i], 2 * EPI_WARPS);
        }
        mb_init(fin, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc_pair(tslot, ACC_COLS);   // one warp of each CTA, collectively
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers are initialised before either signals the other's
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (warp != 0) pdl_wait();   // the producer waits after requesting its first weight tiles

    if (warp == 0) {
        if (lane == 0) {   // ---- TMA producer of this CTA's halves
            auto b0_of = [&](int nt) { return GLU ? (rank ? up_off : 0) + nt * 128 : nt * BN + (int)rank * 128; };
            // the B tiles of the first stages before waiting for the preceding kernel, as in
            // gemm_tc_kernel
            uint32_t npre = 0;
            for (int u = pair; u < units && npre < (uint32_t)STAGES; u += npairs)
                for (int kb = 0; kb < nkb && npre < (uint32_t)STAGES; ++kb, ++npre) {
                    if (rank == 0) mb_expect(&full[npre], 2 * (A_BYTES + B_BYTES));
                    tma_2d_pair(sB + npre * B_BYTES, &tmB, kb * BK, b0_of(u / tiles_m), peer_addr(&full[npre], 0));
                }
            pdl_wait();
            uint32_t g = 0;
            bool ok = true;
            for (int u = pair; u < units && ok; u += npairs) {
                const int m0 = (u % tiles_m) * 2 * BM + (int)rank * BM, nt = u / tiles_m;
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const uint32_t s = g % STAGES, r = g / STAGES;
                    const uint32_t fb = peer_addr(&full[s], 0);
                    if (g >= npre) {
                        if (!mb_wait_ab(&empty[s], (r & 1) ^ 1, 1, abort)) {
                            ok = false;
                            break;
                        }
                        if (rank == 0) mb_expect(&full[s], 2 * (A_BYTES + B_BYTES));
                        tma_2d_pair(sB + s * B_BYTES, &tmB, kb * BK, b0_of(nt), fb);
                    }
                    tma_2d_pair(sA + s * A_BYTES, &tmA, kb * BK, m0, fb);
                }
            }
            // the last copies issued must land before the CTA exits: CTA 0 sees them on its
            // stage barriers, CTA 1 through the MMAs that consumed them releasing its stages
            for (uint32_t q = g > (uint32_t)STAGES ? g - STAGES : 0; q < g; ++q) {
                if (rank == 0) mb_wait(&full[q % STAGES], (q / STAGES) & 1, 4);
                else mb_wait(&empty[q % STAGES], (q / STAGES) & 1, 4);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {   // ---- MMA issuer of the pair
            constexpr uint32_t idesc = idesc_bf16(2 * BM, BN);
            uint32_t g = 0;
            bool ok = true;
            int j = 0;
            for (int u = pair; u < units && ok; u += npairs, ++j) {
                const int buf = j & 1;
                if (!mb_wait_cluster_ab(&acc_empty[buf], ((j >> 1) & 1) ^ 1, 5, abort)) break;
                tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const uint32_t s = g % STAGES, r = g / STAGES;
                    if (!mb_wait_ab(&full[s], r & 1, 2, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(sA + s * A_BYTES), bd = sw128_desc(sB + s * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_pair(dacc, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    mma_commit_pair(peer_addr(&empty[s], 0));
                    mma_commit_pair(peer_addr(&empty[s], 1));
                }
                if (ok) {
                    mma_commit_pair(peer_addr(&acc_full[buf], 0));
                    mma_commit_pair(peer_addr(&acc_full[buf], 1));
                }
            }
            mma_commit_pair(peer_addr(fin, 0));   // TMEM is freed only after every MMA has completed
            mma_commit_pair(peer_addr(fin, 1));
            mb_wait(fin, 0, 6);
        } else if (lane == 0) {
            mb_wait(fin, 0, 6);   // CTA 1: the pair's MMAs read this CTA's stages and write its TMEM
        }
    } else {   // ---- epilogue: warps 2..9 cover TMEM lane quarters 2, 3, 0, 1 twice (column halves 0, 1)
        const int q = warp & 3;
        const uint32_t ae0 = peer_addr(&acc_empty[0], 0), ae1 = peer_addr(&acc_empty[1], 0);
        int j = 0;
        for (int u = pair; u < units; u += npairs, ++j) {
            const int m0 = (u % tiles_m) * 2 * BM + (int)rank * BM, nt = u / tiles_m;
            const int buf = j & 1;
            if (!mb_wait_ab(&acc_full[buf], (j >> 1) & 1, 3, abort)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (uint32_t)(buf * BN) + ((uint32_t)(32 * q) << 16);
            epilogue_row<BN, MODE>(taddr, m0 + 32 * q, lane, M, nt, 0, ldc, Cf, Cb, epi, bias, relu, (warp - 2) >> 2,
                                   &tmC, sE + (warp - 2) * EPI_BOX);
            tc_fence_before();   // this warp's accumulator reads are complete
            __syncwarp();
            if (lane == 0) mb_arrive_cluster(buf ? ae1 : ae0);
        }
        if (TE && lane == 0) bulk_wait_all();   // the staged boxes are written out before the CTA ends
    }
    tc_fence_before();
    cluster_sync();   // neither CTA leaves while the other may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, ACC_COLS);
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

// 2-D map of the output C (row-major [rows, cols], row stride ld elements) for the bulk
// epilogue: boxes of 32 rows x 128 bytes (32 fp32 or 64 bf16 columns), 128-byte swizzle.
bool make_out_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, bool f32) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * (f32 ? 4 : 2)};
    cuuint32_t box[2] = {f32 ? 32u : 64u, 32u};
    cuuint32_t es[2] = {1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, int STAGES>
cudaError_t launch_bn(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc, int M, int N, int K,
                      int up_off, float* Cf, bf16_t* Cb, int ldc, int splits, cudaStream_t s,
                      const QkvRopeEpi& epi = QkvRopeEpi{}, const float* bias = nullptr, int relu = 0) {
    constexpr int smem = STAGES * (BM * BK * 2 + BN * BK * 2) + (tma_epilogue(BN, MODE) ? EPI_WARPS * EPI_BOX : 0) +
                         1024 + 256;
    auto kern = gemm_tc_kernel<BN, MODE, STAGES>;
    static int resident = 0;   // CTAs of this instantiation that fit on the device at once
    if (!resident) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int dev = 0, sms = 0, per_sm = 0;
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, GEMM_THREADS, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        resident = sms * per_sm;
    }
    const int tile_n = (MODE == GEMM_SWIGLU_BF16) ? BN / 2 : BN;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = N / tile_n;
    const long long units = (long long)tiles_m * tiles_n * splits;
    const int grid = (int)(units < resident ? units : resident);   // persistent: each CTA walks units
    return launch_pdl(kern, dim3(grid), dim3(GEMM_THREADS), smem, s, ma, mb, mc, M, K, up_off, Cf, Cb, ldc, epi,
                      tiles_m, tiles_n, splits, bias, relu);
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

template <int MODE, int STAGES>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc, int M, int N, int K,
                        int up_off, float* Cf, bf16_t* Cb, int ldc, cudaStream_t s,
                        const QkvRopeEpi& epi = QkvRopeEpi{}, const float* bias = nullptr, int relu = 0) {
    constexpr int smem = STAGES * (2 * BM * BK * 2) + (tma_epilogue(256, MODE) ? EPI_WARPS * EPI_BOX : 0) + 1024 + 256;
    auto kern = gemm_tc2_kernel<MODE, STAGES>;
    static int pairs = 0;   // clusters of this instantiation that fit on the device at once
    if (!pairs) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (unsigned)device_sms());
        cfg.blockDim = dim3(GEMM_THREADS);
        cfg.dynamicSmemBytes = smem;
        int n = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        pairs = n;
    }
    const int tiles_m = (M + 2 * BM - 1) / (2 * BM), tiles_n = N / (MODE == GEMM_SWIGLU_BF16 ? 128 : 256);
    const long long units = (long long)tiles_m * tiles_n;
    const int grid = 2 * (int)(units < pairs ? units : pairs);   // persistent: each pair walks units
    return launch_pdl(kern, dim3(grid), dim3(GEMM_THREADS), smem, s, ma, mb, mc, M, K, up_off, Cf, Cb, ldc, epi,
                      tiles_m, tiles_n, bias, relu);
}

// Tile height of the 256-wide tiles.  A CTA pair (256 x 256) moves 1.5x fewer operand bytes
// into each SM per FLOP than one CTA (128 x 256), but measured slower at every prompt length
// tried (the 4096-row projections 5-10%, 415 and 1100 rows up to 14%): the k-block loop is
// bound by the latency of a stage's loads, not their bytes, and a pair's stage completes
// only when both CTAs' loads have landed on CTA 0's barrier (~1.7 us after issue against
// ~0.9 us for one CTA).  So one CTA is the default; set_gemm_tile_rows(256) forces the pair.
int g_tile_rows = 0;   // 0 = chosen per shape; 128 or 256 = forced
bool use_pair_tiles(int M) {
    (void)M;
    return g_tile_rows == 256;
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

int set_gemm_tile_rows(int bm) {
    const int prev = g_tile_rows;
    g_tile_rows = bm;
    return prev;
}

int gemm_tile_rows() { return g_tile_rows; }

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
    CUtensorMap ma, mb, mc{};   // mc: the output, for the bulk-output epilogues
    const int w_rows = (mode == GEMM_SWIGLU_BF16) ? up_off + N : N;
    const bool wide = mode != GEMM_ATOMIC_F32 && mode != GEMM_PARTIAL_F32 && use_wide_tiles(M, N, mode);
    if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, BM)) return cudaErrorInvalidValue;
    if (!make_map(&mb, W, (uint64_t)w_rows, (uint64_t)K, (uint64_t)K, (uint32_t)b_box_rows(wide ? 256 : 128, mode)))
        return cudaErrorInvalidValue;
    if (tma_epilogue(wide ? 256 : 128, mode)) {
        const bool f32 = mode == GEMM_STORE_F32 || mode == GEMM_ADD_F32;
        if (!make_out_map(&mc, f32 ? static_cast<const void*>(Cf) : static_cast<const void*>(Cb), (uint64_t)M,
                          (uint64_t)N, (uint64_t)ldc, f32))
            return cudaErrorInvalidValue;
    }
    if (wide && use_pair_tiles(M)) {   // the B map's 128-row boxes serve the pair's halves too
        switch (mode) {
            case GEMM_STORE_F32: return launch_pair<GEMM_STORE_F32, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, s, QkvRopeEpi{}, bias, relu);
            case GEMM_ADD_F32: return launch_pair<GEMM_ADD_F32, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, s, QkvRopeEpi{}, bias, relu);
            case GEMM_SWIGLU_BF16: return launch_pair<GEMM_SWIGLU_BF16, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, s);
            case GEMM_STORE_BF16: return launch_pair<GEMM_STORE_BF16, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, s, QkvRopeEpi{}, bias, relu);
            default: return cudaErrorInvalidValue;
        }
    }
    if (wide) switch (mode) {
        case GEMM_STORE_F32: return launch_bn<256, GEMM_STORE_F32, 4>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_ADD_F32: return launch_bn<256, GEMM_ADD_F32, 4>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_SWIGLU_BF16: return launch_bn<256, GEMM_SWIGLU_BF16, 4>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        case GEMM_STORE_BF16: return launch_bn<256, GEMM_STORE_BF16, 4>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        default: return cudaErrorInvalidValue;
    }
    switch (mode) {
        case GEMM_STORE_F32: return launch_bn<128, GEMM_STORE_F32, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_ADD_F32: return launch_bn<128, GEMM_ADD_F32, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        case GEMM_SWIGLU_BF16: return launch_bn<128, GEMM_SWIGLU_BF16, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        case GEMM_STORE_BF16: return launch_bn<128, GEMM_STORE_BF16, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s, QkvRopeEpi{}, bias, relu);
        // The lockstep batch's split-K CTAs run few k-blocks each: a 3-stage ring (97 KB) lets
        // two share an SM.  The prefill's split-K launches have about one unit per SM and start
        // while the preceding kernel still holds SMs; in a build whose register count let two
        // of their CTAs share an SM, the 64-position prefill took 1.55 against 1.33 ms (CTAs
        // doubling up on the first SMs to free), so their 6-stage ring (193 KB) keeps one CTA
        // per SM.
        case GEMM_ATOMIC_F32: return launch_bn<128, GEMM_ATOMIC_F32, 3>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s);
        case GEMM_PARTIAL_F32: return launch_bn<128, GEMM_PARTIAL_F32, 6>(ma, mb, mc, M, N, K, up_off, Cf, Cb, ldc, splits, s);
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
    CUtensorMap ma, mb, mc{};   // the per-head epilogue stores directly: mc is unused
    if (!make_map(&ma, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, BM)) return cudaErrorInvalidValue;
    if (!make_map(&mb, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    if (use_wide_tiles(M, N, GEMM_QKV_ROPE) && use_pair_tiles(M))   // two heads per tile, on a CTA pair
        return launch_pair<GEMM_QKV_ROPE, 6>(ma, mb, mc, M, N, K, 0, nullptr, nullptr, 0, s, epi);
    if (use_wide_tiles(M, N, GEMM_QKV_ROPE))   // two heads per 256-column tile
        return launch_bn<256, GEMM_QKV_ROPE, 4>(ma, mb, mc, M, N, K, 0, nullptr, nullptr, 0, 1, s, epi);
    return launch_bn<128, GEMM_QKV_ROPE, 6>(ma, mb, mc, M, N, K, 0, nullptr, nullptr, 0, 1, s, epi);
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
