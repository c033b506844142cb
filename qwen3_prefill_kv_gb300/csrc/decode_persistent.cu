// One batch-1 decode step of the whole decoder in a single persistent kernel.
//
// What it computes is one incremental step of "Qwen3ASR ncnn多平台移植" §5 (embed the token,
// RoPE at its absolute position, attend over the cached history plus itself, append its
// K/V, LM head, greedy pick) over the blocks of the "LLM decoder (Qwen3-0.6B, frozen,
// BF16)" table of "Forward map - funasr_nano" (rms_norm, packed QKV, per-head Q/K RMSNorm,
// NeoX RoPE, GQA, o_proj + residual, rms_norm, packed gate_up SwiGLU, down_proj +
// residual; final rms_norm; tied lm_head).
//
// How (GB300): one CTA per SM, launched cooperatively so that every CTA is resident.
//  * Warp NCW is a producer.  It streams this CTA's slices of every weight matrix (and,
//    for the CTA that owns an attention unit, its chunk of the K/V cache) into a ring of
//    16 KB shared-memory slots with 1-D TMA bulk copies (cp.async.bulk + mbarrier
//    complete_tx), in exactly the order the consumers use them, running ahead across
//    phase boundaries so HBM keeps streaming while the consumers wait on data.
//  * Warps 0..NCW-1 are consumers: GEMV rows from shared memory against the input
//    vector (fp32, also in shared memory, pre-multiplied by its RMSNorm gain), attention
//    over the streamed K/V chunk, lm_head rows + argmax.  They walk the step's phases in
//    one loop that is not unrolled, so each code path exists once and the kernel's hot
//    code stays small (instruction fetch, not arithmetic, bounded the first versions).
//  * Phases exchange vectors through global memory as 64-bit words {tag, fp32 value}
//    written with one relaxed 64-bit store; a reader polls the words themselves (several
//    16-byte polls in flight per thread) until every tag equals the phase's tag, so a
//    hand-off costs about one L2 round trip and there are no grid barriers.  Each phase's writers read the whole output of the previous
//    phase before writing, which makes single-buffered tags safe.
//  * Every wait is bounded.  On timeout a CTA sets the error word, stops issuing copies,
//    waits (bounded) for its own copies in flight and returns; the host reports
//    QDEC_E_TIMEOUT.
#include "common.cuh"

namespace qdec {

namespace {

constexpr int NCW = 7;                    // consumer warps (8 warps in all: 2 per SM sub-partition, 255 registers)
constexpr int NCT = 32 * NCW;             // consumer threads
constexpr int NT = NCT + 32;              // + one producer warp
constexpr uint32_t SLOT = 16384;          // ring slot bytes
constexpr int MAX_PR = (3072 / 2 + NCT - 1) / NCT;   // tagged word pairs per consumer thread (n <= 3072)
constexpr int PB = 4;                     // polls a thread keeps in flight (registers: 4 per pair)
constexpr uint32_t SPIN_FAST = 256;       // tagged-vector polls before backing off with nanosleep
constexpr uint32_t SPIN_LIMIT = kDecodeSpinDefault; // default polls (each ~0.3-1 us) before a wait gives up: about a
                                          // second; DecodeParams::spin_limit carries the step's own limit, and
                                          // the exit drain of copies in flight always uses this one
enum { PH_QKV = 0, PH_O = 1, PH_X1 = 2, PH_H = 3, PH_X2 = 4, PH_PER_LAYER = 5 };
enum { ERR_LL = 1, ERR_FULL = 2, ERR_EMPTY = 3, ERR_DRAIN = 4, ERR_PEER = 5 };
enum { F_ABORT = 0, F_ISSUED = 1 };

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t ring, full, empty, xbuf, xown, att, red, kred, flags, total;
};

constexpr int KS_ROWS = 8;   // rows of one K-split block

// Floats of one input-vector buffer: kmax rounded up to whole 256-column chunks (the
// permuted layout below fills chunk positions past the vector's end).
__host__ __device__ inline int xbuf_floats(int kmax) { return (kmax + 255) / 256 * 256; }

__host__ __device__ inline Layout make_layout(int nslot, int kmax, int xown_max, int att_floats) {
    Layout L;
    size_t o = 0;
    L.ring = o;  o += (size_t)nslot * SLOT;
    L.full = o;  o += (size_t)nslot * 8;
    L.empty = o; o += (size_t)nslot * 8;
    o = align_up(o, 16); L.xbuf = o; o += (size_t)xbuf_floats(kmax) * 2 * 4;   // double-buffered
    o = align_up(o, 16); L.xown = o; o += (size_t)xown_max * 4;
    o = align_up(o, 16); L.att = o;  o += (size_t)att_floats * 4;
    o = align_up(o, 16); L.red = o;  o += 64 * 4;
    o = align_up(o, 16); L.kred = o; o += 2 * NCW * KS_ROWS * 4;   // double-buffered
    L.flags = o; o += 16 * 4;
    L.total = o;
    return L;
}

__host__ __device__ inline void split_range(int n, int c, int nc, int& a, int& b) {
    a = (int)((long long)n * c / nc);
    b = (int)((long long)n * (c + 1) / nc);
}

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// True when all four barriers have completed the given phases.  One asm block, so the four
// tests are in flight together (each result is needed only at the end).
__device__ __forceinline__ bool mbar_test_wait4(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                                uint32_t p2, uint64_t* b3, uint32_t p3) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2, q3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
        "and.pred q0, q0, q1;\n\t"
        "and.pred q2, q2, q3;\n\t"
        "and.pred q0, q0, q2;\n\t"
        "selp.u32 %0, 1, 0, q0;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1), "r"(smem_u32(b2)), "r"(p2), "r"(smem_u32(b3)),
          "r"(p3)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// The same with an L2 eviction-priority policy (createpolicy)
__device__ __forceinline__ void tma_load_1d_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
// L2 prefetch of `bytes` (a multiple of 16) at src (16-byte aligned) with a policy
__device__ __forceinline__ void l2_prefetch_hint(const void* src, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

__device__ __forceinline__ void ll_store(unsigned long long* p, uint32_t tag, float v) {
    const unsigned long long w = ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// Two adjacent tagged words (each 8-byte half is single-copy atomic on its own).
__device__ __forceinline__ void ll_load2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ int volatile_load(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// 2^x with the MUFU instruction (relative error about 2^-22); -inf gives +0.  The attention
// units keep scores, maxima and partial maxima in log2 units (q is pre-scaled by log2 e).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Optional phase trace: globaltimer (ns) at slot `idx` of this CTA's row.
__device__ __forceinline__ void trace_mark(const DecodeParams& p, int idx) {
    if (p.trace) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        p.trace[(size_t)blockIdx.x * (11 * p.NL + 8) + idx] = t;
    }
}
// Wait-cycle accumulators of consumer thread 0 live in shared memory (flags[4..7]) and are
// written to the trace once, at the end of the step.
__device__ __forceinline__ void trace_add(int* flags, int which, unsigned long long v) {
    reinterpret_cast<unsigned long long*>(flags + 4)[which] += v;
}

__device__ __forceinline__ float dot8(const uint4 w, const float* x) {
    float a = bf_lo(w.x) * x[0];
    a = fmaf(bf_hi(w.x), x[1], a);
    a = fmaf(bf_lo(w.y), x[2], a);
    a = fmaf(bf_hi(w.y), x[3], a);
    a = fmaf(bf_lo(w.z), x[4], a);
    a = fmaf(bf_hi(w.z), x[5], a);
    a = fmaf(bf_lo(w.w), x[6], a);
    a = fmaf(bf_hi(w.w), x[7], a);
    return a;
}

// Shared-memory position of input element e in the permuted layout of a phase's input
// vector: within each 256-column chunk, the elements lane l covers (l*8 .. l*8+7) sit at
// l*4 .. l*4+3 and 128 + l*4 .. 128 + l*4+3, so both 16-byte loads of a warp read 512
// contiguous bytes (no bank conflicts).  Even e and e + 1 stay adjacent.
__device__ __forceinline__ int xperm(int e) {
    return (e & ~255) | ((e & 4) << 5) | ((e & 248) >> 1) | (e & 3);
}
// The 8 input values of lane `lane` in chunk c.
__device__ __forceinline__ void load_x8(const float* xs, int c, int lane, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(xs + c * 256 + lane * 4);
    const float4 b = *reinterpret_cast<const float4*>(xs + c * 256 + 128 + lane * 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <int EPL>
__device__ __forceinline__ void load_lane_bf16(const bf16_t* row, int lane, float* out) {
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

// Per-CTA work plan; producer and consumers derive identical values.
struct Plan {
    int q0, q1;    // rows of Wqkv
    int x0, x1;    // rows of Wo / Wd (residual rows this CTA owns)
    int f0, f1;    // gate/up pairs
    int v0, v1;    // lm_head rows
    bool unit;     // owns an attention unit
    int ug, uj;    // kv head and chunk of the unit
    int c0, c1;    // key positions of the unit: [c0, c1)
    int old_end;   // keys [c0, old_end) are read from the cache; position pos is the new key
    int rps_h, rps_o, rps_f, pps_gu, pps_kv;   // rows / pairs / positions per ring slot
};

__device__ inline Plan make_plan(const DecodeParams& p, int c, int nc) {
    Plan P;
    const int qkv_rows = (p.HQ + 2 * p.HKV) * p.D;
    split_range(qkv_rows, c, nc, P.q0, P.q1);
    split_range(p.H, c, nc, P.x0, P.x1);
    split_range(p.F, c, nc, P.f0, P.f1);
    split_range(p.V, c, nc, P.v0, P.v1);
    const int n_units = p.HKV * p.n_chunks;
    const int u = (int)(((long long)c * n_units + nc - 1) / nc);
    P.unit = (u < n_units) && ((int)((long long)u * nc / n_units) == c);
    P.ug = P.unit ? u / p.n_chunks : 0;
    P.uj = P.unit ? u % p.n_chunks : 0;
    const int L = p.pos + 1;
    P.c0 = P.uj * p.chunk;
    P.c1 = min(L, P.c0 + p.chunk);
    P.old_end = min(P.c1, p.pos);
    if (!P.unit) P.c0 = P.c1 = P.old_end = 0;
    P.rps_h = (int)(SLOT / (p.H * 2));
    P.rps_o = (int)(SLOT / (p.HQ * p.D * 2));
    P.rps_f = (int)(SLOT / (p.F * 2));
    P.pps_gu = (int)(SLOT / (p.H * 4));
    P.pps_kv = min(64, (int)(SLOT / (p.D * 2)));
    return P;
}

struct Ctx {
    char* ring;
    uint64_t* full;
    uint64_t* empty;
    float* xbuf;
    float* xown;
    float* att;
    float* red;
    float* kred;
    int* flags;
    int nslot;
    int kmax;      // floats per xbuf buffer (xbuf holds two), a multiple of 256
};

// Sets the CTA's abort flag and the global error word (first error wins).
__device__ inline void raise_error(const Ctx& S, const DecodeParams& p, int code) {
    reinterpret_cast<volatile int*>(S.flags)[F_ABORT] = 1;
    atomicCAS(p.err, 0, code);
}

// True once this CTA or any other has failed; latches the CTA's flag so that every
// consumer thread takes the same (wait-free) path after its next barrier.  The global
// error word costs an L2 round trip, so waits consult it only every `global_every`-th
// call of their slow path (errors are rare; normal waits must not pay for the check).
__device__ inline bool should_abort(const Ctx& S, const DecodeParams& p, bool check_global) {
    volatile int* f = reinterpret_cast<volatile int*>(S.flags);
    if (f[F_ABORT]) return true;
    if (check_global && volatile_load(p.err) != 0) {
        f[F_ABORT] = 1;
        return true;
    }
    return false;
}

// Bounded wait on an mbarrier phase; returns false at once after an abort.
__device__ inline bool wait_bar(const Ctx& S, const DecodeParams& p, uint64_t* bar, uint32_t parity, int code) {
    if (mbar_test_wait(bar, parity)) return true;
    if (reinterpret_cast<volatile int*>(S.flags)[F_ABORT]) return false;
    for (uint32_t it = 0; it < p.spin_limit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;   // suspends the thread for a while when not ready
        if ((it & 1023) == 1023 && should_abort(S, p, (it & 16383) == 16383)) return false;
    }
    raise_error(S, p, code);
    return false;
}

// A tagged vector to fetch: n (even) words from src (16-byte aligned).
struct LLSeg {
    const unsigned long long* src;
    int n;
};

// All consumer threads: the segments' words, concatenated, into dst once every tag equals
// `tag` (times gain[i] when `gain` is given; the sum of squares is of the raw values),
// at dst[i] or, with PERM, at dst[xperm(i)].  A thread owns word pairs ct, ct + NCT, ...; each poll issues all of its pending
// 16-byte loads before it looks at any result, so one round of polls costs one L2 round
// trip per PB pairs (not one per word).  Returns the thread's partial sum of squares through *ss.
template <int NSEG, bool PERM = false>
__device__ __forceinline__ bool ll_fetch(const Ctx& S, const DecodeParams& p, const LLSeg (&seg)[NSEG], uint32_t tag,
                                float* dst, float* ss, const bf16_t* gain = nullptr) {
    const int ct = threadIdx.x;
    if (reinterpret_cast<volatile int*>(S.flags)[F_ABORT]) return false;
    const long long t0 = (p.trace && ct == 0) ? clock64() : 0;
    int npairs = 0;
#pragma unroll
    for (int q = 0; q < NSEG; ++q) npairs += seg[q].n >> 1;
    // address of the pair k of this thread (recomputed per poll: no pointer array held in registers)
    auto at = [&](int k) -> const unsigned long long* {
        int e = 2 * (ct + k * NCT);
        const unsigned long long* a = seg[0].src + e;
#pragma unroll
        for (int q = 1; q < NSEG; ++q) {
            e -= seg[q - 1].n;
            if (e >= 0) a = seg[q].src + e;
        }
        return a;
    };
    uint32_t pending = 0;
#pragma unroll 1
    for (int k = 0; k < MAX_PR; ++k) {
        if (ct + k * NCT < npairs) {
            pending |= 1u << k;
            // the gains are read once the values arrive: have them in L1 by then
            if (gain) asm volatile("prefetch.global.L1 [%0];" ::"l"(gain + 2 * (ct + k * NCT)));
        }
    }
    float acc = 0.f;
    for (uint32_t it = 0; pending; ++it) {
#pragma unroll 1
        for (int k0 = 0; k0 < MAX_PR; k0 += PB) {
            unsigned long long w0[PB], w1[PB];
#pragma unroll
            for (int kk = 0; kk < PB; ++kk) {
                const int k = k0 + kk;
                if (k < MAX_PR && (pending & (1u << k))) ll_load2(at(k), w0[kk], w1[kk]);
            }
#pragma unroll
            for (int kk = 0; kk < PB; ++kk) {
                const int k = k0 + kk;
                if (k < MAX_PR && (pending & (1u << k)) && (uint32_t)(w0[kk] >> 32) == tag &&
                    (uint32_t)(w1[kk] >> 32) == tag) {
                    const float a = __uint_as_float((uint32_t)w0[kk]), b = __uint_as_float((uint32_t)w1[kk]);
                    const int e = 2 * (ct + k * NCT);
                    const uint32_t gp = gain ? __ldg(reinterpret_cast<const unsigned int*>(gain + e)) : 0x3f803f80u;
                    *reinterpret_cast<float2*>(dst + (PERM ? xperm(e) : e)) = make_float2(a * bf_lo(gp), b * bf_hi(gp));
                    acc = fmaf(a, a, fmaf(b, b, acc));
                    pending &= ~(1u << k);
                }
            }
        }
        if (!pending) break;
        if (it >= p.spin_limit) {
            raise_error(S, p, ERR_LL);
            return false;
        }
        if ((it & 255) == 255 && should_abort(S, p, (it & 4095) == 4095)) return false;
        if (it >= SPIN_FAST) __nanosleep(32);
    }
    *ss += acc;
    if (p.trace && ct == 0) trace_add(S.flags, 1, (unsigned long long)(clock64() - t0));
    return true;
}

// Input vector of a GEMV phase into shared memory, permuted (xperm): xs = gain * x (x
// without a gain), and the RMSNorm scale r = rsqrt(mean x^2 + eps) (1 without a gain) that the
// phase applies to its dot products, so rms_norm(x) * gain . w = r * (gain * x . w).
// Source: `row` (bf16, the embedding row) when non-null, else the tagged vector `ll`.
// The buffer and the reduction slots alternate between calls (`par`): a phase reads xs
// until the next call's barrier, which every consumer thread passes first.
__device__ inline float prep_input(const Ctx& S, const DecodeParams& p, const unsigned long long* ll,
                                   const bf16_t* row, int n, uint32_t tag, const bf16_t* gain, const float*& xs,
                                   int& par) {
    float* xb = S.xbuf + (size_t)par * S.kmax;
    float* rd = S.red + par * 8;
    par ^= 1;
    const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
    float ss = 0.f;
    if (row) {
        for (int i = ct; i < n; i += NCT) {
            const float v = bf1(row[i]);
            xb[xperm(i)] = gain ? v * bf1(gain[i]) : v;
            ss = fmaf(v, v, ss);
        }
    } else {
        const LLSeg seg[1] = {{ll, n}};
        ll_fetch<1, true>(S, p, seg, tag, xb, &ss, gain);
    }
    ss = warp_sum(ss);
    if (lane == 0) rd[warp] = ss;
    consumer_sync();
    xs = xb;
    if (!gain) return 1.f;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) tot += rd[w];
    return rsqrtf(tot / (float)n + p.eps);
}

// Consumer view of the ring: every consumer warp walks the same stage sequence.  The
// slot and the barrier parity of the next stage are tracked incrementally (no division).
struct Ring {
    int slot = 0;          // slot of the next stage to consume
    uint32_t parity = 0;   // parity of that slot's pending full-barrier phase
    // Slot data of the stage d ahead of the next one (d < nslot).
    __device__ const char* ptr(const Ctx& S, int d) const {
        const int s = slot + d;
        return S.ring + (size_t)(s >= S.nslot ? s - S.nslot : s) * SLOT;
    }
    // Waits for the data of the stage d ahead; after an abort it returns without waiting
    // (the contents are then garbage, and nothing computed from them is published).
    __device__ void wait(const Ctx& S, const DecodeParams& p, int d) const {
        int s = slot + d;
        uint32_t par = parity;
        if (s >= S.nslot) {
            s -= S.nslot;
            par ^= 1u;
        }
        const long long t0 = (p.trace && threadIdx.x == 0) ? clock64() : 0;
        wait_bar(S, p, &S.full[s], par, ERR_FULL);
        if (p.trace && threadIdx.x == 0) trace_add(S.flags, 0, (unsigned long long)(clock64() - t0));
    }
    __device__ const char* acquire(const Ctx& S, const DecodeParams& p) {
        wait(S, p, 0);
        return ptr(S, 0);
    }
    // Waits for the stages 0 .. g-1 ahead (g < nslot): their barriers are tested four at a
    // time in one go, and only an incomplete group falls back to the bounded per-stage waits.
    __device__ void wait_group(const Ctx& S, const DecodeParams& p, int g) const {
        for (int s0 = 0; s0 < g; s0 += 4) {
            uint64_t* b[4];
            uint32_t par[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int s = slot + min(s0 + j, g - 1);
                par[j] = parity;
                if (s >= S.nslot) {
                    s -= S.nslot;
                    par[j] ^= 1u;
                }
                b[j] = &S.full[s];
            }
            if (!mbar_test_wait4(b[0], par[0], b[1], par[1], b[2], par[2], b[3], par[3]))
                for (int j = s0; j < min(s0 + 4, g); ++j) wait(S, p, j);
        }
    }
    // Hands back the next g stages (see release).
    __device__ void release_group(const Ctx& S, int g) {
        __syncwarp();
        const bool give = (threadIdx.x & 31) == 0 && !reinterpret_cast<volatile int*>(S.flags)[F_ABORT];
        for (int j = 0; j < g; ++j) {
            if (give) mbar_arrive(&S.empty[slot]);
            if (++slot == S.nslot) {
                slot = 0;
                parity ^= 1u;
            }
        }
    }
    // After an abort a slot is never handed back: its copy may still be in flight, and the
    // producer must not reuse it (the final drain waits for it instead).
    __device__ void release(const Ctx& S) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0 && !reinterpret_cast<volatile int*>(S.flags)[F_ABORT])
            mbar_arrive(&S.empty[slot]);
        if (++slot == S.nslot) {
            slot = 0;
            parity ^= 1u;
        }
    }
};

// Where the rows of a matrix phase go.
enum { EMIT_LL = 0, EMIT_RESID = 1, EMIT_LOGITS = 2 };
struct PhaseOut {
    int kind;
    unsigned long long* ll;   // EMIT_LL / EMIT_RESID: tagged destination of row 0
    uint32_t tag;
    float* logits;            // EMIT_LOGITS: logits of row 0
    int row0;                 // EMIT_LOGITS: vocabulary index of row 0
};

// Row i's value v: a tagged element (EMIT_RESID first adds it into the residual row this
// CTA owns), or a logit with the running (value, index) maximum of lane 0.
__device__ __forceinline__ void emit_value(const Ctx& S, const PhaseOut& o, int i, float v, float& best, int& besti) {
    if (o.kind == EMIT_LOGITS) {
        o.logits[i] = v;
        if (am_better(v, o.row0 + i, best, besti)) {
            best = v;
            besti = o.row0 + i;
        }
    } else {
        if (o.kind == EMIT_RESID) {
            v += S.xown[i];
            S.xown[i] = v;
        }
        ll_store(o.ll + i, o.tag, v);
    }
}

// Rows [r0, r1) of a matrix phase whose ring stages hold `per` rows each (GLU: `per`
// gate/up pairs; a stage with n pairs holds n gate rows, then the n matching up rows);
// stage s0 of the phase is the ring's next stage.  Each warp computes R rows at a time
// with independent accumulators, so the dot products and the shuffle reductions of
// several rows overlap.  The input vector xs is in shared memory; lane l covers columns
// l*8 + 256 i.  Row values are r * (w . xs), or for GLU silu(r * gate . xs) * (r * up . xs).
template <bool GLU, int R>
__device__ inline void group_rows(const Ring& ring, const Ctx& S, int s0, int r0, int r1, int rows, int per,
                                  float inv_per, int K, const float* xs, float r, const PhaseOut& out, float& best,
                                  int& besti) {
    constexpr int NA = GLU ? 2 : 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int base = r0 + warp; base < r1; base += NCW * R) {
        const uint4* w[R][NA];
        bool valid[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            // rows past the end re-read row `base` (always valid): no branches in the dot products
            const int rr = base + NCW * j;
            valid[j] = rr < r1;
            const int rw = valid[j] ? rr : base;
            const int st = __float2int_rz(((float)rw + 0.5f) * inv_per), off = rw - st * per;
            const int ns = min(per, rows - st * per);
            const char* sp = ring.ptr(S, st - s0);
            w[j][0] = reinterpret_cast<const uint4*>(sp + (size_t)off * K * 2);
            if (GLU) w[j][NA - 1] = reinterpret_cast<const uint4*>(sp + (size_t)(ns + off) * K * 2);
        }
        float acc[R][NA];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int a = 0; a < NA; ++a) acc[j][a] = 0.f;
#pragma unroll 1
        for (int c = 0; c * 256 + lane * 8 < K; ++c) {
            float x[8];
            load_x8(xs, c, lane, x);
            const int k8 = c * 32 + lane;
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int a = 0; a < NA; ++a) acc[j][a] += dot8(w[j][a][k8], x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int a = 0; a < NA; ++a) acc[j][a] += __shfl_xor_sync(0xffffffffu, acc[j][a], o);
        // every lane holds every sum: lane j emits row j (the stores go out together)
        float v = 0.f;
        bool mine = false;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            if (lane == j) {
                v = GLU ? silu(r * acc[j][0]) * (r * acc[j][NA - 1]) : r * acc[j][0];
                mine = valid[j];
            }
        }
        if (mine) emit_value(S, out, base + NCW * lane, v, best, besti);
    }
}

// Rows [r0, r1) with K split over the warps: warp w takes the 256-column chunks w, w + NCW,
// ... of every row in a block of up to KS_ROWS rows, so each warp reads its slice of the
// input vector once; the warps' partial sums meet in shared memory and one thread per row
// adds them and emits the row.  For groups with too few rows to give every warp whole rows
// (o_proj, down_proj).  Every consumer thread calls it (it holds a barrier per block).
__device__ inline void ksplit_rows(const Ring& ring, const Ctx& S, int s0, int r0, int r1, int per, float inv_per,
                                   int K, const float* xs, float r, const PhaseOut& out, float& best, int& besti,
                                   int& kpar) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b0 = r0; b0 < r1; b0 += KS_ROWS) {
        const int nr = min(KS_ROWS, r1 - b0);
        const uint4* w[KS_ROWS];
#pragma unroll
        for (int j = 0; j < KS_ROWS; ++j) {
            const int rw = b0 + min(j, nr - 1);
            const int st = __float2int_rz(((float)rw + 0.5f) * inv_per), off = rw - st * per;
            w[j] = reinterpret_cast<const uint4*>(ring.ptr(S, st - s0) + (size_t)off * K * 2);
        }
        float acc[KS_ROWS];
#pragma unroll
        for (int j = 0; j < KS_ROWS; ++j) acc[j] = 0.f;
#pragma unroll 1
        for (int c = warp; c * 256 < K; c += NCW) {
            if (c * 256 + lane * 8 < K) {
                float x[8];
                load_x8(xs, c, lane, x);
                const int k8 = c * 32 + lane;
#pragma unroll
                for (int j = 0; j < KS_ROWS; ++j)
                    if (j < nr) acc[j] += dot8(w[j][k8], x);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int j = 0; j < KS_ROWS; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
        float* kr = S.kred + kpar * (NCW * KS_ROWS);
        kpar ^= 1;
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < KS_ROWS; ++j)
            if (lane == j) v = acc[j];
        if (lane < KS_ROWS) kr[warp * KS_ROWS + lane] = v;
        consumer_sync();
        if ((int)threadIdx.x < nr) {
            float t = 0.f;
#pragma unroll
            for (int q = 0; q < NCW; ++q) t += kr[q * KS_ROWS + threadIdx.x];
            emit_value(S, out, b0 + threadIdx.x, r * t, best, besti);
        }
    }
}

// Rows [0, rows) of one matrix phase: up to `group` stages are acquired together (one wait,
// then all their rows), then handed back.  The row routine is chosen per group: GLU pairs,
// 4 rows a pass when the group has enough rows for every warp, K split over the warps
// when it has few rows and a long K, else 1 row a pass.
__device__ inline void gemv_phase(Ring& ring, const Ctx& S, const DecodeParams& p, bool glu, int rows, int per, int K,
                                  const float* xs, float r, int group, const PhaseOut& out, float& best, int& besti,
                                  int& kpar) {
    const int maxg = min(group, S.nslot - 1);
    const int nst = (rows + per - 1) / per;
    // stage of row i = floor(i / per) as (i + 0.5) * (1 / per) truncated: exact for i < 2^20, per <= 2^10
    const float inv_per = 1.f / (float)per;
    for (int s0 = 0; s0 < nst; s0 += maxg) {
        const int g = min(maxg, nst - s0);
        ring.wait_group(S, p, g);
        const int r0 = s0 * per, r1 = min(rows, (s0 + g) * per);
        if (glu) group_rows<true, 3>(ring, S, s0, r0, r1, rows, per, inv_per, K, xs, r, out, best, besti);
        else if (r1 - r0 >= 3 * NCW) group_rows<false, 4>(ring, S, s0, r0, r1, rows, per, inv_per, K, xs, r, out, best, besti);
        else if (K >= 512 && r1 - r0 < 2 * NCW) ksplit_rows(ring, S, s0, r0, r1, per, inv_per, K, xs, r, out, best, besti, kpar);
        else group_rows<false, 1>(ring, S, s0, r0, r1, rows, per, inv_per, K, xs, r, out, best, besti);
        ring.release_group(S, g);
    }
}

// ------------------------------------------------------------------ the kernel
template <int D, int G>
__global__ void __launch_bounds__(NT, 1) decode_persistent_kernel(const DecodeParams p) {
    extern __shared__ __align__(1024) char smem[];
    const int nc = gridDim.x, c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HQD = p.HQ * p.D;
    const int kmax = max(max(p.H, HQD), max(p.F, (G + 2) * D));
    const int xown_max = (p.H + nc - 1) / nc + 1;
    const Layout LO = make_layout(p.nslot, kmax, xown_max, NCW * G * (D + 2));
    Ctx S;
    S.ring = smem + LO.ring;
    S.full = reinterpret_cast<uint64_t*>(smem + LO.full);
    S.empty = reinterpret_cast<uint64_t*>(smem + LO.empty);
    S.xbuf = reinterpret_cast<float*>(smem + LO.xbuf);
    S.xown = reinterpret_cast<float*>(smem + LO.xown);
    S.att = reinterpret_cast<float*>(smem + LO.att);
    S.red = reinterpret_cast<float*>(smem + LO.red);
    S.kred = reinterpret_cast<float*>(smem + LO.kred);
    S.flags = reinterpret_cast<int*>(smem + LO.flags);
    S.nslot = p.nslot;
    S.kmax = xbuf_floats(kmax);
    const Plan P = make_plan(p, c, nc);
    const uint32_t tags_per_step = (uint32_t)p.NL * PH_PER_LAYER + 1;
    auto tag = [&](int l, int ph) { return p.epoch * tags_per_step + (uint32_t)(l * PH_PER_LAYER + ph); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nslot; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], NCW);
        }
        S.flags[F_ABORT] = 0;
        S.flags[F_ISSUED] = 0;
        reinterpret_cast<unsigned long long*>(S.flags + 4)[0] = 0;
        reinterpret_cast<unsigned long long*>(S.flags + 4)[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int token = p.token >= 0 ? p.token : volatile_load(p.argmax);
    const bf16_t* erow = p.embed + (size_t)token * p.H;

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // One pass over the step's phases in consumption order; each phase is described
            // by its source rows [i0, i1) (`per` a stage, `stride` elements apart) and either
            // two stages per item group (a K chunk, then its V chunk) or one stage with two
            // sources (gate rows, then the matching up rows).
            int slot = 0, issued = 0;
            uint32_t parity = 0;
            bool ok = true;
            const int n_ph = p.NL * PH_PER_LAYER + 1;
            // The step streams every weight once (1.2 GB against a 129 MB L2): weight stages
            // carry an evict-first policy, so they do not push out the KV history and the
            // lm_head rows prefetched below.  The lm_head phase streams its 311 MB at the HBM
            // roofline after the last layer, while the layers before it, bound by their
            // hand-offs, use a fraction of HBM: during each of the last LM_PF_LAYERS layers
            // this CTA prefetches another 1/LM_PF_DEN of its lm_head rows into L2 (evict-last).
            constexpr int LM_PF_LAYERS = 3, LM_PF_DEN = 12;
            uint64_t pol_w, pol_keep;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
#pragma unroll 1
            for (int t = 0; t < n_ph && ok; ++t) {
                const int l = min(t / PH_PER_LAYER, p.NL - 1);
                const int e = (t == n_ph - 1) ? PH_PER_LAYER : t - l * PH_PER_LAYER;
                const DecodeLayer* Lw = p.layers + l;
                if (e == 0 && l >= p.NL - LM_PF_LAYERS && l < p.NL) {
                    const int nv = P.v1 - P.v0, k = l - (p.NL - LM_PF_LAYERS);
                    const int a = P.v0 + (int)((long long)nv * k / LM_PF_DEN);
                    const int b = P.v0 + (int)((long long)nv * (k + 1) / LM_PF_DEN);
                    for (int r = a; r < b; r += 32)   // 32 rows (64 KB at H = 1024) a request
                        l2_prefetch_hint(p.embed + (size_t)r * p.H, (uint32_t)(min(32, b - r) * p.H * 2), pol_keep);
                }
                const bf16_t *src0, *src1 = nullptr, *src_up = nullptr;
                int i0, i1, per, stride, nsub = 1;
                if (e == 0) {
                    src0 = Lw->wqkv; i0 = P.q0; i1 = P.q1; per = P.rps_h; stride = p.H;
                } else if (e == 1) {
                    const size_t off = (size_t)P.ug * p.max_seq * D;
                    src0 = Lw->kc + off; src1 = Lw->vc + off; i0 = P.c0; i1 = P.old_end; per = P.pps_kv; stride = D;
                    nsub = 2;
                } else if (e == 2) {
                    src0 = Lw->wo; i0 = P.x0; i1 = P.x1; per = P.rps_o; stride = HQD;
                } else if (e == 3) {
                    src0 = Lw->wgu; src_up = Lw->wgu + (size_t)p.F * p.H; i0 = P.f0; i1 = P.f1; per = P.pps_gu;
                    stride = p.H;
                } else if (e == 4) {
                    src0 = Lw->wd; i0 = P.x0; i1 = P.x1; per = P.rps_f; stride = p.F;
                } else {
                    src0 = p.embed; i0 = P.v0; i1 = P.v1; per = P.rps_h; stride = p.H;
                }
                for (int i = i0; i < i1 && ok; i += per) {
                    const uint32_t bytes = (uint32_t)min(per, i1 - i) * (uint32_t)stride * 2u;
                    for (int sub = 0; sub < nsub; ++sub) {
                        if (!wait_bar(S, p, &S.empty[slot], parity ^ 1u, ERR_EMPTY) ||
                            reinterpret_cast<volatile int*>(S.flags)[F_ABORT]) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(&S.full[slot], src_up ? 2u * bytes : bytes);
                        char* dst = S.ring + (size_t)slot * SLOT;
                        if (e == 1) {   // the KV history: default policy
                            tma_load_1d(dst, (sub == 0 ? src0 : src1) + (size_t)i * stride, bytes, &S.full[slot]);
                        } else {
                            tma_load_1d_hint(dst, src0 + (size_t)i * stride, bytes, &S.full[slot], pol_w);
                            if (src_up)
                                tma_load_1d_hint(dst + bytes, src_up + (size_t)i * stride, bytes, &S.full[slot], pol_w);
                        }
                        ++issued;
                        if (++slot == S.nslot) {
                            slot = 0;
                            parity ^= 1u;
                        }
                    }
                }
                if (e == 4) trace_mark(p, 10 * p.NL + 4 + l);
            }
            reinterpret_cast<volatile int*>(S.flags)[F_ISSUED] = issued;
        }
    } else {
        // ------------------------------------------------------------ consumers
        // Control flow below depends only on the plan, never on errors: every consumer
        // thread executes the same barriers whatever happens.
        Ring ring;
        const float* xs = nullptr;   // input vector of the current phase (shared memory)
        int par = 0;   // alternates the staging buffer between input preparations
        if (c == 0 && threadIdx.x == 0) p.history[p.pos] = token;
        for (int r = P.x0 + threadIdx.x; r < P.x1; r += NCT) S.xown[r - P.x0] = bf1(erow[r]);
        consumer_sync();
        const bool tr = p.trace && threadIdx.x == 0;
        if (tr) trace_mark(p, 10 * p.NL + 0);

        float best = -INFINITY;   // lm_head: this thread's running maximum of the rows it emitted
        int besti = 0x7fffffff;
        int kpar = 0;             // alternates the K-split partial buffers
        // One pass over the step's phases: per layer QKV rows, attention, o_proj rows,
        // gate_up pairs, down_proj rows; then the lm_head rows.  A single copy of each code
        // path serves every phase (the loop is not unrolled), which keeps the kernel's hot
        // code small enough to stay in the instruction cache.
        const int n_ph = p.NL * PH_PER_LAYER + 1;
#pragma unroll 1
        for (int t = 0; t < n_ph; ++t) {
            const int l = min(t / PH_PER_LAYER, p.NL - 1);
            const int e = (t == n_ph - 1) ? PH_PER_LAYER : t - l * PH_PER_LAYER;
            const DecodeLayer* Lw = p.layers + l;
            if (e == PH_O) {
                // ---- attention unit (kv head ug, key chunk [c0, c1)) -> tagged o
                if (P.unit) {
                    constexpr int EPL = D / 32;
                    const int g = P.ug;
                    const uint32_t tq = tag(l, PH_QKV);
                    const int half = D / 2;
                    constexpr int PPL = (D / 2 + 31) / 32;   // NeoX pairs per lane
                    // gains and cos/sin of the first head this warp normalises, loaded before the waits
                    float pg_a[PPL], pg_b[PPL];
                    float2 pcs[PPL];
                    {
                        const bf16_t* gn0 = warp < G ? Lw->g_q : Lw->g_k;
    #pragma unroll
                        for (int k = 0; k < PPL; ++k) {
                            const int i = lane + 32 * k;
                            pg_a[k] = i < half ? bf1(gn0[i]) : 0.f;
                            pg_b[k] = i < half ? bf1(gn0[i + half]) : 0.f;
                            pcs[k] = i < half ? p.rope[(size_t)p.pos * half + i] : make_float2(1.f, 0.f);
                        }
                    }
                    float ss = 0.f;
                    float* xa = S.xbuf + (size_t)par * S.kmax;   // q heads, then k, then v
                    par ^= 1;
                    const LLSeg seg[3] = {{p.ll_qkv + (size_t)g * G * D, G * D},
                                          {p.ll_qkv + HQD + (size_t)g * D, D},
                                          {p.ll_qkv + HQD + (size_t)(p.HKV + g) * D, D}};
                    ll_fetch(S, p, seg, tq, xa, &ss);
                    consumer_sync();
                    if (tr) trace_mark(p, l * 10 + 2);
                    // per-head RMSNorm + NeoX RoPE on the G q heads and the k head; bf16 rounding of k, v
                    for (int hh = warp; hh <= G; hh += NCW) {
                        float* hv = xa + hh * D;
                        if (hh != warp) {   // a second head for this warp (G + 1 > NCW): load its gains now
                            const bf16_t* gn1 = hh < G ? Lw->g_q : Lw->g_k;
    #pragma unroll
                            for (int k = 0; k < PPL; ++k) {
                                const int i = lane + 32 * k;
                                pg_a[k] = i < half ? bf1(gn1[i]) : 0.f;
                                pg_b[k] = i < half ? bf1(gn1[i + half]) : 0.f;
                            }
                        }
                        float a[PPL], b[PPL];
                        float s2 = 0.f;
    #pragma unroll
                        for (int k = 0; k < PPL; ++k) {
                            const int i = lane + 32 * k;
                            a[k] = i < half ? hv[i] : 0.f;
                            b[k] = i < half ? hv[i + half] : 0.f;
                            s2 += a[k] * a[k] + b[k] * b[k];
                        }
                        s2 = warp_sum(s2);
                        const float r = rsqrtf(s2 / (float)D + p.eps);
    #pragma unroll
                        for (int k = 0; k < PPL; ++k) {
                            const int i = lane + 32 * k;
                            if (i < half) {
                                const float x1 = a[k] * r * pg_a[k], x2 = b[k] * r * pg_b[k];
                                const float2 cs = pcs[k];
                                float o1 = x1 * cs.x - x2 * cs.y, o2 = x2 * cs.x + x1 * cs.y;
                                if (hh == G) {   // the cache holds bf16 keys: use the rounded values
                                    o1 = bf1(f2bf(o1));
                                    o2 = bf1(f2bf(o2));
                                }
                                hv[i] = o1;
                                hv[i + half] = o2;
                            }
                        }
                    }
                    for (int d = threadIdx.x; d < D; d += NCT) xa[(G + 1) * D + d] = bf1(f2bf(xa[(G + 1) * D + d]));
                    consumer_sync();
                    const bool has_new = (P.c0 <= p.pos) && (p.pos < P.c1);
                    if (has_new) {
                        for (int d = threadIdx.x; d < D; d += NCT) {
                            Lw->kc[((size_t)g * p.max_seq + p.pos) * D + d] = f2bf(xa[G * D + d]);
                            Lw->vc[((size_t)g * p.max_seq + p.pos) * D + d] = f2bf(xa[(G + 1) * D + d]);
                        }
                    }
                    const float scale = rsqrtf((float)D) * 1.4426950408889634f;   // scores in log2 units
                    float qv[G][EPL], m[G], lsum[G], o[G][EPL];
    #pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
    #pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            qv[gi][e] = xa[gi * D + lane * EPL + e] * scale;
                            o[gi][e] = 0.f;
                        }
                        m[gi] = -INFINITY;
                        lsum[gi] = 0.f;
                    }
                    // online softmax over the streamed keys: per stage, warp w takes positions w + NCW k
                    constexpr int KPW = (64 + NCW - 1) / NCW;   // positions per warp per stage (pps_kv <= 64)
                    for (int q = P.c0; q < P.old_end; q += P.pps_kv) {
                        const int np = min(P.pps_kv, P.old_end - q);
                        const char* ks = ring.acquire(S, p);
                        float s[KPW][G];
    #pragma unroll
                        for (int k = 0; k < KPW; ++k) {
                            const int t = min(warp + NCW * k, np - 1);   // clamped: computed, then masked
                            float kf[EPL];
                            load_lane_bf16<EPL>(reinterpret_cast<const bf16_t*>(ks) + (size_t)t * D, lane, kf);
    #pragma unroll
                            for (int gi = 0; gi < G; ++gi) {
                                float d0 = 0.f;
    #pragma unroll
                                for (int e = 0; e < EPL; ++e) d0 = fmaf(qv[gi][e], kf[e], d0);
                                s[k][gi] = d0;
                            }
                        }
    #pragma unroll
                        for (int sh = 16; sh > 0; sh >>= 1)
    #pragma unroll
                            for (int k = 0; k < KPW; ++k)
    #pragma unroll
                                for (int gi = 0; gi < G; ++gi) s[k][gi] += __shfl_xor_sync(0xffffffffu, s[k][gi], sh);
    #pragma unroll
                        for (int k = 0; k < KPW; ++k)
                            if (warp + NCW * k >= np)
    #pragma unroll
                                for (int gi = 0; gi < G; ++gi) s[k][gi] = -INFINITY;
                        ring.release(S);
    #pragma unroll
                        for (int gi = 0; gi < G; ++gi) {
                            float mx = -INFINITY;
    #pragma unroll
                            for (int k = 0; k < KPW; ++k) mx = fmaxf(mx, s[k][gi]);
                            const float mn = fmaxf(m[gi], mx);
                            if (mn != -INFINITY) {
                                const float corr = ex2(m[gi] - mn);   // 0 when m was -inf
                                lsum[gi] *= corr;
    #pragma unroll
                                for (int e = 0; e < EPL; ++e) o[gi][e] *= corr;
                                m[gi] = mn;
    #pragma unroll
                                for (int k = 0; k < KPW; ++k) {
                                    s[k][gi] = ex2(s[k][gi] - mn);   // masked scores (-inf) give 0
                                    lsum[gi] += s[k][gi];
                                }
                            } else {
    #pragma unroll
                                for (int k = 0; k < KPW; ++k) s[k][gi] = 0.f;
                            }
                        }
                        const char* vs = ring.acquire(S, p);
    #pragma unroll
                        for (int k = 0; k < KPW; ++k) {
                            const int t = min(warp + NCW * k, np - 1);   // masked positions carry weight 0
                            float vf[EPL];
                            load_lane_bf16<EPL>(reinterpret_cast<const bf16_t*>(vs) + (size_t)t * D, lane, vf);
    #pragma unroll
                            for (int gi = 0; gi < G; ++gi)
    #pragma unroll
                                for (int e = 0; e < EPL; ++e) o[gi][e] = fmaf(s[k][gi], vf[e], o[gi][e]);
                        }
                        ring.release(S);
                    }
                    if (has_new && warp == 0) {   // the token's own key and value
                        float kf[EPL], vf[EPL];
    #pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            kf[e] = xa[G * D + lane * EPL + e];
                            vf[e] = xa[(G + 1) * D + lane * EPL + e];
                        }
    #pragma unroll
                        for (int gi = 0; gi < G; ++gi) {
                            float d0 = 0.f;
    #pragma unroll
                            for (int e = 0; e < EPL; ++e) d0 = fmaf(qv[gi][e], kf[e], d0);
                            const float sc = warp_sum(d0);
                            const float mn = fmaxf(m[gi], sc);
                            const float corr = ex2(m[gi] - mn);
                            const float pr = ex2(sc - mn);
                            lsum[gi] = lsum[gi] * corr + pr;
    #pragma unroll
                            for (int e = 0; e < EPL; ++e) o[gi][e] = fmaf(pr, vf[e], o[gi][e] * corr);
                            m[gi] = mn;
                        }
                    }
                    // merge the warps' (m, l, o)
    #pragma unroll
                    for (int gi = 0; gi < G; ++gi) {
                        float* a = S.att + ((size_t)warp * G + gi) * (D + 2);
                        if (lane == 0) {
                            a[0] = m[gi];
                            a[1] = lsum[gi];
                        }
    #pragma unroll
                        for (int e = 0; e < EPL; ++e) a[2 + lane * EPL + e] = o[gi][e];
                    }
                    consumer_sync();
                    const uint32_t to = tag(l, PH_O);
                    const bool single = p.n_chunks == 1;
                    for (int idx = threadIdx.x; idx < G * D; idx += NCT) {
                        const int gi = idx / D, d = idx % D;
                        float M = -INFINITY;
    #pragma unroll
                        for (int w = 0; w < NCW; ++w) M = fmaxf(M, S.att[((size_t)w * G + gi) * (D + 2)]);
                        float lt = 0.f, ot = 0.f;
    #pragma unroll
                        for (int w = 0; w < NCW; ++w) {
                            const float* a = S.att + ((size_t)w * G + gi) * (D + 2);
                            const float f = (a[0] == -INFINITY) ? 0.f : ex2(a[0] - M);
                            lt += f * a[1];
                            ot += f * a[2 + d];
                        }
                        const int h = g * G + gi;
                        if (single) {
                            ll_store(p.ll_o + (size_t)h * D + d, to, ot / lt);
                        } else {
                            float* part = p.attn_part + ((size_t)h * p.n_chunks + P.uj) * (D + 2);
                            part[2 + d] = ot;
                            if (d == 0) {
                                part[0] = M;
                                part[1] = lt;
                            }
                        }
                    }
                    if (!single) {
                        __threadfence();
                        consumer_sync();
                        if (threadIdx.x == 0) {
                            const unsigned int tk = atomicAdd(&p.attn_count[l * p.HKV + g], 1u);
                            S.flags[2] = (tk == (unsigned int)p.n_chunks - 1) ? 1 : 0;
                        }
                        consumer_sync();
                        if (S.flags[2]) {   // the last chunk of this kv head merges all chunks
                            __threadfence();
                            for (int idx = threadIdx.x; idx < G * D; idx += NCT) {
                                const int gi = idx / D, d = idx % D;
                                const int h = g * G + gi;
                                const float* base = p.attn_part + (size_t)h * p.n_chunks * (D + 2);
                                float M = -INFINITY;
                                for (int j = 0; j < p.n_chunks; ++j) M = fmaxf(M, __ldcg(base + (size_t)j * (D + 2)));
                                float lt = 0.f, ot = 0.f;
                                for (int j = 0; j < p.n_chunks; ++j) {
                                    const float* a = base + (size_t)j * (D + 2);
                                    const float mj = __ldcg(a);
                                    const float f = (mj == -INFINITY) ? 0.f : ex2(mj - M);
                                    lt += f * __ldcg(a + 1);
                                    ot += f * __ldcg(a + 2 + d);
                                }
                                ll_store(p.ll_o + (size_t)h * D + d, to, ot / lt);
                            }
                            if (threadIdx.x == 0) p.attn_count[l * p.HKV + g] = 0u;
                        }
                    }
                    consumer_sync();
                    if (tr) trace_mark(p, l * 10 + 3);
                }
                continue;
            }
            // ---- a matrix phase: input vector (RMS-normalised where a gain is given) -> rows
            const unsigned long long* in_ll = p.ll_x;
            const bf16_t* in_row = nullptr;
            const bf16_t* gain = nullptr;
            int n_in = p.H, rows, per, K = p.H, group = 8;
            uint32_t in_tag = 0;
            bool glu = false;
            PhaseOut o{EMIT_LL, nullptr, 0u, nullptr, 0};
            if (e == 0) {          // QKV rows, input rms_norm(x) * g_in
                in_row = l == 0 ? erow : nullptr;
                in_tag = l == 0 ? 0u : tag(l - 1, PH_X2);
                gain = Lw->g_in;
                rows = P.q1 - P.q0; per = P.rps_h;
                o.ll = p.ll_qkv + P.q0; o.tag = tag(l, PH_QKV);
            } else if (e == 2) {   // o_proj rows + residual, input: attention output
                in_ll = p.ll_o; n_in = HQD; in_tag = tag(l, PH_O);
                rows = P.x1 - P.x0; per = P.rps_o; K = HQD;
                o.kind = EMIT_RESID; o.ll = p.ll_x + P.x0; o.tag = tag(l, PH_X1);
            } else if (e == 3) {   // gate_up pairs + SwiGLU, input rms_norm(x) * g_post
                in_tag = tag(l, PH_X1); gain = Lw->g_post;
                rows = P.f1 - P.f0; per = P.pps_gu; glu = true;
                o.ll = p.ll_h + P.f0; o.tag = tag(l, PH_H);
            } else if (e == 4) {   // down_proj rows + residual, input: h
                in_ll = p.ll_h; n_in = p.F; in_tag = tag(l, PH_H);
                rows = P.x1 - P.x0; per = P.rps_f; K = p.F;
                o.kind = EMIT_RESID; o.ll = p.ll_x + P.x0; o.tag = tag(l, PH_X2);
            } else {               // tied lm_head rows + argmax, input rms_norm(x) * final_norm
                in_tag = tag(p.NL - 1, PH_X2); gain = p.final_norm;
                rows = P.v1 - P.v0; per = P.rps_h; group = 3;   // bandwidth-bound: hand slots back sooner
                o.kind = EMIT_LOGITS; o.logits = p.logits + P.v0; o.row0 = P.v0;
            }
            if (rows > 0) {
                const float r = prep_input(S, p, in_ll, in_row, n_in, in_tag, gain, xs, par);
                if (tr) trace_mark(p, e == PH_PER_LAYER ? 10 * p.NL + 1 : l * 10 + 2 * e);
                gemv_phase(ring, S, p, glu, rows, per, K, xs, r, group, o, best, besti, kpar);
                if (tr && e != PH_PER_LAYER) trace_mark(p, l * 10 + 2 * e + 1);
            }
        }
        if (tr) trace_mark(p, 10 * p.NL + 2);
        // each thread holds the best of the logits it emitted: reduce over the warp, the CTA, then the grid
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, besti, o);
            if (am_better(ov, oi, best, besti)) {
                best = ov;
                besti = oi;
            }
        }
        float* bv = S.red + 16;
        int* bi = reinterpret_cast<int*>(S.red + 32);
        if (lane == 0) {
            bv[warp] = best;
            bi[warp] = besti;
        }
        consumer_sync();
        if (warp == 0) {
            // lane 0 publishes this CTA's best and takes a ticket; the last CTA's warp 0 reads
            // the grid's partials 32 at a time (the loads overlap) and reduces them
            unsigned int tk = 0;
            if (lane == 0) {
                float b = bv[0];
                int ib = bi[0];
                for (int w = 1; w < NCW; ++w)
                    if (am_better(bv[w], bi[w], b, ib)) { b = bv[w]; ib = bi[w]; }
                p.am_part[c].v = b;
                p.am_part[c].i = ib;
                __threadfence();
                tk = atomicAdd(p.am_count, 1u);
            }
            tk = __shfl_sync(0xffffffffu, tk, 0);
            if (tk == (unsigned int)nc - 1) {
                __threadfence();
                float b = -INFINITY;
                int ib = 0x7fffffff;
                for (int j = lane; j < nc; j += 32) {
                    const float v = __ldcg(&p.am_part[j].v);
                    const int i = __ldcg(&p.am_part[j].i);
                    if (am_better(v, i, b, ib)) { b = v; ib = i; }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, b, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, ib, o);
                    if (am_better(ov, oi, b, ib)) { b = ov; ib = oi; }
                }
                if (lane == 0) {
                    if (volatile_load(p.err) == 0) {
                        *p.argmax = (ib == 0x7fffffff) ? 0 : ib;
                        *p.pos_out = p.pos + 1;
                    }
                    *p.am_count = 0u;
                }
            }
        }
        if (threadIdx.x == 0) {
            trace_mark(p, 10 * p.NL + 3);
            if (p.trace) {
                p.trace[(size_t)blockIdx.x * (11 * p.NL + 8) + 11 * p.NL + 5] = reinterpret_cast<unsigned long long*>(S.flags + 4)[0];
                p.trace[(size_t)blockIdx.x * (11 * p.NL + 8) + 11 * p.NL + 6] = reinterpret_cast<unsigned long long*>(S.flags + 4)[1];
            }
        }
    }
    __syncthreads();
    // After an error, wait (bounded) for this CTA's copies still in flight before exiting.
    if (threadIdx.x == 0 && reinterpret_cast<volatile int*>(S.flags)[F_ABORT]) {
        const int issued = reinterpret_cast<volatile int*>(S.flags)[F_ISSUED];
        const int first = max(0, issued - p.nslot);
        for (int st = first; st < issued; ++st) {
            const uint32_t slot = (uint32_t)st % (uint32_t)p.nslot, round = (uint32_t)st / (uint32_t)p.nslot;
            bool done = false;
            for (uint32_t it = 0; it < SPIN_LIMIT && !done; ++it) {
                done = mbar_try_wait(&S.full[slot], round & 1u);
                if (!done) __nanosleep(128);
            }
            if (!done) atomicCAS(p.err, 0, ERR_DRAIN);
        }
    }
    __syncthreads();
}

using KernelFn = void (*)(const DecodeParams);

KernelFn pick_kernel(int D, int G) {
    if (D == 128 && G == 1) return decode_persistent_kernel<128, 1>;
    if (D == 128 && G == 2) return decode_persistent_kernel<128, 2>;
    if (D == 128 && G == 4) return decode_persistent_kernel<128, 4>;
    if (D == 128 && G == 8) return decode_persistent_kernel<128, 8>;
    if (D == 64 && G == 2) return decode_persistent_kernel<64, 2>;
    if (D == 32 && G == 2) return decode_persistent_kernel<32, 2>;
    return nullptr;
}

}  // namespace

cudaError_t decode_persistent_plan(const Shape& sh, int device, DecodeLaunch* out) {
    *out = DecodeLaunch{};
    const int G = sh.HQ / sh.HKV;
    const int kmax_in = sh.H > sh.HQ * sh.D ? (sh.H > sh.F ? sh.H : sh.F) : (sh.HQ * sh.D > sh.F ? sh.HQ * sh.D : sh.F);
    KernelFn fn = pick_kernel(sh.D, G);
    if (!fn) return cudaErrorNotSupported;
    // a tagged vector is fetched by at most MAX_PR pairs per consumer thread
    if (kmax_in > 2 * MAX_PR * NCT || (G + 2) * sh.D > 2 * MAX_PR * NCT) return cudaErrorNotSupported;
    // every matrix row and every GU pair must fit one ring slot
    if ((size_t)sh.H * 4 > SLOT || (size_t)sh.HQ * sh.D * 2 > SLOT || (size_t)sh.F * 2 > SLOT) return cudaErrorNotSupported;
    int sms = 0, max_smem = 0, coop = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    if (e != cudaSuccess) return e;
    if (!coop) return cudaErrorNotSupported;
    if (sms < sh.HKV) return cudaErrorNotSupported;   // at most one attention unit per CTA
    const int kmax = kmax_in > (G + 2) * sh.D ? kmax_in : (G + 2) * sh.D;
    const int xown_max = (sh.H + sms - 1) / sms + 1;
    const int att = NCW * G * (sh.D + 2);
    const size_t fixed = make_layout(0, kmax, xown_max, att).total + 16 * 64;   // slack for per-slot barriers
    if ((size_t)max_smem < fixed + 2 * SLOT) return cudaErrorNotSupported;
    int nslot = (int)(((size_t)max_smem - fixed) / SLOT);
    if (nslot > 16) nslot = 16;
    const size_t smem = make_layout(nslot, kmax, xown_max, att).total;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    out->grid = sms;
    out->smem = (int)smem;
    out->nslot = nslot;
    out->threads = NT;
    out->max_chunks = sms / sh.HKV > 0 ? sms / sh.HKV : 1;
    out->fn = reinterpret_cast<const void*>(fn);
    return cudaSuccess;
}

void decode_persistent_chunks(const DecodeLaunch& cfg, int L, int keys, int* n_chunks, int* chunk) {
    // about `keys` keys per attention unit, at most one unit per CTA.  Default (keys = 0):
    // one unit up to 160 keys (a split costs a merge of ~1 us per layer), else ~64 keys per
    // unit (measured on GB300 at KV length 416-543: 256 keys 0.754, 128 keys 0.705, 64 keys
    // 0.684, 32 keys 0.735 ms/token; at length <= 128 one unit beats two by 4%)
    // The default rounds a split unit up to whole 64-position ring stages (at KV length ~4100,
    // 17 units of 256 keys measured 4% faster than 19 units of 232).
    int n;
    if (keys > 0) n = (L + keys - 1) / keys;
    else n = L <= 160 ? 1 : (L + 63) / 64;
    if (n > cfg.max_chunks) n = cfg.max_chunks;
    if (n < 1) n = 1;
    int ch = (L + n - 1) / n;
    const int align = (keys == 0 && n > 1) ? 64 : 8;
    ch = (ch + align - 1) / align * align;
    n = (L + ch - 1) / ch;
    *n_chunks = n;
    *chunk = ch;
}

cudaError_t launch_decode_persistent(const DecodeParams& p, const DecodeLaunch& cfg, cudaStream_t s) {
    (void)cudaGetLastError();
    DecodeParams q = p;
    q.nslot = cfg.nslot;
    void* args[] = {&q};
    return cudaLaunchCooperativeKernel(cfg.fn, dim3(cfg.grid), dim3(cfg.threads), args, (size_t)cfg.smem, s);
}

}  // namespace qdec
