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
//  * Warps 0..NCW-1 are consumers: GEMV rows from shared memory with the input vector
//    in registers (fp32), attention over the streamed K/V chunk, lm_head rows + argmax.
//  * Phases exchange vectors through global memory as 64-bit words {tag, fp32 value}
//    written with one relaxed 64-bit store; a reader polls the words themselves until
//    every tag equals the phase's tag, so a hand-off costs one L2 round trip and there
//    are no grid barriers.  Each phase's writers read the whole output of the previous
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
constexpr int MAX_EL = (3072 + NCT - 1) / NCT;   // tagged elements per consumer thread (n <= 3072)
constexpr uint32_t SPIN_FAST = 256;       // tagged-vector polls before backing off with nanosleep
constexpr uint32_t SPIN_LIMIT = 1u << 21; // polls (each ~0.3-1 us) before a wait gives up: about a second
enum { PH_QKV = 0, PH_O = 1, PH_X1 = 2, PH_H = 3, PH_X2 = 4, PH_PER_LAYER = 5 };
enum { ERR_LL = 1, ERR_FULL = 2, ERR_EMPTY = 3, ERR_DRAIN = 4, ERR_PEER = 5 };
enum { F_ABORT = 0, F_ISSUED = 1 };

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t ring, full, empty, xbuf, xown, att, red, flags, total;
};

__host__ __device__ inline Layout make_layout(int nslot, int kmax, int xown_max, int att_floats) {
    Layout L;
    size_t o = 0;
    L.ring = o;  o += (size_t)nslot * SLOT;
    L.full = o;  o += (size_t)nslot * 8;
    L.empty = o; o += (size_t)nslot * 8;
    o = align_up(o, 16); L.xbuf = o; o += (size_t)kmax * 2 * 4;   // double-buffered
    o = align_up(o, 16); L.xown = o; o += (size_t)xown_max * 4;
    o = align_up(o, 16); L.att = o;  o += (size_t)att_floats * 4;
    o = align_up(o, 16); L.red = o;  o += 64 * 4;
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
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

__device__ __forceinline__ void ll_store(unsigned long long* p, uint32_t tag, float v) {
    const unsigned long long w = ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ll_load(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ int volatile_load(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

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
    int* flags;
    int nslot;
    int kmax;      // floats per xbuf buffer (xbuf holds two)
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
    for (uint32_t it = 0; it < SPIN_LIMIT; ++it) {
        if (mbar_try_wait(bar, parity)) return true;   // suspends the thread for a while when not ready
        if ((it & 1023) == 1023 && should_abort(S, p, (it & 16383) == 16383)) return false;
    }
    raise_error(S, p, code);
    return false;
}

// All consumer threads: dst[i] = value of ll[i] once its tag equals `tag`, i < n.
// Returns the thread's partial sum of squares through *ss.  n <= MAX_EL * NCT.
__device__ inline bool ll_fetch(const Ctx& S, const DecodeParams& p, const unsigned long long* ll, int n,
                                uint32_t tag, float* dst, float* ss) {
    const int ct = threadIdx.x;
    if (reinterpret_cast<volatile int*>(S.flags)[F_ABORT]) return false;
    const long long t0 = (p.trace && ct == 0) ? clock64() : 0;
    uint32_t pending = 0;
#pragma unroll
    for (int k = 0; k < MAX_EL; ++k)
        if (ct + k * NCT < n) pending |= 1u << k;
    float acc = 0.f;
    for (uint32_t it = 0; pending; ++it) {
#pragma unroll
        for (int k = 0; k < MAX_EL; ++k) {
            if (pending & (1u << k)) {
                const int i = ct + k * NCT;
                const unsigned long long w = ll_load(ll + i);
                if ((uint32_t)(w >> 32) == tag) {
                    const float v = __uint_as_float((uint32_t)w);
                    dst[i] = v;
                    acc = fmaf(v, v, acc);
                    pending &= ~(1u << k);
                }
            }
        }
        if (!pending) break;
        if (it >= SPIN_LIMIT) {
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

// Input vector of a GEMV phase, optionally RMS-normalised with `gain`, into each warp's
// registers xr (lane holds elements lane*8 + 256 i + j).  Source: `row` (bf16, the
// embedding row) when non-null, else the tagged vector `ll`.  The staging buffer and the
// reduction slots alternate between calls (`par`), so no trailing barrier is needed.
template <int NI>
__device__ inline void prep_input(const Ctx& S, const DecodeParams& p, const unsigned long long* ll,
                                  const bf16_t* row, int n, uint32_t tag, const bf16_t* gain, float (&xr)[NI][8],
                                  int& par) {
    float* xb = S.xbuf + (size_t)par * S.kmax;
    float* rd = S.red + par * 8;
    par ^= 1;
    const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
    uint4 gw[NI];   // gains in the register layout, loaded before the wait
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int k = lane * 8 + 256 * i;
        gw[i] = (gain && k < n) ? *reinterpret_cast<const uint4*>(gain + k) : make_uint4(0, 0, 0, 0);
    }
    float ss = 0.f;
    if (row) {
        for (int i = ct; i < n; i += NCT) {
            const float v = bf1(row[i]);
            xb[i] = v;
            ss = fmaf(v, v, ss);
        }
    } else {
        ll_fetch(S, p, ll, n, tag, xb, &ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) rd[warp] = ss;
    consumer_sync();
    float r = 1.f;
    if (gain) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) tot += rd[w];
        r = rsqrtf(tot / (float)n + p.eps);
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int k = lane * 8 + 256 * i;   // n is a multiple of 8: a lane's 8 values are all in or all out
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (k < n) {
            a = *reinterpret_cast<const float4*>(xb + k);
            b = *reinterpret_cast<const float4*>(xb + k + 4);
        }
        if (gain) {
            const uint4 g = gw[i];
            a.x *= r * bf_lo(g.x); a.y *= r * bf_hi(g.x); a.z *= r * bf_lo(g.y); a.w *= r * bf_hi(g.y);
            b.x *= r * bf_lo(g.z); b.y *= r * bf_hi(g.z); b.z *= r * bf_lo(g.w); b.w *= r * bf_hi(g.w);
        }
        xr[i][0] = a.x; xr[i][1] = a.y; xr[i][2] = a.z; xr[i][3] = a.w;
        xr[i][4] = b.x; xr[i][5] = b.y; xr[i][6] = b.z; xr[i][7] = b.w;
    }
}

// Consumer view of the ring: every consumer warp walks the same stage sequence.
struct Ring {
    uint32_t stage = 0;   // next stage to consume
    __device__ const char* slot_ptr(const Ctx& S, uint32_t st) const {
        return S.ring + (size_t)(st % (uint32_t)S.nslot) * SLOT;
    }
    // Waits for stage st's data; after an abort it returns without waiting (the contents
    // are then garbage, and nothing computed from them is published).
    __device__ void wait_stage(const Ctx& S, const DecodeParams& p, uint32_t st) const {
        const uint32_t slot = st % (uint32_t)S.nslot, round = st / (uint32_t)S.nslot;
        const long long t0 = (p.trace && threadIdx.x == 0) ? clock64() : 0;
        wait_bar(S, p, &S.full[slot], round & 1u, ERR_FULL);
        if (p.trace && threadIdx.x == 0) trace_add(S.flags, 0, (unsigned long long)(clock64() - t0));
    }
    __device__ const char* acquire(const Ctx& S, const DecodeParams& p) {
        wait_stage(S, p, stage);
        return slot_ptr(S, stage);
    }
    // After an abort a slot is never handed back: its copy may still be in flight, and the
    // producer must not reuse it (the final drain waits for it instead).
    __device__ void release(const Ctx& S) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0 && !reinterpret_cast<volatile int*>(S.flags)[F_ABORT])
            mbar_arrive(&S.empty[stage % (uint32_t)S.nslot]);
        ++stage;
    }
};

// Rows [0, rows) of one matrix phase, spread over consecutive ring stages of `per` rows
// (GLU: `per` gate/up pairs; a stage with n pairs holds n gate rows, then the n matching
// up rows).  Up to 8 stages are acquired together; each warp then computes R rows at a
// time with independent accumulators, so the dot products and the shuffle reductions of
// several rows overlap.  emit(row, value) runs on lane 0; value is silu(gate) * up for GLU.
// NK = number of 256-column chunks (K = 256 NK when EXACT).
template <int NK, bool EXACT, bool GLU, int R, int NI, typename Emit>
__device__ inline void phase_rows(Ring& ring, const Ctx& S, const DecodeParams& p, int rows, int per, int K,
                                  const float (&xr)[NI][8], Emit emit, int group) {
    static_assert(NK <= NI, "register vector too short");
    constexpr int NA = GLU ? 2 : 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int maxg = min(group, S.nslot - 1);
    const int nst = (rows + per - 1) / per;
    for (int s0 = 0; s0 < nst; s0 += maxg) {
        const int g = min(maxg, nst - s0);
        const uint32_t st0 = ring.stage;
        for (int s = 0; s < g; ++s) ring.wait_stage(S, p, st0 + s);
        const int r0 = s0 * per, r1 = min(rows, (s0 + g) * per);
        for (int base = r0 + warp; base < r1; base += NCW * R) {
            const uint4* w[R][NA];
            bool valid[R];
#pragma unroll
            for (int j = 0; j < R; ++j) {
                // rows past the end re-read row `base` (always valid): no branches in the dot products
                const int rr = base + NCW * j;
                valid[j] = rr < r1;
                const int r = valid[j] ? rr : base;
                const int st = r / per, off = r - st * per;
                const int ns = min(per, rows - st * per);
                const char* sp = ring.slot_ptr(S, st0 + (uint32_t)(st - s0));
                w[j][0] = reinterpret_cast<const uint4*>(sp + (size_t)off * K * 2);
                if (GLU) w[j][NA - 1] = reinterpret_cast<const uint4*>(sp + (size_t)(ns + off) * K * 2);
            }
            float acc[R][NA];
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int a = 0; a < NA; ++a) acc[j][a] = 0.f;
#pragma unroll
            for (int i = 0; i < NK; ++i) {
                const int k = lane * 8 + 256 * i;
                if (EXACT || k < K) {
#pragma unroll
                    for (int j = 0; j < R; ++j)
#pragma unroll
                        for (int a = 0; a < NA; ++a) acc[j][a] += dot8(w[j][a][k >> 3], xr[i]);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int j = 0; j < R; ++j)
#pragma unroll
                    for (int a = 0; a < NA; ++a) acc[j][a] += __shfl_xor_sync(0xffffffffu, acc[j][a], o);
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < R; ++j)
                    if (valid[j]) emit(base + NCW * j, GLU ? silu(acc[j][0]) * acc[j][NA - 1] : acc[j][0]);
            }
        }
        for (int s = 0; s < g; ++s) ring.release(S);
    }
}

template <int NK, bool EXACT, bool GLU, int NI, typename Emit>
__device__ inline void phase_rows_r(Ring& ring, const Ctx& S, const DecodeParams& p, int rows, int per, int K,
                                    const float (&xr)[NI][8], Emit emit, int group) {
    // several rows per warp pass when a stage group has them (independent accumulators
    // overlap), fewer otherwise (clamped rows are wasted work)
    const int rows_in_group = min(rows, min(group, S.nslot - 1) * per);
    if (rows_in_group >= 3 * NCW) phase_rows<NK, EXACT, GLU, GLU ? 2 : 4>(ring, S, p, rows, per, K, xr, emit, group);
    else if (rows_in_group >= 2 * NCW) phase_rows<NK, EXACT, GLU, 2>(ring, S, p, rows, per, K, xr, emit, group);
    else phase_rows<NK, EXACT, GLU, 1>(ring, S, p, rows, per, K, xr, emit, group);
}

// `group`: stages acquired together (8 for latency-bound phases: one wait, then all the
// rows; 3 for the bandwidth-bound lm_head, which hands slots back as it goes).
template <bool GLU, int NI, typename Emit>
__device__ inline void phase_any(Ring& ring, const Ctx& S, const DecodeParams& p, int rows, int per, int K,
                                 const float (&xr)[NI][8], Emit emit, int group = 8) {
    if constexpr (NI >= 12) {
        if (K == 3072) { phase_rows_r<12, true, GLU>(ring, S, p, rows, per, K, xr, emit, group); return; }
    }
    if constexpr (NI >= 8) {
        if (K == 2048) { phase_rows_r<8, true, GLU>(ring, S, p, rows, per, K, xr, emit, group); return; }
    }
    if constexpr (NI >= 4) {
        if (K == 1024) { phase_rows_r<4, true, GLU>(ring, S, p, rows, per, K, xr, emit, group); return; }
    }
    phase_rows_r<NI, false, GLU>(ring, S, p, rows, per, K, xr, emit, group);
}

// ------------------------------------------------------------------ the kernel
template <int D, int G, int NI>
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
    S.flags = reinterpret_cast<int*>(smem + LO.flags);
    S.nslot = p.nslot;
    S.kmax = kmax;
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
            uint32_t stage = 0;
            bool ok = true;
            auto issue = [&](const void* s0, uint32_t b0, const void* s1, uint32_t b1) {
                if (!ok) return;
                const uint32_t slot = stage % (uint32_t)S.nslot, round = stage / (uint32_t)S.nslot;
                if (!wait_bar(S, p, &S.empty[slot], (round & 1u) ^ 1u, ERR_EMPTY) ||
                    reinterpret_cast<volatile int*>(S.flags)[F_ABORT]) {
                    ok = false;
                    return;
                }
                mbar_expect_tx(&S.full[slot], b0 + b1);
                char* dst = S.ring + (size_t)slot * SLOT;
                tma_load_1d(dst, s0, b0, &S.full[slot]);
                if (b1) tma_load_1d(dst + b0, s1, b1, &S.full[slot]);
                ++stage;
            };
            for (int l = 0; l < p.NL && ok; ++l) {
                const DecodeLayer Lw = p.layers[l];   // by value: registers survive the asm memory clobbers
                for (int r = P.q0; r < P.q1; r += P.rps_h) {
                    const int n = min(P.rps_h, P.q1 - r);
                    issue(Lw.wqkv + (size_t)r * p.H, (uint32_t)n * p.H * 2, nullptr, 0);
                }
                for (int q = P.c0; q < P.old_end; q += P.pps_kv) {
                    const int n = min(P.pps_kv, P.old_end - q);
                    const size_t off = ((size_t)P.ug * p.max_seq + q) * D;
                    issue(Lw.kc + off, (uint32_t)n * D * 2, nullptr, 0);
                    issue(Lw.vc + off, (uint32_t)n * D * 2, nullptr, 0);
                }
                for (int r = P.x0; r < P.x1; r += P.rps_o) {
                    const int n = min(P.rps_o, P.x1 - r);
                    issue(Lw.wo + (size_t)r * HQD, (uint32_t)n * HQD * 2, nullptr, 0);
                }
                for (int j = P.f0; j < P.f1; j += P.pps_gu) {
                    const int n = min(P.pps_gu, P.f1 - j);
                    issue(Lw.wgu + (size_t)j * p.H, (uint32_t)n * p.H * 2, Lw.wgu + (size_t)(p.F + j) * p.H,
                          (uint32_t)n * p.H * 2);
                }
                for (int r = P.x0; r < P.x1; r += P.rps_f) {
                    const int n = min(P.rps_f, P.x1 - r);
                    issue(Lw.wd + (size_t)r * p.F, (uint32_t)n * p.F * 2, nullptr, 0);
                }
                trace_mark(p, 10 * p.NL + 4 + l);
            }
            for (int r = P.v0; r < P.v1 && ok; r += P.rps_h) {
                const int n = min(P.rps_h, P.v1 - r);
                issue(p.embed + (size_t)r * p.H, (uint32_t)n * p.H * 2, nullptr, 0);
            }
            reinterpret_cast<volatile int*>(S.flags)[F_ISSUED] = (int)stage;
        }
    } else {
        // ------------------------------------------------------------ consumers
        // Control flow below depends only on the plan, never on errors: every consumer
        // thread executes the same barriers whatever happens.
        Ring ring;
        float xr[NI][8];
        int par = 0;   // alternates the staging buffer between input preparations
        if (c == 0 && threadIdx.x == 0) p.history[p.pos] = token;
        for (int r = P.x0 + threadIdx.x; r < P.x1; r += NCT) S.xown[r - P.x0] = bf1(erow[r]);
        consumer_sync();
        const bool tr = p.trace && threadIdx.x == 0;
        if (tr) trace_mark(p, 10 * p.NL + 0);

        for (int l = 0; l < p.NL; ++l) {
            const DecodeLayer Lw = p.layers[l];   // by value: registers survive the asm memory clobbers
            // ---- P1: QKV rows (input: rms_norm(x) * g_in) -> tagged qkv
            if (P.q1 > P.q0) {
                prep_input<NI>(S, p, p.ll_x, l == 0 ? erow : nullptr, p.H, l == 0 ? 0u : tag(l - 1, PH_X2),
                               Lw.g_in, xr, par);
                if (tr) trace_mark(p, l * 10 + 0);
                const uint32_t t = tag(l, PH_QKV);
                unsigned long long* dst = p.ll_qkv + P.q0;
                phase_any<false>(ring, S, p, P.q1 - P.q0, P.rps_h, p.H, xr,
                                 [&](int i, float v) { ll_store(dst + i, t, v); });
                if (tr) trace_mark(p, l * 10 + 1);
            }
            // ---- P2: attention unit (kv head ug, key chunk [c0, c1))
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
                    const bf16_t* gn0 = warp < G ? Lw.g_q : Lw.g_k;
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
                ll_fetch(S, p, p.ll_qkv + (size_t)g * G * D, G * D, tq, xa, &ss);
                ll_fetch(S, p, p.ll_qkv + HQD + (size_t)g * D, D, tq, xa + G * D, &ss);
                ll_fetch(S, p, p.ll_qkv + HQD + (size_t)(p.HKV + g) * D, D, tq, xa + (G + 1) * D, &ss);
                consumer_sync();
                if (tr) trace_mark(p, l * 10 + 2);
                // per-head RMSNorm + NeoX RoPE on the G q heads and the k head; bf16 rounding of k, v
                for (int hh = warp; hh <= G; hh += NCW) {
                    float* hv = xa + hh * D;
                    if (hh != warp) {   // a second head for this warp (G + 1 > NCW): load its gains now
                        const bf16_t* gn1 = hh < G ? Lw.g_q : Lw.g_k;
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
                        Lw.kc[((size_t)g * p.max_seq + p.pos) * D + d] = f2bf(xa[G * D + d]);
                        Lw.vc[((size_t)g * p.max_seq + p.pos) * D + d] = f2bf(xa[(G + 1) * D + d]);
                    }
                }
                const float scale = rsqrtf((float)D);
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
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int k = 0; k < KPW; ++k)
#pragma unroll
                            for (int gi = 0; gi < G; ++gi) s[k][gi] += __shfl_xor_sync(0xffffffffu, s[k][gi], o);
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
                            const float corr = expf(m[gi] - mn);   // 0 when m was -inf
                            lsum[gi] *= corr;
#pragma unroll
                            for (int e = 0; e < EPL; ++e) o[gi][e] *= corr;
                            m[gi] = mn;
#pragma unroll
                            for (int k = 0; k < KPW; ++k) {
                                s[k][gi] = (s[k][gi] == -INFINITY) ? 0.f : expf(s[k][gi] - mn);
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
                        const float corr = expf(m[gi] - mn);
                        const float pr = expf(sc - mn);
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
                        const float f = (a[0] == -INFINITY) ? 0.f : expf(a[0] - M);
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
                                const float f = (mj == -INFINITY) ? 0.f : expf(mj - M);
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
            // ---- P3: o_proj rows + residual (input: attention output o)
            if (P.x1 > P.x0) {
                prep_input<NI>(S, p, p.ll_o, nullptr, HQD, tag(l, PH_O), nullptr, xr, par);
                if (tr) trace_mark(p, l * 10 + 4);
                const uint32_t t = tag(l, PH_X1);
                phase_any<false>(ring, S, p, P.x1 - P.x0, P.rps_o, HQD, xr, [&](int i, float v) {
                    const float nx = S.xown[i] + v;
                    S.xown[i] = nx;
                    ll_store(p.ll_x + P.x0 + i, t, nx);
                });
                if (tr) trace_mark(p, l * 10 + 5);
            }
            // ---- P4: gate_up pairs + SwiGLU (input: rms_norm(x) * g_post) -> tagged h
            if (P.f1 > P.f0) {
                prep_input<NI>(S, p, p.ll_x, nullptr, p.H, tag(l, PH_X1), Lw.g_post, xr, par);
                if (tr) trace_mark(p, l * 10 + 6);
                const uint32_t t = tag(l, PH_H);
                unsigned long long* dst = p.ll_h + P.f0;
                phase_any<true>(ring, S, p, P.f1 - P.f0, P.pps_gu, p.H, xr,
                                [&](int i, float v) { ll_store(dst + i, t, v); });
                if (tr) trace_mark(p, l * 10 + 7);
            }
            // ---- P5: down_proj rows + residual (input: h)
            if (P.x1 > P.x0) {
                prep_input<NI>(S, p, p.ll_h, nullptr, p.F, tag(l, PH_H), nullptr, xr, par);
                if (tr) trace_mark(p, l * 10 + 8);
                const uint32_t t = tag(l, PH_X2);
                phase_any<false>(ring, S, p, P.x1 - P.x0, P.rps_f, p.F, xr, [&](int i, float v) {
                    const float nx = S.xown[i] + v;
                    S.xown[i] = nx;
                    ll_store(p.ll_x + P.x0 + i, t, nx);
                });
                if (tr) trace_mark(p, l * 10 + 9);
            }
        }
        // ---- final RMSNorm + tied lm_head + argmax
        float best = -INFINITY;
        int besti = 0x7fffffff;
        if (P.v1 > P.v0) {
            prep_input<NI>(S, p, p.ll_x, nullptr, p.H, tag(p.NL - 1, PH_X2), p.final_norm, xr, par);
            if (tr) trace_mark(p, 10 * p.NL + 1);
            phase_any<false>(ring, S, p, P.v1 - P.v0, P.rps_h, p.H, xr, [&](int i, float v) {
                const int row = P.v0 + i;
                p.logits[row] = v;
                if (am_better(v, row, best, besti)) {
                    best = v;
                    besti = row;
                }
            }, 3);
        }
        if (tr) trace_mark(p, 10 * p.NL + 2);
        // lane 0 of each warp holds its best; reduce over the CTA, then over the grid
        float* bv = S.red + 16;
        int* bi = reinterpret_cast<int*>(S.red + 32);
        if (lane == 0) {
            bv[warp] = best;
            bi[warp] = besti;
        }
        consumer_sync();
        if (threadIdx.x == 0) {
            float b = bv[0];
            int ib = bi[0];
            for (int w = 1; w < NCW; ++w)
                if (am_better(bv[w], bi[w], b, ib)) { b = bv[w]; ib = bi[w]; }
            p.am_part[c].v = b;
            p.am_part[c].i = ib;
            __threadfence();
            const unsigned int tk = atomicAdd(p.am_count, 1u);
            if (tk == (unsigned int)nc - 1) {
                __threadfence();
                for (int j = 0; j < nc; ++j) {
                    const float v = __ldcg(&p.am_part[j].v);
                    const int i = __ldcg(&p.am_part[j].i);
                    if (am_better(v, i, b, ib)) { b = v; ib = i; }
                }
                if (volatile_load(p.err) == 0) {
                    *p.argmax = (ib == 0x7fffffff) ? 0 : ib;
                    *p.pos_out = p.pos + 1;
                }
                *p.am_count = 0u;
            }
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

KernelFn pick_kernel(int D, int G, int ni) {
    if (ni <= 4) {
        if (D == 32 && G == 2) return decode_persistent_kernel<32, 2, 4>;
        if (D == 64 && G == 2) return decode_persistent_kernel<64, 2, 4>;
        if (D == 128 && G == 2) return decode_persistent_kernel<128, 2, 4>;
    }
    if (ni <= 12) {
        if (D == 128 && G == 1) return decode_persistent_kernel<128, 1, 12>;
        if (D == 128 && G == 2) return decode_persistent_kernel<128, 2, 12>;
        if (D == 128 && G == 4) return decode_persistent_kernel<128, 4, 12>;
        if (D == 128 && G == 8) return decode_persistent_kernel<128, 8, 12>;
        if (D == 64 && G == 2) return decode_persistent_kernel<64, 2, 12>;
        if (D == 32 && G == 2) return decode_persistent_kernel<32, 2, 12>;
    }
    return nullptr;
}

}  // namespace

cudaError_t decode_persistent_plan(const Shape& sh, int device, DecodeLaunch* out) {
    *out = DecodeLaunch{};
    const int G = sh.HQ / sh.HKV;
    const int kmax_in = sh.H > sh.HQ * sh.D ? (sh.H > sh.F ? sh.H : sh.F) : (sh.HQ * sh.D > sh.F ? sh.HQ * sh.D : sh.F);
    const int ni = (kmax_in + 255) / 256;
    KernelFn fn = pick_kernel(sh.D, G, ni);
    if (!fn) return cudaErrorNotSupported;
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

void decode_persistent_chunks(const DecodeLaunch& cfg, int L, int* n_chunks, int* chunk) {
    // about 256 keys per attention unit, at most one unit per CTA
    int n = (L + 255) / 256;
    if (n > cfg.max_chunks) n = cfg.max_chunks;
    if (n < 1) n = 1;
    int ch = (L + n - 1) / n;
    ch = (ch + 7) / 8 * 8;
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
