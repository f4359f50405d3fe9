// Paged decode attention for sm_103a.
//
// What it computes (the block-indexed attention of the PagedAttention paper,
// section 4.1, as printed on the zhaifeiyue.github.io detail page, and the
// ricepunchb garden's section 3.3: per-block scores at kernel level, then a
// reduction that completes the softmax):
//
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K[t]) V[t],  t < ctx[s],
//   K[t] = k_cache[table[s][t / B]][h][t % B]  (V likewise).
//
// Design (GB300-first; the pages' A100 kernel notes are prior art only):
//   * The batch's work is the ordered space of steps (s, h, j): step j of
//     (sequence s, head h) covers SUB consecutive tokens of one physical
//     block (SUB = 16 for head_dim 128), i.e. one contiguous K chunk and one
//     contiguous V chunk of at most 4 KiB each in the [block][head][B][D]
//     pools.  A persistent grid (a few CTAs per SM) splits that space into
//     equal contiguous ranges, so every CTA moves the same number of bytes
//     whatever the mix of context lengths (split-K with balanced splits), or
//     into fixed-length chunks when a split length is requested.
//   * Per CTA: one producer warp walks its range, reads block-table entries
//     32 at a time (and prefetches the next 32), and issues 1-D TMA bulk
//     copies (cp.async.bulk) of each step's K and V chunk into a ring of
//     shared-memory stages guarded by mbarriers (full: transaction bytes;
//     empty: released by the consuming warp).  No multicast: every CTA
//     fetches its own blocks.
//   * Two consumer warps take the steps round-robin (small CTAs: 96 threads
//     and a 32 KiB ring, five resident per SM, measured best for short and
//     mixed context lengths; the count and ring size are compile-time knobs).
//     Per step a warp reads
//     the K chunk from shared memory with conflict-free 16-byte loads (lane l
//     reads bytes [16 l, 16 l + 16) of every 512-byte row), forms q . k
//     partial dot products in fp32, and finishes them with a reduce-scatter
//     butterfly (8 shuffles for 16 tokens) that leaves each lane holding one
//     token's score.  An online softmax (running max m, running sum l, both
//     in log2 units) rescales the fp32 accumulator, and the V chunk is
//     accumulated with the per-token weights.  Masked positions (>= ctx) are
//     excluded by selection, never by multiplying, so unwritten pool memory
//     (any bit pattern) cannot leak into the result.
//   * At the end of each piece (a (s, h) run inside one chunk) the warps'
//     states are merged through shared memory.  A piece that covers its whole
//     (s, h) writes the normalised output; otherwise it writes (m, l, acc) to
//     workspace slot s*H + h + chunk, and the merge kernel combines the
//     slots of each split (s, h) with the log-sum-exp rule.
//   * CUDA cores, not tensor cores: decode attention is a matrix-vector
//     product, about 0.5 flop per byte of K/V, bound by HBM bandwidth.
//   * One decode step in one call (kModeAppend): the newest token of every
//     sequence (position ctx - 1) comes with the call; the producer copies its
//     K and V rows from k_new / v_new into their place in the row's last stage
//     instead of the cache's slot, and the consumer warp that takes that step
//     stores them from the stage into the slot.  No other step of the call
//     reads the slot, so the write needs no ordering against the attention.
//   * Every wait is bounded.  The pipeline waits (ring stages, claimed-chunk
//     queue, the consumer warps' meeting at a piece end) give up after the
//     launch's limit (1 s unless the caller shortened it): the warp sets the
//     timeout bit of the device error word and a CTA abort flag, after which
//     every wait of the CTA gives up at once and the warps run out their
//     remaining work without computing it.  A consumer releases a ring stage
//     only once it has seen the stage's copy land, so the producer never
//     re-arms a stage whose copy is in flight, and before the producer warp
//     exits it waits (1 s bound, always) for every copy it issued, so no copy
//     lands in a CTA that has ended.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "pkv_internal.h"

namespace pkv {
namespace dec {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr uint32_t kWaitLimitIters = 1u << 26;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted in
// bytes on `bar`.  Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 2-D tiled bulk tensor copy global -> this CTA's shared memory (the map's
// swizzle applies), completion counted in bytes on `bar`.
__device__ __forceinline__ void tensor_g2s(void* dst, const CUtensorMap* map, int x, int y,
                                           uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) once more than limit_ns have passed (checked every 32
// polls), after kWaitLimitIters polls, or, when `abort` is given, once *abort
// becomes nonzero.
static __device__ __noinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                 uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it < kWaitLimitIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (abort && *abort) return false;
            if (global_ns() - t0 > limit_ns) return false;
        }
    }
    return false;
}

// Common case inline (the phase has already completed); the bounded loop only
// when it has not.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded(bar, parity, abort, limit_ns);
}

// A wait of a pipeline role gave up: record the timeout (unless another warp
// already aborted the CTA, which is the reason this one gave up) and abort.
__device__ __forceinline__ void note_timeout(volatile int* abort, int32_t* err) {
    if (!*abort) atomicOr(err, PKV_DEVERR_TIMEOUT);
    *abort = 1;
}

// Programmatic dependent launch: wait for the preceding kernel in the stream
// (no-op when launched without the dependency), or let the next one start.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ element types
template <typename T>
struct Elem;

template <>
struct Elem<__half> {
    static __device__ __forceinline__ void to_f32x8(const uint4& u, float (&f)[8]) {
        const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
    static __device__ __forceinline__ __half zero() { return __float2half_rn(0.f); }
};

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ void to_f32x8(const uint4& u, float (&f)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) {
        return __float2bfloat16_rn(x);
    }
    static __device__ __forceinline__ __nv_bfloat16 zero() { return __float2bfloat16_rn(0.f); }
};

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// ------------------------------------------------------------ configuration
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 2          // consumer warps per CTA
#endif
#ifndef PKV_DECODE_RING_BYTES
#define PKV_DECODE_RING_BYTES 32768 // shared-memory ring per CTA (4 stages of 8 KiB at D=128)
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 1       // launch-bounds hint: resident CTAs per SM
#endif


template <int D, int B>
struct Cfg {
    static constexpr int NW = PKV_DECODE_WARPS;         // consumer warps
    static constexpr int THREADS = (NW + 1) * 32;       // + one producer warp
    static constexpr int SUB = step_tokens(D);          // tokens per step
    static constexpr int SPB = B > SUB ? B / SUB : 1;   // steps per block
    static constexpr int BPS = B < SUB ? SUB / B : 1;   // blocks per step
    static constexpr int TPC = B < SUB ? B : SUB;       // tokens per bulk copy
    static constexpr int CHUNK = SUB * D * 2;           // bytes of K (or V) per step
    static constexpr int STAGE = 2 * CHUNK;
    // Step g uses stage g % NSTAGE and is consumed by warp g % NW.  NSTAGE must
    // be a multiple of NW: then the previous use of a stage (step g - NSTAGE)
    // belongs to the same warp, which has already waited for it, so a warp
    // never polls a full barrier whose previous phase is still pending (the
    // parity test would report that previous phase as complete).
    static constexpr int NSTAGE = (PKV_DECODE_RING_BYTES / STAGE) / NW * NW;
    static constexpr int NL = CHUNK / 512;              // 16-B loads per lane per chunk
    static constexpr int TPL = 256 / D;                 // tokens per 512-B row
    static constexpr int LPT = D / 8;                   // lanes per token row
    static constexpr int LOG_LPT = ilog2(LPT);
    static constexpr int LOG_NL = ilog2(NL);
    static constexpr int RS = LOG_LPT - LOG_NL;
    static constexpr int MROW = D + 4;                  // merge row: acc[D], m, l, pad
    static constexpr size_t RING = (size_t)NSTAGE * STAGE;
    static constexpr size_t BAR_OFF = RING;     // full[NSTAGE], empty[NSTAGE], pair[2]
    static constexpr size_t MERGE_OFF = BAR_OFF + 16 * (size_t)NSTAGE + 16;
    static constexpr size_t MISC_OFF = MERGE_OFF + 4 * (size_t)(2 * NW * MROW);
    // misc: the abort flag (16 B), then one scan partial per warp
    static constexpr size_t MISC_BYTES = (16 + 4 * (NW + 1) + 15) / 16 * 16;
    // claimed-chunk queue, producer -> consumers: QN entries, each a chunk id,
    // an mbarrier and the query slice of the chunk's first row.  QN > 2 NSTAGE
    // + 1 so an entry is never rewritten before every consumer warp read it.
    static constexpr int QN = 16;
    // per stage: the byte offset in the pools of the cache slot that the
    // stage's newest token (taken from the call's k_new / v_new) goes to,
    // -1 when the stage holds none (written by the producer with the copy)
    static constexpr size_t APP_OFF = MISC_OFF + MISC_BYTES;
    static constexpr size_t QBAR_OFF = APP_OFF + 8 * (size_t)NSTAGE;
    static constexpr size_t QID_OFF = QBAR_OFF + 8 * QN;
    static constexpr size_t QBUF_OFF = QID_OFF + 4 * QN;
    static constexpr size_t CTX_OFF = QBUF_OFF + (size_t)QN * D * 2;
    static_assert(NL >= 1 && NL <= LPT, "step layout");
    static_assert(NSTAGE >= NW && NSTAGE % NW == 0, "ring depth: a multiple of the warps");
    static_assert(QN > 2 * NSTAGE + 1, "claim queue depth");
    static_assert(QBAR_OFF % 8 == 0 && QBUF_OFF % 16 == 0, "claim queue alignment");
    static_assert(TPL * NL == SUB, "tokens per step");
    static_assert(B % SUB == 0 || SUB % B == 0, "steps and blocks nest");
    static_assert(BPS <= 32 && 32 % BPS == 0, "a step's blocks share one table window");
    static __host__ __device__ size_t smem(int S) {
        return CTX_OFF + 4 * (size_t)S + 4 * (size_t)(S + 1);
    }
};

// ------------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// NL partial dot products, one per 16-B load, each spread over the LPT lanes
// of a token row.  Halving exchanges on lane bits LOG_LPT-1, LOG_LPT-2, ...
// leave lane (dl = lane mod LPT) with the full dot product of load
// dl >> (LOG_LPT - LOG_NL); plain butterflies on the remaining low bits make
// the 2^RS lanes that share a load agree bit for bit.
template <int NL, int LOG_LPT>
__device__ __forceinline__ float reduce_scatter(float (&v)[NL], int dl) {
    constexpr int LOG_NL = ilog2(NL);
#pragma unroll
    for (int step = 0; step < LOG_NL; ++step) {
        const int bit = LOG_LPT - 1 - step;
        const int half = (NL >> step) >> 1;
        const bool upper = (dl >> bit) & 1;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = upper ? v[half + i] : v[i];
            const float give = upper ? v[i] : v[half + i];
            v[i] = keep + __shfl_xor_sync(kFull, give, 1 << bit);
        }
    }
    float z = v[0];
#pragma unroll
    for (int bit = LOG_LPT - LOG_NL - 1; bit >= 0; --bit) z += __shfl_xor_sync(kFull, z, 1 << bit);
    return z;
}

// ------------------------------------------------------------ the step space
struct Pos {
    int s, h, j;
};

// Largest s with H * base[s] <= x; requires x < H * base[S] (so that
// sequence s has at least one step).
__device__ __forceinline__ Pos locate(int64_t x, const int* base, int S, int H) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)H * base[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    const int ns = base[lo + 1] - base[lo];
    const int64_t r = x - (int64_t)H * base[lo];
    Pos p;
    p.s = lo;
    p.h = (int)(r / ns);
    p.j = (int)(r - (int64_t)p.h * ns);
    return p;
}

__device__ __forceinline__ void next_segment(Pos& p, const int* base, int S, int H) {
    p.j = 0;
    if (++p.h == H) {
        p.h = 0;
        do {
            ++p.s;
        } while (p.s < S && base[p.s + 1] == base[p.s]);
    }
}

// Exclusive prefix of steps per sequence: base[s] = sum_{s' < s} ceil(ctx[s'] / SUB)
// - skip[s'] (skip: the steps a group reads for the sequence, or null).
template <int SUB>
__device__ void scan_steps(const int* ctx, int* base, int S, int* scratch,
                           const int* skip = nullptr) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
    const int per = (S + nt - 1) / nt;
    const int b = min(tid * per, S), e = min(b + per, S);
    int local = 0;
    for (int i = b; i < e; ++i) local += (ctx[i] + SUB - 1) / SUB - (skip ? skip[i] : 0);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[w] = incl;
    __syncthreads();
    int run = incl - local;
    for (int i = 0; i < w; ++i) run += scratch[i];
    for (int i = b; i < e; ++i) {
        base[i] = run;
        run += (ctx[i] + SUB - 1) / SUB - (skip ? skip[i] : 0);
    }
    if (tid == nt - 1) base[S] = run;
    __syncthreads();
}

// ------------------------------------------------------------ the split
// Chunks of the step space [0, total).  Fixed split length: chunks of Ls
// steps, a contiguous run of them per CTA.  Balanced: one static chunk of Ls
// steps per CTA over [0, X), then Kd dynamic chunks of Ld steps over
// [X, total) claimed at run time.  Chunk indices grow along the step space
// (static c < G, dynamic G + k), so a piece of row (s, h) in chunk k owns
// partial slot s * H + h + k and the slots of one row are contiguous.  The
// main and the merge kernels build the same split.
struct Split {
    int64_t total, X, Ls, Ld, Kd;
    int G;
    bool fixed;
    __device__ __forceinline__ int64_t chunk(int64_t x) const {
        return x < X ? x / Ls : G + (x - X) / Ld;
    }
    __device__ __forceinline__ int64_t chunk_end(int64_t x) const {
        if (x < X) {
            const int64_t e = (x / Ls + 1) * Ls;
            return e < X ? e : X;
        }
        const int64_t e = X + ((x - X) / Ld + 1) * Ld;
        return e < total ? e : total;
    }
    __device__ __forceinline__ int64_t last_chunk() const {
        if (total == 0) return -1;
        return chunk(total - 1);
    }
};

__device__ __forceinline__ Split make_split(int64_t total, int G, int64_t L_steps,
                                            int min_chunk) {
    Split sp;
    sp.total = total;
    sp.G = G;
    if (L_steps > 0) {
        sp.fixed = true;
        sp.Ls = L_steps;
        sp.X = total;
        sp.Ld = 1;
        sp.Kd = 0;
        return sp;
    }
    sp.fixed = false;
    int64_t Ls = (total * PKV_DECODE_STATIC_EIGHTHS / 8) / G;
    if (PKV_DECODE_DYN_PER_CTA == 0) Ls = (total + G - 1) / G;
    if (Ls < min_chunk) Ls = min_chunk;
    sp.Ls = Ls;
    sp.X = (int64_t)G * Ls < total ? (int64_t)G * Ls : total;
    const int64_t rem = total - sp.X;
    if (rem > 0) {
        int64_t kd = (int64_t)PKV_DECODE_DYN_PER_CTA * G;
        if (kd > rem) kd = rem;
        if (kd < 1) kd = 1;
        sp.Ld = (rem + kd - 1) / kd;
        sp.Kd = (rem + sp.Ld - 1) / sp.Ld;
    } else {
        sp.Ld = 1;
        sp.Kd = 0;
    }
    return sp;
}

// Claim the next dynamic chunk.  The claim word holds (epoch << 24 | count);
// the first CTA stamps it with this call's epoch (count 0) in its prologue,
// and every claim is one atomicAdd.  A claimant waits (bounded)
// until the word carries this call's epoch, so a word left by an earlier call
// or never written is not counted.  Returns the claimed index, or -1 if the
// stamp never came.
__device__ __forceinline__ int64_t claim_chunk(unsigned long long* word, uint64_t epoch,
                                               bool& stamped) {
    if (!stamped) {
        const uint64_t t0 = global_ns();
        for (uint32_t it = 0;; ++it) {
            const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(word);
            if ((w >> 24) == epoch) break;
            if (it >= kWaitLimitIters || global_ns() - t0 > kWaitLimitNs) return -1;
            __nanosleep(64);
        }
        stamped = true;
    }
    const unsigned long long old = atomicAdd(word, 1ull);
    if ((old >> 24) != epoch) return -1;
    return (int64_t)(old & 0xffffffull);
}

// ------------------------------------------------------------ shared prefixes
// Sequences adjacent in the batch whose tables begin with the same full blocks
// (forks: parallel sampling, beam search) form groups; the group pass below
// finds them and cuts each group's common prefix into units (a head and at
// most group_unit_steps steps).  In the main kernel a unit's K/V steps are
// staged once and one warp attends every member's query to them together:
// scores S^T = K Q^T (16 tokens x 8 members per tensor-core product) and the
// output O^T += V^T P^T, with the online softmax per member; the unit ends in
// one partial (m, l, acc) per member, which the merge kernel combines with
// the member's own (suffix) partials.  Results are the same attention: the
// prefix is a contiguous run of each member's tokens, and the split-K rule
// combines any partition of a row's tokens.

// D = A B + C, m16n8k16, A row-major, B column-major, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&c)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// Transpose of an 8x8 16-bit matrix held one row pair per thread (the
// fragment layout of the tensor-core products).
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (std::is_same<T, __half>::value) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
}

// Block-wide scans over S values held one per sequence in shared memory, each
// thread a contiguous range (in place).  `scratch` holds one int per warp.
static __device__ void block_scan_max_incl(int* v, int S, int* scratch) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
    const int per = (S + nt - 1) / nt;
    const int b = min(tid * per, S), e = min(b + per, S);
    int local = -1;
    for (int i = b; i < e; ++i) local = max(local, v[i]);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl = max(incl, y);
    }
    if (lane == 31) scratch[w] = incl;
    __syncthreads();
    int run = -1;
    for (int i = 0; i < w; ++i) run = max(run, scratch[i]);
    const int y = __shfl_up_sync(kFull, incl, 1);
    if (lane >= 1) run = max(run, y);
    for (int i = b; i < e; ++i) {
        run = max(run, v[i]);
        v[i] = run;
    }
    __syncthreads();
}
// out[i] = sum_{i' < i} v[i'] for i <= S (out may alias nothing).
static __device__ void block_scan_sum_excl(const int* v, int* out, int S, int* scratch) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
    const int per = (S + nt - 1) / nt;
    const int b = min(tid * per, S), e = min(b + per, S);
    int local = 0;
    for (int i = b; i < e; ++i) local += v[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[w] = incl;
    __syncthreads();
    int run = incl - local;
    for (int i = 0; i < w; ++i) run += scratch[i];
    for (int i = b; i < e; ++i) {
        out[i] = run;
        run += v[i];
    }
    if (tid == nt - 1) out[S] = run;
    __syncthreads();
}

// out1[i] = sum_{i' < i} v1[i'], out2 likewise, for i <= S, in one pass.
static __device__ void block_scan_sum2_excl(const int* v1, const int* v2, int* out1, int* out2,
                                            int S, int* scratch) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
    const int per = (S + nt - 1) / nt;
    const int b = min(tid * per, S), e = min(b + per, S);
    int l1 = 0, l2 = 0;
    for (int i = b; i < e; ++i) {
        l1 += v1[i];
        l2 += v2[i];
    }
    int i1 = l1, i2 = l2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y1 = __shfl_up_sync(kFull, i1, o), y2 = __shfl_up_sync(kFull, i2, o);
        if (lane >= o) {
            i1 += y1;
            i2 += y2;
        }
    }
    if (lane == 31) {
        scratch[w] = i1;
        scratch[32 + w] = i2;
    }
    __syncthreads();
    int r1 = i1 - l1, r2 = i2 - l2;
    for (int i = 0; i < w; ++i) {
        r1 += scratch[i];
        r2 += scratch[32 + i];
    }
    for (int i = b; i < e; ++i) {
        out1[i] = r1;
        out2[i] = r2;
        r1 += v1[i];
        r2 += v2[i];
    }
    if (tid == nt - 1) {
        out1[S] = r1;
        out2[S] = r2;
    }
    __syncthreads();
}

// The group pass: kGroupPassCtas CTAs of kGroupPassThreads threads.  For each sequence s
// >= 1 it counts the leading table entries equal to sequence s-1's among the
// full blocks of both (the shared prefix), forms groups of adjacent
// sequences, and writes per sequence its group prefix (in steps), member
// index and first partial slot, and the list of units, into the workspace.
// Groups only ever read the same blocks a member would read itself: when the
// workspace cannot hold the units or their partials, nothing is grouped.
constexpr int kGroupPassThreads = 1024;
constexpr int kGroupPassCtas = 8;      // all find the groups; they share the unit writes

template <int D, int B>
__global__ void __launch_bounds__(kGroupPassThreads) paged_decode_groups(const DecodeArgs a) {
    constexpr int SUB = step_tokens(D);
    constexpr int LG = group_unit_steps(D, B);
    extern __shared__ int gsm[];
    const int S = a.S, H = a.H, tid = threadIdx.x, nt = blockDim.x;
    int* cs = gsm;                 // [S] clamped context lengths, later a leader's size
    int* nf = cs + S;              // [S] full blocks s and s-1 both hold, later member slots
    int* first = nf + S;           // [S] leading equal entries, then shared steps
    int* rs = first + S;           // [S] start of s's run of followers
    int* units = rs + S;           // [S] units of a leader's group, else 0
    int* gP = units + S;           // [S] a leader's group prefix (steps)
    int* ub = gP + S;              // [S + 1] pair prefix, then unit prefix
    int* mb = ub + S + 1;          // [S + 1] member-slot prefix
    int* scratch = mb + S + 1;     // [64]

    grid_launch_dependents();      // the main kernel waits for this grid to end
    grid_dependency_wait();
    const int cap = a.ctx_cap;
    for (int s = tid; s < S; s += nt) {
        int c = a.context_lens[s];
        cs[s] = c < 0 ? 0 : (c > cap ? cap : c);
    }
    __syncthreads();
    for (int s = tid; s < S; s += nt) {
        const int n = s >= 1 ? min(cs[s], cs[s - 1]) / B : 0;
        nf[s] = n;
        first[s] = n;
    }
    __syncthreads();
    // the first entry that differs: tps threads per sequence, each taking
    // every tps-th entry, sixteen entries' loads issued together
    {
        constexpr int kBatch = 16;
        const int tps = S < nt ? nt / S : 1;
        const int r = tid % tps;
        for (int s = 1 + tid / tps; s < S; s += nt / tps) {
            const int n = nf[s];
            const int32_t* r0 = a.block_tables + (int64_t)s * a.max_blocks;
            const int32_t* r1 = r0 - a.max_blocks;
            for (int j0 = r; j0 < n; j0 += kBatch * tps) {
                int32_t x[kBatch], y[kBatch];
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int j = j0 + k * tps;
                    x[k] = j < n ? __ldg(r0 + j) : 0;
                    y[k] = j < n ? __ldg(r1 + j) : 0;
                }
                int fm = n;
#pragma unroll
                for (int k = kBatch - 1; k >= 0; --k)
                    if (x[k] != y[k]) fm = j0 + k * tps;
                if (fm < n) atomicMin(&first[s], fm);
            }
        }
    }
    __syncthreads();
    // followers (a long enough prefix shared with s - 1) and runs of them
    for (int s = tid; s < S; s += nt) {
        const int steps = s >= 1 ? (first[s] * B) / SUB : 0;
        first[s] = steps;
        rs[s] = (s >= 1 && steps >= kGroupMinSteps) ? -1 : s;
    }
    __syncthreads();
    block_scan_max_incl(rs, S, scratch);
    // groups: every kGroupMax-th sequence of a run leads the next ones
    int* gG = cs;                  // (context lengths no longer needed)
    for (int s = tid; s < S; s += nt) {
        int g = 1, P = 0;
        if ((s - rs[s]) % kGroupMax == 0) {
            P = kGroupMaxPrefixSteps;
            for (int f = s + 1; f < S && f - s < kGroupMax && rs[f] == rs[s]; ++f) {
                ++g;
                P = min(P, first[f]);
            }
        }
        if (g < 2) {
            g = 1;
            P = 0;
        }
        gG[s] = g;
        gP[s] = P;
        units[s] = g >= 2 ? H * ((P + LG - 1) / LG) : 0;
        nf[s] = g * units[s];          // member slots of a leader's group
    }
    __syncthreads();
    block_scan_sum2_excl(units, nf, ub, mb, S, scratch);
    const bool fits = (int64_t)ub[S] <= a.ws_l.gunit_cap && (int64_t)mb[S] <= a.ws_l.gslot_cap;
    const int U = fits ? ub[S] : 0;
    int* gh = reinterpret_cast<int*>(a.ws + a.ws_l.gh_off);
    int* gseq = reinterpret_cast<int*>(a.ws + a.ws_l.gseq_off);
    int* gslot = reinterpret_cast<int*>(a.ws + a.ws_l.gslot_off);
    GroupUnit* gu = reinterpret_cast<GroupUnit*>(a.ws + a.ws_l.gunit_off);
    if (blockIdx.x == 0) {
        if (tid == 0) {
            gh[0] = U;
            gh[1] = fits ? mb[S] : 0;
        }
        for (int s = tid; s < S; s += nt) {
            const int L = s - (s - rs[s]) % kGroupMax;
            const int g = gG[L];
            int info = 0, slot = 0;
            if (fits && g >= 2) {
                const int n = s - L;
                info = gP[L] | (n << 20) | ((g - 1) << 24);
                slot = mb[L] + n * units[L];
            }
            gseq[s] = info;
            gslot[s] = slot;
        }
    }
    // the units, this CTA's share: (leader, head, part); a prefix of P steps
    // in nc parts, the first P mod nc of them one step longer
    for (int u0 = blockIdx.x * nt + (tid & ~31); u0 < U; u0 += gridDim.x * nt) {
        // the leader of the warp's first unit by one search (lane 0), then
        // each lane steps forward to its own (a leader owns H * nc >= H units)
        const int lane = tid & 31, u = u0 + lane;
        int L = 0;
        if (lane == 0) {
            int lo = 0, hi = S - 1;              // largest s with ub[s] <= u0
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (ub[mid] <= u0) lo = mid;
                else hi = mid - 1;
            }
            L = lo;
        }
        L = __shfl_sync(kFull, L, 0);
        if (u >= U) continue;
        while (ub[L + 1] <= u) ++L;
        const int P = gP[L], nc = (P + LG - 1) / LG;
        const int r = u - ub[L], h = r / nc, c = r - h * nc;
        const int q = P / nc, rem = P - q * nc;
        GroupUnit x;
        x.L = L;
        x.h = h;
        x.j0 = c * q + (c < rem ? c : rem);
        x.len = q + (c < rem ? 1 : 0);
        x.g = gG[L];
        x.slot0 = mb[L] + h * nc + c;
        x.mstride = units[L];
        x.pad = 0;
        gu[u] = x;
    }
}

// One unit of a group in one consumer warp: the warp owns steps g0 + NW i +
// warp (i < n) of the ring; it attends every member of `x` to the unit's
// steps (i < x.len; the rest are empty steps that only pass through), then
// writes one partial per member.
template <typename T, int D, int B>
__device__ __forceinline__ void group_unit_consume(const DecodeArgs& a, const GroupUnit& x,
                                                   bool valid, int n, uint32_t g0,
                                                   unsigned char* ring, uint64_t* full,
                                                   uint64_t* empty, volatile int* abort_flag,
                                                   int warp, int lane) {
    using C = Cfg<D, B>;
    constexpr int NKT = D / 16;          // k-tiles of a score product
    constexpr int NMT = D / 16;          // m-tiles of the output product
    constexpr int NTT = C::SUB / 16;     // 16-token tiles per step
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    const int mem = lane >> 2, c4 = lane & 3;
    uint32_t qb[NKT][2];
    if (valid && mem < x.g) {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            static_cast<const T*>(a.q) + ((int64_t)(x.L + mem) * a.H + x.h) * D);
#pragma unroll
        for (int kt = 0; kt < NKT; ++kt) {
            qb[kt][0] = __ldg(qrow + kt * 8 + c4);
            qb[kt][1] = __ldg(qrow + kt * 8 + 4 + c4);
        }
    } else {
#pragma unroll
        for (int kt = 0; kt < NKT; ++kt) qb[kt][0] = qb[kt][1] = 0u;
    }
    float o[NMT][4];
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // ldmatrix row addresses: K as the A operand (rows = tokens), V^T (rows = dims).
    // A step's K (and V) is stored per 64-column half of D as SUB rows of 128
    // bytes, 16-byte chunk c of row r at chunk c ^ (r mod 8) (the copies'
    // 128-byte swizzle).
    const int krow = ((lane >> 3) & 1) * 8 + (lane & 7), kcol = (lane >> 4) * 8;
    const int vrow = (lane >> 4) * 8 + (lane & 7), vcol = ((lane >> 3) & 1) * 8;
    auto swz = [](int row, int col) -> uint32_t {      // col: element index in [0, D)
        return (uint32_t)((col >> 6) * (C::SUB * 128) + row * 128 +
                          ((((col & 63) >> 3) ^ (row & 7)) << 4));
    };
    for (int i = 0; i < n; ++i) {
        const uint32_t g = g0 + (uint32_t)(C::NW * i + warp);
        const int stage = (int)(g % C::NSTAGE);
        const uint32_t par = (g / C::NSTAGE) & 1u;
        const bool got = !*abort_flag && wait_phase(&full[stage], par, abort_flag, a.wait_ns);
        const bool have = __all_sync(kFull, got);
        if (!have && lane == 0) note_timeout(abort_flag, a.err);
        if (have && valid && i < x.len) {
            const uint32_t ks = smem_addr(ring + (size_t)stage * C::STAGE);
            const uint32_t vs = ks + C::CHUNK;
            float sc[NTT][4];
#pragma unroll
            for (int tt = 0; tt < NTT; ++tt) {
                sc[tt][0] = sc[tt][1] = sc[tt][2] = sc[tt][3] = 0.f;
#pragma unroll
                for (int kt = 0; kt < NKT; ++kt) {
                    uint32_t af[4];
                    ldsm_x4(af, ks + swz(tt * 16 + krow, kt * 16 + kcol));
                    mma16816<T>(sc[tt], af, qb[kt][0], qb[kt][1]);
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int tt = 0; tt < NTT; ++tt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[tt][e] *= a.scale_log2;
                mx0 = fmaxf(mx0, fmaxf(sc[tt][0], sc[tt][2]));
                mx1 = fmaxf(mx1, fmaxf(sc[tt][1], sc[tt][3]));
            }
#pragma unroll
            for (int o_ = 4; o_ < 32; o_ <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o_));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o_));
            }
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            uint32_t pb[NTT][2], pr[NTT][2];
#pragma unroll
            for (int tt = 0; tt < NTT; ++tt) {
                const float p0 = exp2f(sc[tt][0] - n0), p1 = exp2f(sc[tt][1] - n1);
                const float p2 = exp2f(sc[tt][2] - n0), p3 = exp2f(sc[tt][3] - n1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                const uint32_t hlo = pack2<T>(p0, p1), hhi = pack2<T>(p2, p3);
                pb[tt][0] = movm_t(hlo);
                pb[tt][1] = movm_t(hhi);
                if constexpr (BF) {
                    // bf16 keeps 8 significant bits: the weights go in as a
                    // high part and the bf16 residual, two products
                    const float2 q01 = unpack2<T>(hlo), q23 = unpack2<T>(hhi);
                    pr[tt][0] = movm_t(pack2<T>(p0 - q01.x, p1 - q01.y));
                    pr[tt][1] = movm_t(pack2<T>(p2 - q23.x, p3 - q23.y));
                }
            }
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
                for (int tt = 0; tt < NTT; ++tt) {
                    uint32_t af[4];
                    ldsm_x4_t(af, vs + swz(tt * 16 + vrow, mt * 16 + vcol));
                    mma16816<T>(o[mt], af, pb[tt][0], pb[tt][1]);
                    if constexpr (BF) mma16816<T>(o[mt], af, pr[tt][0], pr[tt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && have) mbar_arrive(&empty[stage]);
    }
    if (!valid || __any_sync(kFull, *abort_flag)) return;
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, o_);
        l1 += __shfl_xor_sync(kFull, l1, o_);
    }
    float2* gml = reinterpret_cast<float2*>(a.ws + a.ws_l.gml_off);
    float* gacc = reinterpret_cast<float*>(a.ws + a.ws_l.gacc_off);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int member = 2 * c4 + e;
        if (member >= x.g) continue;
        const int64_t slot = (int64_t)x.slot0 + (int64_t)member * x.mstride;
        if (mem == 0) gml[slot] = make_float2(e ? m1 : m0, e ? l1 : l0);
        float* dst = gacc + slot * D + mem;
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
            dst[mt * 16] = o[mt][e];
            dst[mt * 16 + 8] = o[mt][2 + e];
        }
    }
}

// ------------------------------------------------------------ the main kernel
// (with shared prefixes the tensor-core path raises the register count; the
// bound keeps five CTAs per SM, as the plain kernel has)
template <typename T, int D, int B, int MODE>
__global__ void __launch_bounds__(Cfg<D, B>::THREADS,
                                  MODE == kModeShared ? 5 : PKV_DECODE_MIN_CTAS)
    paged_decode_main(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
    using C = Cfg<D, B>;
    constexpr bool CONTIG = MODE == kModeContig;
    constexpr bool GROUPS = MODE == kModeShared;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + C::NSTAGE;
    uint64_t* pair = empty + C::NSTAGE;        // the consumer warps' meeting, per merge buffer
    float* merge = reinterpret_cast<float*>(smem + C::MERGE_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
    int* scratch = reinterpret_cast<int*>(smem + C::MISC_OFF) + 4;   // NW + 1 ints
    int* s_ctx = reinterpret_cast<int*>(smem + C::CTX_OFF);
    int* s_base = s_ctx + a.S;
    // the newest tokens come with the call (k_new / v_new)
    constexpr bool append = MODE == kModeAppend;
    int64_t* app_word = reinterpret_cast<int64_t*>(smem + C::APP_OFF);
    // shared prefixes: the steps a group reads for each sequence, then the unit count
    int* s_pfx = s_base + a.S + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S, H = a.H;

    // 1. context lengths (validated and clamped) and the step prefix
    grid_dependency_wait();
    const int cap = a.ctx_cap;
    for (int s = tid; s < S; s += C::THREADS) {
        int c = a.context_lens[s];
        if (c < 0 || c > cap) {
            atomicOr(a.err, PKV_DEVERR_BAD_CONTEXT);
            c = c < 0 ? 0 : cap;
        }
        s_ctx[s] = c;
        if constexpr (GROUPS)
            s_pfx[s] = reinterpret_cast<const int*>(a.ws + a.ws_l.gseq_off)[s] & kGroupMaxPrefixSteps;
    }
    if constexpr (GROUPS) {
        if (tid == 0) s_pfx[S] = reinterpret_cast<const int*>(a.ws + a.ws_l.gh_off)[0];
    }
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + C::QBAR_OFF);
    int* qid = reinterpret_cast<int*>(smem + C::QID_OFF);
    unsigned char* qbuf = smem + C::QBUF_OFF;
    if (tid == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < C::QN; ++i) mbar_init(&qfull[i], 1);
        mbar_init(&pair[0], C::NW);
        mbar_init(&pair[1], C::NW);
        fence_mbar_init();
        *abort_flag = 0;
    }
    __syncthreads();
    scan_steps<C::SUB>(s_ctx, s_base, S, scratch, GROUPS ? s_pfx : nullptr);
    const int U = GROUPS ? s_pfx[S] : 0;                 // group units
    const bool has_units = GROUPS && (int)blockIdx.x < U;

    // 2. the split of the step space, and this CTA's static range
    const Split sp = make_split((int64_t)H * s_base[S], (int)gridDim.x, a.L_steps,
                                a.min_chunk_steps);
    const int64_t total = sp.total;
    const bool ws_ok = (int64_t)S * H + sp.last_chunk() + 1 <= a.ws_l.cap;
    if (blockIdx.x == 0) {
        int64_t* hdr = reinterpret_cast<int64_t*>(a.ws);
        int* wbase = reinterpret_cast<int*>(a.ws + a.ws_l.base_off);
        for (int i = tid; i <= S; i += C::THREADS) wbase[i] = s_base[i];
        if (tid == 0) {
            hdr[0] = ws_ok ? sp.Ls : 0;
            hdr[1] = total;
            if (!ws_ok) atomicOr(a.err, PKV_DEVERR_WORKSPACE);
#if PKV_DECODE_DYN_PER_CTA != 0
            // stamp the claim word (header word 2) with this call's epoch,
            // count 0.  The previous call on this stream has finished (the
            // dependency wait above), so no claim of its can land after this.
            if (ws_ok && !sp.fixed && sp.Kd > 0) {
                *reinterpret_cast<volatile unsigned long long*>(hdr + 2) =
                    (unsigned long long)a.epoch << 24;
                __threadfence();
            }
#endif
        }
    }
    grid_launch_dependents();
    if (!ws_ok || (total == 0 && !has_units)) return;
    int64_t xb = 0, xe = 0;
    if (total == 0) {
        // group units only
    } else if (sp.fixed) {
        const int64_t K = (total + sp.Ls - 1) / sp.Ls;
        const int64_t kb = (int64_t)blockIdx.x * K / gridDim.x;
        const int64_t ke = (int64_t)(blockIdx.x + 1) * K / gridDim.x;
        xb = kb * sp.Ls;
        xe = ke * sp.Ls < total ? ke * sp.Ls : total;
        if (xb >= xe && !has_units) return;
        if (xb > xe) xb = xe;
    } else {
        xb = (int64_t)blockIdx.x * sp.Ls;
        xe = xb + sp.Ls < sp.X ? xb + sp.Ls : sp.X;
        if (xb > xe) xb = xe;                    // no static share: claimed chunks only
        if (xb >= xe && sp.Kd == 0 && !has_units) return;
    }
    if (warp == C::NW) {
        // ================================================= producer warp
        const char* kpool = static_cast<const char*>(a.k_cache);
        const char* vpool = static_cast<const char*>(a.v_cache);
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        // block-table cache, warp-wide: the current 32-entry window, the next
        // window of the same sequence, and the first window of the next
        // sequence (both prefetched so no table read sits on the copy path)
        int tc_s = -1, tc_win = 0, tc_val = 0, tn_val = 0, ts_s = -1, ts_val = 0, ts_win = 0;
        bool tn_ok = false;
        bool stop = false;
        // issue the copies of the steps [rb, re), in order, into the ring
        auto issue_range = [&](int64_t rb, int64_t re) {
            if (rb >= re) return;
            Pos p = locate(rb, s_base, S, H);
            for (int64_t x = rb; x < re && !stop;) {
                const int ns = s_base[p.s + 1] - s_base[p.s];
                const int64_t left = re - x;
                const int run = (int64_t)(ns - p.j) < left ? ns - p.j : (int)left;
                // (a member of a group starts after the steps its group reads)
                const int skip = GROUPS ? s_pfx[p.s] : 0;
                for (int i = 0; i < run; ++i) {
                    const int j = p.j + i + skip;
                    // first logical block of the step, and the step's token offset in it
                    const int jb = C::BPS > 1 ? j * C::BPS : j / C::SPB;
                    const int sub = C::BPS > 1 ? 0 : j - jb * C::SPB;
                    int phys_raw[C::BPS];
                    if constexpr (!CONTIG) {
                    const int nblk = (s_ctx[p.s] + B - 1) / B;
                    const int32_t* row = a.block_tables + (int64_t)p.s * a.max_blocks;
                    const int win = jb & ~31;
                    if (p.s != tc_s || win != tc_win) {
                        if (p.s == tc_s && win == tc_win + 32 && tn_ok) {
                            tc_val = tn_val;
                        } else if (p.s == ts_s && win == ts_win) {
                            tc_val = ts_val;
                        } else {
                            tc_val = (win + lane < nblk) ? __ldg(row + win + lane) : 0;
                        }
                        if (p.s != tc_s) {
                            int s2 = p.s + 1;
                            while (s2 < S && s_base[s2 + 1] == s_base[s2]) ++s2;
                            ts_s = -1;
                            if (s2 < S) {
                                const int nb2 = (s_ctx[s2] + B - 1) / B;
                                const int j2 = GROUPS ? s_pfx[s2] : 0;
                                ts_win = (C::BPS > 1 ? j2 * C::BPS : j2 / C::SPB) & ~31;
                                ts_val = ts_win + lane < nb2
                                             ? __ldg(a.block_tables + (int64_t)s2 * a.max_blocks +
                                                     ts_win + lane)
                                             : 0;
                                ts_s = s2;
                            }
                        }
                        tc_s = p.s;
                        tc_win = win;
                        tn_ok = win + 32 < nblk;
                        if (tn_ok) tn_val = (win + 32 + lane < nblk) ? __ldg(row + win + 32 + lane) : 0;
                    }
#pragma unroll
                    for (int b = 0; b < C::BPS; ++b)
                        phys_raw[b] = __shfl_sync(kFull, tc_val, jb + b - win);
                    }  // !CONTIG
                    int ok = 1;
                    if (lane == 0) {
                        // (after an abort a stage the consumers released is still
                        // safe to fill -- its copy landed -- and the first one they
                        // did not release stops this loop; the drain below waits
                        // for everything issued)
                        ok = wait_phase(&empty[stage], phase ^ 1u, abort_flag, a.wait_ns) ? 1 : 0;
                        if (ok) {
                            // only the step's valid tokens move (the last step of a
                            // row is usually partial); the rest of the stage keeps
                            // stale bytes that the consumers mask out
                            const int tok0 = j * C::SUB;
                            // With the newest tokens given, the row's last step
                            // takes its last token (the newest, tn within the
                            // step) from k_new / v_new instead of the cache, and
                            // the stage's word tells the consumer the token's
                            // slot, which it then writes from the stage.
                            const bool app = append && j == ns - 1;
                            const int tn = s_ctx[p.s] - 1 - tok0;
                            uint32_t bytes[C::BPS];
                            uint32_t tx = 0;
#pragma unroll
                            for (int b = 0; b < C::BPS; ++b) {
                                int valid = s_ctx[p.s] - (tok0 + b * C::TPC);
                                valid = valid < 0 ? 0 : (valid > C::TPC ? C::TPC : valid);
                                if (app && b == tn / C::TPC) --valid;   // (its last valid token)
                                bytes[b] = (uint32_t)valid * (uint32_t)(D * 2);
                                tx += 2 * bytes[b];
                            }
                            unsigned char* dst = ring + (size_t)stage * C::STAGE;
                            if (app) {
                                tx += 2 * (uint32_t)(D * 2);
                                const int bn = tn / C::TPC;
                                int64_t phys = 0;
                                if constexpr (!CONTIG) phys = phys_raw[bn];
                                int64_t w = -1;
                                if (phys >= 0 && phys < a.num_blocks)
                                    w = ((phys * H + p.h) * B + (int64_t)sub * C::SUB +
                                         (tn - bn * C::TPC)) *
                                        (int64_t)D * 2;
                                else    // (its block may have nothing else to copy)
                                    atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                                app_word[stage] = w;            // before the arrive (release)
                            }
                            mbar_arrive_expect_tx(&full[stage], tx);
                            if (app) {
                                const int64_t nrow = ((int64_t)p.s * H + p.h) * D * 2;
                                bulk_g2s(dst + tn * D * 2, static_cast<const char*>(a.k_new) + nrow,
                                         D * 2, &full[stage]);
                                bulk_g2s(dst + C::CHUNK + tn * D * 2,
                                         static_cast<const char*>(a.v_new) + nrow, D * 2,
                                         &full[stage]);
                            }
#pragma unroll
                            for (int b = 0; b < C::BPS; ++b) {
                                if (bytes[b] == 0) continue;
                                int64_t off;
                                if constexpr (CONTIG) {
                                    // [seq][head][token][D]: the step's tokens are one run
                                    off = (((int64_t)p.s * H + p.h) * a.kv_stride + tok0) *
                                          (int64_t)D * 2;
                                } else {
                                    int64_t phys = phys_raw[b];
                                    if (phys < 0 || phys >= a.num_blocks) {
                                        atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                                        phys = 0;
                                    }
                                    off = ((phys * H + p.h) * B + (int64_t)sub * C::SUB) *
                                          (int64_t)D * 2;
                                }
                                const uint32_t doff = (uint32_t)(b * C::TPC * D * 2);
                                bulk_g2s(dst + doff, kpool + off, bytes[b], &full[stage]);
                                bulk_g2s(dst + C::CHUNK + doff, vpool + off, bytes[b], &full[stage]);
                            }
                        }
                    }
                    ok = __shfl_sync(kFull, ok, 0);
                    if (!ok) {
                        if (lane == 0) note_timeout(abort_flag, a.err);
                        stop = true;
                        break;
                    }
                    ++issued;
                    if (++stage == C::NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (stop) break;
                x += run;
                p.j += run;
                if (p.j == ns && x < re) next_segment(p, s_base, S, H);
            }
        };
        if constexpr (GROUPS) {
            // group units first: a batch of NW units (this CTA's next ones,
            // one per consumer warp), interleaved step by step so that step g
            // belongs to warp g mod NW; a unit that has run out is padded with
            // empty steps (an arrival without bytes)
            const GroupUnit* gu = reinterpret_cast<const GroupUnit*>(a.ws + a.ws_l.gunit_off);
            for (int u0 = blockIdx.x; u0 < U && !stop; u0 += C::NW * (int)gridDim.x) {
                GroupUnit ux[C::NW];
                int tw[C::NW], jb0[C::NW], n = 0;
#pragma unroll
                for (int w = 0; w < C::NW; ++w) {
                    const int u = u0 + w * (int)gridDim.x;
                    if (u < U) {
                        ux[w] = gu[u];
                    } else {
                        ux[w].L = 0;
                        ux[w].h = 0;
                        ux[w].j0 = 0;
                        ux[w].len = 0;
                    }
                    n = max(n, ux[w].len);
                    jb0[w] = C::BPS > 1 ? ux[w].j0 * C::BPS : ux[w].j0 / C::SPB;
                    const int nblk = (s_ctx[ux[w].L] + B - 1) / B;
                    tw[w] = (ux[w].len > 0 && jb0[w] + lane < nblk)
                                ? __ldg(a.block_tables + (int64_t)ux[w].L * a.max_blocks + jb0[w] +
                                        lane)
                                : 0;
                }
                for (int i = 0; i < n && !stop; ++i) {
#pragma unroll
                    for (int w = 0; w < C::NW; ++w) {
                        if (stop) break;
                        const bool real = i < ux[w].len;
                        const int j = ux[w].j0 + i;
                        const int jb = C::BPS > 1 ? j * C::BPS : j / C::SPB;
                        const int sub = C::BPS > 1 ? 0 : j - jb * C::SPB;
                        int phys_raw[C::BPS];
#pragma unroll
                        for (int b = 0; b < C::BPS; ++b)
                            phys_raw[b] = __shfl_sync(kFull, tw[w], (jb + b - jb0[w]) & 31);
                        int ok = 1;
                        if (lane == 0) {
                            ok = wait_phase(&empty[stage], phase ^ 1u, abort_flag, a.wait_ns) ? 1 : 0;
                            if (ok && !real) {
                                mbar_arrive(&full[stage]);
                            } else if (ok) {
                                // a prefix step is whole (every member holds all of
                                // its tokens); it is copied by tiled tensor copies
                                // with the 128-byte swizzle: per 64-column half of
                                // D, the step's rows of 128 bytes, chunk c of row r
                                // at chunk c ^ (r mod 8), so that the tensor-core
                                // fragment loads hit distinct banks
                                unsigned char* dst = ring + (size_t)stage * C::STAGE;
                                mbar_arrive_expect_tx(&full[stage], 2u * C::CHUNK);
#pragma unroll
                                for (int b = 0; b < C::BPS; ++b) {
                                    int64_t phys = phys_raw[b];
                                    if (phys < 0 || phys >= a.num_blocks) {
                                        atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                                        phys = 0;
                                    }
                                    const int y = (int)((phys * H + ux[w].h) * B +
                                                        (int64_t)sub * C::SUB);
#pragma unroll
                                    for (int hh = 0; hh < D / 64; ++hh) {
                                        const uint32_t doff =
                                            (uint32_t)(hh * C::SUB * 128 + b * C::TPC * 128);
                                        tensor_g2s(dst + doff, &tmk, hh * 64, y, &full[stage]);
                                        tensor_g2s(dst + C::CHUNK + doff, &tmv, hh * 64, y,
                                                   &full[stage]);
                                    }
                                }
                            }
                        }
                        ok = __shfl_sync(kFull, ok, 0);
                        if (!ok) {
                            if (lane == 0) note_timeout(abort_flag, a.err);
                            stop = true;
                            break;
                        }
                        ++issued;
                        if (++stage == C::NSTAGE) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
        // the static range first; then (balanced split) claimed chunks, each
        // handed to the consumers through the queue with the query slice of
        // its first row
        issue_range(xb, xe);
#if PKV_DECODE_DYN_PER_CTA != 0
        // (the claim state lives only here, not across the static range's loop)
        int published = 0;
        bool stamped = false;
        unsigned long long* claim_word = reinterpret_cast<unsigned long long*>(a.ws) + 2;
        const char* qbytes = static_cast<const char*>(a.q);
        while (!stop && !sp.fixed && sp.Kd > 0) {
            int64_t k = -1;
            if (lane == 0) {
                k = claim_chunk(claim_word, a.epoch, stamped);
                if (k < 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
            }
            k = __shfl_sync(kFull, k, 0);
            const bool more = k >= 0 && k < sp.Kd;
            const int slot = published % C::QN;
            if (lane == 0) {
                qid[slot] = more ? (int)k : -1;
                if (more) {
                    const Pos p0 = locate(sp.X + k * sp.Ld, s_base, S, H);
                    mbar_arrive_expect_tx(&qfull[slot], D * 2);
                    bulk_g2s(qbuf + (size_t)slot * D * 2,
                             qbytes + ((int64_t)p0.s * H + p0.h) * (int64_t)D * 2, D * 2,
                             &qfull[slot]);
                } else {
                    mbar_arrive(&qfull[slot]);
                }
            }
            ++published;
            __syncwarp();
            if (!more) break;
            const int64_t rb = sp.X + k * sp.Ld;
            issue_range(rb, rb + sp.Ld < total ? rb + sp.Ld : total);
        }
        __syncwarp();
        if (lane == 0) {
            // the query slices this warp copied (the latest use of each queue
            // entry): landed before the CTA may end, whatever the consumers did
            for (int e = published > C::QN ? published - C::QN : 0; e < published; ++e)
                wait_bounded(&qfull[e % C::QN], (uint32_t)(e / C::QN) & 1u, nullptr, kWaitLimitNs);
        }
#endif
        __syncwarp();
        if (lane == 0) {
            // the same for the ring: the latest copy into each stage (earlier
            // ones landed before their stage was released for reuse)
            const int n = issued < C::NSTAGE ? issued : C::NSTAGE;
            int st = stage;
            uint32_t ph = phase;
            for (int i = 0; i < n; ++i) {
                if (--st < 0) {
                    st = C::NSTAGE - 1;
                    ph ^= 1u;
                }
                wait_bounded(&full[st], ph, nullptr, kWaitLimitNs);
            }
        }
        return;
    }

    // ===================================================== consumer warps
    const int hi = lane >> C::LOG_LPT;          // token within a 512-B row
    const int dl = lane & (C::LPT - 1);         // 8-element slice of head_dim
    const int own = dl >> C::RS;                // load whose score this lane ends up with
    const bool leader = (dl & ((1 << C::RS) - 1)) == 0;
    const T* qptr = static_cast<const T*>(a.q);
    T* optr = static_cast<T*>(a.out);
    float2* ws_ml = reinterpret_cast<float2*>(a.ws + a.ws_l.ml_off);
    float* ws_acc = reinterpret_cast<float*>(a.ws + a.ws_l.acc_off);

    uint32_t g0 = 0;
    int pbuf = 0;
    uint32_t npiece = 0;                        // pieces met so far (pair barrier phases)
    // the static range, then the claimed chunks the producer publishes; one
    // copy of the loop serves both.  q_first is the query slice of a range's
    // first row; the next piece's slice is loaded one piece ahead, and the
    // chunk id and the chunk's end are carried along (no division per piece).
    int64_t rb = xb, re = xe;
    uint4 q_first = make_uint4(0u, 0u, 0u, 0u);
    if (xb < xe) {
        const Pos p0 = locate(xb, s_base, S, H);
        q_first = ld_nc_v4(qptr + ((int64_t)p0.s * H + p0.h) * D + dl * 8);
    }
#if PKV_DECODE_DYN_PER_CTA != 0
    int qe = 0;
#endif
    if constexpr (GROUPS) {
        // group units: the same batches as the producer's, this warp's unit
        const GroupUnit* gu = reinterpret_cast<const GroupUnit*>(a.ws + a.ws_l.gunit_off);
        for (int u0 = blockIdx.x; u0 < U; u0 += C::NW * (int)gridDim.x) {
            int n = 0;
#pragma unroll
            for (int w = 0; w < C::NW; ++w) {
                const int u = u0 + w * (int)gridDim.x;
                if (u < U) n = max(n, gu[u].len);
            }
            const int um = u0 + warp * (int)gridDim.x;
            const bool valid = um < U;
            GroupUnit x;
            if (valid) {
                x = gu[um];
            } else {
                x.L = x.h = x.j0 = x.len = x.g = x.slot0 = x.mstride = x.pad = 0;
            }
            group_unit_consume<T, D, B>(a, x, valid, n, g0, ring, full, empty, abort_flag, warp,
                                        lane);
            g0 += (uint32_t)(C::NW * n);
        }
    }
    while (true) {
        if (rb >= re) {
#if PKV_DECODE_DYN_PER_CTA == 0
            break;
#else
            if (sp.fixed || sp.Kd == 0 || *abort_flag) break;
            const int slot = qe % C::QN;
            const bool got = wait_phase(&qfull[slot], (uint32_t)(qe / C::QN) & 1u, abort_flag,
                                        a.wait_ns);
            if (!__all_sync(kFull, got)) {
                if (lane == 0) note_timeout(abort_flag, a.err);
                break;
            }
            ++qe;
            const int k = qid[slot];
            if (k < 0) break;
            q_first = *reinterpret_cast<const uint4*>(qbuf + (size_t)slot * D * 2 + dl * 16);
            rb = sp.X + (int64_t)k * sp.Ld;
            re = rb + sp.Ld < total ? rb + sp.Ld : total;
#endif
        }
        Pos p = locate(rb, s_base, S, H);
        int64_t x = rb;
        int64_t chunk = sp.chunk(rb);
        int64_t cend = sp.chunk_end(rb);
        uint4 q_next = q_first;
        while (x < re) {
            if (x == cend) {                         // fixed split: the next chunk of the run
                ++chunk;
                cend = cend + sp.Ls < re ? cend + sp.Ls : re;
            }
            const int ns = s_base[p.s + 1] - s_base[p.s];
            int64_t len64 = ns - p.j;
            if (cend - x < len64) len64 = cend - x;
            if (re - x < len64) len64 = re - x;
            const int len = (int)len64;
            const int skip = GROUPS ? s_pfx[p.s] : 0;   // steps its group read
            const bool whole = (p.j == 0 && len == ns && skip == 0);
            const int ctx = s_ctx[p.s];
            const int64_t row = (int64_t)p.s * H + p.h;
    
            const uint4 q_raw = q_next;
            if (x + len < re && p.j + len == ns) {
                Pos pn = p;
                next_segment(pn, s_base, S, H);
                q_next = ld_nc_v4(qptr + ((int64_t)pn.s * H + pn.h) * D + dl * 8);
            }
            float qf[8];
            {
                Elem<T>::to_f32x8(q_raw, qf);
    #pragma unroll
                for (int e = 0; e < 8; ++e) qf[e] *= a.scale_log2;
            }
            float m = -INFINITY, l = 0.f;
            float acc[8];
    #pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    
            const int first = (int)((uint32_t)(warp + C::NW - (int)(g0 % C::NW)) % C::NW);
            for (int i = first; i < len; i += C::NW) {
                const uint32_t g = g0 + (uint32_t)i;
                const int stage = (int)(g % C::NSTAGE);
                const uint32_t par = (g / C::NSTAGE) & 1u;
                // `have`: every lane saw the stage's copy land.  Only then is
                // the stage released; after an abort the warp runs through
                // its steps without waiting (and its results are not used).
                const bool got = !*abort_flag && wait_phase(&full[stage], par, abort_flag, a.wait_ns);
                const bool have = __all_sync(kFull, got);
                if (!have && lane == 0) note_timeout(abort_flag, a.err);
                const uint4* Ks = reinterpret_cast<const uint4*>(ring + (size_t)stage * C::STAGE);
                const uint4* Vs = Ks + C::CHUNK / 16;
                const int nvalid = ctx - (p.j + i + skip) * C::SUB;   // >= 1
    
                float part[C::NL];
    #pragma unroll
                for (int t = 0; t < C::NL; ++t) {
                    const uint4 kv = Ks[t * 32 + lane];
                    float kf[8];
                    Elem<T>::to_f32x8(kv, kf);
                    float d = 0.f;
    #pragma unroll
                    for (int e = 0; e < 8; ++e) d = fmaf(qf[e], kf[e], d);
                    part[t] = d;
                }
                float z = reduce_scatter<C::NL, C::LOG_LPT>(part, dl);
                if (own * C::TPL + hi >= nvalid) z = -INFINITY;
                const float m_new = fmaxf(m, warp_max(z));
                const float alpha = exp2f(m - m_new);
                const float pz = exp2f(z - m_new);
                l = fmaf(l, alpha, leader ? pz : 0.f);
    #pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] *= alpha;
    #pragma unroll
                for (int t = 0; t < C::NL; ++t) {
                    const float pt = __shfl_sync(kFull, pz, (hi << C::LOG_LPT) | (t << C::RS));
                    if (t * C::TPL + hi < nvalid) {
                        const uint4 vv = Vs[t * 32 + lane];
                        float vf[8];
                        Elem<T>::to_f32x8(vv, vf);
    #pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] = fmaf(pt, vf[e], acc[e]);
                    }
                }
                m = m_new;
                if constexpr (append) {
                    // the row's last step with a new token: write its K and V
                    // rows from the stage into the token's cache slot (lanes
                    // 0 .. LPT-1 the K row, the next LPT the V row, 16 bytes
                    // each), before the stage is released
                    const int64_t w =
                        have && i == len - 1 && p.j + len == ns ? app_word[stage] : -1;
                    if (w >= 0 && lane < 2 * C::LPT) {
                        const int isv = lane >= C::LPT ? 1 : 0;
                        const int c16 = (lane & (C::LPT - 1)) * 16;
                        const uint4 val = *reinterpret_cast<const uint4*>(
                            ring + (size_t)stage * C::STAGE + isv * C::CHUNK +
                            (nvalid - 1) * D * 2 + c16);
                        char* pool = const_cast<char*>(
                            static_cast<const char*>(isv ? a.v_cache : a.k_cache));
                        *reinterpret_cast<uint4*>(pool + w + c16) = val;
                    }
                }
                __syncwarp();
                if (lane == 0 && have) mbar_arrive(&empty[stage]);
            }
    
            // fold the token groups of the warp, then merge the warps
    #pragma unroll
            for (int o = C::LPT; o < 32; o <<= 1)
    #pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
            l = warp_sum(l);
            float* mrow = merge + (pbuf * C::NW + warp) * C::MROW;
            if (lane < C::LPT) {
                float4* d4 = reinterpret_cast<float4*>(mrow + dl * 8);
                d4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                d4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            if (lane == 0) {
                mrow[D] = m;
                mrow[D + 1] = l;
            }
            // meet the other consumer warps (bounded: an aborted CTA's warps
            // may no longer agree on their pieces)
            __syncwarp();
            if (lane == 0) mbar_arrive(&pair[pbuf]);
            const bool met_l = !*abort_flag &&
                               wait_phase(&pair[pbuf], (npiece >> 1) & 1u, abort_flag, a.wait_ns);
            const bool met = __all_sync(kFull, met_l);
            if (!met && lane == 0) note_timeout(abort_flag, a.err);
            ++npiece;
            if (met) {
                const float* mb = merge + pbuf * C::NW * C::MROW;
                float M = -INFINITY;
    #pragma unroll
                for (int w = 0; w < C::NW; ++w) M = fmaxf(M, mb[w * C::MROW + D]);
                float sc[C::NW];
                float ls = 0.f;
    #pragma unroll
                for (int w = 0; w < C::NW; ++w) {
                    sc[w] = exp2f(mb[w * C::MROW + D] - M);
                    ls = fmaf(sc[w], mb[w * C::MROW + D + 1], ls);
                }
                for (int d = tid; d < D; d += C::NW * 32) {
                    float av = 0.f;
    #pragma unroll
                    for (int w = 0; w < C::NW; ++w) av = fmaf(sc[w], mb[w * C::MROW + d], av);
                    if (whole) {
                        optr[row * D + d] = Elem<T>::from_f32(av / ls);
                    } else {
                        const int64_t slot = row + chunk;
                        ws_acc[slot * D + d] = av;
                        if (d == 0) ws_ml[slot] = make_float2(M, ls);
                    }
                }
            }
            pbuf ^= 1;
            x += len;
            g0 += (uint32_t)len;
            p.j += len;
            if (p.j == ns && x < re) next_segment(p, s_base, S, H);
        }
        rb = re;
    }
}

// ------------------------------------------------------------ the merge kernel
// One warp per (sequence, head).  Before waiting for the main kernel, every
// CTA rebuilds the step prefix from context_lens (an input the main kernel
// only reads) and so knows which of its rows fell inside one chunk -- the main
// kernel wrote those -- and returns for them at once.  A zero-length sequence
// gets a zero row.  The other rows wait, then combine their partials with the
// log-sum-exp rule, online and 8 partials per batch of loads:
//   M = max_k m_k,  out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k.
constexpr int kMergeBatch = 8;

template <typename T, int D, int B, int MODE>
__global__ void __launch_bounds__(128) paged_decode_merge(const DecodeArgs a) {
    using C = Cfg<D, B>;
    constexpr bool GROUPS = MODE == kModeShared;
    constexpr int LG = group_unit_steps(D, B);
    extern __shared__ int msm[];            // base[S + 1], then 8 scan partials
    int* base = msm;
    int* scratch = msm + a.S + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S, H = a.H;
    const int* gseq = reinterpret_cast<const int*>(a.ws + a.ws_l.gseq_off);
    // With groups every CTA waits first: the steps a group read for each
    // sequence (written by the group pass) enter the step prefix.
    if constexpr (GROUPS) grid_dependency_wait();

    // the step prefix, as the main kernel forms it (same clamping)
    {
        const int cap = a.ctx_cap;
        const int per = (S + 127) / 128;
        const int b = min(tid * per, S), e = min(b + per, S);
        auto steps = [&](int i) {
            int c = a.context_lens[i];
            c = c < 0 ? 0 : (c > cap ? cap : c);
            return (c + C::SUB - 1) / C::SUB - (GROUPS ? (gseq[i] & kGroupMaxPrefixSteps) : 0);
        };
        int local = 0;
        for (int i = b; i < e; ++i) local += steps(i);
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) scratch[warp] = incl;
        __syncthreads();
        int run = incl - local;
        for (int i = 0; i < warp; ++i) run += scratch[i];
        for (int i = b; i < e; ++i) {
            base[i] = run;
            run += steps(i);
        }
        if (tid == 127) base[S] = run;
        __syncthreads();
    }
    // The first CTA always waits for the main kernel, even where its rows need
    // no merge: then this grid cannot complete before the main kernel has,
    // which the next call's claim-word stamp and any later reader of the
    // output rely on.  The other CTAs wait only where they merge, so those
    // with nothing to do leave at once.
    const bool anchor = blockIdx.x == 0;
    if (!GROUPS && anchor) grid_dependency_wait();
    const int64_t sh = (int64_t)blockIdx.x * 4 + warp;
    if (sh >= (int64_t)S * H) return;
    const int s = (int)(sh / H), h = (int)(sh - (int64_t)s * H);
    const int ns = base[s + 1] - base[s];
    const int pfx = GROUPS ? (gseq[s] & kGroupMaxPrefixSteps) : 0;   // steps its group read
    const Split sp = make_split((int64_t)H * base[S], a.main_grid, a.L_steps, a.min_chunk_steps);
    const int64_t x0 = (int64_t)H * base[s] + (int64_t)h * ns;
    const int64_t kf = ns ? sp.chunk(x0) : 0, kl = ns ? sp.chunk(x0 + ns - 1) : 0;
    if (ns > 0 && kf == kl && pfx == 0) return;          // written by the main kernel

    if (!GROUPS && !anchor) grid_dependency_wait();
    // the main kernel writes 0 here when it could not run (workspace too small)
    if (reinterpret_cast<const int64_t*>(a.ws)[0] != sp.Ls) return;
    constexpr int PER = D / 32;
    T* o = static_cast<T*>(a.out) + sh * D + lane * PER;
    if (ns == 0 && pfx == 0) {
#pragma unroll
        for (int e = 0; e < PER; ++e) o[e] = Elem<T>::zero();
        return;
    }
    float M = -INFINITY, ls = 0.f, acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    // fold partial slots [first, first + count) of (mlw, accw) into the state
    auto absorb = [&](const float2* mlw, const float* accw, int64_t first, int count) {
        for (int k0 = 0; k0 < count; k0 += kMergeBatch) {
            float2 mv[kMergeBatch];
            float av[kMergeBatch][PER];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                if (k0 + u < count) {
                    const int64_t k = first + k0 + u;
                    mv[u] = mlw[k];
                    const float* r = accw + k * D + lane * PER;
                    if constexpr (PER == 4) {
                        const float4 f = *reinterpret_cast<const float4*>(r);
                        av[u][0] = f.x; av[u][1] = f.y; av[u][2] = f.z; av[u][3] = f.w;
                    } else {
                        const float2 f = *reinterpret_cast<const float2*>(r);
                        av[u][0] = f.x; av[u][1] = f.y;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                if (k0 + u < count) {
                    if (mv[u].x > M) {
                        const float r = exp2f(M - mv[u].x);
                        ls *= r;
#pragma unroll
                        for (int e = 0; e < PER; ++e) acc[e] *= r;
                        M = mv[u].x;
                    }
                    const float sc = exp2f(mv[u].x - M);
                    ls = fmaf(sc, mv[u].y, ls);
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[e] = fmaf(sc, av[u][e], acc[e]);
                }
            }
        }
    };
    if (GROUPS && pfx > 0) {
        // the group's partials of this member and head: one per unit
        const int nc = (pfx + LG - 1) / LG;
        const int64_t g0 =
            (int64_t)reinterpret_cast<const int*>(a.ws + a.ws_l.gslot_off)[s] + (int64_t)h * nc;
        absorb(reinterpret_cast<const float2*>(a.ws + a.ws_l.gml_off),
               reinterpret_cast<const float*>(a.ws + a.ws_l.gacc_off), g0, nc);
    }
    if (ns > 0)
        absorb(reinterpret_cast<const float2*>(a.ws + a.ws_l.ml_off) + sh,
               reinterpret_cast<const float*>(a.ws + a.ws_l.acc_off) + sh * D, kf,
               (int)(kl - kf + 1));
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = Elem<T>::from_f32(acc[e] / ls);
}

// ------------------------------------------------------------ host glue
constexpr int kLimitDevices = 64;

template <typename T, int D, int B, int MODE = kModePaged>
struct Launcher {
    using C = Cfg<D, B>;
    static constexpr bool GROUPS = MODE == kModeShared;
    static size_t smem_bytes(int S) { return C::smem(S) + (GROUPS ? 4 * (size_t)(S + 1) : 0); }
    static size_t merge_smem(int S) { return 4 * (size_t)(S + 1 + 8); }
    static size_t groups_smem(int S) { return 4 * (8 * (size_t)S + 2 + 64); }
    // The dynamic shared memory limit of a kernel also steers the L1/shared
    // carveout the driver picks for it: with the limit at the device maximum
    // every launch got the largest carveout (228 KiB, the least L1), whatever
    // its batch needed.  So each kernel's limit is kept at exactly the size
    // of the launch in hand, re-set when the batch size changes, with the
    // lock held across the launch so that concurrent host threads with
    // different batch sizes cannot undercut each other.
    struct Limits {
        std::mutex mu;
        int main[kLimitDevices] = {};
        int merge[kLimitDevices] = {};
        int groups[kLimitDevices] = {};
    };
    static Limits& limits() {
        static Limits l;
        return l;
    }
    static cudaError_t set_limit(int* cur, const void* fn, size_t bytes) {
        if (*cur == (int)bytes) return cudaSuccess;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
        if (e == cudaSuccess) *cur = (int)bytes;
        return e;
    }
    static cudaError_t occupancy(int* ctas, size_t smem) {
        int dev = 0, max_optin = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kLimitDevices) return cudaErrorInvalidDevice;
        e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        if (smem > (size_t)max_optin) {
            *ctas = 0;
            return cudaSuccess;
        }
        Limits& L = limits();
        std::lock_guard<std::mutex> lk(L.mu);
        e = set_limit(&L.main[dev], (const void*)paged_decode_main<T, D, B, MODE>, smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, paged_decode_main<T, D, B, MODE>,
                                                             C::THREADS, smem);
    }
    // Every kernel is launched as a programmatic dependent of its predecessor
    // in the stream: each waits (griddepcontrol.wait) before it reads anything,
    // so only the launch latency overlaps the predecessor.  With shared
    // prefixes the group pass (kGroupPassCtas CTAs) runs first.
    static cudaError_t launch(const DecodeArgs& args, int grid, cudaStream_t stream,
                              const CUtensorMap& tk, const CUtensorMap& tv) {
        DecodeArgs a = args;
        a.main_grid = grid;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kLimitDevices) return cudaErrorInvalidDevice;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        Limits& L = limits();
        std::lock_guard<std::mutex> lk(L.mu);
        if constexpr (GROUPS) {
            cfg.gridDim = dim3(kGroupPassCtas);
            cfg.blockDim = dim3(kGroupPassThreads);
            cfg.dynamicSmemBytes = groups_smem(a.S);
            e = set_limit(&L.groups[dev], (const void*)paged_decode_groups<D, B>,
                          cfg.dynamicSmemBytes);
            if (e != cudaSuccess) return e;
            e = cudaLaunchKernelEx(&cfg, paged_decode_groups<D, B>, a);
            if (e != cudaSuccess) return e;
        }
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = smem_bytes(a.S);
        e = set_limit(&L.main[dev], (const void*)paged_decode_main<T, D, B, MODE>, cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, paged_decode_main<T, D, B, MODE>, tk, tv, a);
        if (e != cudaSuccess) return e;
        const int64_t warps = (int64_t)a.S * a.H;
        cfg.gridDim = dim3((unsigned)((warps + 3) / 4));
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = merge_smem(a.S);
        e = set_limit(&L.merge[dev], (const void*)paged_decode_merge<T, D, B, MODE>, cfg.dynamicSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, paged_decode_merge<T, D, B, MODE>, a);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    static const DecodeKernel* get() {
        static const DecodeKernel k = {&launch, &smem_bytes, &occupancy, C::THREADS};
        return &k;
    }
};

}  // namespace dec
}  // namespace pkv
