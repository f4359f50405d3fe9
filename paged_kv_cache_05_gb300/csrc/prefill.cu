// Prompt-phase (prefill) attention over the paged cache, on the fifth-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes (wywy.jp notes, "prompt phase": every prompt token is
// known, so attention runs as matrix-matrix work; the block-indexed attention
// of the zhaifeiyue.github.io detail page, paper section 4.1, per query row):
// sequence s has qlen new tokens, already written to the cache at positions
// ctx - qlen .. ctx - 1; query token i (position p = ctx - qlen + i) attends
// positions 0 .. p (causal):
//   out[i][h] = sum_{t <= p} softmax_t(scale * q[i][h] . K[t][h]) V[t][h].
//
// Design.  Persistent CTAs, one per SM, walk the work items (128 query rows
// of one (sequence, head); one query row per tensor-memory lane) longest
// first; loads and products run ahead across item boundaries.  Eleven warps:
//   warps 0, 10 TMA producers: the query tile of each item and the K tiles
//               (warp 0), the V tiles (warp 10), 128 keys per tile, block by
//               block through the block table (2-D tiled copies with the
//               128-byte swizzle), each in a ring of two stages; a K stage is
//               refilled once its S product is done, a V stage once its P V is;
//   warp 1      owns the tensor memory and issues the MMAs from one thread:
//               S_j = Q K_j^T into one of two S buffers (128 x 128 fp32), and
//               O += P_j V_j into the O accumulator (128 x D fp32);
//   warps 2..9  softmax, two warps per row quarter, each taking half of the
//               keys of a tile and half of O's columns: read S_j from tensor
//               memory, causal mask (diagonal tiles only), online softmax in
//               log2 units (the two halves agree on the running max through
//               tensor memory), write P_j (16-bit) to shared memory in the
//               MMA's operand layout, rescale O in tensor memory when the
//               running max grows.
// S_{j+1} is computed while the softmax works on S_j.  The running max is
// only raised when a row's max grows by more than 2^8 (the weights then stay
// below 256), so most tiles need no O rescale; the result is the same softmax.
// For bf16, P = high part + residual (two products), so the weights keep
// about 16 bits.
//
// Operand layouts (shared memory, 1024-byte aligned atoms of 8 rows x 128 B,
// 16-byte chunk c of row r stored at chunk c ^ (r % 8)):
//   Q, K: K-major (row = token, 64 elements of the head dimension per slab);
//   P:    K-major (row = query, 64 keys per slab);
//   V:    the same bytes as K, read as an MN-major operand (N = head dimension).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr int kBM = 128;            // query rows per CTA (MMA M, tensor-memory lanes)
constexpr int kBN = 128;            // keys per tile (MMA N of S, K of P V)
constexpr int kWarps = 11;          // K producer, MMA issuer, 8 softmax warps, V producer
constexpr int kThreads = kWarps * 32;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256, 256+D), exchange
constexpr uint32_t kColO = 256;
constexpr uint32_t kColX = 384;      // per-row exchange between the two softmax halves
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past this growth
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;

template <int D>
struct PCfg {
    static constexpr int SLABS = D / 64;               // 128-byte slabs per K/Q row
    static constexpr int SLAB_Q = kBM * 128;           // bytes of one Q slab
    static constexpr int SLAB_KV = kBN * 128;          // bytes of one K (or V) slab
    static constexpr int SLAB_P = kBM * 128;           // bytes of one P slab (64 keys)
    static constexpr int KV_BYTES = SLABS * SLAB_KV;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + SLABS * SLAB_Q;
    static constexpr int V_OFF = K_OFF + 2 * KV_BYTES;
    static constexpr int P_OFF = V_OFF + 2 * KV_BYTES;
    static constexpr int PLO_OFF = P_OFF + 2 * SLAB_P;   // bf16 residual of P
    static constexpr int bar_off(bool split) { return PLO_OFF + (split ? 2 * SLAB_P : 0); }
    // dynamic shared memory: 1 KiB of alignment slack, the buffers, 256 B of
    // barriers; never below 116 KiB so that one CTA holds an SM (each CTA
    // allocates 512 tensor-memory columns, the SM's whole tensor memory)
    static constexpr size_t smem(bool split) {
        const size_t n = 1024 + (size_t)bar_off(split) + 256;
        return n < (116u << 10) ? (116u << 10) : n;
    }
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity.  Gives up (false) after
// 1 s, after kWaitLimitIters polls, or once *abort is set (when given).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it < kWaitLimitIters; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (abort && *abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try(bar, parity)) return true;
    return wait_slow(bar, parity, abort);
}

// 2-D / 3-D tiled bulk tensor copies global -> shared, completion in bytes on `bar`.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                       uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), the fixed version bit 46, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both f16 (0)
// or both bf16 (1), A K-major, B K-major or MN-major, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc(uint32_t ab_type, bool b_mn_major, int n, int m) {
    return (1u << 4) | (ab_type << 7) | (ab_type << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive columns of this warp's 32 lanes (thread i: lane base + i),
// load and wait in one statement so that no use of the registers can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Store 32 columns of this warp's lanes and wait for the store to complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
        "%27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One column of this warp's lanes, stored (and waited for) / loaded.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(v))
        : "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
    uint32_t v;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v)
        : "r"(taddr)
        : "memory");
    return __uint_as_float(v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// ------------------------------------------------------------ element types
template <typename T>
struct Pk;

template <>
struct Pk<__half> {
    static constexpr uint32_t kType = 0;
    static constexpr bool kSplit = false;     // fp16 weights keep 11 bits
    static __device__ __forceinline__ uint32_t pack(float lo, float hi, uint32_t& res) {
        __half2 v = __floats2half2_rn(lo, hi);
        res = 0u;
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ uint32_t pack_out(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

template <>
struct Pk<__nv_bfloat16> {
    static constexpr uint32_t kType = 1;
    static constexpr bool kSplit = true;      // bf16 weights: high part + residual
    static __device__ __forceinline__ uint32_t pack(float lo, float hi, uint32_t& res) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        const __nv_bfloat162 r = __floats2bfloat162_rn(lo - __low2float(h), hi - __high2float(h));
        res = *reinterpret_cast<const uint32_t*>(&r);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    static __device__ __forceinline__ uint32_t pack_out(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

struct PrefillArgs {
    void* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;
    float scale_log2;
    int S, H, B, max_blocks, max_query_len, num_tokens;
    int q_tiles;             // query tiles per sequence: ceil(max_query_len / kBM)
    int64_t num_blocks;
    int32_t* err;
};

// barrier slots (8 bytes each) in the barrier region
enum : int {
    kBarQFull = 0,
    kBarQEmpty = 1,
    kBarKFull = 2,    // + stage
    kBarKEmpty = 4,   // + stage
    kBarVFull = 6,    // + stage
    kBarVEmpty = 8,   // + stage
    kBarSFull = 10,   // + buffer
    kBarPFull = 12,
    kBarPvDone = 13,
    kBarMmaDone = 14,
    kBarXch = 15,     // + lane quarter: the two softmax warps of a quarter
    kBarCount = 19
};

// One work item: 128 query rows of one (sequence, head).
struct Item {
    int s, h, q0, qlen, ctx, q_begin, rows, pos0, n_tiles;
};

// Work items in longest-first order: index w -> query tile q_tiles-1 - w/(S H),
// then sequence, then head.  False for an empty item (past the sequence's
// query rows) or a sequence whose lengths are out of range (flagged once).
__device__ __forceinline__ bool item_at(const PrefillArgs& a, int64_t w, bool flag, Item& it) {
    const int64_t sh = (int64_t)a.S * a.H;
    const int t = a.q_tiles - 1 - (int)(w / sh);
    const int64_t rem = w - (w / sh) * sh;
    it.s = (int)(rem / a.H);
    it.h = (int)(rem - (int64_t)it.s * a.H);
    it.q0 = a.query_start[it.s];
    it.qlen = a.query_start[it.s + 1] - it.q0;
    it.ctx = a.context_lens[it.s];
    if (it.ctx < 0 || it.ctx > a.max_blocks * a.B || it.qlen < 0 || it.qlen > it.ctx ||
        it.q0 < 0 || (int64_t)it.q0 + it.qlen > a.num_tokens) {
        if (flag && t == 0 && it.h == 0) atomicOr(a.err, PKV_DEVERR_BAD_CONTEXT);
        return false;
    }
    if (flag && t == 0 && it.h == 0 && it.qlen > a.max_query_len)
        atomicOr(a.err, PKV_DEVERR_BAD_CONTEXT);     // rows past the last tile stay unwritten
    it.q_begin = t * kBM;
    if (it.q_begin >= it.qlen) return false;
    it.rows = min(kBM, it.qlen - it.q_begin);
    it.pos0 = it.ctx - it.qlen + it.q_begin;         // position of the item's first query
    it.n_tiles = (it.pos0 + it.rows - 1) / kBN + 1;  // key tiles up to the causal limit
    return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tc(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    using C = PCfg<D>;
    constexpr bool kSplit = Pk<T>::kSplit;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;                 // 1024-aligned
    unsigned char* gbase = smem_raw + (base - raw);               // same, generic
    const uint32_t sQ = base + C::Q_OFF, sK = base + C::K_OFF, sV = base + C::V_OFF;
    const uint32_t sP = base + C::P_OFF, sPlo = base + C::PLO_OFF;
    const uint32_t bars = base + C::bar_off(kSplit);
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::bar_off(kSplit) + 8 * kBarCount);
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(gbase + C::bar_off(kSplit) + 8 * kBarCount + 4);

    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_items = (int64_t)a.q_tiles * a.S * a.H;
    const int64_t w0 = blockIdx.x, dw = gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < kBarCount; ++i)
            mbar_init(bar(i), i == kBarPFull ? (uint32_t)kSoftmaxThreads : i >= kBarXch ? 64u : 1u);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() {
        if (!*abort_flag) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0 || warp == kWarps - 1) {
        // ============================================ TMA producers
        // warp 0: the query tiles and the K tiles; the last warp: the V tiles.
        // Both walk the same items and the same global tile sequence g; tile g
        // uses stage g & 1 of its ring.
        const bool kq = warp == 0;
        if (lane == 0) {
            const CUtensorMap* map = kq ? &tm_k : &tm_v;
            const uint32_t ring = kq ? sK : sV;
            const int full0 = kq ? kBarKFull : kBarVFull, empty0 = kq ? kBarKEmpty : kBarVEmpty;
            int64_t g = 0;
            int items = 0;
            bool ok = true;
            for (int64_t w = w0; ok && w < n_items; w += dw) {
                Item it;
                if (!item_at(a, w, false, it)) continue;
                if (kq) {
                    // the query tile, once the previous item's S products are done
                    if (items > 0 && !mbar_wait(bar(kBarQEmpty), (items - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar(kBarQFull), (uint32_t)(C::SLABS * C::SLAB_Q));
                    for (int sl = 0; sl < C::SLABS; ++sl)
                        tma_3d(sQ + sl * C::SLAB_Q, &tm_q, sl * 64, it.h, it.q0 + it.q_begin,
                               bar(kBarQFull));
                }
                ++items;
                const int32_t* row_tab = a.block_tables + (int64_t)it.s * a.max_blocks;
                for (int j = 0; j < it.n_tiles; ++j, ++g) {
                    const int st = (int)(g & 1);
                    if (g >= 2 &&
                        !mbar_wait(bar(empty0 + st), (uint32_t)(((g >> 1) - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int tok0 = j * kBN;
                    const int tok1 = min(tok0 + kBN, it.ctx);  // tokens of the tile in the context
                    const int jb0 = tok0 / a.B, jb1 = (tok1 - 1) / a.B;
                    mbar_expect_tx(bar(full0 + st), (uint32_t)((jb1 - jb0 + 1) * a.B * 128 * C::SLABS));
                    for (int jb = jb0; jb <= jb1; ++jb) {
                        int64_t phys = row_tab[jb];
                        if (phys < 0 || phys >= a.num_blocks) {
                            if (kq) atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                            phys = 0;                           // keeps the byte count; flagged
                        }
                        const int y = (int)((phys * a.H + it.h) * a.B);
                        const uint32_t koff = (uint32_t)(jb * a.B - tok0) * 128u;
                        for (int sl = 0; sl < C::SLABS; ++sl)
                            tma_2d(ring + st * C::KV_BYTES + sl * C::SLAB_KV + koff, map, sl * 64,
                                   y, bar(full0 + st));
                    }
                }
            }
            if (!ok) fail();
            if (*abort_flag) {
                // let the copies in flight land before the CTA can exit
                if (kq && items > 0) mbar_wait(bar(kBarQFull), (items - 1) & 1, nullptr);
                for (int64_t t = g - 2 < 0 ? 0 : g - 2; t < g; ++t)
                    mbar_wait(bar(full0 + (int)(t & 1)), (uint32_t)((t >> 1) & 1), nullptr);
            }
        }
    } else if (warp == 1) {
        // ======================================================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc(Pk<T>::kType, false, kBN, kBM);
            constexpr uint32_t ID_PV = idesc(Pk<T>::kType, true, D, kBM);
            // S_g for global tile g (j = its index in the item, item = the
            // item count); the last S of an item frees the query buffer
            auto issue_s = [&](int64_t g, int j, int n_tiles, int item) -> bool {
                if (j == 0 && !mbar_wait(bar(kBarQFull), (uint32_t)(item & 1), abort_flag))
                    return false;
                const int st = (int)(g & 1);
                if (!mbar_wait(bar(kBarKFull + st), (uint32_t)((g >> 1) & 1), abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)st * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * C::SLAB_Q + (uint32_t)(kk & 3) * 32u;
                    const uint32_t koff =
                        (uint32_t)(kk >> 2) * C::SLAB_KV + (uint32_t)(kk & 3) * 32u;
                    umma(d, sdesc(sQ + off, 16, 1024),
                         sdesc(sK + st * C::KV_BYTES + koff, 16, 1024), ID_S, kk > 0);
                }
                umma_commit(bar(kBarSFull + st));
                umma_commit(bar(kBarKEmpty + st));
                if (j == n_tiles - 1) umma_commit(bar(kBarQEmpty));
                return true;
            };
            // S runs up to two tiles ahead of P V, across item boundaries: a
            // cursor (item, tile) over the same sequence the others walk
            int64_t sw = w0;                 // item of the next S
            Item sit;
            int sj = 0, sitem = 0;           // tile within it, item count
            int64_t gs = 0;                  // global index of the next S
            bool s_has = false;
            auto s_next_item = [&]() {
                s_has = false;
                while (sw < n_items) {
                    const bool v = item_at(a, sw, true, sit);
                    sw += dw;
                    if (v) {
                        s_has = true;
                        sj = 0;
                        return;
                    }
                }
            };
            auto s_issue_one = [&]() -> bool {
                if (!s_has) return true;
                if (!issue_s(gs, sj, sit.n_tiles, sitem)) return false;
                ++gs;
                if (++sj == sit.n_tiles) {
                    ++sitem;
                    s_next_item();
                }
                return true;
            };
            s_next_item();
            bool ok = s_issue_one() && s_issue_one();
            int64_t g = 0;
            for (int64_t w = w0; ok && w < n_items; w += dw) {
                Item it;
                if (!item_at(a, w, false, it)) continue;
                for (int j = 0; j < it.n_tiles; ++j, ++g) {
                    if (!mbar_wait(bar(kBarPFull), (uint32_t)(g & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int st = (int)(g & 1);
                    if (!mbar_wait(bar(kBarVFull + st), (uint32_t)((g >> 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t vst = sV + st * C::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint32_t poff =
                            (uint32_t)(kk >> 2) * C::SLAB_P + (uint32_t)(kk & 3) * 32u;
                        const uint64_t vd = sdesc(vst + (uint32_t)kk * 2048u, C::SLAB_KV, 1024);
                        umma(tmem + kColO, sdesc(sP + poff, 16, 1024), vd, ID_PV,
                             (j > 0 || kk > 0));
                        if constexpr (kSplit)
                            umma(tmem + kColO, sdesc(sPlo + poff, 16, 1024), vd, ID_PV, 1u);
                    }
                    umma_commit(bar(kBarVEmpty + st));
                    umma_commit(bar(kBarPvDone));
                    if (!s_issue_one()) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) fail();
            // every MMA issued has completed before the CTA moves on
            umma_commit(bar(kBarMmaDone));
            mbar_wait(bar(kBarMmaDone), 0, nullptr);
        }
    } else {
        // ======================================================= softmax
        // Warps 2..9.  Warps w and w + 4 share a lane quarter (the rows
        // 32 (w % 4) .. + 31) and split the keys of each tile: half 0 takes
        // keys 0..63 (P slab 0) and O's first D/2 columns, half 1 the rest.
        // The two agree on the running max through tensor memory once per tile.
        const int q4 = warp & 3;                     // this warp's lane quarter
        const int half = (warp - 2) >> 2;
        const int row = q4 * 32 + lane;              // query row of the item = TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const int stid = tid - 64;                   // 0..255 among the softmax threads
        const uint32_t xbar = bar(kBarXch + q4);     // the two warps' exchange barrier
        int xphase = 0;
        // publish v in this half's slot, wait for the other half, return its value
        auto exchange = [&](float v, int slot_self, int slot_other, float& other) -> bool {
            tmem_st1(tl + kColX + (uint32_t)slot_self, v);
            tc_fence_before();
            mbar_arrive(xbar);
            const bool got = mbar_wait(xbar, (uint32_t)(xphase & 1), abort_flag);
            ++xphase;
            if (!got) return false;
            tc_fence_after();
            other = tmem_ld1(tl + kColX + (uint32_t)slot_other);
            return true;
        };
        const float sl2 = a.scale_log2;
        const bool pos_scale = sl2 >= 0.f;
        bool ok = true;
        int64_t g = 0;
        for (int64_t w = w0; ok && w < n_items; w += dw) {
            Item it;
            if (!item_at(a, w, false, it)) continue;
            const int qpos = it.pos0 + row;          // causal limit of the row
            float m = -INFINITY, l = 0.f;            // l: this half's share of the row sum
            for (int j = 0; j < it.n_tiles; ++j, ++g) {
                const int st = (int)(g & 1);
                if (!mbar_wait(bar(kBarSFull + st), (uint32_t)((g >> 1) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sb = tl + (uint32_t)st * kBN + (uint32_t)half * 64;
                const int kb = j * kBN + half * 64;      // first key of this half
                const bool full = kb + 63 <= it.pos0;    // every key visible to every row
                // row max of this half (scaled scores; masked keys excluded)
                float mx = -INFINITY;
                if (full) {
                    float ext = pos_scale ? -INFINITY : INFINITY;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t r[32];
                        tmem_ld32(sb + c * 32, r);
                        if (pos_scale) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) ext = fmaxf(ext, __uint_as_float(r[e]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) ext = fminf(ext, __uint_as_float(r[e]));
                        }
                    }
                    mx = ext * sl2;
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t r[32];
                        tmem_ld32(sb + c * 32, r);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (kb + c * 32 + e <= qpos)
                                mx = fmaxf(mx, __uint_as_float(r[e]) * sl2);
                    }
                }
                {
                    // slots alternate with the exchange parity, so a slot is
                    // rewritten only after the other half has passed the next one
                    float other;
                    const int par = xphase & 1;
                    if (!exchange(mx, half * 2 + par, (half ^ 1) * 2 + par, other)) {
                        ok = false;
                        break;
                    }
                    mx = fmaxf(mx, other);
                }
                float m_new = m;
                if (mx > m + kRescaleLog2 || (m == -INFINITY && mx > -INFINITY)) m_new = mx;
                const bool rescale = j > 0 && m_new != m;
                const float alpha = rescale ? ex2(m - m_new) : 1.f;
                // weights of this half, packed to 16 bits (and the bf16 residual)
                uint32_t pk[32];
                uint32_t pr[kSplit ? 32 : 1];
                float rs = 0.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
                    tmem_ld32(sb + c * 32, r);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float p0 = ex2(fmaf(__uint_as_float(r[e]), sl2, -m_new));
                        float p1 = ex2(fmaf(__uint_as_float(r[e + 1]), sl2, -m_new));
                        if (!full) {
                            const int k0 = kb + c * 32 + e;
                            p0 = k0 <= qpos ? p0 : 0.f;
                            p1 = k0 + 1 <= qpos ? p1 : 0.f;
                        }
                        rs += p0 + p1;
                        uint32_t res;
                        pk[(c * 32 + e) >> 1] = Pk<T>::pack(p0, p1, res);
                        if constexpr (kSplit) pr[(c * 32 + e) >> 1] = res;
                    }
                }
                l = l * alpha + rs;
                m = m_new;
                // P's buffer and O are free once the previous P V has completed
                // (for an item's first tile the previous item's end waited)
                if (j > 0) {
                    if (!mbar_wait(bar(kBarPvDone), (uint32_t)((g - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                // V rows past the context (partial last block, blocks never
                // loaded) are zeroed: their weights are 0, but 0 * NaN would not be
                const int kbase = j * kBN;
                if (kbase + kBN > it.ctx) {
                    if (!mbar_wait(bar(kBarVFull + st), (uint32_t)((g >> 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int z0 = it.ctx - kbase > 0 ? it.ctx - kbase : 0;
                    const int n16 = (kBN - z0) * 8;       // 16-byte chunks per slab
                    unsigned char* vs = gbase + C::V_OFF + st * C::KV_BYTES;
                    for (int i = stid; i < n16 * C::SLABS; i += kSoftmaxThreads) {
                        const int sl = i / n16, wv = i - sl * n16;
                        *reinterpret_cast<uint4*>(vs + sl * C::SLAB_KV + (z0 * 128) + wv * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // this half of the P row -> P slab `half` (K-major, 128-byte swizzle)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t off = (uint32_t)half * C::SLAB_P + (uint32_t)row * 128u +
                                         ((uint32_t)(ch ^ (row & 7)) << 4);
                    st_shared_v4(sP + off, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2],
                                 pk[4 * ch + 3]);
                    if constexpr (kSplit)
                        st_shared_v4(sPlo + off, pr[4 * ch], pr[4 * ch + 1], pr[4 * ch + 2],
                                     pr[4 * ch + 3]);
                }
                // O *= alpha for rows whose running max rose: this half's columns
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        const uint32_t ta = tl + kColO + (uint32_t)(half * (D / 2) + c * 32);
                        uint32_t r[32];
                        tmem_ld32(ta, r);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st32(ta, r);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                mbar_arrive(bar(kBarPFull));
            }
            if (!ok) break;
            // the two halves of the row sum, then the item's output rows
            float other;
            if (!exchange(l, 4 + half, 4 + (half ^ 1), other) ||
                !mbar_wait(bar(kBarPvDone), (uint32_t)((g - 1) & 1), abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            l += other;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T* orow = static_cast<T*>(a.out) +
                      ((int64_t)(it.q0 + it.q_begin + row) * a.H + it.h) * D + half * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[32];
                tmem_ld32(tl + kColO + (uint32_t)(half * (D / 2) + c * 32), r);
                if (row < it.rows) {
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wv[e] = Pk<T>::pack_out(__uint_as_float(r[2 * e]) * inv,
                                                __uint_as_float(r[2 * e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
                }
            }
        }
        if (!ok) fail();
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tiled map of 16-bit elements, 128-byte swizzle, box inner extent 64 elements.
bool make_map(CUtensorMap* m, bool bf16, uint32_t rank, const void* gaddr, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank,
              const_cast<void*>(gaddr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D>
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = PCfg<D>::smem(Pk<T>::kSplit);
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_tc<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    // persistent: one CTA per SM (shared memory and tensor memory allow no
    // more), each walking the work items grid-stride, longest first
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)a.q_tiles * a.S * a.H;
    const int sms = pkv::sm_count(dev);
    if (sms < 1) return cudaErrorInvalidDevice;
    cfg.gridDim = dim3((unsigned)(items < sms ? items : sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, paged_prefill_tc<T, D>, tq, tk, tv, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

bool aligned(const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) & (al - 1)) == 0; }

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_prefill(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       float scale, int num_seqs, int num_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                       int max_query_len, int num_query_tokens, pkv_dtype dtype,
                                       cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_prefill";
    if (num_seqs < 0 || num_seqs > 65535)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_seqs must be in [0, 65535]", fn);
    if (num_heads < 1 || num_heads > 65535)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_heads must be in [1, 65535]", fn);
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "%s: head_dim must be 64 or 128", fn);
    if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64)
        return pkv::fail(PKV_ERR_INVALID, "%s: block_size must be 8, 16, 32 or 64", fn);
    if (max_blocks_per_seq < 1 || num_blocks < 1 || max_query_len < 0 || num_query_tokens < 0)
        return pkv::fail(PKV_ERR_INVALID, "%s: bad sizes", fn);
    if ((int64_t)max_blocks_per_seq * block_size >= (1LL << 31))
        return pkv::fail(PKV_ERR_INVALID, "%s: context capacity overflows", fn);
    // the tiled copies address cache rows (block, head, token) with 32-bit coordinates
    if (num_blocks * num_heads * block_size >= (1LL << 31))
        return pkv::fail(PKV_ERR_INVALID, "%s: pool too large for 32-bit row coordinates", fn);
    if (dtype != PKV_F16 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_INVALID, "%s: dtype", fn);
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0 || max_query_len == 0 || num_query_tokens == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return pkv::fail(PKV_ERR_INVALID, "%s: out, q and the caches must be 16-byte aligned", fn);
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no CUDA device", fn);

    const bool bf16 = dtype == PKV_BF16;
    const cuuint64_t D = (cuuint64_t)head_dim;
    CUtensorMap tq, tk, tv;
    {
        // q: [tokens][heads][D], one box = 128 tokens x 64 elements of one head
        const cuuint64_t dims[3] = {D, (cuuint64_t)num_heads, (cuuint64_t)num_query_tokens};
        const cuuint64_t strides[2] = {D * 2, (cuuint64_t)num_heads * D * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
        if (!make_map(&tq, bf16, 3, q, dims, strides, box))
            return pkv::fail(PKV_ERR_CUDA, "%s: tensor map of q", fn);
    }
    {
        // caches: rows (block, head, token) of D elements, one box = one block's
        // tokens x 64 elements
        const cuuint64_t dims[2] = {D, (cuuint64_t)(num_blocks * num_heads * block_size)};
        const cuuint64_t strides[1] = {D * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)block_size};
        if (!make_map(&tk, bf16, 2, k_cache, dims, strides, box) ||
            !make_map(&tv, bf16, 2, v_cache, dims, strides, box))
            return pkv::fail(PKV_ERR_CUDA, "%s: tensor map of the caches", fn);
    }
    PrefillArgs a;
    a.out = out;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.S = num_seqs;
    a.H = num_heads;
    a.B = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.max_query_len = max_query_len;
    a.num_tokens = num_query_tokens;
    a.q_tiles = (max_query_len + kBM - 1) / kBM;
    a.num_blocks = num_blocks;
    a.err = err;
    cudaError_t e;
    if (!bf16)
        e = head_dim == 128 ? launch_prefill<__half, 128>(tq, tk, tv, a, stream)
                            : launch_prefill<__half, 64>(tq, tk, tv, a, stream);
    else
        e = head_dim == 128 ? launch_prefill<__nv_bfloat16, 128>(tq, tk, tv, a, stream)
                            : launch_prefill<__nv_bfloat16, 64>(tq, tk, tv, a, stream);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

}  // extern "C"
