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
// Design.  Persistent CTAs, one per SM, in pairs (clusters of two, one TPC);
// an item is 256 query rows of one (sequence, head): two query tiles of 128
// rows, one row per tensor-memory lane, that share every K/V tile of 128
// keys.  Each pair takes a contiguous run, of equal estimated cost, of the
// units (sequence, head pair, item; items from the last down), the two CTAs
// the same item of adjacent heads.  The item's tiles go to two slots X = 0, 1
// (a softmax group, its query buffer and tensor-memory columns each), the
// later 128 rows, which see one more (diagonal) key tile, to slot 1 in even
// items and slot 0 in odd ones, and at each key tile the slot with more key
// tiles is served first: the group that ends an item first leads the next.
// Eleven warps:
//   warps 0, 10 TMA producers: the query tiles of each item (the first-served
//               slot's before the item's first K tile) and the K tiles (warp
//               0), the V tiles (warp 10), block by block through the block
//               table (2-D tiled copies with the 128-byte swizzle), each in a
//               ring of 2-4 stages;
//   warp 1      owns the tensor memory and issues the MMAs from one thread:
//               S_X = Q_X K^T (128 x 128 fp32 in tensor memory) and
//               O_X += P_X V with P_X read from tensor memory, where the
//               softmax wrote it over S_X;
//   warps 2..5  softmax of slot 0, warps 6..9 of slot 1, one row per thread:
//               read S from tensor memory, causal mask (diagonal tiles only),
//               online softmax in log2 units, write P (16-bit, packed in
//               pairs) back over S, rescale O when the running max grows.
// The two groups ping-pong: while one group's softmax runs, the tensor cores
// compute the other group's products.  The MMAs of one thread complete in
// issue order, so S_X(j+1) (issued after O_X += P_X(j) V) finding its
// barrier complete means that P V has completed too.  The running max is
// only raised when a row's max grows by more than 2^8 (the weights then stay
// below 256), so most tiles need no O rescale; the result is the same
// softmax.  For bf16, P = high part + residual (two products), so the
// weights keep about 16 bits.
//
// Operand layouts: Q, K in shared memory K-major (row = token, 64 elements
// of the head dimension per 128-byte slab, 1024-byte atoms of 8 rows, 16-byte
// chunk c of row r at chunk c ^ (r % 8)); V the same bytes read as an
// MN-major operand (N = head dimension); P in tensor memory, row = lane, keys
// 32 q + 2c and 32 q + 2c + 1 in column 32 q + c (bf16 residuals 16 further).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "pkv_internal.h"

namespace {

constexpr int kBM = 128;            // query rows per tile (MMA M, tensor-memory lanes)
constexpr int kRows = 2 * kBM;      // query rows per work item (two query tiles)
constexpr int kBN = 128;            // keys per K/V tile (MMA N of S, K of P V)
constexpr int kWarps = 11;          // K producer, MMA issuer, 2 x 4 softmax warps, V producer
constexpr int kThreads = kWarps * 32;
// With the prompt's K/V read from the input tensors (FUSED), a twelfth warp
// writes them into the paged cache.
constexpr int kWriterWarp = kWarps;
__host__ __device__ constexpr int threads_for(bool fused) { return (kWarps + (fused ? 1 : 0)) * 32; }
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: S_X (and P_X over it) at X kBN, O_X at kColO + X D;
// P_X: keys 32 q .. + 31 packed in pairs in the columns 32 q .. + 15 of S_X,
// their bf16 residuals in 32 q + 16 .. + 31
constexpr uint32_t kColO = 2 * kBN;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past this growth
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;

template <int D, bool SPLIT>
struct PCfg {
    static constexpr int SLABS = D / 64;               // 128-byte slabs per K/Q row
    static constexpr int SLAB_Q = kBM * 128;           // bytes of one Q slab (one tile)
    static constexpr int SLAB_KV = kBN * 128;          // bytes of one K (or V) slab
    static constexpr int Q_BYTES = SLABS * SLAB_Q;     // one tile's Q
    static constexpr int KV_BYTES = SLABS * SLAB_KV;
    // K and V ring depth: as deep as shared memory allows
    static constexpr int NST = D == 128 ? 2 : 4;
    static constexpr int Q_OFF = 0;                    // Q_A, Q_B
    static constexpr int K_OFF = Q_OFF + 2 * Q_BYTES;
    static constexpr int V_OFF = K_OFF + NST * KV_BYTES;
    static constexpr int BAR_OFF = V_OFF + NST * KV_BYTES;
    // dynamic shared memory: 1 KiB of alignment slack, the buffers, 256 B of
    // barriers; never below 116 KiB so that one CTA holds an SM (each CTA
    // allocates 512 tensor-memory columns, the SM's whole tensor memory)
    static constexpr size_t SMEM_NEED = 1024 + (size_t)BAR_OFF + 512;
    static constexpr size_t SMEM = SMEM_NEED < (116u << 10) ? (116u << 10) : SMEM_NEED;
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(kColO + 2 * D <= kTmemCols, "tensor memory columns");
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

// One test of the phase.  With SUSPEND a thread whose phase is not complete
// is suspended (up to the hint, 1 ms) until it completes, so waiting threads
// do not take issue slots from the softmax warps beside them; without it the
// test returns at once (for the MMA issuer, whose reaction time is on the
// critical path).
template <bool SUSPEND>
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    if (SUSPEND)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(1000000u)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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
// 1 s, after kWaitLimitIters tests, or once *abort is set (when given; a
// suspended test notices it after its hint at the latest).
template <bool SUSPEND>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; it < kWaitLimitIters; ++it) {
        if (mbar_try<SUSPEND>(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (abort && *abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    return false;
}

template <bool SUSPEND = true>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try<SUSPEND>(bar, parity)) return true;
    return wait_slow<SUSPEND>(bar, parity, abort);
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

// 2-D tiled bulk tensor copy shared -> global (the map's swizzle applies to
// the shared-memory side), in this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until the shared memory read by this thread's committed bulk stores
// may be reused / until those stores have completed
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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

// The same with A read from tensor memory (M rows = lanes, K packed in pairs
// along the columns).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
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

// 64 columns, load issued without waiting (tmem_wait64 completes it)
__device__ __forceinline__ void tmem_ld64_nw(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr)
                 : "memory");
}
// wait for this thread's tensor-memory loads; r counts as written here, so
// nothing reads it earlier
__device__ __forceinline__ void tmem_wait64(uint32_t (&r)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63]) : : "memory");
}

// Store 16 columns of this warp's lanes and wait for the store to complete.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
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

// Pairs of fp32 values in one 64-bit register, and the packed fp32 FMA and
// add that work on both halves at once.
__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 32 bytes to global memory in one instruction (32-byte aligned address)
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// max / min of three values in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
    void* k_cache;               // (FUSED: the cache writer's plain stores)
    void* v_cache;
    int out_v8;                  // out is 32-byte aligned: 32-byte stores
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;
    float scale_log2;
    int S, H, B, max_blocks, max_query_len, num_tokens;
    int q_items;             // work items per sequence: ceil(max_query_len / kRows)
    int64_t num_blocks;
    int32_t* err;
};

// barrier slots (8 bytes each) in the barrier region
enum : int {
    kBarQFull = 0,    // + slot: its query tile of the item loaded
    kBarQEmpty = 2,   // + slot: its last S of the item done
    kBarKFull = 4,    // + stage (up to 4)
    kBarKEmpty = 8,   // + stage
    kBarVFull = 12,   // + stage
    kBarVEmpty = 16,  // + stage
    kBarSFull = 20,   // + group: S_X computed (and every earlier product)
    kBarPFull = 22,   // + group: P_X written, O_X rescaled
    kBarPvDone = 24,  // + group: an item's last O_X += P_X V completed
    kBarMmaDone = 26,
    kBarKStored = 27, // + stage: the cache writer is done with a K stage (FUSED)
    kBarVStored = 31, // + stage: ... with a V stage
    kBarCount = 35
};

// One work item: 256 query rows (two query tiles) of one (sequence, head).
struct Item {
    int s, h, q0, qlen, ctx, q_begin;
    int sw;                          // slot x holds rows (x ^ sw) * 128 .. + 127 of the item
    int rows[2], pos0[2], n[2];      // per slot: rows, first position, key tiles
    int n_kv;                        // key tiles loaded: the larger of n[0], n[1]
    int f;                           // the slot served first at each key tile
};

// Lengths of one sequence and its number of items (0 for a sequence whose
// lengths are out of range, or, with whole, not a whole prompt).
struct SeqInfo {
    int q0, qlen, ctx, ni;
};
__device__ __forceinline__ bool seq_info(const PrefillArgs& a, int s, bool whole, SeqInfo& si) {
    si.q0 = a.query_start[s];
    si.qlen = a.query_start[s + 1] - si.q0;
    si.ctx = a.context_lens[s];
    si.ni = 0;
    if (si.ctx < 0 || si.ctx > a.max_blocks * a.B || si.qlen < 0 || si.qlen > si.ctx ||
        si.q0 < 0 || (int64_t)si.q0 + si.qlen > a.num_tokens || (whole && si.qlen != si.ctx))
        return false;
    const int n = (si.qlen + kRows - 1) / kRows;   // rows past the last item stay unwritten
    si.ni = n < a.q_items ? n : a.q_items;
    return true;
}

// Item t of a sequence: per slot (query group) its tile's rows, first
// position and key tiles.  Odd items put the later 128 rows (the tile with the
// extra, diagonal key tile) in slot 0, even ones in slot 1, and the slot with
// more key tiles is served first: the group that finishes an item first (the
// one with fewer key tiles) takes the longer tile of the next item and leads
// it, while the other still works through its diagonal tile and output rows.
__device__ __forceinline__ void item_tiles(const SeqInfo& si, int t, Item& it) {
    it.q_begin = t * kRows;
    it.sw = t & 1;
    for (int x = 0; x < 2; ++x) {
        const int b = it.q_begin + (x ^ it.sw) * kBM;
        it.rows[x] = si.qlen - b < kBM ? (si.qlen - b > 0 ? si.qlen - b : 0) : kBM;
        it.pos0[x] = si.ctx - si.qlen + b;            // position of the tile's first query
        it.n[x] = it.rows[x] > 0 ? (it.pos0[x] + it.rows[x] - 1) / kBN + 1 : 0;
    }
    it.n_kv = it.n[1] > it.n[0] ? it.n[1] : it.n[0];
    it.f = it.n[1] > it.n[0] ? 1 : 0;
}

// Estimated cost of an item, in tenths of a 128 x 128 tile product issued
// beside the other query tile's: a key tile both query tiles see costs 20, one
// that only one of them sees 17 (its softmax, products and hand-offs then run
// with nothing to overlap them), and the item's fixed work (its query load,
// first products and output) 24.  Fitted to the per-CTA times of 16 prompts
// of 543-1729 tokens (40 heads x 128) under several schedules.
constexpr int kPairCost = 20, kSoloCost = 17, kItemCost = 24;
__device__ __forceinline__ int item_cost(const SeqInfo& si, int t) {
    Item it;
    item_tiles(si, t, it);
    const int lo = it.n[0] < it.n[1] ? it.n[0] : it.n[1];
    const int hi = it.n[0] < it.n[1] ? it.n[1] : it.n[0];
    return kPairCost * lo + kSoloCost * (hi - lo) + kItemCost;
}

// Work schedule.  A unit is item t of heads 2 hp and 2 hp + 1 of sequence s,
// one head for each CTA of a pair (clusters of two); the units are ordered by
// sequence, head pair, then t from the last item down, and each CTA pair takes
// a contiguous run of them of equal estimated cost: unit u, whose cost c_u
// follows P_u of cost before it, belongs to pair k when
// th(k) <= 2 P_u + c_u < th(k + 1), th(k) = floor(2 k P_total / pairs), where
// P_total is the cost of all units.  A CTA thus works on one (sequence, head)
// at a time, item after item, each item finding in L2 the K/V tiles the one
// before it loaded, and the two CTAs of a pair run the same item shapes side
// by side.
struct Sched {
    int s, hp;         // first unit that may belong to the pair: (s, hp, last item)
    int64_t P;         // cost of the units before it
    int64_t lo, hi;    // the pair's thresholds th(k), th(k + 1)
};

struct Walker {
    int s, hp, ti;     // the next unit: (sequence, head pair, items from the last)
    int64_t P;         // cost of the units before it
    __device__ __forceinline__ void init(const Sched& sc) {
        s = sc.s;
        hp = sc.hp;
        ti = 0;
        P = sc.P;
    }
    // the pair's next unit, as this CTA's item (its head 2 hp + rank)
    __device__ __forceinline__ bool next(const PrefillArgs& a, const Sched& sc, bool whole,
                                         Item& it) {
        const int HP = (a.H + 1) >> 1;
        const int rank = (int)(blockIdx.x & 1u);
        while (s < a.S) {
            SeqInfo si;
            seq_info(a, s, whole, si);
            if (si.ni == 0) {                         // no items: the next sequence
                ++s;
                hp = 0;
                ti = 0;
                continue;
            }
            const int t = si.ni - 1 - ti;
            const int c = item_cost(si, t);
            item_tiles(si, t, it);
            const int64_t v = 2 * P + c;
            if (v >= sc.hi) {
                s = a.S;
                return false;
            }
            const int h = 2 * hp + rank;
            const bool mine = v >= sc.lo && h < a.H;
            it.s = s;
            it.h = h;
            it.q0 = si.q0;
            it.qlen = si.qlen;
            it.ctx = si.ctx;
            P += c;
            if (++ti == si.ni) {
                ti = 0;
                if (++hp == HP) {
                    ++s;
                    hp = 0;
                }
            }
            if (mine) return true;
        }
        return false;
    }
};

// Locates the pair's first unit (one warp; every CTA computes the same
// total).  CTA 0 flags each sequence whose lengths are out of range, or
// whose rows pass max_query_len (those rows stay unwritten).
__device__ __forceinline__ void plan(const PrefillArgs& a, bool whole, Sched* out, int lane) {
    const int HP = (a.H + 1) >> 1;
    long long tot = 0;
    for (int s0 = 0; s0 < a.S; s0 += 32) {
        const int s = s0 + lane;
        if (s >= a.S) break;
        SeqInfo si;
        const bool good = seq_info(a, s, whole, si);
        if (blockIdx.x == 0 && (!good || si.qlen > a.max_query_len))
            atomicOr(a.err, PKV_DEVERR_BAD_CONTEXT);
        for (int t = 0; t < si.ni; ++t) tot += item_cost(si, t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    tot *= HP;
    const int64_t np = gridDim.x >> 1, k = blockIdx.x >> 1;
    const int64_t A = 2 * (int64_t)tot;
    const int64_t lo = k * (A / np) + (k * (A % np)) / np;
    const int64_t hi = (k + 1) * (A / np) + ((k + 1) * (A % np)) / np;
    // the first sequence whose units reach past lo
    int fs = a.S;
    int64_t fP = 0, fT = 0;
    long long carry = 0;
    for (int s0 = 0; s0 < a.S && fs == a.S; s0 += 32) {
        const int s = s0 + lane;
        long long ts = 0;
        if (s < a.S) {
            SeqInfo si;
            seq_info(a, s, whole, si);
            for (int t = 0; t < si.ni; ++t) ts += item_cost(si, t);
        }
        long long e = ts * HP;                        // inclusive scan of the sequences' cost
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long u = __shfl_up_sync(0xffffffffu, e, o);
            if (lane >= o) e += u;
        }
        e += carry;
        const unsigned hit = __ballot_sync(0xffffffffu, s < a.S && 2 * e > lo);
        if (hit) {
            const int f = __ffs(hit) - 1;
            fs = s0 + f;
            fT = __shfl_sync(0xffffffffu, ts, f);
            fP = __shfl_sync(0xffffffffu, e, f) - fT * HP;
        }
        carry = __shfl_sync(0xffffffffu, e, 31);
    }
    if (lane == 0) {
        int hp0 = 0;
        if (fs < a.S && fT > 0 && lo > 2 * fP) {
            const int64_t h = (lo - 2 * fP) / (2 * fT);
            hp0 = (int)(h < HP - 1 ? h : HP - 1);
        }
        out->s = fs;
        out->hp = hp0;
        out->P = fP + (int64_t)hp0 * fT;
        out->lo = lo;
        out->hi = hi;
    }
}

template <typename T, int D, bool FUSED>
__global__ void __launch_bounds__(threads_for(FUSED), 1)
    paged_prefill_tc(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_kin,
                     const __grid_constant__ CUtensorMap tm_vin, const PrefillArgs a) {
    constexpr bool kSplit = Pk<T>::kSplit;
    using C = PCfg<D, kSplit>;
    constexpr int NST = C::NST;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;                 // 1024-aligned
    unsigned char* gbase = smem_raw + (base - raw);               // same, generic
    const uint32_t sQ = base + C::Q_OFF, sK = base + C::K_OFF, sV = base + C::V_OFF;
    const uint32_t bars = base + C::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::BAR_OFF + 8 * kBarCount);
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(gbase + C::BAR_OFF + 8 * kBarCount + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Sched* sched = reinterpret_cast<Sched*>(gbase + C::BAR_OFF + 8 * kBarCount + 8);

    if (tid == 0) {
        for (int i = 0; i < kBarCount; ++i)
            mbar_init(bar(i), (i == kBarPFull || i == kBarPFull + 1) ? 128u : 1u);
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
    if (warp == 2) plan(a, FUSED, sched, lane);
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
        // warp 0: the query tiles and the K tiles; the last warp: the V tiles
        // (separate warps: a lane waiting on a barrier would hold up the
        // other's issue).  Both walk the same items and the same global
        // key-tile sequence g; tile g uses stage g % NST of its ring.
        if (lane == 0) {
            const bool kq = warp == 0;
            const CUtensorMap* map = kq ? &tm_k : &tm_v;
            const CUtensorMap* in_map = kq ? &tm_kin : &tm_vin;
            const uint32_t ring = kq ? sK : sV;
            const int full0 = kq ? kBarKFull : kBarVFull, empty0 = kq ? kBarKEmpty : kBarVEmpty;
            const int stored0 = kq ? kBarKStored : kBarVStored;
            int64_t g = 0;
            int qn[2] = {0, 0};               // query tiles loaded, per slot
            bool ok = true;
            Walker wk;
            wk.init(*sched);
            Item it;
            while (ok && wk.next(a, *sched, FUSED, it)) {
                // slot x's query tile of the item, once the slot's last S of the
                // previous item is done: the first-served slot's before the
                // item's first K tile, the other's after it
                auto load_q = [&](int x) -> bool {
                    const int n = x ? qn[1] : qn[0];
                    if (n > 0 && !mbar_wait(bar(kBarQEmpty + x), (uint32_t)((n - 1) & 1), abort_flag))
                        return false;
                    mbar_expect_tx(bar(kBarQFull + x), (uint32_t)C::Q_BYTES);
                    for (int sl = 0; sl < C::SLABS; ++sl)
                        tma_3d(sQ + x * C::Q_BYTES + sl * C::SLAB_Q, &tm_q, sl * 64, it.h,
                               it.q0 + it.q_begin + (x ^ it.sw) * kBM, bar(kBarQFull + x));
                    if (x) ++qn[1]; else ++qn[0];
                    return true;
                };
                if (kq && !load_q(it.f)) {
                    ok = false;
                    break;
                }
                const int32_t* row_tab = a.block_tables + (int64_t)it.s * a.max_blocks;
                for (int j = 0; j < it.n_kv; ++j, ++g) {
                    if (kq && j == 1 && !load_q(1 - it.f)) {
                        ok = false;
                        break;
                    }
                    const int st = (int)(g % NST);
                    if (g >= NST &&
                        !mbar_wait(bar(empty0 + st), (uint32_t)((g / NST - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    if constexpr (FUSED) {
                        // the prompt's keys straight from the input tensor: 128
                        // token rows per box (rows past the prompt are masked,
                        // V's zeroed); the stage is free once the cache writer
                        // is done with its previous tile too
                        if (g >= NST && !mbar_wait(bar(stored0 + st), (uint32_t)((g / NST - 1) & 1),
                                                   abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(bar(full0 + st), (uint32_t)(kBN * 128 * C::SLABS));
                        for (int sl = 0; sl < C::SLABS; ++sl)
                            tma_3d(ring + st * C::KV_BYTES + sl * C::SLAB_KV, in_map, sl * 64, it.h,
                                   it.q0 + j * kBN, bar(full0 + st));
                        continue;
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
                if (ok && kq && it.n_kv == 1 && !load_q(1 - it.f)) ok = false;
            }
            if (!ok) fail();
            // let the latest copy into every stage (and the last query tiles)
            // land before the CTA can exit, whatever the other roles did (on a
            // normal run these have long landed)
            for (int x = 0; kq && x < 2; ++x)
                if (qn[x] > 0) mbar_wait(bar(kBarQFull + x), (uint32_t)((qn[x] - 1) & 1), nullptr);
            for (int64_t t = g - NST < 0 ? 0 : g - NST; t < g; ++t)
                mbar_wait(bar(full0 + (int)(t % NST)), (uint32_t)((t / NST) & 1), nullptr);
        }
    } else if (FUSED && warp == kWriterWarp) {
        // ====================================================== cache writer
        // Walks the same key tiles as the producers and observes every K and
        // V stage as it fills (so it never falls two phases behind a
        // barrier); for a diagonal tile (the last key tile of a query tile,
        // which no other item owns) it writes the tile's tokens into the
        // cache: whole blocks by tiled bulk stores from the swizzled stage,
        // the tokens of a partial last block by plain stores; then it hands
        // the stage back (the producers wait for that as well as for the MMAs).
        bool ok = true;
        int64_t g = 0;
        unsigned char* kc = static_cast<unsigned char*>(a.k_cache);
        unsigned char* vc = static_cast<unsigned char*>(a.v_cache);
        Walker wk;
        wk.init(*sched);
        Item it;
        while (ok && wk.next(a, *sched, FUSED, it)) {
            const int32_t* row_tab = a.block_tables + (int64_t)it.s * a.max_blocks;
            for (int j = 0; j < it.n_kv; ++j, ++g) {
                const int st = (int)(g % NST);
                const uint32_t par = (uint32_t)((g / NST) & 1);
                int got = 1;
                if (lane == 0)
                    got = mbar_wait(bar(kBarKFull + st), par, abort_flag) &&
                          mbar_wait(bar(kBarVFull + st), par, abort_flag);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                const bool diag = j == it.n[0] - 1 || (it.n[1] > 0 && j == it.n[1] - 1);
                if (diag) {
                    const int tok0 = j * kBN, tok1 = min(tok0 + kBN, it.ctx);
                    const int jb0 = tok0 / a.B, jbf = tok1 / a.B;   // whole blocks [jb0, jbf)
                    const uint32_t ks = sK + st * C::KV_BYTES, vs = sV + st * C::KV_BYTES;
                    if (lane == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        for (int jb = jb0; jb < jbf; ++jb) {
                            const int64_t phys = row_tab[jb];
                            if (phys < 0 || phys >= a.num_blocks) {
                                atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                                continue;
                            }
                            const int y = (int)((phys * a.H + it.h) * a.B);
                            const uint32_t off = (uint32_t)(jb * a.B - tok0) * 128u;
                            for (int sl = 0; sl < C::SLABS; ++sl) {
                                tma_store_2d(&tm_k, sl * 64, y, ks + sl * C::SLAB_KV + off);
                                tma_store_2d(&tm_v, sl * 64, y, vs + sl * C::SLAB_KV + off);
                            }
                        }
                        bulk_commit();
                    }
                    const int rem = tok1 - jbf * a.B;        // tokens of a partial last block
                    if (rem > 0) {
                        const int64_t phys = row_tab[jbf];
                        if (phys >= 0 && phys < a.num_blocks) {
                            const int r0 = jbf * a.B - tok0;  // its first row in the stage
                            const int64_t dst0 = ((phys * a.H + it.h) * a.B) * (int64_t)D * 2;
                            for (int i = lane; i < rem * C::SLABS * 8; i += 32) {
                                const int r = i / (C::SLABS * 8), c = i - r * (C::SLABS * 8);
                                const int sl = c >> 3, ch = c & 7, sr = r0 + r;
                                const uint32_t so = (uint32_t)(sl * C::SLAB_KV + sr * 128 +
                                                               ((ch ^ (sr & 7)) << 4));
                                const int64_t go = dst0 + ((int64_t)r * D + sl * 64 + ch * 8) * 2;
                                uint4 kv4, vv4;
                                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                             : "=r"(kv4.x), "=r"(kv4.y), "=r"(kv4.z), "=r"(kv4.w)
                                             : "r"(ks + so));
                                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                             : "=r"(vv4.x), "=r"(vv4.y), "=r"(vv4.z), "=r"(vv4.w)
                                             : "r"(vs + so));
                                *reinterpret_cast<uint4*>(kc + go) = kv4;
                                *reinterpret_cast<uint4*>(vc + go) = vv4;
                            }
                        } else if (lane == 0) {
                            atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                        }
                    }
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_arrive(bar(kBarKStored + st));
                    mbar_arrive(bar(kBarVStored + st));
                }
            }
        }
        if (lane == 0) {
            if (!ok) fail();
            bulk_wait0();                   // every store complete before the CTA ends
        }
    } else if (warp == 1) {
        // ======================================================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc(Pk<T>::kType, false, kBN, kBM);
            constexpr uint32_t ID_PV = idesc(Pk<T>::kType, true, D, kBM);
            // descriptors of each buffer's start, computed once; an operand's
            // descriptor is its buffer's plus the (16-byte unit) offset, which
            // never carries out of the 14-bit address field (addresses stay
            // below 256 KiB)
            const uint64_t dQ = sdesc(sQ, 16, 1024), dK = sdesc(sK, 16, 1024);
            const uint64_t dV = sdesc(sV, C::SLAB_KV, 1024);
            int64_t gpx[2] = {0, 0};         // P V products issued per group
            int items = 0;
            // S_X = Q_X K^T for the key tile in stage st into S_X's columns
            auto s_mma = [&](int x, int st) {
                const uint64_t dk = dK + (uint64_t)((st * C::KV_BYTES) >> 4);
                const uint64_t dq = dQ + (uint64_t)((x * C::Q_BYTES) >> 4);
                const uint32_t d = tmem + (uint32_t)(x * kBN);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = ((kk >> 2) * C::SLAB_Q + (kk & 3) * 32) >> 4;
                    const uint32_t ko = ((kk >> 2) * C::SLAB_KV + (kk & 3) * 32) >> 4;
                    umma(d, dq + qo, dk + ko, ID_S, kk > 0);
                }
                umma_commit(bar(kBarSFull + x));
            };
            bool ok = true;
            int64_t g = 0;
            // The next item is looked up while the current one runs: its
            // lengths are global loads whose latency would otherwise fall
            // between two items, when nothing is queued on the tensor pipe.
            Walker wk;
            wk.init(*sched);
            auto next_item = [&](Item& nit) -> bool { return wk.next(a, *sched, FUSED, nit); };
            Item nit;
            bool have = next_item(nit);
            while (ok && have) {
                const Item it = nit;
                const int s2 = 1 - it.f;             // the slot served second
                const int n2 = s2 ? it.n[1] : it.n[0];   // its key tiles
                // S of key tile 0, the slot served first first; a slot's query
                // tile is released after its last S (here when it has one key
                // tile or none)
                {
                    const int st = (int)(g % NST);
                    if (!mbar_wait(bar(kBarKFull + st), (uint32_t)((g / NST) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int xi = 0; ok && xi < 2; ++xi) {
                        const int x = xi ? s2 : it.f;
                        const int nx = x ? it.n[1] : it.n[0];
                        if (!mbar_wait(bar(kBarQFull + x), (uint32_t)(items & 1), abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (nx > 0) s_mma(x, st);
                        if (nx <= 1) umma_commit(bar(kBarQEmpty + x));
                    }
                    if (!ok) break;
                    umma_commit(bar(kBarKEmpty + st));
                }
                have = next_item(nit);
                for (int j = 0; ok && j < it.n_kv; ++j, ++g) {
                    const int st = (int)(g % NST);
                    if (!mbar_wait(bar(kBarVFull + st), (uint32_t)((g / NST) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint64_t dv = dV + (uint64_t)((st * C::KV_BYTES) >> 4);
                    const int stn = (int)((g + 1) % NST);
                    bool k_next = false;             // next key tile's K waited for
                    for (int xi = 0; xi < 2; ++xi) {
                        const int x = xi ? s2 : it.f;
                        const int nx = x ? it.n[1] : it.n[0];
                        if (j >= nx) continue;
                        const uint32_t par = (uint32_t)((x ? gpx[1] : gpx[0]) & 1);
                        // O_X += P_X(j) V_j, P_X from tensor memory
                        if (!mbar_wait<false>(bar(kBarPFull + x), par, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t pa = tmem + (uint32_t)(x * kBN);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            // keys 16 kk .. + 15: quarter kk / 2, 8 columns per step
                            const uint32_t pc = (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8);
                            const uint64_t vd = dv + (uint64_t)((kk * 2048) >> 4);
                            umma_ts(tmem + kColO + x * D, pa + pc, vd, ID_PV, (j > 0 || kk > 0));
                            if constexpr (kSplit)
                                umma_ts(tmem + kColO + x * D, pa + pc + 16, vd, ID_PV, 1u);
                        }
                        if (x) ++gpx[1]; else ++gpx[0];
                        if (j == nx - 1) umma_commit(bar(kBarPvDone + x));
                        // V_j's stage is free once its last P V (the second
                        // slot's, or the first's where the second has no tile
                        // j) completes, before the next S
                        if (x == s2 || j >= n2) umma_commit(bar(kBarVEmpty + st));
                        // then S_X of the next key tile over P_X (in issue order)
                        if (j + 1 < nx) {
                            if (!k_next) {
                                if (!mbar_wait(bar(kBarKFull + stn), (uint32_t)(((g + 1) / NST) & 1),
                                               abort_flag)) {
                                    ok = false;
                                    break;
                                }
                                k_next = true;
                                tc_fence_after();
                            }
                            s_mma(x, stn);
                            if (j + 2 == nx) umma_commit(bar(kBarQEmpty + x));
                            if (x == s2 || j + 1 >= n2) umma_commit(bar(kBarKEmpty + stn));
                        }
                    }
                    if (!ok) break;
                }
                ++items;
            }
            if (!ok) fail();
            // every MMA issued has completed before the CTA moves on
            umma_commit(bar(kBarMmaDone));
            mbar_wait(bar(kBarMmaDone), 0, nullptr);
        }
    } else {
        // ======================================================= softmax
        // Warps 2..5: slot 0, warps 6..9: slot 1; one row per thread (warp w
        // reaches the lanes 32 (w % 4) .. + 31 of tensor memory).
        const int x = (warp - 2) >> 2;               // the group's slot
        const int q4 = warp & 3;                     // this warp's lane quarter
        const int row = q4 * 32 + lane;              // row of the tile = TMEM lane
        const int gtid = (warp - 2 - 4 * x) * 32 + lane;   // 0..127 within the group
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t tS = tl + (uint32_t)(x * kBN);      // S_X, then P_X over it
        const uint32_t tO = tl + kColO + (uint32_t)(x * D);
        const float sl2 = a.scale_log2;
        const bool pos_scale = sl2 >= 0.f;
        bool ok = true;
        int64_t gx = 0;                              // this group's tiles so far
        int64_t g = 0;                               // key tiles so far (V stage)
        int items = 0;
        Walker wk;
        wk.init(*sched);
        Item it;
        while (ok && wk.next(a, *sched, FUSED, it)) {
            const int nx = x ? it.n[1] : it.n[0];
            const int pos0 = x ? it.pos0[1] : it.pos0[0];
            const int rows = x ? it.rows[1] : it.rows[0];
            // the group that zeroes V rows past the context (only the item's
            // last key tile has any): the first slot served whose rows reach
            // that tile, since its P V is issued before the other's
            const bool f_last = (it.f ? it.n[1] : it.n[0]) == it.n_kv;
            const bool zeroer = x == it.f ? f_last : !f_last;
            const int qpos = pos0 + row;             // causal limit of the row
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < nx; ++j, ++gx) {
                // S_X(j) complete (and with it the previous O_X += P_X V)
                if (!mbar_wait(bar(kBarSFull + x), (uint32_t)(gx & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int kb = j * kBN;
                const bool full = kb + kBN - 1 <= pos0;   // every key visible to every row
                // Row max of the visible scaled scores.  A full tile: both
                // 64-column halves loaded before one wait, two max chains per
                // half.  A tile crossing the diagonal runs once per query tile,
                // so its code is kept small (it would otherwise miss in the
                // instruction cache every time): a rolled loop over the 32-key
                // quarters, skipping those no row of the warp sees.
                float mx = -INFINITY;
                if (full) {
                    uint32_t rr[2][64];
                    tmem_ld64_nw(tS, rr[0]);
                    tmem_ld64_nw(tS + 64u, rr[1]);
                    tmem_wait64(rr[0]);
                    tmem_wait64(rr[1]);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t (&r)[64] = rr[hh];
                        float e0 = pos_scale ? -INFINITY : INFINITY, e1 = e0;
                        if (pos_scale) {
#pragma unroll
                            for (int e = 0; e < 64; e += 4) {
                                e0 = max3(e0, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
                                e1 = max3(e1, __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 64; e += 4) {
                                e0 = min3(e0, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
                                e1 = min3(e1, __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
                            }
                        }
                        mx = fmaxf(mx, (pos_scale ? fmaxf(e0, e1) : fminf(e0, e1)) * sl2);
                    }
                } else {
                    float e0 = -INFINITY, e1 = -INFINITY;
#pragma unroll 1
                    for (int q = 0; q < kBN / 32; ++q) {
                        const int lq = qpos - kb - q * 32;   // last visible key of the quarter
                        if (__all_sync(0xffffffffu, lq < 0)) continue;
                        uint32_t r[32];
                        tmem_ld32(tS + (uint32_t)(q * 32), r);
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            e0 = max3(e0, e <= lq ? __uint_as_float(r[e]) * sl2 : -INFINITY,
                                      e + 1 <= lq ? __uint_as_float(r[e + 1]) * sl2 : -INFINITY);
                            e1 = max3(e1, e + 2 <= lq ? __uint_as_float(r[e + 2]) * sl2 : -INFINITY,
                                      e + 3 <= lq ? __uint_as_float(r[e + 3]) * sl2 : -INFINITY);
                        }
                    }
                    mx = fmaxf(e0, e1);
                }
                float m_new = m;
                if (mx > m + kRescaleLog2 || (m == -INFINITY && mx > -INFINITY)) m_new = mx;
                const bool rescale = j > 0 && m_new != m;
                const float alpha = rescale ? ex2(m - m_new) : 1.f;
                // weights, packed in pairs over S, a quarter of 32 keys at a
                // time: keys 32 q .. + 31 go to the columns 32 q .. + 15 (high
                // parts) and + 16 .. + 31 (bf16 residuals), which held that
                // quarter's scores, read again here
                uint64_t rs2 = f2(0.f, 0.f);
                const uint64_t sc2 = f2(sl2, sl2), nm2 = f2(-m_new, -m_new);
                // The full-tile loop carries no mask code and is unrolled; the
                // diagonal one compares each key with the row's last visible
                // key, is rolled (small code, as for the max), and writes zero
                // weights for a quarter no row of the warp sees.
                auto weights = [&](auto masked) {
                    constexpr bool kMask = decltype(masked)::value;
                    const int lim = qpos - kb;       // last visible key of the tile
                    auto quarter = [&](const int q) {
                        if (kMask && __all_sync(0xffffffffu, lim < q * 32)) {
                            uint32_t z[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) z[e] = 0u;
                            tmem_st16(tS + (uint32_t)(q * 32), z);
                            if constexpr (kSplit) tmem_st16(tS + (uint32_t)(q * 32 + 16), z);
                            return;
                        }
                        uint32_t r[32];
                        tmem_ld32(tS + (uint32_t)(q * 32), r);
                        uint32_t pk[16];
                        uint32_t pr[kSplit ? 16 : 1];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const uint64_t x2 = fma2(
                                f2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sc2, nm2);
                            float p0, p1;
                            f2_split(x2, p0, p1);
                            p0 = ex2(p0);
                            p1 = ex2(p1);
                            if constexpr (kMask) {
                                p0 = q * 32 + e <= lim ? p0 : 0.f;
                                p1 = q * 32 + e + 1 <= lim ? p1 : 0.f;
                            }
                            rs2 = add2(rs2, f2(p0, p1));
                            uint32_t res;
                            pk[e >> 1] = Pk<T>::pack(p0, p1, res);
                            if constexpr (kSplit) pr[e >> 1] = res;
                        }
                        tmem_st16(tS + (uint32_t)(q * 32), pk);
                        if constexpr (kSplit) tmem_st16(tS + (uint32_t)(q * 32 + 16), pr);
                    };
                    if constexpr (kMask) {
#pragma unroll 1
                        for (int q = 0; q < kBN / 32; ++q) quarter(q);
                    } else {
#pragma unroll
                        for (int q = 0; q < kBN / 32; ++q) quarter(q);
                    }
                };
                if (full)
                    weights(std::false_type{});
                else
                    weights(std::true_type{});
                float rs0, rs1;
                f2_split(rs2, rs0, rs1);
                l = l * alpha + (rs0 + rs1);
                m = m_new;
                // O_X *= alpha for rows whose running max rose (warp-wide access)
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tO + c * 32, o);
                    }
                }
                // V rows past the context (partial last block, blocks never
                // loaded) are zeroed: their weights are 0, but 0 * NaN would not be
                const int64_t gk = g + j;
                if (zeroer && kb + kBN > it.ctx) {
                    const int st = (int)(gk % NST);
                    if (!mbar_wait(bar(kBarVFull + st), (uint32_t)((gk / NST) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int z0 = it.ctx - kb > 0 ? it.ctx - kb : 0;
                    const int n16 = (kBN - z0) * 8;       // 16-byte chunks per slab
                    unsigned char* vs = gbase + C::V_OFF + st * C::KV_BYTES;
                    for (int i = gtid; i < n16 * C::SLABS; i += 128) {
                        const int sl = i / n16, wv = i - sl * n16;
                        *reinterpret_cast<uint4*>(vs + sl * C::SLAB_KV + (z0 * 128) + wv * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + x));
            }
            if (!ok) break;
            g += it.n_kv;
            if (nx == 0) continue;
            // the item's output rows of this tile, once its last P V is done
            if (!mbar_wait(bar(kBarPvDone + x), (uint32_t)(items & 1), abort_flag)) {
                ok = false;
                break;
            }
            ++items;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T* orow = static_cast<T*>(a.out) +
                      ((int64_t)(it.q0 + it.q_begin + (x ^ it.sw) * kBM + row) * a.H + it.h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                if (row < rows) {
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wv[e] = Pk<T>::pack_out(__uint_as_float(o[2 * e]) * inv,
                                                __uint_as_float(o[2 * e + 1]) * inv);
                    if (a.out_v8) {
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            st_global_v8(orow + c * 32 + e * 16, wv + 8 * e);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] =
                                make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
                    }
                }
            }
            tc_fence_before();
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

template <typename T, int D, bool FUSED>
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tkin, const CUtensorMap& tvin,
                           const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = PCfg<D, Pk<T>::kSplit>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_tc<T, D, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // Clusters of two CTAs, so that CTAs 2k and 2k + 1, which take the same
    // items of adjacent heads, run on the two SMs of one TPC.  How the CTAs
    // are paired matters on GB300: placed at random (as a programmatic
    // dependent of a reshape_and_cache, whose CTAs let it launch as they
    // start), most CTAs ran 1.3-1.5x longer on the same items; the default
    // placement pairs them by chance, and the cluster launch pairs them
    // always and ran 4% faster than the default (333 against 348 us on 16
    // prompts of 543-1729 tokens, 40 x 128).  Not a programmatic dependent
    // either: that still cost 13 us after a reshape_and_cache.
    cudaLaunchConfig_t cfg = {};
    // persistent: one CTA per SM (shared memory and tensor memory allow no
    // more), each pair walking its run of the units
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // an even number of CTAs (pairs), no more than two per unit of work
    const int64_t units = (int64_t)a.q_items * a.S * ((a.H + 1) / 2);
    const int sms = pkv::sm_count(dev);
    if (sms < 1) return cudaErrorInvalidDevice;
    const int64_t pairs = sms / 2 > 1 ? sms / 2 : 1;
    cfg.gridDim = dim3((unsigned)(2 * (units < pairs ? units : pairs)));
    cfg.blockDim = dim3(threads_for(FUSED));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (cfg.gridDim.x % 2 == 0) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, paged_prefill_tc<T, D, FUSED>, tq, tk, tv, tkin, tvin, a);
    if (e == cudaErrorInvalidClusterSize && cfg.numAttrs == 1) {
        // the device refused the pairing: the same kernel, CTAs placed one
        // by one
        cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, paged_prefill_tc<T, D, FUSED>, tq, tk, tv, tkin, tvin, a);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

bool aligned(const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) & (al - 1)) == 0; }

}  // namespace

namespace {

pkv_status prefill_common(const char* fn, void* out, const void* q, const void* k_in,
                          const void* v_in, void* k_cache, void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          const int32_t* query_start, float scale, int num_seqs, int num_heads,
                          int head_dim, int block_size, int max_blocks_per_seq,
                          int64_t num_blocks, int max_query_len, int num_query_tokens,
                          pkv_dtype dtype, cudaStream_t stream) {
    const bool fused = k_in != nullptr || v_in != nullptr;
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
    {
        // the work schedule sums item costs in 64 bits: a bound far above any
        // call whose tensors fit in memory
        const double units = (double)((num_heads + 1) / 2) * num_seqs *
                             (double)(((int64_t)max_query_len + kRows - 1) / kRows);
        const double unit_cost =
            kPairCost * ((double)max_blocks_per_seq * block_size / kBN + 1.0) + kItemCost;
        if (units * unit_cost >= 0x1p60)
            return pkv::fail(PKV_ERR_INVALID, "%s: too much work for one call", fn);
    }
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0 || max_query_len == 0 || num_query_tokens == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start ||
        (fused && (!k_in || !v_in)))
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        (fused && (!aligned(k_in, 16) || !aligned(v_in, 16))))
        return pkv::fail(PKV_ERR_INVALID, "%s: out, q, k, v and the caches must be 16-byte aligned",
                         fn);
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no CUDA device", fn);

    const bool bf16 = dtype == PKV_BF16;
    const cuuint64_t D = (cuuint64_t)head_dim;
    CUtensorMap tq, tk, tv, tkin, tvin;
    {
        // q (and the prompt's k, v): [tokens][heads][D], one box = 128 tokens
        // x 64 elements of one head
        const cuuint64_t dims[3] = {D, (cuuint64_t)num_heads, (cuuint64_t)num_query_tokens};
        const cuuint64_t strides[2] = {D * 2, (cuuint64_t)num_heads * D * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBM};
        if (!make_map(&tq, bf16, 3, q, dims, strides, box))
            return pkv::fail(PKV_ERR_CUDA, "%s: tensor map of q", fn);
        if (fused) {
            if (!make_map(&tkin, bf16, 3, k_in, dims, strides, box) ||
                !make_map(&tvin, bf16, 3, v_in, dims, strides, box))
                return pkv::fail(PKV_ERR_CUDA, "%s: tensor maps of k and v", fn);
        } else {
            tkin = tq;                       // unused
            tvin = tq;
        }
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
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out_v8 = aligned(out, 32) ? 1 : 0;
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
    a.q_items = (max_query_len + kRows - 1) / kRows;
    a.num_blocks = num_blocks;
    a.err = err;
    cudaError_t e;
    if (fused) {
        if (!bf16)
            e = head_dim == 128
                    ? launch_prefill<__half, 128, true>(tq, tk, tv, tkin, tvin, a, stream)
                    : launch_prefill<__half, 64, true>(tq, tk, tv, tkin, tvin, a, stream);
        else
            e = head_dim == 128
                    ? launch_prefill<__nv_bfloat16, 128, true>(tq, tk, tv, tkin, tvin, a, stream)
                    : launch_prefill<__nv_bfloat16, 64, true>(tq, tk, tv, tkin, tvin, a, stream);
    } else {
        if (!bf16)
            e = head_dim == 128
                    ? launch_prefill<__half, 128, false>(tq, tk, tv, tkin, tvin, a, stream)
                    : launch_prefill<__half, 64, false>(tq, tk, tv, tkin, tvin, a, stream);
        else
            e = head_dim == 128
                    ? launch_prefill<__nv_bfloat16, 128, false>(tq, tk, tv, tkin, tvin, a, stream)
                    : launch_prefill<__nv_bfloat16, 64, false>(tq, tk, tv, tkin, tvin, a, stream);
    }
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_prefill(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       float scale, int num_seqs, int num_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                       int max_query_len, int num_query_tokens, pkv_dtype dtype,
                                       cudaStream_t stream) {
    return prefill_common("pkv_paged_attention_prefill", out, q, nullptr, nullptr,
                          const_cast<void*>(k_cache), const_cast<void*>(v_cache), block_tables,
                          context_lens, query_start, scale, num_seqs, num_heads, head_dim,
                          block_size, max_blocks_per_seq, num_blocks, max_query_len,
                          num_query_tokens, dtype, stream);
}

pkv_status pkv_paged_attention_prefill_write(void* out, const void* q, const void* k,
                                             const void* v, void* k_cache, void* v_cache,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens,
                                             const int32_t* query_start, float scale,
                                             int num_seqs, int num_heads, int head_dim,
                                             int block_size, int max_blocks_per_seq,
                                             int64_t num_blocks, int max_query_len,
                                             int num_query_tokens, pkv_dtype dtype,
                                             cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_prefill_write";
    if (!k || !v) return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    return prefill_common(fn, out, q, k, v, k_cache, v_cache, block_tables, context_lens,
                          query_start, scale, num_seqs, num_heads, head_dim, block_size,
                          max_blocks_per_seq, num_blocks, max_query_len, num_query_tokens, dtype,
                          stream);
}

}  // extern "C"
