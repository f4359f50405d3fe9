// C ABI of the decode attention: argument checks, workspace sizing, grid choice.
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <random>

#include <cudaTypedefs.h>

#include "pkv_internal.h"

namespace {

constexpr int kMaxDevices = 64;
// Lower bound of a balanced chunk, in steps: keeps tiny batches from being cut
// into one-step pieces that would all need the merge pass.
constexpr int kMinChunkSteps = 8;
#ifndef PKV_DECODE_WAVES
#define PKV_DECODE_WAVES 1
#endif

struct OccEntry {
    const pkv::DecodeKernel* k;
    size_t smem;
    int ctas;
};

std::mutex g_mu;
OccEntry g_occ[kMaxDevices][8] = {};

// Bound of the decode kernels' pipeline waits, in ns (pkv_set_decode_wait_limit).
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
constexpr uint64_t kMaxWaitNs = 10000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// A 40-bit tag per call.  The call's first CTA stamps the workspace's claim
// word with it, and a claimant starts claiming only once it sees the tag, so
// a word left by an earlier call, or never written, is not taken for this
// call's.  The sequence starts at a random point so that words left by
// another process do not match either.
uint64_t next_epoch() {
    static std::atomic<uint64_t> counter{[] {
        std::random_device rd;
        const uint64_t t = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
        return ((uint64_t)rd() << 20) ^ t;
    }()};
    return (counter.fetch_add(1) + 1) & ((1ull << 40) - 1);
}

// CTAs per SM for kernel k with `smem` bytes, cached per device.
cudaError_t ctas_per_sm(const pkv::DecodeKernel* k, int dev, size_t smem, int* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    OccEntry* row = g_occ[dev];
    for (int i = 0; i < 8; ++i)
        if (row[i].k == k && row[i].smem == smem) {
            *out = row[i].ctas;
            return cudaSuccess;
        }
    int n = 0;
    cudaError_t e = k->occupancy(&n, smem);
    if (e != cudaSuccess) return e;
    for (int i = 7; i > 0; --i) row[i] = row[i - 1];
    row[0] = {k, smem, n};
    *out = n;
    return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The driver's tiled tensor-map encoder (a host computation), looked up once.
PFN_cuTensorMapEncodeTiled_v12000 map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A pool [num_blocks][H][B][D] seen as rows of D 16-bit elements; boxes of
// 64 columns x box_rows rows, 128-byte swizzle (the shared-prefix steps).
bool pool_map(CUtensorMap* m, bool bf16, const void* pool, int64_t rows, int D, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = map_encoder();
    if (!fn || rows >= (1LL << 31)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host-only checks shared by the workspace query and the launch.
pkv_status check_shape(int S, int H, int D, int B, int max_blocks, int partition_size,
                       const char* fn) {
    if (S < 0 || S > PKV_MAX_SEQS)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_seqs must be in [0, %d]", fn, PKV_MAX_SEQS);
    if (H < 1) return pkv::fail(PKV_ERR_INVALID, "%s: num_heads must be >= 1", fn);
    if (D != 64 && D != 128) return pkv::fail(PKV_ERR_INVALID, "%s: head_dim must be 64 or 128", fn);
    if (B != 8 && B != 16 && B != 32 && B != 64)
        return pkv::fail(PKV_ERR_INVALID, "%s: block_size must be 8, 16, 32 or 64", fn);
    if (max_blocks < 1) return pkv::fail(PKV_ERR_INVALID, "%s: max_blocks_per_seq must be >= 1", fn);
    const int sub = pkv::step_tokens(D);
    const int64_t steps = (int64_t)S * pkv::max_steps_per_seq(D, B, max_blocks);
    if (steps >= (1LL << 31) || steps * H >= (1LL << 62))
        return pkv::fail(PKV_ERR_INVALID, "%s: batch too large (step count overflows)", fn);
    if (partition_size < 0 || (partition_size > 0 && partition_size % sub != 0))
        return pkv::fail(PKV_ERR_INVALID,
                         "%s: partition_size must be 0 or a positive multiple of %d tokens", fn,
                         sub);
    return PKV_OK;
}

// Capacities of the shared-prefix regions (group units, group partial slots):
// a sequence belongs to at most one group, whose prefix (at most the
// sequence's steps) is cut into units of group_unit_steps(D, B) steps.
// False when grouping is not offered for these sizes (the plain kernel runs).
bool group_caps(int S, int H, int D, int B, int max_blocks, int64_t* units, int64_t* slots) {
    if (S < 2 || S > pkv::kGroupMaxSeqs) return false;
    const int64_t lg = pkv::group_unit_steps(D, B);
    const int64_t nc = (pkv::max_steps_per_seq(D, B, max_blocks) + lg - 1) / lg;
    *slots = (int64_t)S * H * nc;
    *units = (int64_t)(S / 2) * H * nc;
    return *slots < (1LL << 31);
}

int64_t max_chunks(int S, int H, int D, int B, int max_blocks, int partition_size) {
    if (partition_size == 0) return (int64_t)PKV_MAX_GRID * (1 + PKV_DECODE_DYN_PER_CTA);
    const int64_t L = partition_size / pkv::step_tokens(D);
    const int64_t steps = (int64_t)S * H * pkv::max_steps_per_seq(D, B, max_blocks);
    return (steps + L - 1) / L;
}

// The checks and launch shared by the paged and the contiguous entry points.
// `a` arrives with the layout's fields set (tables, ctx_cap, kv_stride,
// num_blocks); B and max_blocks are the layout's step geometry.
pkv_status launch_decode(const char* fn, const pkv::DecodeKernel* k, pkv::DecodeArgs a,
                         void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* context_lens, float scale, int num_seqs, int num_heads,
                         int head_dim, int block_size, int max_blocks, int partition_size,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream,
                         int64_t gunit_cap = 0, int64_t gslot_cap = 0,
                         const CUtensorMap* tk = nullptr, const CUtensorMap* tv = nullptr) {
    if (!out || !q || !k_cache || !v_cache || !context_lens || !workspace)
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return pkv::fail(PKV_ERR_INVALID, "%s: out, q and the caches must be 16-byte aligned", fn);
    if (!aligned(context_lens, 4))
        return pkv::fail(PKV_ERR_INVALID, "%s: int32 arrays must be 4-byte aligned", fn);
    if (!aligned(workspace, 256))
        return pkv::fail(PKV_ERR_INVALID, "%s: workspace must be 256-byte aligned", fn);
    const int64_t mc = max_chunks(num_seqs, num_heads, head_dim, block_size, max_blocks,
                                  partition_size);
    const pkv::WsLayout wl = pkv::ws_layout(num_seqs, num_heads, head_dim, mc, gunit_cap, gslot_cap);
    if (workspace_bytes < wl.total)
        return pkv::fail(PKV_ERR_INVALID, "%s: workspace too small (%zu < %zu bytes)", fn,
                         workspace_bytes, wl.total);

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    if (dev < 0 || dev >= kMaxDevices) return pkv::fail(PKV_ERR_INVALID, "%s: device id", fn);
    const size_t smem = k->smem_bytes(num_seqs);
    int per_sm = 0;
    e = ctas_per_sm(k, dev, smem, &per_sm);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "decode: occupancy");
    if (per_sm < 1)
        return pkv::fail(PKV_ERR_INVALID, "%s: %d sequences need %zu bytes of shared memory", fn,
                         num_seqs, smem);
    int grid = pkv::sm_count(dev) * per_sm * PKV_DECODE_WAVES;
    if (grid < 1) return pkv::fail(PKV_ERR_CUDA, "%s: no multiprocessors", fn);
    if (grid > PKV_MAX_GRID) grid = PKV_MAX_GRID;
    {
        // small batches: no more CTAs than balanced chunks of the minimum length
        // the batch could fill (the bound uses the table width, not the
        // device-side lengths)
        const int64_t steps_bound = (int64_t)num_seqs * num_heads *
                                    pkv::max_steps_per_seq(head_dim, block_size, max_blocks);
        const int64_t useful = (steps_bound + kMinChunkSteps - 1) / kMinChunkSteps;
        if (useful < grid) grid = (int)(useful > 0 ? useful : 1);
    }
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no device error word", fn);

    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.context_lens = context_lens;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.S = num_seqs;
    a.H = num_heads;
    a.L_steps = partition_size > 0 ? partition_size / pkv::step_tokens(head_dim) : 0;
    a.min_chunk_steps = kMinChunkSteps;
    a.main_grid = grid;
    a.epoch = next_epoch();
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a.ws = static_cast<char*>(workspace);
    a.ws_l = wl;
    a.err = err;
    CUtensorMap none;
    memset(&none, 0, sizeof(none));
    e = k->launch(a, grid, stream, tk ? *tk : none, tv ? *tv : none);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int block_size,
                                     int max_blocks_per_seq, int partition_size, size_t* bytes) {
    const char* fn = "pkv_decode_workspace_size";
    if (!bytes) return pkv::fail(PKV_ERR_INVALID, "%s: bytes is NULL", fn);
    pkv_status st = check_shape(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                partition_size, fn);
    if (st != PKV_OK) return st;
    const int64_t mc = max_chunks(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                  partition_size);
    *bytes = pkv::ws_layout(num_seqs, num_heads, head_dim, mc).total;
    return PKV_OK;
}

pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float scale, int num_seqs,
                                      int num_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int64_t num_blocks,
                                      pkv_dtype dtype, int partition_size, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_decode";
    pkv_status st = check_shape(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                partition_size, fn);
    if (st != PKV_OK) return st;
    if (num_blocks < 1) return pkv::fail(PKV_ERR_INVALID, "%s: num_blocks must be >= 1", fn);
    if (dtype != PKV_F16 && dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "%s: unknown dtype", fn);
    if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables) return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(block_tables, 4))
        return pkv::fail(PKV_ERR_INVALID, "%s: int32 arrays must be 4-byte aligned", fn);
    const pkv::DecodeKernel* k = dtype == PKV_F16 ? pkv::decode_kernel_f16(head_dim, block_size)
                                                  : pkv::decode_kernel_bf16(head_dim, block_size);
    if (!k) return pkv::fail(PKV_ERR_INVALID, "%s: unsupported head_dim/block_size", fn);
    pkv::DecodeArgs a = {};
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.ctx_cap = max_blocks_per_seq * block_size;
    a.kv_stride = 0;
    a.num_blocks = num_blocks;
    a.mode = pkv::kModePaged;
    return launch_decode(fn, k, a, out, q, k_cache, v_cache, context_lens, scale, num_seqs,
                         num_heads, head_dim, block_size, max_blocks_per_seq, partition_size,
                         workspace, workspace_bytes, stream);
}

pkv_status pkv_paged_attention_decode_append(void* out, const void* q, const void* k_new,
                                             const void* v_new, void* k_cache, void* v_cache,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens, float scale,
                                             int num_seqs, int num_heads, int head_dim,
                                             int block_size, int max_blocks_per_seq,
                                             int64_t num_blocks, pkv_dtype dtype,
                                             int partition_size, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_decode_append";
    pkv_status st = check_shape(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                partition_size, fn);
    if (st != PKV_OK) return st;
    if (num_blocks < 1) return pkv::fail(PKV_ERR_INVALID, "%s: num_blocks must be >= 1", fn);
    if (dtype != PKV_F16 && dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "%s: unknown dtype", fn);
    if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables || !k_new || !v_new)
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(block_tables, 4))
        return pkv::fail(PKV_ERR_INVALID, "%s: int32 arrays must be 4-byte aligned", fn);
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return pkv::fail(PKV_ERR_INVALID, "%s: k_new and v_new must be 16-byte aligned", fn);
    const pkv::DecodeKernel* k = dtype == PKV_F16
                                     ? pkv::decode_kernel_append_f16(head_dim, block_size)
                                     : pkv::decode_kernel_append_bf16(head_dim, block_size);
    if (!k) return pkv::fail(PKV_ERR_INVALID, "%s: unsupported head_dim/block_size", fn);
    pkv::DecodeArgs a = {};
    a.block_tables = block_tables;
    a.k_new = k_new;
    a.v_new = v_new;
    a.max_blocks = max_blocks_per_seq;
    a.ctx_cap = max_blocks_per_seq * block_size;
    a.kv_stride = 0;
    a.num_blocks = num_blocks;
    a.mode = pkv::kModeAppend;
    return launch_decode(fn, k, a, out, q, k_cache, v_cache, context_lens, scale, num_seqs,
                         num_heads, head_dim, block_size, max_blocks_per_seq, partition_size,
                         workspace, workspace_bytes, stream);
}

pkv_status pkv_contiguous_workspace_size(int num_seqs, int num_heads, int head_dim,
                                         int max_context_len, int partition_size,
                                         size_t* bytes) {
    const char* fn = "pkv_contiguous_workspace_size";
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "%s: head_dim must be 64 or 128", fn);
    if (max_context_len < 1)
        return pkv::fail(PKV_ERR_INVALID, "%s: max_context_len must be >= 1", fn);
    const int sub = pkv::step_tokens(head_dim);
    return pkv_decode_workspace_size(num_seqs, num_heads, head_dim, sub,
                                     (max_context_len + sub - 1) / sub, partition_size, bytes);
}

pkv_status pkv_contiguous_attention_decode(void* out, const void* q, const void* k,
                                           const void* v, const int32_t* context_lens,
                                           float scale, int num_seqs, int num_heads,
                                           int head_dim, int max_context_len, pkv_dtype dtype,
                                           int partition_size, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream) {
    const char* fn = "pkv_contiguous_attention_decode";
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "%s: head_dim must be 64 or 128", fn);
    if (max_context_len < 1)
        return pkv::fail(PKV_ERR_INVALID, "%s: max_context_len must be >= 1", fn);
    const int sub = pkv::step_tokens(head_dim);
    const int mb = (max_context_len + sub - 1) / sub;
    pkv_status st = check_shape(num_seqs, num_heads, head_dim, sub, mb, partition_size, fn);
    if (st != PKV_OK) return st;
    if (dtype != PKV_F16 && dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "%s: unknown dtype", fn);
    if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0) return PKV_OK;
    const pkv::DecodeKernel* kern = dtype == PKV_F16 ? pkv::decode_kernel_contig_f16(head_dim)
                                                     : pkv::decode_kernel_contig_bf16(head_dim);
    if (!kern) return pkv::fail(PKV_ERR_INVALID, "%s: unsupported head_dim", fn);
    pkv::DecodeArgs a = {};
    a.block_tables = nullptr;
    a.max_blocks = mb;
    a.ctx_cap = max_context_len;
    a.kv_stride = max_context_len;
    a.num_blocks = 1;
    a.mode = pkv::kModeContig;
    return launch_decode(fn, kern, a, out, q, k, v, context_lens, scale, num_seqs, num_heads,
                         head_dim, sub, mb, partition_size, workspace, workspace_bytes, stream);
}

pkv_status pkv_decode_shared_workspace_size(int num_seqs, int num_heads, int head_dim,
                                            int block_size, int max_blocks_per_seq,
                                            int partition_size, size_t* bytes) {
    const char* fn = "pkv_decode_shared_workspace_size";
    if (!bytes) return pkv::fail(PKV_ERR_INVALID, "%s: bytes is NULL", fn);
    pkv_status st = check_shape(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                partition_size, fn);
    if (st != PKV_OK) return st;
    int64_t gu = 0, gs = 0;
    if (!group_caps(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, &gu, &gs))
        gu = gs = 0;
    const int64_t mc = max_chunks(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                  partition_size);
    *bytes = pkv::ws_layout(num_seqs, num_heads, head_dim, mc, gu, gs).total;
    return PKV_OK;
}

pkv_status pkv_paged_attention_decode_shared(void* out, const void* q, const void* k_cache,
                                             const void* v_cache, const int32_t* block_tables,
                                             const int32_t* context_lens, float scale,
                                             int num_seqs, int num_heads, int head_dim,
                                             int block_size, int max_blocks_per_seq,
                                             int64_t num_blocks, pkv_dtype dtype,
                                             int partition_size, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_decode_shared";
    pkv_status st = check_shape(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                partition_size, fn);
    if (st != PKV_OK) return st;
    if (num_blocks < 1) return pkv::fail(PKV_ERR_INVALID, "%s: num_blocks must be >= 1", fn);
    if (dtype != PKV_F16 && dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "%s: unknown dtype", fn);
    if (!std::isfinite(scale)) return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables) return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(block_tables, 4))
        return pkv::fail(PKV_ERR_INVALID, "%s: int32 arrays must be 4-byte aligned", fn);
    int64_t gu = 0, gs = 0;
    bool groups =
        group_caps(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, &gu, &gs);
    CUtensorMap tk, tv;
    if (groups) {
        // the prefix steps' tiled copies address pool rows with 32-bit coordinates
        const int64_t rows = num_blocks * num_heads * (int64_t)block_size;
        const int sub = pkv::step_tokens(head_dim);
        const int box = block_size < sub ? block_size : sub;
        groups = pool_map(&tk, dtype == PKV_BF16, k_cache, rows, head_dim, box) &&
                 pool_map(&tv, dtype == PKV_BF16, v_cache, rows, head_dim, box);
    }
    const pkv::DecodeKernel* k =
        groups ? (dtype == PKV_F16 ? pkv::decode_kernel_shared_f16(head_dim, block_size)
                                   : pkv::decode_kernel_shared_bf16(head_dim, block_size))
               : (dtype == PKV_F16 ? pkv::decode_kernel_f16(head_dim, block_size)
                                   : pkv::decode_kernel_bf16(head_dim, block_size));
    if (!k) return pkv::fail(PKV_ERR_INVALID, "%s: unsupported head_dim/block_size", fn);
    pkv::DecodeArgs a = {};
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.ctx_cap = max_blocks_per_seq * block_size;
    a.kv_stride = 0;
    a.num_blocks = num_blocks;
    a.mode = groups ? pkv::kModeShared : pkv::kModePaged;
    return launch_decode(fn, k, a, out, q, k_cache, v_cache, context_lens, scale, num_seqs,
                         num_heads, head_dim, block_size, max_blocks_per_seq, partition_size,
                         workspace, workspace_bytes, stream, groups ? gu : 0, groups ? gs : 0,
                         groups ? &tk : nullptr, groups ? &tv : nullptr);
}

pkv_status pkv_set_decode_wait_limit(uint64_t ns, uint64_t* previous) {
    if (ns > kMaxWaitNs)
        return pkv::fail(PKV_ERR_INVALID,
                         "pkv_set_decode_wait_limit: %llu ns is above the %llu ns maximum",
                         (unsigned long long)ns, (unsigned long long)kMaxWaitNs);
    const uint64_t old = g_wait_ns.exchange(ns);
    if (previous) *previous = old;
    return PKV_OK;
}

}  // extern "C"
