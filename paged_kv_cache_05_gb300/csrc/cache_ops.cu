// Cache maintenance kernels: the new-token write (reshape_and_cache) and the
// block-granular copy used by copy-on-write (copy_blocks).
//
// Both are pure bit copies bound by HBM bandwidth: 16-byte vector loads and
// stores, consecutive threads on consecutive 16-byte pieces of a row.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Programmatic dependent launch: wait for the preceding kernel in the stream
// before touching memory (a no-op without the dependency), then let the next
// kernel's CTAs be scheduled while this one runs.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, cudaStream_t stream,
                       Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// One row = one (token, head): VPR 16-byte pieces of K and as many of V (8
// at head_dim 64, 16 at 128), VPR consecutive threads per row.  The grid is
// at most one wave (as many CTAs per SM as can be resident) and strides over
// the rows, two rows per thread per pass so that four 16-byte loads are in
// flight before the stores.  Destination: slot / B is the physical block,
// slot % B the offset inside it (ricepunchb garden, section 3.2).
constexpr int kRowThreads = 256;

template <int VPR>
__global__ void __launch_bounds__(kRowThreads) reshape_and_cache_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slots, int T, int H, int B,
    int64_t num_slots, int32_t* err) {
    pdl_wait_then_release();
    constexpr int RPP = kRowThreads / VPR;           // rows per CTA per pass
    const int piece = threadIdx.x % VPR;
    const int64_t rows = (int64_t)T * H;
    const int64_t stride = (int64_t)gridDim.x * RPP;
    for (int64_t r0 = (int64_t)blockIdx.x * RPP + threadIdx.x / VPR; r0 < rows; r0 += 2 * stride) {
        uint4 kv[2], vv[2];
        int64_t dst[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t row = r0 + u * stride;
            dst[u] = -1;
            if (row >= rows) continue;
            const int t = (int)(row / H);
            const int h = (int)(row - (int64_t)t * H);
            const int64_t slot = slots[t];
            if (slot < 0) continue;
            if (slot >= num_slots) {
                if (h == 0 && piece == 0) atomicOr(err, PKV_DEVERR_BAD_SLOT);
                continue;
            }
            const int64_t blk = slot / B, off = slot - blk * B;
            dst[u] = ((blk * H + h) * B + off) * VPR + piece;
            kv[u] = ld_nc_v4(k + row * VPR + piece);
            vv[u] = ld_nc_v4(v + row * VPR + piece);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (dst[u] < 0) continue;
            k_cache[dst[u]] = kv[u];
            v_cache[dst[u]] = vv[u];
        }
    }
}

// grid = (pieces, pairs, 2): blockIdx.z picks the K or the V pool; each thread
// moves kUnroll 16-byte vectors of the whole-block copy src -> dst.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ pairs,
    int64_t vecs_per_block, int64_t num_blocks, int32_t* err) {
    pdl_wait_then_release();
    const int p = blockIdx.y;
    const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            atomicOr(err, PKV_DEVERR_BAD_BLOCK);
        return;
    }
    uint4* pool = blockIdx.z == 0 ? k_cache : v_cache;
    const uint4* s = pool + src * vecs_per_block;
    uint4* d = pool + dst * vecs_per_block;
    const int64_t base = (int64_t)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x;
    uint4 buf[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kCopyThreads;
        if (i < vecs_per_block) buf[u] = ld_nc_v4(s + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kCopyThreads;
        if (i < vecs_per_block) d[i] = buf[u];
    }
}

// Block swap between two pools, one of which may live in pinned host memory
// (reached over NVLink-C2C / PCIe through unified addressing): grid =
// (pieces, pairs, 2), blockIdx.z picks K or V.  Plain (coherent) loads, since
// the source may be host memory; each thread keeps kCopyUnroll vectors in flight.
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(
    uint4* __restrict__ dst_k, uint4* __restrict__ dst_v, const uint4* __restrict__ src_k,
    const uint4* __restrict__ src_v, const int32_t* __restrict__ pairs, int64_t vecs_per_block,
    int64_t src_blocks, int64_t dst_blocks, int32_t* err) {
    pdl_wait_then_release();
    const int p = blockIdx.y;
    const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            atomicOr(err, PKV_DEVERR_BAD_BLOCK);
        return;
    }
    const uint4* s = (blockIdx.z == 0 ? src_k : src_v) + src * vecs_per_block;
    uint4* d = (blockIdx.z == 0 ? dst_k : dst_v) + dst * vecs_per_block;
    const int64_t base = (int64_t)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x;
    uint4 buf[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kCopyThreads;
        if (i < vecs_per_block) buf[u] = s[i];
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kCopyThreads;
        if (i < vecs_per_block) d[i] = buf[u];
    }
}

}  // namespace

namespace pkv {

cudaError_t launch_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                               const int32_t* pairs, int P, int H, int D, int B,
                               int64_t src_blocks, int64_t dst_blocks, int32_t* err,
                               cudaStream_t stream) {
    const int64_t vecs = (int64_t)H * B * D / 8;
    const int64_t per_cta = kCopyThreads * kCopyUnroll;
    dim3 grid((unsigned)((vecs + per_cta - 1) / per_cta), (unsigned)P, 2);
    cudaError_t e = launch_pdl(swap_blocks_kernel, grid, dim3(kCopyThreads), stream,
                               static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v),
                               static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v),
                               pairs, vecs, src_blocks, dst_blocks, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slots, int T, int H, int D, int B,
                                     int64_t num_blocks, int32_t* err, cudaStream_t stream) {
    // one wave at most, striding over the rows: 107 us for the 694 MB of a
    // 16,947-token prompt batch (40 x 128, fp16) on GB300, against 122 us for
    // one thread per piece and one CTA per 256 pieces
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = sm_count(dev);
    if (sms < 1) return cudaErrorInvalidDevice;
    // resident CTAs per SM, from the compiled kernel (registers decide it)
    static int per_sm[2] = {0, 0};
    int& occ = per_sm[D == 64 ? 0 : 1];
    if (occ == 0) {
        int n = 0;
        e = D == 64 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                          &n, reshape_and_cache_kernel<8>, kRowThreads, 0)
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                          &n, reshape_and_cache_kernel<16>, kRowThreads, 0);
        if (e != cudaSuccess) return e;
        occ = n < 1 ? 1 : n;
    }
    const int64_t rows = (int64_t)T * H;
    const int rpp = kRowThreads / (D / 8);
    int64_t blocks = (rows + rpp - 1) / rpp;
    if (blocks > (int64_t)sms * occ) blocks = (int64_t)sms * occ;
    if (blocks < 1) blocks = 1;
    const uint4* k4 = static_cast<const uint4*>(k);
    const uint4* v4 = static_cast<const uint4*>(v);
    uint4* kc4 = static_cast<uint4*>(k_cache);
    uint4* vc4 = static_cast<uint4*>(v_cache);
    if (D == 64)
        e = launch_pdl(reshape_and_cache_kernel<8>, dim3((unsigned)blocks), dim3(kRowThreads),
                       stream, k4, v4, kc4, vc4, slots, T, H, B, num_blocks * B, err);
    else
        e = launch_pdl(reshape_and_cache_kernel<16>, dim3((unsigned)blocks), dim3(kRowThreads),
                       stream, k4, v4, kc4, vc4, slots, T, H, B, num_blocks * B, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int P, int H,
                               int D, int B, int64_t num_blocks, int32_t* err,
                               cudaStream_t stream) {
    const int64_t vecs = (int64_t)H * B * D / 8;
    const int64_t per_cta = kCopyThreads * kCopyUnroll;
    dim3 grid((unsigned)((vecs + per_cta - 1) / per_cta), (unsigned)P, 2);
    cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), stream,
                               static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs,
                               vecs, num_blocks, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pkv

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Device memory, pinned (registered) host memory or managed memory: what a
// kernel may dereference.  Pageable host memory is refused.
bool device_reachable(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeHost ||
           at.type == cudaMemoryTypeManaged;
}

pkv_status check_common(int H, int D, int B, int64_t num_blocks, pkv_dtype dtype,
                        const char* fn) {
    if (H < 1) return pkv::fail(PKV_ERR_INVALID, "%s: num_heads must be >= 1", fn);
    if (D != 64 && D != 128) return pkv::fail(PKV_ERR_INVALID, "%s: head_dim must be 64 or 128", fn);
    if (B != 8 && B != 16 && B != 32 && B != 64)
        return pkv::fail(PKV_ERR_INVALID, "%s: block_size must be 8, 16, 32 or 64", fn);
    if (num_blocks < 1) return pkv::fail(PKV_ERR_INVALID, "%s: num_blocks must be >= 1", fn);
    if (dtype != PKV_F16 && dtype != PKV_BF16)
        return pkv::fail(PKV_ERR_INVALID, "%s: unknown dtype", fn);
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_heads,
                                 int head_dim, int block_size, int64_t num_blocks,
                                 pkv_dtype dtype, cudaStream_t stream) {
    const char* fn = "pkv_reshape_and_cache";
    pkv_status st = check_common(num_heads, head_dim, block_size, num_blocks, dtype, fn);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return pkv::fail(PKV_ERR_INVALID, "%s: num_tokens < 0", fn);
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID, "%s: k, v and the caches must be 16-byte aligned", fn);
    if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7) != 0)
        return pkv::fail(PKV_ERR_INVALID, "%s: slot_mapping must be 8-byte aligned", fn);
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no CUDA device", fn);
    cudaError_t e = pkv::launch_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                                  num_heads, head_dim, block_size, num_blocks, err,
                                                  stream);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                           int num_heads, int head_dim, int block_size, int64_t num_blocks,
                           pkv_dtype dtype, cudaStream_t stream) {
    const char* fn = "pkv_copy_blocks";
    pkv_status st = check_common(num_heads, head_dim, block_size, num_blocks, dtype, fn);
    if (st != PKV_OK) return st;
    if (num_pairs < 0 || num_pairs > 65535)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_pairs must be in [0, 65535]", fn);
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !pairs) return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return pkv::fail(PKV_ERR_INVALID, "%s: the caches must be 16-byte aligned", fn);
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no CUDA device", fn);
    cudaError_t e = pkv::launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_heads,
                                            head_dim, block_size, num_blocks, err, stream);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

pkv_status pkv_swap_blocks(void* dst_k_cache, void* dst_v_cache, const void* src_k_cache,
                           const void* src_v_cache, const int32_t* pairs, int num_pairs,
                           int num_heads, int head_dim, int block_size, int64_t src_num_blocks,
                           int64_t dst_num_blocks, pkv_dtype dtype, cudaStream_t stream) {
    const char* fn = "pkv_swap_blocks";
    pkv_status st = check_common(num_heads, head_dim, block_size,
                                 src_num_blocks < dst_num_blocks ? src_num_blocks : dst_num_blocks,
                                 dtype, fn);
    if (st != PKV_OK) return st;
    if (num_pairs < 0 || num_pairs > 65535)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_pairs must be in [0, 65535]", fn);
    if (num_pairs == 0) return PKV_OK;
    if (!dst_k_cache || !dst_v_cache || !src_k_cache || !src_v_cache || !pairs)
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned16(dst_k_cache) || !aligned16(dst_v_cache) || !aligned16(src_k_cache) ||
        !aligned16(src_v_cache))
        return pkv::fail(PKV_ERR_INVALID, "%s: the pools must be 16-byte aligned", fn);
    if (!device_reachable(dst_k_cache) || !device_reachable(dst_v_cache) ||
        !device_reachable(src_k_cache) || !device_reachable(src_v_cache) ||
        !device_reachable(pairs))
        return pkv::fail(PKV_ERR_INVALID,
                         "%s: pools and pairs must be device, pinned host or managed memory", fn);
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no CUDA device", fn);
    cudaError_t e = pkv::launch_swap_blocks(dst_k_cache, dst_v_cache, src_k_cache, src_v_cache,
                                            pairs, num_pairs, num_heads, head_dim, block_size,
                                            src_num_blocks, dst_num_blocks, err, stream);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

}  // extern "C"
