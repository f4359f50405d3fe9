// Decode attention for callers that cannot allocate device memory.
//
// pkv_paged_attention_decode needs a caller-provided workspace.  Some callers
// cannot provide one: a serving loop whose device memory is planned once at
// start-up and may not grow afterwards, or a plugin whose enqueue callback is
// not allowed to allocate (and has no workspace handed to it).  This entry
// point gives them the same computation with its scratch in a fixed array of
// the library's own static device memory, so the call itself allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
#include <mutex>

#include "pkv_internal.h"

namespace {

// The scratch: PKV_NOALLOC_SCRATCH_BYTES per device, reserved when the library
// is loaded on that device and held until the process exits.  Every call on a
// device shares it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Host code cannot use g_noalloc_scratch's name as a device address; look the
// address up once per device, with that device current.
pkv_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "pkv_paged_attention_decode_noalloc: device");
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::fail(PKV_ERR_INVALID, "pkv_paged_attention_decode_noalloc: device id %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return pkv::cuda_fail(e, "pkv_paged_attention_decode_noalloc: scratch address");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale,
                                              int num_seqs, int num_heads, int head_dim,
                                              int block_size, int max_blocks_per_seq,
                                              int64_t num_blocks, pkv_dtype dtype,
                                              int partition_size, cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_decode_noalloc";
    size_t need = 0;
    pkv_status st = pkv_decode_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                              max_blocks_per_seq, partition_size, &need);
    if (st != PKV_OK) return st;
    if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES)
        return pkv::fail(PKV_ERR_INVALID,
                         "%s: these sizes need %zu bytes of scratch but the static array holds "
                         "%zu; use pkv_paged_attention_decode with a workspace",
                         fn, need, (size_t)PKV_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    // The scratch needs no clearing.  Within one call the header, the step
    // prefix and the partials are written before they are read.  The one word
    // read before this call writes it, the claim word of the dynamic chunks,
    // carries the tag of the call that stamped it; a claimant ignores a word
    // whose tag is not its own call's, so what an earlier call left there is
    // never counted.  The remaining argument checks (num_blocks, dtype, scale,
    // pointers) and the empty batch are handled by the workspace entry point,
    // so both entry points answer the same arguments with the same status.
    return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                      num_seqs, num_heads, head_dim, block_size,
                                      max_blocks_per_seq, num_blocks, dtype, partition_size,
                                      scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
