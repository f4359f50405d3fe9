// Internal declarations shared by the library's translation units (host side,
// plus the workspace layout that host and device code must agree on).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "pagedkv.h"

namespace pkv {

// ---- status / last error ---------------------------------------------------
pkv_status fail(pkv_status st, const char* fmt, ...);
pkv_status cuda_fail(cudaError_t e, const char* what);
void clear_last_error();

// ---- device error word (one per device, lives in errors.cu) -----------------
// Returns the device address of the error word of the current device.
int32_t* device_error_word();

// ---- device facts, cached per device ---------------------------------------
int sm_count(int device);

// ---- decode work split -------------------------------------------------------
// Balanced split: each CTA streams a static share of STATIC_EIGHTHS/8 of the
// steps; the rest is cut into DYN_PER_CTA chunks per CTA that CTAs claim as
// they finish (0 turns the dynamic tail off).  Shared by host (workspace
// bound) and device (the split).
#ifndef PKV_DECODE_STATIC_EIGHTHS
#define PKV_DECODE_STATIC_EIGHTHS 6
#endif
#ifndef PKV_DECODE_DYN_PER_CTA
#define PKV_DECODE_DYN_PER_CTA 4
#endif

// Tokens per pipeline step: a step moves 4 KiB of K and 4 KiB of V (16 tokens
// at head_dim 128, 32 at head_dim 64), from one block or from several
// consecutive logical blocks when the block size is smaller.
__host__ __device__ constexpr int step_tokens(int D) { return 2048 / D; }

// ---- decode workspace layout -------------------------------------------------
// [0, 64)                  header: int64 static chunk length, int64 total steps,
//                          uint64 claim word of the dynamic chunks (epoch << 24 | count)
// [64, 64 + 4 (S + 1))     int32 step prefix per sequence (written by CTA 0)
// then, 256-aligned:       float2 ml[cap]   (running max in log2 units, sum)
// then, 256-aligned:       float  acc[cap][D] (unnormalised output)
// cap = S * H + (max number of chunks)
//
// The shared-prefix entry point appends, 256-aligned:
//   int32 gh[16]             U (group units), slots used, written by the group pass
//   int32 gseq[S]            per sequence: group prefix steps (bits 0-19), member
//                            index (20-23), group size - 1 (24-26); 0 = no group
//   int32 gslot[S]           per sequence: its first group partial slot (head 0)
//   GroupUnit gunit[gunit_cap]
//   float2 gml[gslot_cap], float gacc[gslot_cap][D]   group partials
struct WsLayout {
    size_t base_off, ml_off, acc_off, total;
    int64_t cap;
    size_t gh_off, gseq_off, gslot_off, gunit_off, gml_off, gacc_off;
    int64_t gunit_cap, gslot_cap;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int S, int H, int D, int64_t max_chunks,
                                              int64_t gunit_cap = 0, int64_t gslot_cap = 0) {
    WsLayout w;
    w.cap = (int64_t)S * H + max_chunks;
    w.base_off = 64;
    w.ml_off = align_up(w.base_off + 4 * (size_t)(S + 1), 256);
    w.acc_off = align_up(w.ml_off + 8 * (size_t)w.cap, 256);
    w.total = align_up(w.acc_off + 4 * (size_t)w.cap * D, 256);
    w.gunit_cap = gunit_cap;
    w.gslot_cap = gslot_cap;
    w.gh_off = w.gseq_off = w.gslot_off = w.gunit_off = w.gml_off = w.gacc_off = w.total;
    if (gslot_cap > 0) {
        w.gh_off = w.total;
        w.gseq_off = w.gh_off + 64;
        w.gslot_off = align_up(w.gseq_off + 4 * (size_t)S, 16);
        w.gunit_off = align_up(w.gslot_off + 4 * (size_t)S, 256);
        w.gml_off = align_up(w.gunit_off + 32 * (size_t)gunit_cap, 256);
        w.gacc_off = align_up(w.gml_off + 8 * (size_t)gslot_cap, 256);
        w.total = align_up(w.gacc_off + 4 * (size_t)gslot_cap * D, 256);
    }
    return w;
}

// ---- shared prefixes -----------------------------------------------------------
// Sequences adjacent in the batch whose block tables begin with the same full
// blocks form a group (at most kGroupMax members, a common prefix of at least
// kGroupMinSteps steps).  The group's common prefix is read once and attended
// by every member together; each member's own blocks are read as usual.
constexpr int kGroupMax = 8;
constexpr int kGroupMinSteps = 4;
constexpr int kGroupMaxSeqs = 4096;
constexpr int kGroupMaxPrefixSteps = (1 << 20) - 1;
// Steps per group unit: a unit's blocks fit one 32-entry table window.
__host__ __device__ constexpr int group_unit_steps(int D, int B) {
    return B < step_tokens(D) ? 32 / (step_tokens(D) / B) : 32;
}
struct GroupUnit {
    int L;        // the group's first sequence (its table is read)
    int h;        // head
    int j0, len;  // steps [j0, j0 + len) of the common prefix
    int g;        // members: sequences L .. L + g - 1
    int slot0;    // partial slot of member 0; member n at slot0 + n * mstride
    int mstride;
    int pad;
};

// Upper bound of the steps one sequence can have.
__host__ __device__ inline int64_t max_steps_per_seq(int D, int B, int max_blocks) {
    return ((int64_t)max_blocks * B + step_tokens(D) - 1) / step_tokens(D);
}

// ---- decode kernel dispatch ---------------------------------------------------
struct DecodeArgs {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    // paged layout only: the newest token's K and V ([S][H][D]), taken by the
    // attention from here and stored into the token's cache slot (null: the
    // cache already holds them)
    const void* k_new;
    const void* v_new;
    float scale_log2;        // softmax scale * log2(e)
    int S, H, max_blocks;
    int ctx_cap;             // largest valid context length (max_blocks * B, or the
                             // contiguous layout's token stride)
    int64_t kv_stride;       // contiguous layout: tokens per (sequence, head) row
    int64_t num_blocks;
    int64_t L_steps;         // fixed chunk length in steps, 0 = balanced
    int min_chunk_steps;     // balanced mode: lower bound of the chunk length
    int main_grid;           // CTAs of the main kernel
    uint64_t epoch;          // 40-bit tag of this call (claims of the dynamic chunks)
    uint64_t wait_ns;        // bound of the pipeline waits (pkv_set_decode_wait_limit)
    int mode;                // decode kind (kModePaged, kModeContig, kModeShared, kModeAppend)
    char* ws;
    WsLayout ws_l;
    int32_t* err;
};

struct DecodeKernel {
    // launch main + merge on `stream`; grid = number of persistent CTAs; tk/tv:
    // tiled maps of the K and V pools (read by the shared-prefix kernels only)
    cudaError_t (*launch)(const DecodeArgs& a, int grid, cudaStream_t stream,
                          const CUtensorMap& tk, const CUtensorMap& tv);
    // dynamic shared memory of the main kernel for S sequences
    size_t (*smem_bytes)(int S);
    // CTAs per SM the main kernel can keep resident with that shared memory
    cudaError_t (*occupancy)(int* ctas_per_sm, size_t smem);
    int threads;
};

const DecodeKernel* decode_kernel_f16(int D, int B);
const DecodeKernel* decode_kernel_bf16(int D, int B);
// the same, writing each sequence's newest token (kModeAppend)
const DecodeKernel* decode_kernel_append_f16(int D, int B);
const DecodeKernel* decode_kernel_append_bf16(int D, int B);
// the same kernels over a contiguous [seq][head][token][D] K/V layout (no block table)
const DecodeKernel* decode_kernel_contig_f16(int D);
const DecodeKernel* decode_kernel_contig_bf16(int D);
// the paged kernels with shared prefixes read once (a group pass launched first)
const DecodeKernel* decode_kernel_shared_f16(int D, int B);
const DecodeKernel* decode_kernel_shared_bf16(int D, int B);
// kModeAppend: the paged layout, with the newest token of every sequence
// taken from the call's k_new / v_new and written into its cache slot
enum : int { kModePaged = 0, kModeContig = 1, kModeShared = 2, kModeAppend = 3 };

// ---- cache kernels -----------------------------------------------------------
cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slots, int T, int H, int D, int B,
                                     int64_t num_blocks, int32_t* err, cudaStream_t stream);
cudaError_t launch_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                               const int32_t* pairs, int P, int H, int D, int B,
                               int64_t src_blocks, int64_t dst_blocks, int32_t* err,
                               cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int P,
                               int H, int D, int B, int64_t num_blocks, int32_t* err,
                               cudaStream_t stream);

}  // namespace pkv
