// Prompt-phase (prefill) attention over the paged cache.
//
// What it computes (wywy.jp notes, "prompt phase": every prompt token is
// known, so attention runs as matrix-matrix work; the block-indexed attention
// of the zhaifeiyue.github.io detail page, paper section 4.1, per query row):
// sequence s has qlen new tokens, already written to the cache at positions
// ctx - qlen .. ctx - 1; query token i (position p = ctx - qlen + i) attends
// positions 0 .. p (causal):
//   out[i][h] = sum_{t <= p} softmax_t(scale * q[i][h] . K[t][h]) V[t][h].
//
// Design: tensor cores (a dense contraction here, unlike decode).  A CTA of
// four warps takes 64 query rows of one (sequence, head); K/V tiles of 64
// tokens are gathered through the block table with cp.async (16-B pieces,
// XOR-swizzled rows so ldmatrix is conflict-free; pieces past the context are
// zero-filled), double-buffered.  Each warp computes S = Q K^T for its 16 rows
// with mma.sync m16n8k16 (fp16/bf16 in, fp32 accumulate), applies the causal
// mask, updates an online softmax in log2 units, and accumulates O += P V with
// P re-packed from the S accumulators (for bf16, P = high part + residual, two
// products, so the weights keep about 16 bits).  Tiles run longest-first.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

constexpr int kBM = 64;        // query rows per CTA
constexpr int kBN = 64;        // keys per K/V tile
constexpr int kWarps = 4;      // 16 query rows per warp
constexpr int kThreads = kWarps * 32;

template <typename T>
struct Mma;

template <>
struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ uint32_t pack_out(float lo, float hi) { return pack(lo, hi); }
    // fp16 softmax weights keep 11 bits: no residual term needed
    static constexpr bool kSplitP = false;
    static __device__ __forceinline__ uint32_t pack_residual(float, float) { return 0u; }
};

template <>
struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ uint32_t pack_out(float lo, float hi) { return pack(lo, hi); }
    // bf16 softmax weights would keep only 8 bits: P = hi + residual, both
    // bf16, and P V takes two products (about 16 bits for the weights)
    static constexpr bool kSplitP = true;
    static __device__ __forceinline__ uint32_t pack_residual(float lo, float hi) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return pack(lo - __low2float(h), hi - __high2float(h));
    }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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

// 16-byte async copy; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] tile: the chunk index
// is XORed with the row's low three bits.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

struct PrefillArgs {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;
    float scale_log2;
    int S, H, B, max_blocks, max_query_len;
    int64_t num_blocks;
    int32_t* err;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) paged_prefill_kernel(const PrefillArgs a) {
    constexpr int CH = D / 8;                     // 16-byte chunks per row
    constexpr int TILE = kBN * D * 2;             // bytes of one K (or V) tile
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* Qs = smem;                     // [kBM][D]
    unsigned char* Ks = smem + kBM * D * 2;       // [2][kBN][D]
    unsigned char* Vs = Ks + 2 * TILE;            // [2][kBN][D]

    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = gridDim.x - 1 - blockIdx.x;  // longest (latest) query tiles first
    const int h = blockIdx.y, s = blockIdx.z;
    const int B = a.B;
    const int q0 = a.query_start[s];
    const int qlen = a.query_start[s + 1] - q0;
    const int ctx = a.context_lens[s];
    if (ctx < 0 || ctx > a.max_blocks * B || qlen < 0 || qlen > ctx) {
        if (tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(a.err, PKV_DEVERR_BAD_CONTEXT);
        return;
    }
    if (qlen > a.max_query_len && tid == 0 && blockIdx.x == 0 && h == 0)
        atomicOr(a.err, PKV_DEVERR_BAD_CONTEXT);     // rows past the grid stay unwritten
    const int q_begin = tile * kBM;
    if (q_begin >= qlen) return;
    const int rows = min(kBM, qlen - q_begin);
    const int pos0 = ctx - qlen + q_begin;           // position of the tile's first query
    const int last = pos0 + rows - 1;                // causal limit of the tile
    const int n_tiles = last / kBN + 1;
    const int nblk = (ctx + B - 1) / B;
    const int32_t* row_tab = a.block_tables + (int64_t)s * a.max_blocks;
    const T* qg = static_cast<const T*>(a.q);
    const T* kg = static_cast<const T*>(a.k_cache);
    const T* vg = static_cast<const T*>(a.v_cache);

    // --- Q tile (rows past qlen zero-filled)
    for (int i = tid; i < kBM * CH; i += kThreads) {
        const int r = i / CH, c = i - r * CH;
        const bool ok = r < rows;
        const T* src = ok ? qg + ((int64_t)(q0 + q_begin + r) * a.H + h) * D + c * 8 : qg;
        cp_async16(smem_u32(Qs) + swz<D>(r, c), src, ok ? 16 : 0);
    }
    // --- K/V tile loader: token t of tile j is cache position j*kBN + t
    auto load_kv = [&](int j, int stage) {
        const uint32_t kb = smem_u32(Ks + stage * TILE), vb = smem_u32(Vs + stage * TILE);
        for (int i = tid; i < kBN * CH; i += kThreads) {
            const int r = i / CH, c = i - r * CH;
            const int pos = j * kBN + r;
            int bytes = 0;
            int64_t off = 0;
            if (pos < ctx) {
                const int jb = pos / B;
                int64_t phys = jb < nblk ? row_tab[jb] : -1;
                if (phys < 0 || phys >= a.num_blocks) {
                    atomicOr(a.err, PKV_DEVERR_BAD_BLOCK);
                } else {
                    off = ((phys * a.H + h) * B + (pos - jb * B)) * D + c * 8;
                    bytes = 16;
                }
            }
            cp_async16(kb + swz<D>(r, c), kg + off, bytes);
            cp_async16(vb + swz<D>(r, c), vg + off, bytes);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // per warp: 16 query rows; thread holds rows g and g + 8 of them
    const int g = lane >> 2, t4 = lane & 3;
    const int qp_lo = pos0 + warp * 16 + g;          // positions of the thread's two rows
    const int qp_hi = qp_lo + 8;
    uint32_t qf[D / 16][4];
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    for (int j = 0; j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
            load_kv(j + 1, (j + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = warp * 16 + (lane & 15);
                ldsm_x4(qf[kk], smem_u32(Qs) + swz<D>(r, 2 * kk + (lane >> 4)));
            }
        }
        const uint32_t kb = smem_u32(Ks + (j & 1) * TILE), vb = smem_u32(Vs + (j & 1) * TILE);

        // S = Q K^T for 16 rows x 64 keys
        float sacc[kBN / 8][4];
#pragma unroll
        for (int n = 0; n < kBN / 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < kBN / 16; ++np) {
                uint32_t b[4];
                const int r = np * 16 + ((lane >> 4) << 3) + (lane & 7);
                ldsm_x4(b, kb + swz<D>(r, 2 * kk + ((lane >> 3) & 1)));
                Mma<T>::run(sacc[2 * np], qf[kk], b[0], b[1]);
                Mma<T>::run(sacc[2 * np + 1], qf[kk], b[2], b[3]);
            }
        }
        // causal mask (keys past the query's position; past ctx is implied),
        // scores in log2 units, online softmax
        float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
        for (int n = 0; n < kBN / 8; ++n) {
            const int kp = j * kBN + n * 8 + 2 * t4;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float lo = sacc[n][e] * a.scale_log2, hi = sacc[n][2 + e] * a.scale_log2;
                lo = (kp + e <= qp_lo) ? lo : -INFINITY;
                hi = (kp + e <= qp_hi) ? hi : -INFINITY;
                sacc[n][e] = lo;
                sacc[n][2 + e] = hi;
                mx_lo = fmaxf(mx_lo, lo);
                mx_hi = fmaxf(mx_hi, hi);
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
        }
        const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
        // a row with no valid key yet keeps -inf (only possible for padding rows)
        const float al_lo = mn_lo == -INFINITY ? 1.f : exp2f(m_lo - mn_lo);
        const float al_hi = mn_hi == -INFINITY ? 1.f : exp2f(m_hi - mn_hi);
        float rs_lo = 0.f, rs_hi = 0.f;
        uint32_t pa[kBN / 16][4];
        uint32_t pr[Mma<T>::kSplitP ? kBN / 16 : 1][4];
#pragma unroll
        for (int n = 0; n < kBN / 8; ++n) {
            const float p0 = mn_lo == -INFINITY ? 0.f : exp2f(sacc[n][0] - mn_lo);
            const float p1 = mn_lo == -INFINITY ? 0.f : exp2f(sacc[n][1] - mn_lo);
            const float p2 = mn_hi == -INFINITY ? 0.f : exp2f(sacc[n][2] - mn_hi);
            const float p3 = mn_hi == -INFINITY ? 0.f : exp2f(sacc[n][3] - mn_hi);
            rs_lo += p0 + p1;
            rs_hi += p2 + p3;
            // accumulator tiles n = 2k, 2k+1 form the A fragment of key step k
            pa[n >> 1][(n & 1) * 2 + 0] = Mma<T>::pack(p0, p1);
            pa[n >> 1][(n & 1) * 2 + 1] = Mma<T>::pack(p2, p3);
            if constexpr (Mma<T>::kSplitP) {
                pr[n >> 1][(n & 1) * 2 + 0] = Mma<T>::pack_residual(p0, p1);
                pr[n >> 1][(n & 1) * 2 + 1] = Mma<T>::pack_residual(p2, p3);
            }
        }
        l_lo = l_lo * al_lo + rs_lo;
        l_hi = l_hi * al_hi + rs_hi;
        m_lo = mn_lo;
        m_hi = mn_hi;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= al_lo;
            o[n][1] *= al_lo;
            o[n][2] *= al_hi;
            o[n][3] *= al_hi;
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t b[4];
                const int r = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
                ldsm_x4_t(b, vb + swz<D>(r, 2 * dp + (lane >> 4)));
                Mma<T>::run(o[2 * dp], pa[kk], b[0], b[1]);
                Mma<T>::run(o[2 * dp + 1], pa[kk], b[2], b[3]);
                if constexpr (Mma<T>::kSplitP) {
                    Mma<T>::run(o[2 * dp], pr[kk], b[0], b[1]);
                    Mma<T>::run(o[2 * dp + 1], pr[kk], b[2], b[3]);
                }
            }
        }
        __syncthreads();   // the stage is refilled by the load issued next iteration
    }

    // row sums across the quad, normalise, store
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
    }
    const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
    const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
    T* og = static_cast<T*>(a.out);
    const int r_lo = warp * 16 + g, r_hi = r_lo + 8;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int d = n * 8 + 2 * t4;
        if (r_lo < rows) {
            uint32_t v = Mma<T>::pack_out(o[n][0] * inv_lo, o[n][1] * inv_lo);
            *reinterpret_cast<uint32_t*>(og + ((int64_t)(q0 + q_begin + r_lo) * a.H + h) * D + d) = v;
        }
        if (r_hi < rows) {
            uint32_t v = Mma<T>::pack_out(o[n][2] * inv_hi, o[n][3] * inv_hi);
            *reinterpret_cast<uint32_t*>(og + ((int64_t)(q0 + q_begin + r_hi) * a.H + h) * D + d) = v;
        }
    }
}

template <typename T, int D>
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    const size_t smem = (size_t)kBM * D * 2 + 4 * (size_t)kBN * D * 2;
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.max_query_len + kBM - 1) / kBM), (unsigned)a.H,
                       (unsigned)a.S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, paged_prefill_kernel<T, D>, a);
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
                                       int max_query_len, pkv_dtype dtype, cudaStream_t stream) {
    const char* fn = "pkv_paged_attention_prefill";
    if (num_seqs < 0 || num_seqs > 65535)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_seqs must be in [0, 65535]", fn);
    if (num_heads < 1 || num_heads > 65535)
        return pkv::fail(PKV_ERR_INVALID, "%s: num_heads must be in [1, 65535]", fn);
    if (head_dim != 64 && head_dim != 128)
        return pkv::fail(PKV_ERR_INVALID, "%s: head_dim must be 64 or 128", fn);
    if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64)
        return pkv::fail(PKV_ERR_INVALID, "%s: block_size must be 8, 16, 32 or 64", fn);
    if (max_blocks_per_seq < 1 || num_blocks < 1 || max_query_len < 0)
        return pkv::fail(PKV_ERR_INVALID, "%s: bad sizes", fn);
    if ((int64_t)max_blocks_per_seq * block_size >= (1LL << 31))
        return pkv::fail(PKV_ERR_INVALID, "%s: context capacity overflows", fn);
    if (dtype != PKV_F16 && dtype != PKV_BF16) return pkv::fail(PKV_ERR_INVALID, "%s: dtype", fn);
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return pkv::fail(PKV_ERR_INVALID, "%s: scale is not finite", fn);
    if (num_seqs == 0 || max_query_len == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return pkv::fail(PKV_ERR_INVALID, "%s: NULL pointer", fn);
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return pkv::fail(PKV_ERR_INVALID, "%s: out, q and the caches must be 16-byte aligned", fn);
    int32_t* err = pkv::device_error_word();
    if (!err) return pkv::fail(PKV_ERR_CUDA, "%s: no CUDA device", fn);
    PrefillArgs a;
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.S = num_seqs;
    a.H = num_heads;
    a.B = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.max_query_len = max_query_len;
    a.num_blocks = num_blocks;
    a.err = err;
    cudaError_t e;
    if (dtype == PKV_F16)
        e = head_dim == 128 ? launch_prefill<__half, 128>(a, stream)
                            : launch_prefill<__half, 64>(a, stream);
    else
        e = head_dim == 128 ? launch_prefill<__nv_bfloat16, 128>(a, stream)
                            : launch_prefill<__nv_bfloat16, 64>(a, stream);
    if (e != cudaSuccess) return pkv::cuda_fail(e, fn);
    return PKV_OK;
}

}  // extern "C"
