/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it follows (page titles as cited):
 *   - "Efficient Memory Management for Large Language Model Serving with
 *     PagedAttention" (wywy.jp notes), glossary entry "PagedAttention": K and V
 *     vectors live in non-contiguous blocks; the kernel multiplies the query
 *     with each block's keys to get scores, then weights the same block's
 *     values.  Same page, "Block table": logical block -> physical block.
 *   - zhaifeiyue.github.io detail page, core formula (the block-indexed
 *     attention A_ij / o_i, paper section 4.1) and the statement that it is
 *     mathematically equivalent to standard attention because the softmax
 *     denominator runs over all blocks.
 *   - ricepunchb garden "KV Cache Optimization", section 3.2 (address
 *     translation): block index = position / B, offset = position mod B,
 *     physical address = table[block index] * B + offset.
 *
 * Layout (the pages leave layout open; this is the reading used everywhere):
 *   k_cache, v_cache : [num_blocks][H][B][D] 16-bit words (fp16 or bf16)
 *   q                : [S][H][D] 16-bit words
 *   block_tables     : int32 [S][max_blocks]
 *   context_lens     : int32 [S]
 *   out              : double [S][H][D]
 *
 * Decode reading: the query of sequence s attends positions 0 .. ctx[s]-1
 * (its own, newest token included).  ctx[s] == 0 yields a zero row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F16 0
#define ORC_BF16 1

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);            /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400), expo - 25); /* (1.frac) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper 16 bits of an IEEE-754 binary32 word. */
double orc_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133);           /* frac * 2^-126 * 2^-7 */
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x80), expo - 134); /* (1.frac) * 2^(e-127) */
    }
    return sign ? -v : v;
}

static double widen(uint16_t w, int dtype) {
    return dtype == ORC_BF16 ? orc_bf16_to_f64(w) : orc_f16_to_f64(w);
}

/* Address translation (garden page, section 3.2): token i of a sequence lives in
 * logical block i / B at offset i mod B; the block table names the physical block. */
static int64_t kv_word_index(const int32_t* table_row, int64_t pos, int h, int d,
                             int H, int B, int D) {
    int64_t logical = pos / B;
    int64_t offset = pos % B;
    int64_t physical = table_row[logical];
    return ((physical * H + h) * B + offset) * D + d;
}

static int check_table_row(const int32_t* row, int32_t ctx, int B, int max_blocks,
                           int64_t num_blocks) {
    int64_t nblk = ((int64_t)ctx + B - 1) / B;
    if (ctx < 0 || nblk > max_blocks) return -1;
    for (int64_t j = 0; j < nblk; ++j)
        if (row[j] < 0 || row[j] >= num_blocks) return -1;
    return 0;
}

/*
 * Contiguous form: gather K_s, V_s through the table, then the textbook
 * softmax(scale * q K^T) V with the usual max subtraction, all in fp64.
 * Sequences [s_begin, s_end) are computed.  Returns 0, or -1 on a bad table.
 */
int orc_paged_attention_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                               const uint16_t* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, double scale, int S, int H,
                               int D, int B, int max_blocks, int64_t num_blocks, int dtype,
                               int s_begin, int s_end) {
    if (s_begin < 0) s_begin = 0;
    if (s_end > S) s_end = S;
    for (int s = s_begin; s < s_end; ++s) {
        const int32_t* row = block_tables + (int64_t)s * max_blocks;
        int32_t n = context_lens[s];
        if (check_table_row(row, n, B, max_blocks, num_blocks)) return -1;
        for (int h = 0; h < H; ++h) {
            double* o = out + ((int64_t)s * H + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) continue;
            double* K = (double*)malloc(sizeof(double) * (size_t)n * D);
            double* V = (double*)malloc(sizeof(double) * (size_t)n * D);
            double* z = (double*)malloc(sizeof(double) * (size_t)n);
            if (!K || !V || !z) { free(K); free(V); free(z); return -2; }
            /* gather into contiguous K and V */
            for (int64_t t = 0; t < n; ++t)
                for (int d = 0; d < D; ++d) {
                    int64_t w = kv_word_index(row, t, h, d, H, B, D);
                    K[t * D + d] = widen(k_cache[w], dtype);
                    V[t * D + d] = widen(v_cache[w], dtype);
                }
            const uint16_t* qrow = q + ((int64_t)s * H + h) * D;
            /* scores z_t = scale * q . K_t */
            double zmax = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += widen(qrow[d], dtype) * K[t * D + d];
                z[t] = scale * acc;
                if (z[t] > zmax) zmax = z[t];
            }
            /* softmax weights and weighted sum of V */
            double denom = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                z[t] = exp(z[t] - zmax);
                denom += z[t];
            }
            for (int64_t t = 0; t < n; ++t)
                for (int d = 0; d < D; ++d) o[d] += z[t] * V[t * D + d];
            for (int d = 0; d < D; ++d) o[d] /= denom;
            free(K); free(V); free(z);
        }
    }
    return 0;
}

/*
 * Block-indexed form, written the way the detail page's formula reads:
 *   A_ij = exp(q K_j / sqrt(d)) / sum_t sum_(tokens of block t) exp(q k / sqrt(d))
 *   o    = sum_j V_j A_ij^T
 * i.e. each block's exponentiated scores are formed block by block, the
 * denominator sums over every block, and no maximum is subtracted.  Positions
 * at or beyond ctx inside the last block are excluded.  It exists to show that
 * the block-wise reduction equals the contiguous softmax (used by tests only).
 */
int orc_paged_attention_decode_blockwise(double* out, const uint16_t* q,
                                         const uint16_t* k_cache, const uint16_t* v_cache,
                                         const int32_t* block_tables,
                                         const int32_t* context_lens, double scale, int S,
                                         int H, int D, int B, int max_blocks,
                                         int64_t num_blocks, int dtype) {
    for (int s = 0; s < S; ++s) {
        const int32_t* row = block_tables + (int64_t)s * max_blocks;
        int32_t n = context_lens[s];
        if (check_table_row(row, n, B, max_blocks, num_blocks)) return -1;
        int64_t nblk = ((int64_t)n + B - 1) / B;
        for (int h = 0; h < H; ++h) {
            double* o = out + ((int64_t)s * H + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) continue;
            const uint16_t* qrow = q + ((int64_t)s * H + h) * D;
            /* denominator: sum over all blocks t of the block's exp-scores */
            double denom = 0.0;
            for (int64_t j = 0; j < nblk; ++j) {
                int64_t phys = row[j];
                for (int b = 0; b < B && j * B + b < n; ++b) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) {
                        int64_t w = ((phys * H + h) * B + b) * D + d;
                        acc += widen(qrow[d], dtype) * widen(k_cache[w], dtype);
                    }
                    denom += exp(scale * acc);
                }
            }
            /* o = sum_j V_j A_ij^T */
            for (int64_t j = 0; j < nblk; ++j) {
                int64_t phys = row[j];
                for (int b = 0; b < B && j * B + b < n; ++b) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) {
                        int64_t w = ((phys * H + h) * B + b) * D + d;
                        acc += widen(qrow[d], dtype) * widen(k_cache[w], dtype);
                    }
                    double a = exp(scale * acc) / denom;
                    for (int d = 0; d < D; ++d) {
                        int64_t w = ((phys * H + h) * B + b) * D + d;
                        o[d] += widen(v_cache[w], dtype) * a;
                    }
                }
            }
        }
    }
    return 0;
}

/*
 * New-token write: each of the T tokens' K and V rows [H][D] goes to the slot
 * the block manager gave it; slot = physical block * B + offset (garden page
 * section 3.2), so the block is slot / B and the offset slot mod B.  A
 * negative slot means "no write".  Returns -1 if a slot is out of the pool.
 */
int orc_reshape_and_cache(const uint16_t* k, const uint16_t* v, uint16_t* k_cache,
                          uint16_t* v_cache, const int64_t* slot_mapping, int T, int H,
                          int D, int B, int64_t num_blocks) {
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * B) return -1;
        int64_t block = slot / B, offset = slot % B;
        for (int h = 0; h < H; ++h)
            for (int d = 0; d < D; ++d) {
                int64_t dst = ((block * H + h) * B + offset) * D + d;
                int64_t src = ((int64_t)t * H + h) * D + d;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
    }
    return 0;
}

/*
 * Block-granular copy for copy-on-write (wywy.jp notes, parallel sampling
 * example: the block engine copies the shared physical block's contents into
 * the newly allocated one).  pairs is int32 [P][2] = (src, dst); the whole
 * block, every head, is copied, in K and in V.
 */
int orc_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int32_t* pairs, int P,
                    int H, int D, int B, int64_t num_blocks) {
    int64_t words = (int64_t)H * B * D;
    for (int p = 0; p < P; ++p) {
        int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return -1;
        for (int64_t w = 0; w < words; ++w) {
            k_cache[dst * words + w] = k_cache[src * words + w];
            v_cache[dst * words + w] = v_cache[src * words + w];
        }
    }
    return 0;
}

/*
 * Swap between two pools (GPU and CPU swap space, wywy.jp notes, "Swapping"):
 * for each pair (src, dst), dst pool block dst = src pool block src, whole
 * blocks, K and V.
 */
int orc_swap_blocks(uint16_t* dst_k, uint16_t* dst_v, const uint16_t* src_k,
                    const uint16_t* src_v, const int32_t* pairs, int P, int H, int D, int B,
                    int64_t src_blocks, int64_t dst_blocks) {
    int64_t words = (int64_t)H * B * D;
    for (int p = 0; p < P; ++p) {
        int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) return -1;
        for (int64_t w = 0; w < words; ++w) {
            dst_k[dst * words + w] = src_k[src * words + w];
            dst_v[dst * words + w] = src_v[src * words + w];
        }
    }
    return 0;
}

/*
 * Prompt phase with the paged cache (wywy.jp notes, "prompt phase": every
 * prompt token is known, their K/V are produced together and attention runs
 * as matrix-matrix work).  Sequence s has qlen = query_start[s+1] -
 * query_start[s] new tokens whose K/V are already in the cache at positions
 * ctx - qlen .. ctx - 1; query token i (row query_start[s] + i of q and out)
 * sits at position p = ctx - qlen + i and attends positions 0 .. p (causal).
 * Each row is the decode definition with context length p + 1.
 */
int orc_paged_attention_prefill(double* out, const uint16_t* q, const uint16_t* k_cache,
                                const uint16_t* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, const int32_t* query_start,
                                double scale, int S, int H, int D, int B, int max_blocks,
                                int64_t num_blocks, int dtype) {
    for (int s = 0; s < S; ++s) {
        const int32_t* row = block_tables + (int64_t)s * max_blocks;
        int32_t n = context_lens[s];
        int32_t q0 = query_start[s], qlen = query_start[s + 1] - query_start[s];
        if (qlen < 0 || qlen > n) return -1;
        if (check_table_row(row, n, B, max_blocks, num_blocks)) return -1;
        for (int i = 0; i < qlen; ++i) {
            int64_t p = (int64_t)n - qlen + i;
            for (int h = 0; h < H; ++h) {
                double* o = out + ((int64_t)(q0 + i) * H + h) * D;
                const uint16_t* qrow = q + ((int64_t)(q0 + i) * H + h) * D;
                double* z = (double*)malloc(sizeof(double) * (size_t)(p + 1));
                if (!z) return -2;
                double zmax = -INFINITY;
                for (int64_t t = 0; t <= p; ++t) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += widen(qrow[d], dtype) *
                               widen(k_cache[kv_word_index(row, t, h, d, H, B, D)], dtype);
                    z[t] = scale * acc;
                    if (z[t] > zmax) zmax = z[t];
                }
                double denom = 0.0;
                for (int64_t t = 0; t <= p; ++t) {
                    z[t] = exp(z[t] - zmax);
                    denom += z[t];
                }
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int64_t t = 0; t <= p; ++t)
                        acc += z[t] * widen(v_cache[kv_word_index(row, t, h, d, H, B, D)], dtype);
                    o[d] = acc / denom;
                }
                free(z);
            }
        }
    }
    return 0;
}
