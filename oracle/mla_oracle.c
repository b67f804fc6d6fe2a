/*
 * mla_oracle.c -- CPU reference for Multi-Head Latent Attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * Everything is plain fp64 loops in the order the pages state the method.
 * Nothing is blocked, fused or reordered.  In particular the decode computes
 * MLA the UNMERGED way: every head's keys and values are expanded from the
 * cached latents and then ordinary masked softmax attention runs on them.  The
 * absorbed form used on the GPU is a different association of the same
 * products and is never used here.
 *
 * Notation (row vectors, as on "Multi-Head Latent Attention (MLA)",
 * section "The construction"):
 *   c_i   = x_i . W_L            latent of token i, d_L values, shared by all heads
 *   kr_i  = RoPE(x_i . W_KR, i)  decoupled rotary key part, d_R values, shared by all heads
 *   k_h,i = [c_i . W_LK_h , kr_i]   per-head key   (W_LK_h is d_L x d_n)
 *   v_h,i =  c_i . W_LV_h           per-head value (W_LV_h is d_L x d_v)
 * Cache row of token i = [c_i | kr_i], d_L + d_R values.
 *
 * Pages followed:
 *   "Latent Space Strikes Again", "The Core Idea": attention formula, latent
 *       compression c_i = U x_i, up-projections k_i = B_K c_i, v_i = B_V c_i.
 *   "Multi-Head Latent Attention (MLA)", "The construction": factorisation
 *       W_K = W_L W_LK, W_V = W_L W_LV, W_Q = W_LQ W_LQQ, cache L = X W_L;
 *       "The RoPE problem": a separate non-latent key/query part carries RoPE.
 *   "How DeepSeek Rewrote the Transformer (MLA)", section 03 "Building
 *       attention from matrices": score, causal mask, divide by sqrt(dim),
 *       row softmax, weighted sum of values, stack heads and multiply by W_O;
 *       section 04 "The KV cache": decode needs only the newest query row;
 *       section 05 "Four megabytes per token": cache holds 2 N DH NH L numbers.
 *   "Multi-Head Latent Attention: How DeepSeek Shrinks AI Memory", "How does
 *       multi-head latent attention work?": 512-value latent plus a 64-value
 *       decoupled position piece per token per layer.
 *
 * Readings where the pages are silent (the same list is kept with the design
 * notes of the repository):
 *   - RoPE formula: interleaved pairs (2j, 2j+1) rotated by angle pos*theta_j,
 *     theta_j = base^(-2j/d_R); (a, b) -> (a cos - b sin, a sin + b cos).
 *   - The key RoPE part is one vector per token shared by all heads; the query
 *     RoPE part is per head.  The cache stores the key part after rotation.
 *   - seq_len counts attended tokens including the current one; key i sits at
 *     position i and the query at position seq_len-1.
 *   - softmax scale is a parameter (default 1/sqrt(d_n + d_R)).
 *
 * Planted mistakes: the `plant` argument of the decode and RoPE routines
 * deliberately breaks one step (used only by tests that show each pin catches
 * a plausible error).  plant == 0 is the real oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PLANT_NONE 0
#define ORACLE_PLANT_DROP_ROPE_TERM 1   /* score ignores q_pe . kr           */
#define ORACLE_PLANT_TRANSPOSE_WLK 2    /* reads W_LK_h with swapped indices */
#define ORACLE_PLANT_ROPE_SIGN 3        /* rotates by -angle                  */
#define ORACLE_PLANT_MASK_OFF_BY_ONE 4  /* attends one token too few          */
#define ORACLE_PLANT_NO_SCALE 5         /* forgets the 1/sqrt(dim) scale      */
#define ORACLE_PLANT_VALUE_FROM_KEY 6   /* uses W_LK_h in place of W_LV_h     */

int mla_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Rotary position embedding of one d_r-vector at position pos (reading above). */
void mla_oracle_rope(const double* in, int d_r, double pos, double base, int plant,
                     double* out) {
    for (int j = 0; j < d_r / 2; ++j) {
        double theta = pow(base, -2.0 * (double)j / (double)d_r);
        double phi = pos * theta;
        if (plant == ORACLE_PLANT_ROPE_SIGN) phi = -phi;
        double c = cos(phi), s = sin(phi);
        double a = in[2 * j], b = in[2 * j + 1];
        out[2 * j] = a * c - b * s;
        out[2 * j + 1] = a * s + b * c;
    }
}

/*
 * Down-projection of new tokens into cache rows ("The construction": L = X W_L;
 * "The RoPE problem": separate rotary key part).
 *   x      [n_tok][d_in]
 *   w_dkv  [d_in][d_l + d_r]   columns 0..d_l-1 are W_L, the rest W_KR
 *   pos    [n_tok]             position of each token
 *   rows   [n_tok][d_l + d_r]  out: [c | RoPE(x W_KR, pos)]
 */
void mla_oracle_latent_rows(const double* x, int n_tok, int d_in, const double* w_dkv,
                            int d_l, int d_r, const int32_t* pos, double base,
                            double* rows) {
    int dr = d_l + d_r;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)(d_r > 0 ? d_r : 1));
    for (int t = 0; t < n_tok; ++t) {
        const double* xt = x + (size_t)t * d_in;
        double* row = rows + (size_t)t * dr;
        for (int j = 0; j < dr; ++j) {
            double acc = 0.0;
            for (int k = 0; k < d_in; ++k) acc += xt[k] * w_dkv[(size_t)k * dr + j];
            row[j] = acc;
        }
        if (d_r > 0) {
            memcpy(tmp, row + d_l, sizeof(double) * d_r);
            mla_oracle_rope(tmp, d_r, (double)pos[t], base, 0, row + d_l);
        }
    }
    free(tmp);
}

/*
 * Query of the current token (page "Latent Space Strikes Again": optional
 * query compression q = B_Q U_Q x; page "Multi-Head Latent Attention (MLA)":
 * W_Q = W_LQ W_LQQ, plus a rotary query part per head).
 *   x     [batch][d_in]
 *   w_dq  [d_in][d_lq] or NULL (then the query comes from x directly, d_lq = d_in)
 *   w_uq  [d_lq][heads][d_n + d_r]   per head: d_n latent-side columns then d_r rotary
 *   pos   [batch]
 *   q_nope [batch][heads][d_n], q_pe [batch][heads][d_r]  (out)
 */
void mla_oracle_query(const double* x, int batch, int d_in, const double* w_dq, int d_lq,
                      const double* w_uq, int heads, int d_n, int d_r, const int32_t* pos,
                      double base, double* q_nope, double* q_pe) {
    int dq = d_n + d_r;
    int width = heads * dq;
    int din2 = w_dq ? d_lq : d_in;
    double* cq = (double*)malloc(sizeof(double) * (size_t)din2);
    double* raw = (double*)malloc(sizeof(double) * (size_t)(d_r > 0 ? d_r : 1));
    for (int b = 0; b < batch; ++b) {
        const double* xb = x + (size_t)b * d_in;
        if (w_dq) {
            for (int j = 0; j < d_lq; ++j) {
                double acc = 0.0;
                for (int k = 0; k < d_in; ++k) acc += xb[k] * w_dq[(size_t)k * d_lq + j];
                cq[j] = acc;
            }
        } else {
            memcpy(cq, xb, sizeof(double) * (size_t)d_in);
        }
        for (int h = 0; h < heads; ++h) {
            for (int j = 0; j < dq; ++j) {
                double acc = 0.0;
                for (int k = 0; k < din2; ++k)
                    acc += cq[k] * w_uq[(size_t)k * width + (size_t)h * dq + j];
                if (j < d_n)
                    q_nope[((size_t)b * heads + h) * d_n + j] = acc;
                else
                    raw[j - d_n] = acc;
            }
            if (d_r > 0)
                mla_oracle_rope(raw, d_r, (double)pos[b], base, 0,
                                q_pe + ((size_t)b * heads + h) * d_r);
        }
    }
    free(cq);
    free(raw);
}

/*
 * Physical row of logical token i of sequence b in a paged cache:
 * block_table[b][i / block_size] * block_size + i % block_size.
 * Returns -1 when the block id is outside [0, num_blocks).
 */
int64_t mla_oracle_slot(const int32_t* block_table, int max_blocks, int block_size,
                        int64_t num_blocks, int b, int i) {
    int32_t blk = block_table[(size_t)b * max_blocks + i / block_size];
    if (blk < 0 || (int64_t)blk >= num_blocks) return -1;
    return (int64_t)blk * block_size + i % block_size;
}

/*
 * Byte-level scatter of dense rows into the paged cache with the index map
 * above (section 04 "The KV cache": appending must leave earlier rows alone).
 * Returns the number of rows skipped because of an invalid block id.
 */
int mla_oracle_scatter_rows(const uint8_t* rows, int n_tok, int64_t row_bytes,
                            const int32_t* seq_idx, const int32_t* pos,
                            const int32_t* block_table, int max_blocks, int block_size,
                            int64_t num_blocks, uint8_t* cache) {
    int skipped = 0;
    for (int t = 0; t < n_tok; ++t) {
        int64_t slot = mla_oracle_slot(block_table, max_blocks, block_size, num_blocks,
                                       seq_idx[t], pos[t]);
        if (slot < 0) { ++skipped; continue; }
        memcpy(cache + slot * row_bytes, rows + (int64_t)t * row_bytes, (size_t)row_bytes);
    }
    return skipped;
}

/*
 * Unmerged MLA decode for one (sequence, head).  Follows section 03 of
 * "How DeepSeek Rewrote the Transformer (MLA)": scores of the newest query row
 * against every cached key, causal mask, divide by sqrt(dim), softmax, weighted
 * sum of values; the keys and values are the per-head up-projections of the
 * cached latents ("Latent Space Strikes Again", step 2).
 *
 * Outputs for this (b, h):
 *   o_v   [d_v]  sum_i p_i v_h,i              (the head's attention output)
 *   o_lat [d_l]  sum_i p_i c_i                (same weights applied to latents)
 *   lse          log sum_i exp(s_i)           (natural log)
 */
/* Widens one stored cache row to fp64.  kind 0: fp64, 1: fp32, 2: bf16 bit
 * patterns (the upper 16 bits of an IEEE fp32, so widening is exact). */
static void load_row(const void* cache, int kind, int64_t slot, int dr, double* out) {
    if (kind == 0) {
        const double* p = (const double*)cache + slot * dr;
        for (int j = 0; j < dr; ++j) out[j] = p[j];
    } else if (kind == 1) {
        const float* p = (const float*)cache + slot * dr;
        for (int j = 0; j < dr; ++j) out[j] = (double)p[j];
    } else {
        const uint16_t* p = (const uint16_t*)cache + slot * dr;
        for (int j = 0; j < dr; ++j) {
            uint32_t bits = (uint32_t)p[j] << 16;
            float f;
            memcpy(&f, &bits, sizeof f);
            out[j] = (double)f;
        }
    }
}

static void decode_one(const void* cache, int kind, int d_l, int d_r, const int32_t* block_table,
                       int max_blocks, int block_size, int64_t num_blocks, int b, int n,
                       const double* q_nope_h, const double* q_pe_h, const double* w_uk_h,
                       const double* w_uv_h, int d_n, int d_v, double scale, int plant,
                       double* o_v, double* o_lat, double* lse) {
    int dr = d_l + d_r;
    int q_pos = n - 1;                       /* query sits at the last position */
    int n_att = n;                           /* keys 0..n-1 exist in the cache  */
    if (plant == ORACLE_PLANT_MASK_OFF_BY_ONE) n_att = n - 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double* k = (double*)malloc(sizeof(double) * (size_t)d_n);
    double* v = (double*)malloc(sizeof(double) * (size_t)d_v);
    double* row = (double*)malloc(sizeof(double) * (size_t)dr);

    /* scores with the causal mask: key i is visible iff i <= query position */
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
        if (i > q_pos || i >= n_att) { s[i] = -INFINITY; continue; }
        int64_t slot = mla_oracle_slot(block_table, max_blocks, block_size, num_blocks, b, i);
        load_row(cache, kind, slot, dr, row);
        /* k_h,i = c_i . W_LK_h  (W_LK_h is d_l x d_n, row-major) */
        for (int j = 0; j < d_n; ++j) {
            double acc = 0.0;
            for (int l = 0; l < d_l; ++l) {
                double w = (plant == ORACLE_PLANT_TRANSPOSE_WLK)
                               ? w_uk_h[(size_t)(j % d_l) * d_n + (l % d_n)]
                               : w_uk_h[(size_t)l * d_n + j];
                acc += row[l] * w;
            }
            k[j] = acc;
        }
        double dot = 0.0;
        for (int j = 0; j < d_n; ++j) dot += q_nope_h[j] * k[j];
        if (plant != ORACLE_PLANT_DROP_ROPE_TERM)
            for (int r = 0; r < d_r; ++r) dot += q_pe_h[r] * row[d_l + r];
        s[i] = (plant == ORACLE_PLANT_NO_SCALE) ? dot : dot * scale;
        if (s[i] > m) m = s[i];
    }
    /* softmax: subtract the max, exponentiate, normalise so the row sums to 1 */
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
        double p = (s[i] == -INFINITY) ? 0.0 : exp(s[i] - m);
        s[i] = p;
        sum += p;
    }
    for (int j = 0; j < d_v; ++j) o_v[j] = 0.0;
    for (int l = 0; l < d_l; ++l) o_lat[l] = 0.0;
    if (sum > 0.0) {
        for (int i = 0; i < n; ++i) {
            double p = s[i] / sum;
            if (p == 0.0) continue;
            int64_t slot = mla_oracle_slot(block_table, max_blocks, block_size, num_blocks, b, i);
            load_row(cache, kind, slot, dr, row);
            /* v_h,i = c_i . W_LV_h, expanded explicitly */
            for (int j = 0; j < d_v; ++j) {
                double acc = 0.0;
                for (int l = 0; l < d_l; ++l) {
                    double w = (plant == ORACLE_PLANT_VALUE_FROM_KEY)
                                   ? w_uk_h[(size_t)l * d_n + (j % d_n)]
                                   : w_uv_h[(size_t)l * d_v + j];
                    acc += row[l] * w;
                }
                v[j] = acc;
            }
            for (int j = 0; j < d_v; ++j) o_v[j] += p * v[j];
            for (int l = 0; l < d_l; ++l) o_lat[l] += p * row[l];
        }
        *lse = m + log(sum);
    } else {
        *lse = -INFINITY;
    }
    free(s);
    free(k);
    free(v);
    free(row);
}

/*
 * Batched unmerged decode.
 *   cache        [num_blocks][block_size][d_l + d_r], stored as cache_kind
 *                (0 fp64, 1 fp32, 2 bf16 bit patterns)
 *   block_table  [batch][max_blocks]
 *   seq_lens     [batch]   attended tokens including the current one
 *   q_nope       [batch][heads][d_n],  q_pe [batch][heads][d_r]
 *   w_uk         [heads][d_l][d_n],    w_uv [heads][d_l][d_v]
 *   w_o          [heads*d_v][d_model] or NULL
 *   pairs        list of n_pairs (b, h) index pairs to compute (b*heads + h),
 *                or NULL for all of them
 * Outputs (entries of unlisted pairs are left untouched):
 *   o_lat [batch][heads][d_l], o_v [batch][heads][d_v], lse [batch][heads]
 *   out   [batch][d_model] = sum_h o_v[b][h] . W_O_h   (only when w_o != NULL
 *         and pairs == NULL)
 * Returns 0, or -1 when a needed block id is invalid or a seq_len is out of range.
 */
int mla_oracle_decode(const void* cache, int cache_kind, int64_t num_blocks, int block_size,
                      const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                      int batch, int heads, int d_l, int d_r, int d_n, int d_v,
                      const double* q_nope, const double* q_pe, const double* w_uk,
                      const double* w_uv, double scale, const double* w_o, int d_model,
                      const int32_t* pairs, int n_pairs, int plant, double* o_lat,
                      double* o_v, double* lse, double* out) {
    /* validate the index map before touching the cache */
    for (int b = 0; b < batch; ++b) {
        int n = seq_lens[b];
        if (n < 1 || n > max_blocks * block_size) return -1;
        for (int i = 0; i < n; i += block_size)
            if (mla_oracle_slot(block_table, max_blocks, block_size, num_blocks, b, i) < 0)
                return -1;
    }
    int total = pairs ? n_pairs : batch * heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int idx = 0; idx < total; ++idx) {
        int bh = pairs ? pairs[idx] : idx;
        int b = bh / heads, h = bh % heads;
        decode_one(cache, cache_kind, d_l, d_r, block_table, max_blocks, block_size, num_blocks, b,
                   seq_lens[b], q_nope + (size_t)bh * d_n, q_pe + (size_t)bh * d_r,
                   w_uk + (size_t)h * d_l * d_n, w_uv + (size_t)h * d_l * d_v, d_n, d_v,
                   scale, plant, o_v + (size_t)bh * d_v, o_lat + (size_t)bh * d_l,
                   lse + bh);
    }
    /* stack the heads and multiply by W_O (section 03, last step) */
    if (w_o && !pairs) {
        for (int b = 0; b < batch; ++b)
            for (int j = 0; j < d_model; ++j) {
                double acc = 0.0;
                for (int h = 0; h < heads; ++h)
                    for (int e = 0; e < d_v; ++e)
                        acc += o_v[((size_t)b * heads + h) * d_v + e] *
                               w_o[((size_t)h * d_v + e) * d_model + j];
                out[(size_t)b * d_model + j] = acc;
            }
    }
    return 0;
}

/*
 * Cache size per token, in numbers, from section 05 "Four megabytes per
 * token": standard attention keeps keys and values for every head of every
 * layer, 2 * DH * NH * L per token (kv_heads = NH for MHA, fewer for GQA/MQA).
 * MLA keeps one latent of d_l plus the d_r rotary part per layer.
 */
double mla_oracle_kv_numbers_per_token(int kv_heads, int head_dim, int layers) {
    return 2.0 * (double)head_dim * (double)kv_heads * (double)layers;
}

double mla_oracle_latent_numbers_per_token(int d_l, int d_r, int layers) {
    return (double)(d_l + d_r) * (double)layers;
}
