/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU oracle for the paged KV-cache
 * hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference legs may load or call this file.  The
 * product library never includes, links or calls it, and this file includes
 * nothing of the product: it shares no header, helper, table or constant with
 * the CUDA path.
 *
 * Every routine is the plain definition of what the method computes, written
 * out with no blocking, fusion or reordering:
 *
 *   - fp16 decode: IEEE 754 binary16 bit layout, decoded by hand.
 *   - slot translation: token t of a sequence lives in physical block
 *     table[t / B] at row t % B; flat slot = table[t / B] * B + t % B
 *     ("Why Naive KV-Caches Waste >60% VRAM", section 1 "Physical Block Pool &
 *     Block Tables": 35 tokens -> ceil(35/16) = 3 blocks; PageFault README,
 *     "The OS analogy": the page-table walk resolves a token address).
 *   - pool layout: per layer, K and V each [N_blocks][block_size][H][D]
 *     ("Why Naive KV-Caches Waste >60% VRAM", "Implementation Walkthrough":
 *     the cache is shaped [N_blocks, block_size, N_heads, D_head]); the layer
 *     index is an outer dimension (PageForge, "Five techniques", 04
 *     layer-combined pooling).
 *   - scatter / gather: copy one token row between a dense buffer and its slot
 *     (PageForge, "Four layers, one pointer": gather_kv assembles scattered
 *     pages into a contiguous buffer, scatter_kv_layer writes new tokens back).
 *   - attention: single-query softmax attention over a sequence's L tokens,
 *     z_t = scale * sum_d q_d K_td, p_t = exp(z_t - max z) / sum exp(z - max z),
 *     out_d = sum_t p_t V_td, in fp64, two-pass (PagedAttention blog, "The
 *     Attention Kernel"; PageFault README, "Four stages": the paged kernel has
 *     the same math as the contiguous stage-1 kernel).
 *   - partial / merge: the attention of a token subrange summarised as
 *     (m, l, acc) and combined with the log-sum-exp rule (PagedAttention blog,
 *     "The Attention Kernel": the reduction across thread blocks combines
 *     partial softmax results with the log-sum-exp trick).
 *   - memory accounting: PageFault README, "Calculate", core formulas.
 *
 * Readings where the pages are silent (head mapping for grouped heads, the
 * query attending to every token including the one just written, L = 0 giving
 * a zero output) are the plain ones; each is listed in the design notes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ fp16 */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Exact in fp64 for every pattern. */
double or_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);              /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac + 1024), expo - 25); /* 1.frac * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Decode a whole array (used to build dense fp64 copies in tests). */
void or_half_to_double_array(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = or_half_to_double(src[i]);
}

/* ----------------------------------------------------- slots and blocks */

int64_t or_blocks_needed(int64_t len, int64_t block_size)
{
    return (len + block_size - 1) / block_size;
}

/* Unused slots in a sequence's last page: (B - L % B) % B. */
int64_t or_tail_waste(int64_t len, int64_t block_size)
{
    return (block_size - len % block_size) % block_size;
}

/* Flat slot of logical token t for a sequence whose block table row is
 * table_row. */
int64_t or_slot(const int32_t *table_row, int64_t block_size, int64_t t)
{
    return (int64_t)table_row[t / block_size] * block_size + t % block_size;
}

/* Element offset of (layer, slot, head 0, dim 0) in a
 * [n_layers][n_blocks][block_size][n_heads][head_dim] pool. */
static int64_t row_offset(int64_t layer, int64_t n_blocks, int64_t block_size,
                          int64_t n_heads, int64_t head_dim, int64_t slot)
{
    return ((layer * n_blocks * block_size) + slot) * n_heads * head_dim;
}

/* --------------------------------------------------- scatter and gather */

/* Token i of the batch (sequence seq_idx[i], logical position pos[i]) is
 * written into its slot of layer `layer`.  k_new / v_new are
 * [n_tokens][n_heads][head_dim]. */
void or_scatter(uint16_t *k_pool, uint16_t *v_pool, int n_blocks,
                int block_size, int n_heads, int head_dim, int layer,
                const uint16_t *k_new, const uint16_t *v_new,
                const int32_t *block_tables, int max_blocks_per_seq,
                const int32_t *seq_idx, const int32_t *pos, int n_tokens)
{
    int64_t row = (int64_t)n_heads * head_dim;
    for (int i = 0; i < n_tokens; ++i) {
        const int32_t *table_row =
            block_tables + (int64_t)seq_idx[i] * max_blocks_per_seq;
        int64_t slot = or_slot(table_row, block_size, pos[i]);
        int64_t off = row_offset(layer, n_blocks, block_size, n_heads,
                                 head_dim, slot);
        memcpy(k_pool + off, k_new + (int64_t)i * row, row * sizeof(uint16_t));
        memcpy(v_pool + off, v_new + (int64_t)i * row, row * sizeof(uint16_t));
    }
}

/* Rebuild contiguous K/V: output row cu_off[s] + t holds token t of
 * sequence s, for t < context_lens[s]. */
void or_gather(const uint16_t *k_pool, const uint16_t *v_pool, int n_blocks,
               int block_size, int n_heads, int head_dim, int layer,
               const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, const int64_t *cu_off, int n_seqs,
               uint16_t *k_out, uint16_t *v_out)
{
    int64_t row = (int64_t)n_heads * head_dim;
    for (int s = 0; s < n_seqs; ++s) {
        const int32_t *table_row =
            block_tables + (int64_t)s * max_blocks_per_seq;
        for (int64_t t = 0; t < context_lens[s]; ++t) {
            int64_t slot = or_slot(table_row, block_size, t);
            int64_t src = row_offset(layer, n_blocks, block_size, n_heads,
                                     head_dim, slot);
            int64_t dst = (cu_off[s] + t) * row;
            memcpy(k_out + dst, k_pool + src, row * sizeof(uint16_t));
            memcpy(v_out + dst, v_pool + src, row * sizeof(uint16_t));
        }
    }
}

/* ------------------------------------------------- block copies, swap */

/* Offset of block `block` of layer `layer` in a pool [n_layers][N][block_elems]. */
static int64_t block_offset(int64_t layer, int64_t n_blocks, int64_t block,
                            int64_t block_elems)
{
    return (layer * n_blocks + block) * block_elems;
}

/* Copy-on-write copies (PagedAttention blog, "Copy-on-Write for Parallel
 * Sampling": a new physical block receives the contents of the shared one).
 * For i < n, block dst[i] takes the contents of block src[i], in every layer,
 * K and V.  block_elems = B * Hkv * D. */
void or_copy_blocks(uint16_t *k_pool, uint16_t *v_pool, int n_layers,
                    int n_blocks, int64_t block_elems, const int32_t *src,
                    const int32_t *dst, int n)
{
    for (int i = 0; i < n; ++i) {
        for (int layer = 0; layer < n_layers; ++layer) {
            int64_t from = block_offset(layer, n_blocks, src[i], block_elems);
            int64_t to = block_offset(layer, n_blocks, dst[i], block_elems);
            memcpy(k_pool + to, k_pool + from, block_elems * sizeof(uint16_t));
            memcpy(v_pool + to, v_pool + from, block_elems * sizeof(uint16_t));
        }
    }
}

/* Swapping (same blog, "Preemption and Swapping": blocks are evicted to CPU
 * memory one by one and copied back later).  The host image of block ids[i]
 * is images[i][layer][kv][block_elems], kv = 0 for K and 1 for V. */
void or_swap_out(const uint16_t *k_pool, const uint16_t *v_pool, int n_layers,
                 int n_blocks, int64_t block_elems, const int32_t *ids, int n,
                 uint16_t *images)
{
    for (int i = 0; i < n; ++i) {
        for (int layer = 0; layer < n_layers; ++layer) {
            int64_t from = block_offset(layer, n_blocks, ids[i], block_elems);
            uint16_t *img = images + (((int64_t)i * n_layers + layer) * 2) * block_elems;
            memcpy(img, k_pool + from, block_elems * sizeof(uint16_t));
            memcpy(img + block_elems, v_pool + from, block_elems * sizeof(uint16_t));
        }
    }
}

void or_swap_in(uint16_t *k_pool, uint16_t *v_pool, int n_layers, int n_blocks,
                int64_t block_elems, const uint16_t *images, const int32_t *ids,
                int n)
{
    for (int i = 0; i < n; ++i) {
        for (int layer = 0; layer < n_layers; ++layer) {
            int64_t to = block_offset(layer, n_blocks, ids[i], block_elems);
            const uint16_t *img = images + (((int64_t)i * n_layers + layer) * 2) * block_elems;
            memcpy(k_pool + to, img, block_elems * sizeof(uint16_t));
            memcpy(v_pool + to, img + block_elems, block_elems * sizeof(uint16_t));
        }
    }
}

/* ------------------------------------------------------------ attention */

/* One query row against L key/value rows given by pointer arrays.
 * Two passes: scores and their maximum, then normalised weights and the
 * weighted sum.  z is caller scratch of length L. */
static void attend_rows(const uint16_t *q, const uint16_t *const *k_rows,
                        const uint16_t *const *v_rows, int64_t L,
                        int head_dim, double scale, double *z, double *out)
{
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (L <= 0) return;
    double zmax = -INFINITY;
    for (int64_t t = 0; t < L; ++t) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += or_half_to_double(q[d]) * or_half_to_double(k_rows[t][d]);
        z[t] = scale * dot;
        if (z[t] > zmax) zmax = z[t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        z[t] = exp(z[t] - zmax);
        denom += z[t];
    }
    for (int64_t t = 0; t < L; ++t) {
        double p = z[t] / denom;
        for (int d = 0; d < head_dim; ++d)
            out[d] += p * or_half_to_double(v_rows[t][d]);
    }
}

/* Largest context length in the batch (sizes the scratch arrays). */
static int64_t max_len(const int32_t *lens, int n)
{
    int64_t m = 0;
    for (int i = 0; i < n; ++i)
        if (lens[i] > m) m = lens[i];
    return m;
}

/* Attention over a contiguous per-sequence cache (the unpaged baseline):
 * K/V rows of sequence s are kc/vc rows cu_off[s] .. cu_off[s] + L_s - 1,
 * each [n_kv_heads][head_dim].  q and out are [n_seqs][n_q_heads][head_dim];
 * q-head hq reads kv-head hq / (n_q_heads / n_kv_heads).  Returns 0, or -1 on
 * a bad argument or allocation failure. */
int or_attention_contiguous(const uint16_t *q, const uint16_t *kc,
                            const uint16_t *vc, const int64_t *cu_off,
                            const int32_t *context_lens, int n_seqs,
                            int n_q_heads, int n_kv_heads, int head_dim,
                            float scale, double *out)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads) return -1;
    int group = n_q_heads / n_kv_heads;
    int64_t lmax = max_len(context_lens, n_seqs);
    const uint16_t **kr = malloc((size_t)(lmax + 1) * sizeof(*kr));
    const uint16_t **vr = malloc((size_t)(lmax + 1) * sizeof(*vr));
    double *z = malloc((size_t)(lmax + 1) * sizeof(double));
    if (!kr || !vr || !z) { free(kr); free(vr); free(z); return -1; }
    int64_t row = (int64_t)n_kv_heads * head_dim;
    for (int s = 0; s < n_seqs; ++s) {
        for (int hq = 0; hq < n_q_heads; ++hq) {
            int hkv = hq / group;
            for (int64_t t = 0; t < context_lens[s]; ++t) {
                kr[t] = kc + (cu_off[s] + t) * row + (int64_t)hkv * head_dim;
                vr[t] = vc + (cu_off[s] + t) * row + (int64_t)hkv * head_dim;
            }
            int64_t qo = ((int64_t)s * n_q_heads + hq) * head_dim;
            attend_rows(q + qo, kr, vr, context_lens[s], head_dim,
                        (double)scale, z, out + qo);
        }
    }
    free(kr); free(vr); free(z);
    return 0;
}

/* Attention read back through the block tables from a host copy of the pool
 * ([n_layers][n_blocks][block_size][n_kv_heads][head_dim]).  Same arithmetic,
 * in the same order, as or_attention_contiguous: only the row addresses come
 * from the page-table walk. */
int or_attention_paged(const uint16_t *q, const uint16_t *k_pool,
                       const uint16_t *v_pool, int n_blocks, int block_size,
                       int n_kv_heads, int head_dim, int layer,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int n_seqs, int n_q_heads,
                       float scale, double *out)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads) return -1;
    int group = n_q_heads / n_kv_heads;
    int64_t lmax = max_len(context_lens, n_seqs);
    const uint16_t **kr = malloc((size_t)(lmax + 1) * sizeof(*kr));
    const uint16_t **vr = malloc((size_t)(lmax + 1) * sizeof(*vr));
    double *z = malloc((size_t)(lmax + 1) * sizeof(double));
    if (!kr || !vr || !z) { free(kr); free(vr); free(z); return -1; }
    for (int s = 0; s < n_seqs; ++s) {
        const int32_t *table_row =
            block_tables + (int64_t)s * max_blocks_per_seq;
        for (int hq = 0; hq < n_q_heads; ++hq) {
            int hkv = hq / group;
            for (int64_t t = 0; t < context_lens[s]; ++t) {
                int64_t slot = or_slot(table_row, block_size, t);
                int64_t off = row_offset(layer, n_blocks, block_size,
                                         n_kv_heads, head_dim, slot) +
                              (int64_t)hkv * head_dim;
                kr[t] = k_pool + off;
                vr[t] = v_pool + off;
            }
            int64_t qo = ((int64_t)s * n_q_heads + hq) * head_dim;
            attend_rows(q + qo, kr, vr, context_lens[s], head_dim,
                        (double)scale, z, out + qo);
        }
    }
    free(kr); free(vr); free(z);
    return 0;
}

/* Attention of one query row over the token subrange [t0, t1) of a
 * contiguous K/V sequence (rows of `row_stride` elements, kv-head columns at
 * head_off), summarised as m = max z, l = sum exp(z - m),
 * acc_d = sum exp(z - m) V_td.  An empty range gives m = -inf, l = 0,
 * acc = 0. */
void or_attention_partial(const uint16_t *q, const uint16_t *k,
                          const uint16_t *v, int64_t row_stride,
                          int64_t head_off, int head_dim, float scale,
                          int64_t t0, int64_t t1, double *m_out,
                          double *l_out, double *acc)
{
    for (int d = 0; d < head_dim; ++d) acc[d] = 0.0;
    double m = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += or_half_to_double(q[d]) *
                   or_half_to_double(k[t * row_stride + head_off + d]);
        double zt = (double)scale * dot;
        if (zt > m) m = zt;
    }
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += or_half_to_double(q[d]) *
                   or_half_to_double(k[t * row_stride + head_off + d]);
        double e = exp((double)scale * dot - m);
        l += e;
        for (int d = 0; d < head_dim; ++d)
            acc[d] += e * or_half_to_double(v[t * row_stride + head_off + d]);
    }
    *m_out = m;
    *l_out = l;
}

/* Log-sum-exp merge of n partial results (m_i, l_i, acc_i[head_dim]):
 * M = max m_i, out_d = sum_i e^(m_i - M) acc_id / sum_i e^(m_i - M) l_i.
 * Partials with l_i = 0 (empty ranges) contribute nothing.  If every partial
 * is empty the output is zero. */
void or_lse_merge(const double *m, const double *l, const double *acc,
                  int n, int head_dim, double *out)
{
    double big = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (l[i] > 0.0 && m[i] > big) big = m[i];
    double denom = 0.0;
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (big == -INFINITY) return;
    for (int i = 0; i < n; ++i) {
        if (!(l[i] > 0.0)) continue;
        double w = exp(m[i] - big);
        denom += w * l[i];
        for (int d = 0; d < head_dim; ++d) out[d] += w * acc[(int64_t)i * head_dim + d];
    }
    for (int d = 0; d < head_dim; ++d) out[d] /= denom;
}

/* ---------------------------------------------------- memory accounting */
/* PageFault README, "Calculate": bytes per token, naive and paged
 * reservations, utilisation and internal fragmentation. */

int64_t or_kv_bytes_per_token(int64_t n_layers, int64_t n_kv_heads,
                              int64_t head_dim, int64_t dtype_bytes)
{
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes;
}

int64_t or_naive_reserved_bytes(int64_t n_seqs, int64_t max_seq_len,
                                int64_t bytes_per_token)
{
    return n_seqs * max_seq_len * bytes_per_token;
}

int64_t or_paged_blocks(const int32_t *lens, int n, int64_t block_size)
{
    int64_t blocks = 0;
    for (int i = 0; i < n; ++i) blocks += or_blocks_needed(lens[i], block_size);
    return blocks;
}

int64_t or_paged_reserved_bytes(const int32_t *lens, int n,
                                int64_t block_size, int64_t bytes_per_token)
{
    return or_paged_blocks(lens, n, block_size) * block_size * bytes_per_token;
}

int64_t or_internal_fragmentation_tokens(const int32_t *lens, int n,
                                         int64_t block_size)
{
    int64_t waste = 0;
    for (int i = 0; i < n; ++i)
        waste += or_blocks_needed(lens[i], block_size) * block_size - lens[i];
    return waste;
}

/* Stored tokens / reserved tokens. */
double or_paged_utilization(const int32_t *lens, int n, int64_t block_size)
{
    int64_t used = 0;
    for (int i = 0; i < n; ++i) used += lens[i];
    int64_t reserved = or_paged_blocks(lens, n, block_size) * block_size;
    return reserved ? (double)used / (double)reserved : 0.0;
}
