/*
 * CPU oracle for sparse-attention token selection over a paged KV cache.
 *
 * TEST INFRASTRUCTURE. This file is the plain, slow reference definition that the
 * CUDA path is checked against. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it; the library never does. It shares no
 * code, header or constant with the CUDA sources.
 *
 * What it computes, step by step, for every query row r of request i
 * (rows [qsl[i], qsl[i+1]); rows past qsl[num_reqs] are padding):
 *
 *   1. ctx = positions[r] + 1. ("Row context == position + 1", vLLM page
 *      flashinfer_mla_sparse_sm90, _kv_lens_host.)
 *   2. ctx <= index_topk: the row selects every token 0 .. ctx-1 (same docstring:
 *      "contexts up to index_topk select everything").
 *   3. otherwise P = ctx / kpool complete pools are visible. Pool j lives in the
 *      request's logical key page j / 64 at row j % 64 (ReVolta PR #59, "Change":
 *      64-key tiles through a page table). Its score is
 *          s_j = sum_{h<4} sum_{d<128} q[r,h,d] * k[j,d]
 *      accumulated sequentially in fp32 (the fp16 x fp16 product is exact in
 *      fp32). A pool whose key page is out of range scores -inf.
 *   4. K = index_topk / kpool pools are kept: the K best under the total order
 *      (score descending, pool index ascending). A full sort by that order is used
 *      on purpose: it is a different algorithm from the GPU's radix select.
 *   5. Expansion: each kept pool p gives tokens p*kpool .. p*kpool+kpool-1, and the
 *      trailing incomplete pool's tokens P*kpool .. ctx-1 are always added
 *      (_kv_lens_host: "the top index_topk pool-expanded tokens plus the trailing
 *      incomplete pool"). Tokens are listed in ascending order and the row is
 *      padded with -1 to the output width.
 *   6. Remap (sparse_utils, triton_convert_req_index_to_global_index):
 *          slot = block_table[i, t / block_size] * block_stride_rows + t % block_size
 *      and -1 when t == -1 or the block is out of bounds: the logical block is past
 *      max_blocks_per_req, or the physical id is outside [0, num_kv_blocks).
 *   7. valid count = number of entries that are not -1 ("the count of valid
 *      (non -1) indices per row").
 *
 * Also here: the MaxSim rerank of a query against packed documents (orc_maxsim), and the
 * sparse MLA decode attention over the selected slots (orc_mla_decode).
 *
 * The remap also has the page's two other modes: prefill rows mapped into a prefill
 * workspace (orc_remap_ws_rows) and a decode-context-parallel rank's filter with optional
 * compaction to the front (orc_remap_dcp_rows).
 *
 * Readings where the pages are silent: the score has no weights, ReLU or scale;
 * only complete pools are scored; ties go to the lower pool index; -0.0 equals
 * +0.0; NaN (outside the input contract) ranks below -inf.
 *
 * Parity pins: see tests/test_oracle_pins.py. Nothing here is unpinned.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_ST_KEYPAGE_OOB 1
#define ORC_ST_CTX_OVER_BOUND 2
#define ORC_ST_BAD_QSL 8

/* IEEE 754 binary16 -> float, from the format's definition (1 sign bit, 5 exponent
 * bits with bias 15, 10 fraction bits). Every binary16 value is exact in float. */
float orc_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    return (float)(sign ? -v : v);
}

void orc_half_to_float_array(const uint16_t *h, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_half_to_float(h[i]);
}

/* Score of one pool against one query row: sum over heads, then over dimensions,
 * in fp32, in that order. Also returns sum |q*k| in fp64, the scale of the score's
 * rounding error. */
float orc_pool_score(const uint16_t *q_row, const uint16_t *key, int heads, int dim,
                     double *abs_terms)
{
    float s = 0.0f;
    double a = 0.0;
    for (int h = 0; h < heads; ++h) {
        for (int d = 0; d < dim; ++d) {
            float qv = orc_half_to_float(q_row[h * dim + d]);
            float kv = orc_half_to_float(key[d]);
            float prod = qv * kv;
            s = s + prod;
            a += fabs((double)qv * (double)kv);
        }
    }
    s = s + 0.0f; /* -0.0 -> +0.0 */
    if (abs_terms)
        *abs_terms = a;
    return s;
}

typedef struct {
    float s;
    int32_t j;
} orc_pool;

/* Total order used for selection: higher score first, lower index first on ties;
 * NaN after everything (it is outside the input contract). */
static int orc_better(const orc_pool *a, const orc_pool *b)
{
    int an = isnan(a->s), bn = isnan(b->s);
    if (an != bn)
        return bn;             /* the non-NaN one is better */
    if (!an && a->s != b->s)
        return a->s > b->s;
    return a->j < b->j;
}

static int orc_cmp_pool(const void *pa, const void *pb)
{
    const orc_pool *a = (const orc_pool *)pa, *b = (const orc_pool *)pb;
    if (a->j == b->j)
        return 0;
    return orc_better(a, b) ? -1 : 1;
}

static int orc_cmp_int(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* The K best pools of scores[0..P) under the order above, returned in ascending
 * pool index. Returns the number written (min(K, P)). */
int orc_topk_pools(const float *scores, int32_t P, int32_t K, int32_t *out)
{
    if (P <= 0 || K <= 0)
        return 0;
    orc_pool *v = (orc_pool *)malloc(sizeof(orc_pool) * (size_t)P);
    if (!v)
        return -1;
    for (int32_t j = 0; j < P; ++j) {
        v[j].s = scores[j];
        v[j].j = j;
    }
    qsort(v, (size_t)P, sizeof(orc_pool), orc_cmp_pool);
    int32_t n = K < P ? K : P;
    for (int32_t i = 0; i < n; ++i)
        out[i] = v[i].j;
    free(v);
    qsort(out, (size_t)n, sizeof(int32_t), orc_cmp_int);
    return n;
}

/* Expansion of a row's kept pools (ascending) into tokens, plus the trailing
 * incomplete pool; -1 padding to width W. Returns the number of tokens, or -1 if
 * they do not fit in W. */
int orc_expand(int64_t ctx, int32_t topk, int32_t kpool, const int32_t *pools,
               int32_t npools, int32_t W, int32_t *tokens)
{
    int32_t n = 0;
    if (ctx > 0 && ctx <= topk) {
        if (ctx > W)
            return -1;
        for (int64_t t = 0; t < ctx; ++t)
            tokens[n++] = (int32_t)t;
    } else if (ctx > topk) {
        int64_t P = ctx / kpool;
        for (int32_t i = 0; i < npools; ++i)
            for (int32_t t = 0; t < kpool; ++t) {
                if (n >= W)
                    return -1;
                tokens[n++] = (int32_t)((int64_t)pools[i] * kpool + t);
            }
        for (int64_t t = P * kpool; t < ctx; ++t) {
            if (n >= W)
                return -1;
            tokens[n++] = (int32_t)t;
        }
    }
    for (int32_t c = n; c < W; ++c)
        tokens[c] = -1;
    return n;
}

/* One token index through one request's block-table row. */
int64_t orc_remap_token(int32_t t, const int32_t *bt_row, int32_t max_blocks,
                        int32_t num_kv_blocks, int32_t block_size, int64_t block_stride_rows)
{
    if (t < 0)
        return -1;
    int32_t b = t / block_size;
    if (b >= max_blocks)
        return -1;
    int32_t ph = bt_row[b];
    if (ph < 0 || ph >= num_kv_blocks)
        return -1;
    return (int64_t)ph * block_stride_rows + (t % block_size);
}

/* Remap of whole rows: token_idx [rows, width] -> slots [rows, width], counts [rows].
 * req_id[r] outside [0, num_reqs) gives an all -1 row. */
void orc_remap_rows(const int32_t *req_id, int32_t num_reqs, const int32_t *block_table,
                    int64_t bt_ld, int32_t max_blocks, int32_t num_kv_blocks,
                    const int32_t *token_idx, int32_t rows, int32_t width,
                    int32_t block_size, int64_t block_stride_rows, int64_t *slots,
                    int32_t *counts)
{
    for (int32_t r = 0; r < rows; ++r) {
        int32_t req = req_id[r];
        int32_t cnt = 0;
        for (int32_t c = 0; c < width; ++c) {
            int64_t s = -1;
            if (req >= 0 && req < num_reqs)
                s = orc_remap_token(token_idx[(int64_t)r * width + c],
                                    block_table + (int64_t)req * bt_ld, max_blocks,
                                    num_kv_blocks, block_size, block_stride_rows);
            slots[(int64_t)r * width + c] = s;
            cnt += (s != -1);
        }
        if (counts)
            counts[r] = cnt;
    }
}

/* Prefill-workspace remap (vLLM page "sparse_utils", triton_convert_req_index_to_global_index
 * with HAS_PREFILL_WORKSPACE): prefill rows map their tokens to offsets in a prefill
 * workspace instead of global cache slots. ws_req[r] is -1 for a decode row (the global
 * remap above) or the row's prefill request w, whose tokens start at ws_starts[w]:
 *     out = t == -1 ? -1 : ws_starts[w] + t
 * The pages give no formula; this is the plainest reading of "mapped to workspace offsets"
 * with "0-indexed workspace starts for each prefill request". A w outside [-1, num_prefills)
 * gives an all -1 row (the same guard as an out-of-range request id). */
void orc_remap_ws_rows(const int32_t *req_id, int32_t num_reqs, const int32_t *block_table,
                       int64_t bt_ld, int32_t max_blocks, int32_t num_kv_blocks,
                       const int32_t *ws_req, const int32_t *ws_starts, int32_t num_prefills,
                       const int32_t *token_idx, int32_t rows, int32_t width,
                       int32_t block_size, int64_t block_stride_rows, int64_t *slots,
                       int32_t *counts)
{
    for (int32_t r = 0; r < rows; ++r) {
        int32_t w = ws_req[r];
        int32_t req = req_id[r];
        int32_t cnt = 0;
        for (int32_t c = 0; c < width; ++c) {
            int32_t t = token_idx[(int64_t)r * width + c];
            int64_t s = -1;
            if (w == -1) {
                if (req >= 0 && req < num_reqs)
                    s = orc_remap_token(t, block_table + (int64_t)req * bt_ld, max_blocks,
                                        num_kv_blocks, block_size, block_stride_rows);
            } else if (w >= 0 && w < num_prefills && t >= 0) {
                s = (int64_t)ws_starts[w] + t;
            }
            slots[(int64_t)r * width + c] = s;
            cnt += (s != -1);
        }
        if (counts)
            counts[r] = cnt;
    }
}

/* Decode context parallelism (vLLM page "sparse_utils", triton_filter_and_convert_dcp_index):
 * dcp_size ranks each hold part of every request's KV, interleaved in groups of
 * `interleave` tokens (block_size is a multiple of interleave, so a group never straddles
 * a block). The page does not print the index formula; the plainest reading of a
 * round-robin interleave is:
 *     owner(t) = (t / interleave) % dcp_size
 *     local(t) = (t / (interleave * dcp_size)) * interleave + t % interleave
 * i.e. each rank stores its groups back to back. Returns local(t), or -1 when t is -1 or
 * another rank owns t. */
int64_t orc_dcp_local_index(int32_t t, int32_t dcp_size, int32_t dcp_rank, int32_t interleave)
{
    if (t < 0)
        return -1;
    int64_t group = t / interleave;
    if (group % dcp_size != dcp_rank)
        return -1;
    return (group / dcp_size) * interleave + t % interleave;
}

/* The rank's slots: the local index goes through the rank's own block table, which on the
 * DCP path is dense (block stride == block size, "dense caches on the DCP path"), with the
 * same -1 guards as the global remap. Tokens owned by other ranks become -1 ("DCP filtering
 * marks non-owned slots -1"). With compact != 0 the row's non -1 slots are moved, in
 * ascending column order, to columns 0 .. count-1 and the rest is -1 (the page: "scatters
 * this rank's owned slots to a contiguous prefix [0, valid_count) ... Prefix order is
 * unspecified"; ascending is one valid order). count = number of non -1 entries. */
void orc_remap_dcp_rows(const int32_t *req_id, int32_t num_reqs, const int32_t *block_table,
                        int64_t bt_ld, int32_t max_blocks, int32_t num_kv_blocks,
                        const int32_t *token_idx, int32_t rows, int32_t width, int32_t block_size,
                        int32_t dcp_size, int32_t dcp_rank, int32_t interleave, int32_t compact,
                        int64_t *slots, int32_t *counts)
{
    for (int32_t r = 0; r < rows; ++r) {
        int32_t req = req_id[r];
        int32_t cnt = 0;
        int64_t *out = slots + (int64_t)r * width;
        for (int32_t c = 0; c < width; ++c) {
            int64_t s = -1;
            int64_t l = orc_dcp_local_index(token_idx[(int64_t)r * width + c], dcp_size, dcp_rank,
                                            interleave);
            if (l >= 0 && l <= INT32_MAX && req >= 0 && req < num_reqs)
                s = orc_remap_token((int32_t)l, block_table + (int64_t)req * bt_ld, max_blocks,
                                    num_kv_blocks, block_size, block_size);
            if (compact) {
                if (s != -1)
                    out[cnt] = s;
            } else {
                out[c] = s;
            }
            cnt += (s != -1);
        }
        if (compact)
            for (int32_t c = cnt; c < width; ++c)
                out[c] = -1;
        if (counts)
            counts[r] = cnt;
    }
}

/* MaxSim rerank (vLLM page "flash_maxsim_rerank", _maxsim_rerank_kernel and
 * flash_maxsim_rerank_direct): one query of lq token embeddings against num_docs documents
 * whose token embeddings lie anywhere in a packed [total_tokens, doc_stride] tensor, doc i
 * being rows offsets[i] .. offsets[i] + lengths[i] - 1. For every query token the best
 * (largest) dot product over the document's tokens is taken, and the document's score is
 * the sum of those maxima over the query tokens:
 *     score_i = sum_{a < lq} max_{j < len_i} sum_{k < d} q[a][k] * doc[off_i + j][k]
 * The page's masking fixes the degenerate cases: a running maximum starts at -inf, so a
 * document with no tokens (length <= 0) scores -inf, and with no query tokens every
 * document scores 0. A row outside [0, total_tokens) reads as a zero vector (it lies
 * outside the page's contract; this is the reading the device path implements).
 * Each dot product is accumulated in double from the exact fp16 x fp16 products, the
 * maxima are summed in double and the score is rounded to float once. abs_bound[i]
 * (optional) = sum_a max_j sum_k |q[a][k] * doc[off_i + j][k]|, the scale of the rounding
 * of an implementation that accumulates in fp32. */
void orc_maxsim(const uint16_t *q, int32_t lq, int32_t d, const uint16_t *docs, int64_t doc_stride,
                int64_t total_tokens, const int32_t *offsets, const int32_t *lengths, int32_t num_docs,
                float *scores, double *abs_bound)
{
    for (int32_t i = 0; i < num_docs; ++i) {
        double total = 0.0, bound = 0.0;
        for (int32_t a = 0; a < lq; ++a) {
            double best = -INFINITY, best_abs = 0.0;
            for (int32_t j = 0; j < lengths[i]; ++j) {
                const int64_t r = (int64_t)offsets[i] + j;
                double s = 0.0, sa = 0.0;
                if (r >= 0 && r < total_tokens) {
                    const uint16_t *row = docs + r * doc_stride;
                    for (int32_t k = 0; k < d; ++k) {
                        double t = (double)orc_half_to_float(q[(int64_t)a * d + k]) * (double)orc_half_to_float(row[k]);
                        s += t;
                        sa += fabs(t);
                    }
                }
                if (s > best)
                    best = s;
                if (sa > best_abs)
                    best_abs = sa;
            }
            total += best;
            bound += best_abs;
        }
        scores[i] = (float)total;
        if (abs_bound)
            abs_bound[i] = bound;
    }
}

/* bfloat16 bit pattern -> double: the top 16 bits of a binary32 (the format's definition). */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Sparse MLA decode attention over selected KV slots (vLLM page
 * "flashinfer_mla_sparse_sm90", _SM90State: FlashInfer's BatchMLAPagedAttentionWrapper planned
 * with page_size 1 -- the selected slots are the page table --, head_dim_ckv = kv_lora_rank,
 * qk_rope_head_dim 0 or 64, no causal mask, sm_scale, bf16 queries, and the exact per-row
 * kv_len of _kv_lens_host; entries past kv_len (the -1 tail) are never read).
 * The MLA computation in its absorbed form (the wrapper's head_dim_ckv output): for row r,
 * head h and each entry j < kv_len[r] whose slot s = slots[r][j] lies in [0, num_slots)
 * (a -1 or out-of-range slot inside kv_len contributes nothing):
 *     logit_j    = sm_scale * (q_nope[r][h] . ckv[s] + q_pe[r][h] . kpe[s])
 *     out[r][h]  = sum_j exp(logit_j - m) * ckv[s_j] / sum_j exp(logit_j - m),  m = max_j logit_j
 *     lse[r][h]  = m + log(sum_j exp(logit_j - m))           (natural logarithm)
 * A row with no such entry gives out = 0 and lse = -inf. Every input is bf16 (given as bit
 * patterns); the dot products, exponentials and sums are taken in double.
 * Layouts: q_nope [rows][heads][dc], q_pe [rows][heads][dr], ckv row s at s * ckv_stride,
 * kpe row s at s * kpe_stride (unused when dr == 0), slots [rows][width], out [rows][heads][dc],
 * lse [rows][heads]. */
void orc_mla_decode(const uint16_t *q_nope, const uint16_t *q_pe, int32_t rows, int32_t heads,
                    int32_t dc, int32_t dr, const uint16_t *ckv, int64_t ckv_stride,
                    const uint16_t *kpe, int64_t kpe_stride, int64_t num_slots, const int32_t *slots,
                    int32_t width, const int32_t *kv_len, double sm_scale, double *out, double *lse)
{
    double *logit = (double *)malloc(sizeof(double) * (size_t)(width > 0 ? width : 1));
    for (int32_t r = 0; r < rows; ++r) {
        const int32_t n = kv_len[r] < width ? kv_len[r] : width;
        for (int32_t h = 0; h < heads; ++h) {
            const uint16_t *qn = q_nope + ((int64_t)r * heads + h) * dc;
            const uint16_t *qp = q_pe + ((int64_t)r * heads + h) * dr;
            double *o = out + ((int64_t)r * heads + h) * dc;
            double m = -INFINITY;
            int any = 0;
            for (int32_t j = 0; j < n; ++j) {
                const int64_t sl = slots[(int64_t)r * width + j];
                if (sl < 0 || sl >= num_slots)
                    continue;
                double acc = 0.0;
                for (int32_t d = 0; d < dc; ++d)
                    acc += orc_bf16_to_double(qn[d]) * orc_bf16_to_double(ckv[sl * ckv_stride + d]);
                for (int32_t d = 0; d < dr; ++d)
                    acc += orc_bf16_to_double(qp[d]) * orc_bf16_to_double(kpe[sl * kpe_stride + d]);
                logit[j] = sm_scale * acc;
                if (logit[j] > m)
                    m = logit[j];
                any = 1;
            }
            for (int32_t d = 0; d < dc; ++d)
                o[d] = 0.0;
            if (!any) {
                lse[(int64_t)r * heads + h] = -INFINITY;
                continue;
            }
            double z = 0.0;
            for (int32_t j = 0; j < n; ++j) {
                const int64_t sl = slots[(int64_t)r * width + j];
                if (sl < 0 || sl >= num_slots)
                    continue;
                const double p = exp(logit[j] - m);
                z += p;
                for (int32_t d = 0; d < dc; ++d)
                    o[d] += p * orc_bf16_to_double(ckv[sl * ckv_stride + d]);
            }
            for (int32_t d = 0; d < dc; ++d)
                o[d] /= z;
            lse[(int64_t)r * heads + h] = m + log(z);
        }
    }
    free(logit);
}

typedef struct {
    int32_t num_reqs, num_rows;
    const int32_t *qsl, *positions;
    const uint16_t *q;            /* [num_rows, heads, dim] fp16 bits */
    int64_t q_row_stride;         /* elements */
    const uint16_t *key_cache;    /* fp16 bits */
    int64_t key_page_stride;      /* elements */
    int32_t num_key_pages;
    const int32_t *key_page_table;
    int64_t kpt_ld;
    int32_t max_key_pages_per_req;
    const int32_t *block_table;
    int64_t bt_ld;
    int32_t max_blocks_per_req, num_kv_blocks, block_size;
    int64_t block_stride_rows;
    int32_t heads, dim, key_page_size, index_topk, kpool, out_width;
    int64_t max_context;
} orc_problem;

typedef struct {
    const orc_problem *p;
    const int32_t *rows;          /* rows to compute (indices into the batch) */
    int32_t nrows;
    int32_t tid, nthreads;
    int64_t *slots;               /* [nrows, out_width] */
    int32_t *counts;              /* [nrows] */
    int32_t *token_idx;           /* [nrows, out_width] or NULL */
    float *scores;                /* [nrows, scores_ld] or NULL */
    double *abs_terms;            /* [nrows, scores_ld] or NULL */
    int64_t scores_ld;
    int32_t status;
    int32_t error;
} orc_job;

static int orc_qsl_ok(const orc_problem *p)
{
    if (p->qsl[0] < 0 || p->qsl[p->num_reqs] > p->num_rows)
        return 0;
    for (int32_t i = 0; i < p->num_reqs; ++i)
        if (p->qsl[i] > p->qsl[i + 1])
            return 0;
    return 1;
}

static int32_t orc_request_of(const orc_problem *p, int32_t r)
{
    for (int32_t i = 0; i < p->num_reqs; ++i)
        if (p->qsl[i] <= r && r < p->qsl[i + 1])
            return i;
    return -1;
}

static void orc_one_row(orc_job *jb, int32_t k)
{
    const orc_problem *p = jb->p;
    const int32_t W = p->out_width;
    int32_t r = jb->rows[k];
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)W);
    int64_t *slot = jb->slots + (int64_t)k * W;
    for (int32_t c = 0; c < W; ++c)
        tok[c] = -1;

    int32_t req = orc_qsl_ok(p) ? orc_request_of(p, r) : -1;
    if (!orc_qsl_ok(p))
        jb->status |= ORC_ST_BAD_QSL;
    int64_t ctx = (int64_t)p->positions[r] + 1;
    if (req >= 0 && ctx > p->max_context) {
        jb->status |= ORC_ST_CTX_OVER_BOUND;
        req = -1;
    }
    if (req >= 0 && ctx > p->index_topk) {
        int32_t P = (int32_t)(ctx / p->kpool);
        int32_t K = p->index_topk / p->kpool;
        float *s = (float *)malloc(sizeof(float) * (size_t)P);
        const uint16_t *qr = p->q + (int64_t)r * p->q_row_stride;
        for (int32_t j = 0; j < P; ++j) {
            int32_t lp = j / p->key_page_size;
            int32_t pg = lp < p->max_key_pages_per_req
                             ? p->key_page_table[(int64_t)req * p->kpt_ld + lp] : -1;
            double a = 0.0;
            if (pg < 0 || pg >= p->num_key_pages) {
                s[j] = -INFINITY;
                jb->status |= ORC_ST_KEYPAGE_OOB;
            } else {
                const uint16_t *key = p->key_cache + (int64_t)pg * p->key_page_stride +
                                      (int64_t)(j % p->key_page_size) * p->dim;
                s[j] = orc_pool_score(qr, key, p->heads, p->dim, &a);
            }
            if (jb->scores && j < jb->scores_ld)
                jb->scores[(int64_t)k * jb->scores_ld + j] = s[j];
            if (jb->abs_terms && j < jb->scores_ld)
                jb->abs_terms[(int64_t)k * jb->scores_ld + j] = a;
        }
        int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
        int32_t n = orc_topk_pools(s, P, K, sel);
        if (orc_expand(ctx, p->index_topk, p->kpool, sel, n, W, tok) < 0)
            jb->error = 1;
        free(sel);
        free(s);
    } else if (req >= 0) {
        if (orc_expand(ctx, p->index_topk, p->kpool, NULL, 0, W, tok) < 0)
            jb->error = 1;
    }
    int32_t cnt = 0;
    for (int32_t c = 0; c < W; ++c) {
        int64_t sl = -1;
        if (req >= 0)
            sl = orc_remap_token(tok[c], p->block_table + (int64_t)req * p->bt_ld,
                                 p->max_blocks_per_req, p->num_kv_blocks, p->block_size,
                                 p->block_stride_rows);
        slot[c] = sl;
        cnt += (sl != -1);
    }
    jb->counts[k] = cnt;
    if (jb->token_idx)
        memcpy(jb->token_idx + (int64_t)k * W, tok, sizeof(int32_t) * (size_t)W);
    free(tok);
}

static void *orc_worker(void *arg)
{
    orc_job *jb = (orc_job *)arg;
    for (int32_t k = jb->tid; k < jb->nrows; k += jb->nthreads)
        orc_one_row(jb, k);
    return NULL;
}

/* The whole selection for the listed rows, on nthreads POSIX threads (rows are
 * independent). Returns the OR of the status bits, or -1 on an internal error
 * (output width too small). */
int32_t orc_select(const orc_problem *p, const int32_t *rows, int32_t nrows,
                   int32_t nthreads, int64_t *slots, int32_t *counts, int32_t *token_idx,
                   float *scores, double *abs_terms, int64_t scores_ld)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    orc_job jobs[256];
    pthread_t th[256];
    for (int32_t t = 0; t < nthreads; ++t) {
        jobs[t] = (orc_job){p, rows, nrows, t, nthreads, slots, counts, token_idx,
                            scores, abs_terms, scores_ld, 0, 0};
    }
    for (int32_t t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    orc_worker(&jobs[0]);
    for (int32_t t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    int32_t st = 0;
    for (int32_t t = 0; t < nthreads; ++t) {
        if (jobs[t].error)
            return -1;
        st |= jobs[t].status;
    }
    return st;
}

/* The scoring step alone (step 3) for the listed rows, over the row's complete pools:
 * scores[k, j] for j < ctx / kpool, -inf on out-of-range key pages; entries at
 * higher j are left untouched. Rows whose request cannot be found are skipped. */
int32_t orc_score_rows(const orc_problem *p, const int32_t *rows, int32_t nrows,
                       float *scores, double *abs_terms, int64_t scores_ld)
{
    int32_t st = 0;
    for (int32_t k = 0; k < nrows; ++k) {
        int32_t r = rows[k];
        int32_t req = orc_request_of(p, r);
        if (req < 0)
            continue;
        int64_t ctx = (int64_t)p->positions[r] + 1;
        int64_t P = ctx > 0 ? ctx / p->kpool : 0;
        if (P > scores_ld)
            P = scores_ld;
        const uint16_t *qr = p->q + (int64_t)r * p->q_row_stride;
        for (int64_t j = 0; j < P; ++j) {
            int32_t lp = (int32_t)(j / p->key_page_size);
            int32_t pg = lp < p->max_key_pages_per_req
                             ? p->key_page_table[(int64_t)req * p->kpt_ld + lp] : -1;
            double a = 0.0;
            float s;
            if (pg < 0 || pg >= p->num_key_pages) {
                s = -INFINITY;
                st |= ORC_ST_KEYPAGE_OOB;
            } else {
                const uint16_t *key = p->key_cache + (int64_t)pg * p->key_page_stride +
                                      (j % p->key_page_size) * p->dim;
                s = orc_pool_score(qr, key, p->heads, p->dim, &a);
            }
            scores[(int64_t)k * scores_ld + j] = s;
            if (abs_terms)
                abs_terms[(int64_t)k * scores_ld + j] = a;
        }
    }
    return st;
}

/* Top-k + expansion alone (steps 2, 4, 5) on given score rows: row k has context
 * ctx[k] and scores[k, 0 .. ctx/kpool). token_idx [nrows, W]; counts = tokens. */
int32_t orc_topk_expand_rows(const float *scores, int64_t scores_ld, const int64_t *ctx,
                             int32_t nrows, int32_t topk, int32_t kpool, int32_t W,
                             int32_t *token_idx, int32_t *counts)
{
    int32_t K = topk / kpool;
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    for (int32_t k = 0; k < nrows; ++k) {
        int32_t *tok = token_idx + (int64_t)k * W;
        int32_t n;
        if (ctx[k] > topk) {
            int64_t P = ctx[k] / kpool;
            int32_t ns = orc_topk_pools(scores + (int64_t)k * scores_ld, (int32_t)P, K, sel);
            n = orc_expand(ctx[k], topk, kpool, sel, ns, W, tok);
        } else {
            n = orc_expand(ctx[k], topk, kpool, NULL, 0, W, tok);
        }
        if (n < 0) {
            free(sel);
            return -1;
        }
        counts[k] = n;
    }
    free(sel);
    return 0;
}
