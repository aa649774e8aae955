/*
 * Plain CPU oracle of the DSpark draft-token fused QK-norm / RoPE / KV insert.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA path and is deliberately slow and literal:
 * one head of one token at a time, fp64 arithmetic.
 *
 * What it computes (DSpark draft model page, dspark_qknorm_rope_kv_insert:
 * "the fused QK-norm/RoPE on qkv, also storing the draft tokens' k/v", with
 * the call's arguments qkv, q_norm_weight, k_norm_weight, cos_sin_cache,
 * positions, num_heads, num_kv_heads, rotary_dim, eps, slot_mapping,
 * kv_cache, block_size, kv_cache_dtype, q_fp8_out, q_fp8_scale).  The page
 * prints no kernel, so the readings below are the plainest ones its
 * arguments and the context-KV writer page support:
 *   qkv [T, (Hq + 2 Hkv) * 128] bf16, per token the Hq query heads, then the
 *   Hkv key heads, then the Hkv value heads (the packed QKV projection).
 *   For every token t (padding included: the slot mapping only steers the
 *   insert) and every query head i and key head h:
 *     1. Gemma RMSNorm of the head, weight q_norm_weight (query heads) or
 *        k_norm_weight (key heads), one [128] weight shared by all heads:
 *        y = x * rsqrt(mean(x^2) + eps) * (1 + w), materialised to bf16 (fp64
 *        here; both bf16 neighbours admissible within 2^-18 of a midpoint,
 *        exactly as the context-KV oracle does);
 *     2. partial NeoX RoPE of the first r dims at positions[t], cos in
 *        [0, r/2) and sin in [r/2, r) of the bf16 cache row, one rounding to
 *        bf16 per output; dims >= r pass through;
 *     3. the result replaces the head in qkv; value heads are left as they are.
 *   q_fp8_out [T, Hq * 128] (when given): e4m3 (OCP, RNE, saturating) of the
 *   bf16 query result divided by q_fp8_scale in fp32.
 *   Insert (when a slot mapping and a cache are given): for every token with
 *   slot >= 0 and every KV head h, the 256-element row K'_h | V_h goes to
 *   kv_cache [num_blocks, Hkv, block_size, 256] at block slot / block_size,
 *   head h, offset slot % block_size -- as bf16, or as e4m3 of x / k_scale
 *   (K) and x / v_scale (V) in fp32 for an fp8 cache, the same encoding the
 *   context-KV writer stores into the same cache.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK_HEAD_DIM 128
#define QK_ROW 256

/* scalar conversions and the norm of one head: defined in ctx_kv_oracle.c */
double dspark_oracle_bf16_decode(uint16_t b);
uint16_t dspark_oracle_bf16_rne(double x);
uint8_t dspark_oracle_e4m3_rne_sat(float xf);
int dspark_oracle_gemma_knorm(const uint16_t *k, const uint16_t *w, float eps,
                              uint16_t *y, uint16_t *y_alt);
void dspark_oracle_rope_pair(uint16_t x1, uint16_t x2, uint16_t c, uint16_t s,
                             uint16_t *o1, uint16_t *o2);

enum { QK_KV_BF16 = 0, QK_KV_FP8_E4M3 = 1 };

enum {
    QK_OK = 0,
    QK_ERR_ARG = -1,
    QK_ERR_SLOT_RANGE = -2,
    QK_ERR_SLOT_DUP = -3,
    QK_ERR_POS_RANGE = -4,
    QK_ERR_SCALE = -5,
    QK_ERR_ALT_CAP = -6,
    QK_ERR_NOMEM = -7,
};

/* Everything one call reads (host memory). */
typedef struct {
    const uint16_t *qkv;          /* bf16 bits [T][(Hq + 2 Hkv) * 128] */
    const uint16_t *q_norm_w;     /* bf16 bits [128] */
    const uint16_t *k_norm_w;     /* bf16 bits [128] */
    const int64_t *positions;     /* [T] */
    const int64_t *slot_mapping;  /* [T], < 0 = padding; NULL = no insert */
    const uint16_t *cos_sin;      /* bf16 bits [max_pos][r] */
    int64_t num_tokens;
    int64_t max_pos;
    int64_t num_blocks;           /* cache blocks (insert only) */
    int32_t num_heads;            /* Hq */
    int32_t num_kv_heads;         /* Hkv */
    int32_t block_size;
    int32_t rotary_dim;
    int32_t kv_dtype;             /* of the cache */
    float eps;
    float k_scale, v_scale;       /* fp8 cache only */
    float q_scale;                /* q_fp8_out only */
} dspark_oracle_qk_inputs;

/* Where an admissible alternate value lives. */
enum { QK_ALT_QKV = 0, QK_ALT_QFP8 = 1, QK_ALT_CACHE = 2 };

typedef struct {
    int32_t *where;   /* QK_ALT_* */
    int64_t *elem;    /* element index in that output */
    uint16_t *val;
    int64_t cap, n;
} qk_alts;

static void alt_push(qk_alts *a, int where, int64_t elem, uint16_t val)
{
    if (a->n < a->cap) {
        a->where[a->n] = where;
        a->elem[a->n] = elem;
        a->val[a->n] = val;
    }
    a->n++;
}

/* Steps 1 and 2 on one head: out[d] is the result built from the correctly
 * rounded norm outputs; cand[d][0..ncand[d]) lists every admissible value of
 * dim d (cand[d][0] == out[d]), following each tie-region norm output
 * through the rotation. */
static void norm_rope_head(const uint16_t *x, const uint16_t *w, float eps, const uint16_t *cs,
                           int r, uint16_t out[QK_HEAD_DIM], uint16_t cand[QK_HEAD_DIM][4],
                           int ncand[QK_HEAD_DIM])
{
    uint16_t y[QK_HEAD_DIM], y_alt[QK_HEAD_DIM];
    dspark_oracle_gemma_knorm(x, w, eps, y, y_alt);
    const int half = r / 2;
    for (int d = 0; d < QK_HEAD_DIM; d++) {
        int nc = 0;
        if (d < r) {
            const int lower = d < half;
            const int i = lower ? d : d - half;
            const int p = lower ? d + half : d - half;
            const uint16_t c = cs[i], s = cs[half + i];
            const uint16_t self_c[2] = {y[d], y_alt[d]};
            const uint16_t part_c[2] = {y[p], y_alt[p]};
            const int ns = y_alt[d] != y[d] ? 2 : 1;
            const int np = y_alt[p] != y[p] ? 2 : 1;
            for (int a = 0; a < ns; a++)
                for (int b = 0; b < np; b++) {
                    uint16_t o1, o2, v;
                    if (lower) {
                        dspark_oracle_rope_pair(self_c[a], part_c[b], c, s, &o1, &o2);
                        v = o1;
                    } else {
                        dspark_oracle_rope_pair(part_c[b], self_c[a], c, s, &o1, &o2);
                        v = o2;
                    }
                    int seen = 0;
                    for (int q = 0; q < nc; q++)
                        seen |= cand[d][q] == v;
                    if (!seen)
                        cand[d][nc++] = v;
                }
        } else {
            cand[d][nc++] = y[d];
            if (y_alt[d] != y[d])
                cand[d][nc++] = y_alt[d];
        }
        ncand[d] = nc;
        out[d] = cand[d][0];
    }
}

static uint8_t e4m3_of_quotient(uint16_t x, float scale)
{
    float xf = (float)dspark_oracle_bf16_decode(x);
    float q = xf / scale; /* fp32 division, correctly rounded */
    return dspark_oracle_e4m3_rne_sat(q);
}

/* Encoded candidates of one element: enc[0] from cand[0]; the distinct
 * others are pushed as alternates of (where, elem). */
static uint16_t encode_with_alts(const uint16_t *cand, int nc, int fp8, float scale, qk_alts *alts,
                                 int where, int64_t elem)
{
    uint16_t enc[4] = {0, 0, 0, 0};
    for (int j = 0; j < nc; j++)
        enc[j] = fp8 ? e4m3_of_quotient(cand[j], scale) : cand[j];
    for (int j = 1; j < nc; j++) {
        int seen = enc[j] == enc[0];
        for (int q = 1; q < j; q++)
            seen |= enc[q] == enc[j];
        if (!seen && alts)
            alt_push(alts, where, elem, enc[j]);
    }
    return enc[0];
}

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* Preconditions: every position inside the cos|sin table (every token is
 * rotated); with an insert, valid slots unique and inside the cache and fp8
 * scales positive and finite; a positive finite q scale for q_fp8_out. */
int dspark_oracle_qk_check(const dspark_oracle_qk_inputs *in, int with_cache, int with_qfp8)
{
    if (!in || in->num_tokens < 0 || in->num_heads <= 0 || in->num_kv_heads <= 0 || in->max_pos <= 0)
        return QK_ERR_ARG;
    if (in->rotary_dim <= 0 || in->rotary_dim > QK_HEAD_DIM || in->rotary_dim % 2)
        return QK_ERR_ARG;
    for (int64_t t = 0; t < in->num_tokens; t++)
        if (in->positions[t] < 0 || in->positions[t] >= in->max_pos)
            return QK_ERR_POS_RANGE;
    if (with_qfp8 && (!(in->q_scale > 0.0f) || isinf(in->q_scale)))
        return QK_ERR_SCALE;
    if (!with_cache || !in->slot_mapping)
        return QK_OK;
    if (in->block_size <= 0 || in->num_blocks <= 0)
        return QK_ERR_ARG;
    if (in->kv_dtype != QK_KV_BF16 && in->kv_dtype != QK_KV_FP8_E4M3)
        return QK_ERR_ARG;
    if (in->kv_dtype == QK_KV_FP8_E4M3 &&
        (!(in->k_scale > 0.0f) || !(in->v_scale > 0.0f) || isinf(in->k_scale) || isinf(in->v_scale)))
        return QK_ERR_SCALE;
    const int64_t cap = in->num_blocks * in->block_size;
    int64_t *sorted = (int64_t *)malloc((size_t)(in->num_tokens ? in->num_tokens : 1) * sizeof(int64_t));
    if (!sorted)
        return QK_ERR_NOMEM;
    int64_t nv = 0;
    int rc = QK_OK;
    for (int64_t t = 0; t < in->num_tokens; t++) {
        int64_t s = in->slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= cap) {
            rc = QK_ERR_SLOT_RANGE;
            break;
        }
        sorted[nv++] = s;
    }
    if (rc == QK_OK) {
        qsort(sorted, (size_t)nv, sizeof(int64_t), cmp_i64);
        for (int64_t i = 1; i < nv; i++)
            if (sorted[i] == sorted[i - 1]) {
                rc = QK_ERR_SLOT_DUP;
                break;
            }
    }
    free(sorted);
    return rc;
}

/*
 * The whole call for tokens [t_begin, t_end).
 *   qkv_out   [T][(Hq + 2 Hkv) * 128] bf16 bits: receives the rows of those
 *             tokens (query and key heads replaced, value heads copied).
 *   q_fp8     [T][Hq * 128] e4m3 codes, or NULL.
 *   cache     [num_blocks][Hkv][block_size][256] of the cache dtype, or NULL
 *             (no insert; also when slot_mapping is NULL).
 * Admissible alternates: (output, element index, value) into the three
 * arrays, up to alt_cap; *n_alt receives the total.
 */
int dspark_oracle_qk_insert(const dspark_oracle_qk_inputs *in, int64_t t_begin, int64_t t_end,
                            uint16_t *qkv_out, uint8_t *q_fp8, void *cache,
                            int32_t *alt_where, int64_t *alt_elem, uint16_t *alt_val,
                            int64_t alt_cap, int64_t *n_alt)
{
    const int with_cache = cache != NULL && in && in->slot_mapping != NULL;
    int rc = dspark_oracle_qk_check(in, with_cache, q_fp8 != NULL);
    if (rc != QK_OK)
        return rc;
    if (!qkv_out || t_begin < 0 || t_end > in->num_tokens || t_begin > t_end)
        return QK_ERR_ARG;
    const int Hq = in->num_heads, Hkv = in->num_kv_heads, r = in->rotary_dim;
    const int64_t width = (int64_t)(Hq + 2 * Hkv) * QK_HEAD_DIM;
    const int fp8 = in->kv_dtype == QK_KV_FP8_E4M3;
    qk_alts alts = {alt_where, alt_elem, alt_val, alt_cap, 0};
    uint16_t out[QK_HEAD_DIM], cand[QK_HEAD_DIM][4];
    int ncand[QK_HEAD_DIM];

    for (int64_t t = t_begin; t < t_end; t++) {
        const uint16_t *row = in->qkv + t * width;
        uint16_t *orow = qkv_out + t * width;
        const uint16_t *cs = in->cos_sin + in->positions[t] * r;
        const int64_t slot = with_cache ? in->slot_mapping[t] : -1;
        int64_t dst = -1; /* first element of head 0's cache row */
        if (slot >= 0) {
            const int64_t block = slot / in->block_size, offset = slot % in->block_size;
            dst = ((block * Hkv) * in->block_size + offset) * QK_ROW;
        }
        /* query heads */
        for (int i = 0; i < Hq; i++) {
            const int64_t e0 = (int64_t)i * QK_HEAD_DIM;
            norm_rope_head(row + e0, in->q_norm_w, in->eps, cs, r, out, cand, ncand);
            for (int d = 0; d < QK_HEAD_DIM; d++) {
                orow[e0 + d] = out[d];
                for (int j = 1; j < ncand[d]; j++)
                    alt_push(&alts, QK_ALT_QKV, t * width + e0 + d, cand[d][j]);
                if (q_fp8)
                    q_fp8[t * (int64_t)Hq * QK_HEAD_DIM + e0 + d] = (uint8_t)encode_with_alts(
                        cand[d], ncand[d], 1, in->q_scale, &alts, QK_ALT_QFP8,
                        t * (int64_t)Hq * QK_HEAD_DIM + e0 + d);
            }
        }
        /* key heads (and, with the insert, their cache rows) */
        for (int h = 0; h < Hkv; h++) {
            const int64_t e0 = (int64_t)(Hq + h) * QK_HEAD_DIM;
            norm_rope_head(row + e0, in->k_norm_w, in->eps, cs, r, out, cand, ncand);
            const int64_t crow = dst >= 0 ? dst + (int64_t)h * in->block_size * QK_ROW : -1;
            for (int d = 0; d < QK_HEAD_DIM; d++) {
                orow[e0 + d] = out[d];
                for (int j = 1; j < ncand[d]; j++)
                    alt_push(&alts, QK_ALT_QKV, t * width + e0 + d, cand[d][j]);
                if (crow >= 0) {
                    uint16_t v = encode_with_alts(cand[d], ncand[d], fp8, in->k_scale, &alts,
                                                  QK_ALT_CACHE, crow + d);
                    if (fp8)
                        ((uint8_t *)cache)[crow + d] = (uint8_t)v;
                    else
                        ((uint16_t *)cache)[crow + d] = v;
                }
            }
        }
        /* value heads: unchanged in qkv; inserted as they are (or encoded) */
        for (int h = 0; h < Hkv; h++) {
            const int64_t e0 = (int64_t)(Hq + Hkv + h) * QK_HEAD_DIM;
            const int64_t crow = dst >= 0 ? dst + (int64_t)h * in->block_size * QK_ROW : -1;
            for (int d = 0; d < QK_HEAD_DIM; d++) {
                const uint16_t v = row[e0 + d];
                orow[e0 + d] = v;
                if (crow >= 0) {
                    if (fp8)
                        ((uint8_t *)cache)[crow + QK_HEAD_DIM + d] = e4m3_of_quotient(v, in->v_scale);
                    else
                        ((uint16_t *)cache)[crow + QK_HEAD_DIM + d] = v;
                }
            }
        }
    }
    if (n_alt)
        *n_alt = alts.n;
    return alts.n > alt_cap ? QK_ERR_ALT_CAP : QK_OK;
}
