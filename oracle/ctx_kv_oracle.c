/*
 * Plain CPU oracle of the DSpark fused context-KV write.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA path and is deliberately slow and literal:
 * one row at a time, fp64 arithmetic, no blocking, no fusion.
 *
 * What it computes (vLLM DSpark context-KV writer page, module docstring, and
 * the DSpark draft model page, MiniMaxM3DSparkModel.precompute_and_store_context_kv):
 * for every context token t whose slot is >= 0, every layer l and every KV
 * head h,
 *   1. k = all_kv[t, l, 0, h, :], v = all_kv[t, l, 1, h, :]   (bf16, D each;
 *      D = 128 on the pages, any head_dim up to 256 here)
 *   2. Gemma RMSNorm of k:  y = k * rsqrt(mean(k^2) + eps) * (1 + w[l]),
 *      materialised to bf16 (the page states fp32 evaluation; this oracle
 *      evaluates in fp64 and reports both bf16 neighbours as admissible when
 *      the value lies within 2^-18 relative of a rounding midpoint, which
 *      covers any fp32 evaluation order)
 *   3. partial NeoX RoPE of the first r dims at position pos[t] from the
 *      bf16 cos|sin row (cos in [0, r/2), sin in [r/2, r)):
 *        y'[i]       = y[i] c_i - y[i + r/2] s_i
 *        y'[i + r/2] = y[i + r/2] c_i + y[i] s_i        for i < r/2,
 *      each output rounded once to bf16; dims >= r pass through
 *   4. store: raw bf16 K'|V, or fp8 e4m3 (OCP, round to nearest even,
 *      saturating at +-448) of x / scale with the division in fp32
 *   5. the 2D-element row K'|V goes to layer l's paged cache
 *      [num_blocks, nkv, block_size, 2D] at block slot / block_size,
 *      head h, offset slot % block_size (any block size >= 1).
 * Slots < 0 are padding: nothing is read or written for them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_HEAD_DIM 128     /* the pages' head dim: the default */
#define ORACLE_MAX_HEAD_DIM 256
#define ORACLE_TIE_REL 3.814697265625e-06 /* 2^-18 */

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_FP8_E4M3 = 1 };

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_ARG = -1,
    ORACLE_ERR_SLOT_RANGE = -2,
    ORACLE_ERR_SLOT_DUP = -3,
    ORACLE_ERR_POS_RANGE = -4,
    ORACLE_ERR_SCALE = -5,
    ORACLE_ERR_ALT_CAP = -6,
    ORACLE_ERR_NOMEM = -7,
};

/* Everything one write call reads (host memory). */
typedef struct {
    const uint16_t *all_kv;       /* bf16 bits [T][L][2][H][D] */
    const uint16_t *knorm_w;      /* bf16 bits [L][D] */
    const int64_t *positions;     /* [T] */
    const int64_t *slot_mapping;  /* [T], < 0 = padding */
    const uint16_t *cos_sin;      /* bf16 bits [max_pos][r] */
    const float *k_scale;         /* [L], read in fp8 mode only */
    const float *v_scale;         /* [L], read in fp8 mode only */
    int64_t num_ctx;
    int64_t max_pos;
    int64_t num_blocks;
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t rotary_dim;
    int32_t kv_dtype;
    float eps;
    /* [L][T] one slot mapping per layer (drafts whose layers span several
     * KV-cache groups, DSpark draft model page, _shared_slot_mapping), or
     * NULL: slot_mapping is shared by every layer. */
    const int64_t *layer_slots;
    /* D, the head dim of K and V (1..256); 0 means the pages' 128.  all_kv
     * is then [T][L][2][H][D], knorm_w [L][D], cache rows 2D elements. */
    int32_t head_dim;
} dspark_oracle_inputs;

static int head_dim_of(const dspark_oracle_inputs *in)
{
    return in->head_dim ? in->head_dim : ORACLE_HEAD_DIM;
}

/* The slot of token t in layer l's cache. */
static int64_t slot_of(const dspark_oracle_inputs *in, int64_t t, int32_t l)
{
    return in->layer_slots ? in->layer_slots[(int64_t)l * in->num_ctx + t] : in->slot_mapping[t];
}

/* ------------------------------------------------------------------ */
/* bf16: 1 sign, 8 exponent, 7 stored mantissa bits (the top half of an
 * IEEE binary32).                                                        */

double dspark_oracle_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a real number (given as a double) to the nearest bf16, ties to
 * even.  8 significant bits; below 2^-126 the spacing stays 2^-133
 * (subnormals); results above the largest finite bf16 become infinity. */
uint16_t dspark_oracle_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e2;
    frexp(a, &e2);               /* a in [2^(e2-1), 2^e2) */
    int ulp_exp = (e2 - 1) - 7;  /* 7 fraction bits */
    if (ulp_exp < -133)
        ulp_exp = -133;
    double q = ldexp(a, -ulp_exp);      /* exact: a power-of-two scaling */
    double whole = floor(q);
    double rem = q - whole;             /* exact */
    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) != 0.0))
        whole += 1.0;
    double r = ldexp(whole, ulp_exp);
    if (r > 3.3895313892515355e38)      /* (2 - 2^-7) * 2^127 */
        return sign | 0x7F80;
    float f = (float)r;                 /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448;
 * exponent field 0 holds subnormals m/8 * 2^-6.                           */

double dspark_oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* fp32 value -> e4m3 code, round to nearest even, saturating to +-448 (also
 * for infinities); NaN -> 0x7F. */
uint8_t dspark_oracle_e4m3_rne_sat(float xf)
{
    double x = (double)xf;
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);
    int e = e2 - 1;                        /* a in [2^e, 2^(e+1)) */
    int ulp_exp = (e < -6 ? -6 : e) - 3;   /* 3 fraction bits; subnormal spacing 2^-9 */
    double q = ldexp(a, -ulp_exp);
    double whole = floor(q);
    double rem = q - whole;
    if (rem > 0.5 || (rem == 0.5 && fmod(whole, 2.0) != 0.0))
        whole += 1.0;
    double v = ldexp(whole, ulp_exp);      /* <= 448 since a < 448 */
    if (v == 0.0)
        return sign;
    frexp(v, &e2);
    e = e2 - 1;
    if (e < -6)
        return sign | (uint8_t)ldexp(v, 9);            /* subnormal: m = v / 2^-9 */
    int m = (int)(ldexp(v, -e) * 8.0) - 8;             /* v = (1 + m/8) 2^e */
    return sign | (uint8_t)(((e + 7) << 3) | m);
}

/* ------------------------------------------------------------------ */
/* Step 2: Gemma RMSNorm of one K row of n elements.  y[d] is the bf16 rounding (ties to
 * even) of the exact value; y_alt[d] is the other bf16 neighbour when the
 * exact value lies within ORACLE_TIE_REL (relative) of a rounding midpoint,
 * else y[d] again.  Returns the number of such ambiguous dims. */
int dspark_oracle_gemma_knorm_n(const uint16_t *k, const uint16_t *w, int n, float eps,
                                uint16_t *y, uint16_t *y_alt)
{
    double ss = 0.0;
    for (int d = 0; d < n; d++) {
        double kd = dspark_oracle_bf16_decode(k[d]);
        ss += kd * kd;
    }
    double inv = 1.0 / sqrt(ss / (double)n + (double)eps);
    int amb = 0;
    for (int d = 0; d < n; d++) {
        double v = dspark_oracle_bf16_decode(k[d]) * inv *
                   (1.0 + dspark_oracle_bf16_decode(w[d]));
        uint16_t dn = dspark_oracle_bf16_rne(v * (1.0 - ORACLE_TIE_REL));
        uint16_t up = dspark_oracle_bf16_rne(v * (1.0 + ORACLE_TIE_REL));
        y[d] = dspark_oracle_bf16_rne(v);
        y_alt[d] = y[d];
        if (dn != up) {
            y_alt[d] = y[d] == dn ? up : dn;
            amb++;
        }
    }
    return amb;
}

/* The same at the pages' head dim, 128. */
int dspark_oracle_gemma_knorm(const uint16_t *k, const uint16_t *w, float eps,
                              uint16_t *y, uint16_t *y_alt)
{
    return dspark_oracle_gemma_knorm_n(k, w, ORACLE_HEAD_DIM, eps, y, y_alt);
}

/* Step 3 for one rotated pair (i, i + r/2): exact products in fp64, one
 * rounding to bf16 per output. */
void dspark_oracle_rope_pair(uint16_t x1, uint16_t x2, uint16_t c, uint16_t s,
                             uint16_t *o1, uint16_t *o2)
{
    double a = dspark_oracle_bf16_decode(x1), b = dspark_oracle_bf16_decode(x2);
    double cc = dspark_oracle_bf16_decode(c), ss = dspark_oracle_bf16_decode(s);
    *o1 = dspark_oracle_bf16_rne(a * cc - b * ss);
    *o2 = dspark_oracle_bf16_rne(b * cc + a * ss);
}

/* Step 4 for one bf16 value: the stored element (bf16 bits or e4m3 code). */
static uint16_t encode_elem(uint16_t x, int kv_dtype, float scale)
{
    if (kv_dtype == ORACLE_KV_BF16)
        return x;
    float xf = (float)dspark_oracle_bf16_decode(x);
    float q = xf / scale; /* fp32 division, correctly rounded */
    return dspark_oracle_e4m3_rne_sat(q);
}

/* ------------------------------------------------------------------ */
/* One output row.  out: 2D stored elements (uint16 bf16 bits, or uint8
 * e4m3 codes when kv_dtype is fp8).  Every other admissible value of a K
 * element (from a bf16 tie in the norm) is appended to alt_dim/alt_val
 * (room for 3 * D entries); *n_alt receives their count. */
int dspark_oracle_row(const dspark_oracle_inputs *in, int64_t t, int32_t l, int32_t h,
                      void *out, int32_t *alt_dim, uint16_t *alt_val, int32_t *n_alt)
{
    const int L = in->num_layers, H = in->num_kv_heads, r = in->rotary_dim;
    const int D = head_dim_of(in);
    if (t < 0 || t >= in->num_ctx || l < 0 || l >= L || h < 0 || h >= H)
        return ORACLE_ERR_ARG;
    if (D < 1 || D > ORACLE_MAX_HEAD_DIM)
        return ORACLE_ERR_ARG;
    const int64_t base = (((t * L + l) * 2 + 0) * H + h) * D;
    const int64_t vbase = (((t * L + l) * 2 + 1) * H + h) * D;
    const uint16_t *k = in->all_kv + base;
    const uint16_t *v = in->all_kv + vbase;
    const uint16_t *w = in->knorm_w + (int64_t)l * D;
    const int64_t pos = in->positions[t];
    if (pos < 0 || pos >= in->max_pos)
        return ORACLE_ERR_POS_RANGE;
    const uint16_t *cs = in->cos_sin + pos * r;
    const float ks = in->kv_dtype == ORACLE_KV_FP8_E4M3 ? in->k_scale[l] : 1.0f;
    const float vs = in->kv_dtype == ORACLE_KV_FP8_E4M3 ? in->v_scale[l] : 1.0f;

    uint16_t y[ORACLE_MAX_HEAD_DIM], y_alt[ORACLE_MAX_HEAD_DIM];
    dspark_oracle_gemma_knorm_n(k, w, D, in->eps, y, y_alt);

    uint16_t res[2 * ORACLE_MAX_HEAD_DIM];
    int na = 0;
    for (int d = 0; d < D; d++) {
        /* candidate K' values of dim d; the first is the primary one, built
         * from the correctly rounded norm outputs */
        uint16_t cand[4];
        int nc = 0;
        if (d < r) {
            const int half = r / 2;
            const int lower = d < half;
            const int i = lower ? d : d - half;        /* frequency index */
            const int p = lower ? d + half : d - half; /* partner dim */
            const uint16_t c = cs[i], s = cs[half + i];
            const uint16_t self_c[2] = {y[d], y_alt[d]};
            const uint16_t part_c[2] = {y[p], y_alt[p]};
            const int ns = y_alt[d] != y[d] ? 2 : 1;
            const int np = y_alt[p] != y[p] ? 2 : 1;
            for (int a = 0; a < ns; a++)
                for (int b = 0; b < np; b++) {
                    uint16_t o1, o2;
                    if (lower) {
                        dspark_oracle_rope_pair(self_c[a], part_c[b], c, s, &o1, &o2);
                        cand[nc++] = o1;
                    } else {
                        dspark_oracle_rope_pair(part_c[b], self_c[a], c, s, &o1, &o2);
                        cand[nc++] = o2;
                    }
                }
        } else {
            cand[nc++] = y[d];
            if (y_alt[d] != y[d])
                cand[nc++] = y_alt[d];
        }
        uint16_t enc[4];
        for (int j = 0; j < nc; j++)
            enc[j] = encode_elem(cand[j], in->kv_dtype, ks);
        res[d] = enc[0];
        for (int j = 1; j < nc; j++) {
            int seen = enc[j] == enc[0];
            for (int q = 1; q < j; q++)
                seen |= enc[q] == enc[j];
            if (!seen) {
                if (alt_dim)
                    alt_dim[na] = d;
                if (alt_val)
                    alt_val[na] = enc[j];
                na++;
            }
        }
    }
    for (int d = 0; d < D; d++)
        res[D + d] = encode_elem(v[d], in->kv_dtype, vs);

    if (in->kv_dtype == ORACLE_KV_FP8_E4M3) {
        uint8_t *o8 = (uint8_t *)out;
        for (int d = 0; d < 2 * D; d++)
            o8[d] = (uint8_t)res[d];
    } else {
        memcpy(out, res, (size_t)(2 * D) * sizeof(uint16_t));
    }
    if (n_alt)
        *n_alt = na;
    return ORACLE_OK;
}

/* Step 5: the row of layer l's cache [num_blocks, H, block_size, 2D] that
 * (slot, h) addresses, counted in 2D-element rows; -1 for padding, -2 when
 * the slot lies beyond the cache. */
int64_t dspark_oracle_dest_row(int64_t slot, int32_t h, int32_t num_kv_heads,
                               int32_t block_size, int64_t num_blocks)
{
    if (slot < 0)
        return -1;
    int64_t block = slot / block_size;
    int64_t offset = slot % block_size;
    if (block >= num_blocks)
        return -2;
    return (block * num_kv_heads + h) * block_size + offset;
}

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* Preconditions of a write: within each layer's cache, valid slots unique
 * and inside the cache; positions of tokens with a valid slot (in any
 * layer) inside the cos|sin table; fp8 scales positive and finite. */
int dspark_oracle_check_inputs(const dspark_oracle_inputs *in)
{
    if (!in || in->num_ctx < 0 || in->num_layers <= 0 || in->num_kv_heads <= 0 ||
        in->block_size <= 0 || in->num_blocks <= 0 || in->max_pos <= 0)
        return ORACLE_ERR_ARG;
    if (head_dim_of(in) < 1 || head_dim_of(in) > ORACLE_MAX_HEAD_DIM)
        return ORACLE_ERR_ARG;
    if (in->rotary_dim <= 0 || in->rotary_dim > head_dim_of(in) || in->rotary_dim % 2)
        return ORACLE_ERR_ARG;
    if (in->kv_dtype != ORACLE_KV_BF16 && in->kv_dtype != ORACLE_KV_FP8_E4M3)
        return ORACLE_ERR_ARG;
    const int64_t cap = in->num_blocks * in->block_size;
    const int L = in->num_layers;
    for (int64_t t = 0; t < in->num_ctx; t++) {
        int any = 0;
        for (int l = 0; l < L; l++) {
            int64_t s = slot_of(in, t, l);
            if (s < 0)
                continue;
            if (s >= cap)
                return ORACLE_ERR_SLOT_RANGE;
            any = 1;
        }
        if (any && (in->positions[t] < 0 || in->positions[t] >= in->max_pos))
            return ORACLE_ERR_POS_RANGE;
    }
    if (in->kv_dtype == ORACLE_KV_FP8_E4M3)
        for (int l = 0; l < L; l++)
            if (!(in->k_scale[l] > 0.0f) || !(in->v_scale[l] > 0.0f) ||
                isinf(in->k_scale[l]) || isinf(in->v_scale[l]))
                return ORACLE_ERR_SCALE;
    int64_t *sorted = (int64_t *)malloc((size_t)(in->num_ctx ? in->num_ctx : 1) * sizeof(int64_t));
    if (!sorted)
        return ORACLE_ERR_NOMEM;
    int rc = ORACLE_OK;
    const int layers_to_check = in->layer_slots ? L : 1;
    for (int l = 0; l < layers_to_check && rc == ORACLE_OK; l++) {
        int64_t nv = 0;
        for (int64_t t = 0; t < in->num_ctx; t++) {
            int64_t s = slot_of(in, t, l);
            if (s >= 0)
                sorted[nv++] = s;
        }
        qsort(sorted, (size_t)nv, sizeof(int64_t), cmp_i64);
        for (int64_t i = 1; i < nv; i++)
            if (sorted[i] == sorted[i - 1]) {
                rc = ORACLE_ERR_SLOT_DUP;
                break;
            }
    }
    free(sorted);
    return rc;
}

/* The whole write for tokens [t_begin, t_end): every valid row computed by
 * dspark_oracle_row and stored into caches[l] (host buffers, one per layer,
 * each [num_blocks, H, block_size, 2D] of the cache dtype).  Admissible
 * alternates are reported as (layer, element index in that layer's cache,
 * value), up to alt_cap of them; *n_alt receives how many there were in
 * total.  Returns ORACLE_ERR_ALT_CAP (after writing everything) when more
 * alternates existed than fit. */
int dspark_oracle_write(const dspark_oracle_inputs *in, void *const *caches,
                        int64_t t_begin, int64_t t_end,
                        int32_t *alt_layer, int64_t *alt_elem, uint16_t *alt_val,
                        int64_t alt_cap, int64_t *n_alt)
{
    int rc = dspark_oracle_check_inputs(in);
    if (rc != ORACLE_OK)
        return rc;
    if (t_begin < 0 || t_end > in->num_ctx || t_begin > t_end)
        return ORACLE_ERR_ARG;
    const int L = in->num_layers, H = in->num_kv_heads;
    const size_t esz = in->kv_dtype == ORACLE_KV_FP8_E4M3 ? 1 : 2;
    const int64_t row_elems = 2 * (int64_t)head_dim_of(in);
    int64_t total_alt = 0;
    int32_t rd[3 * ORACLE_MAX_HEAD_DIM];
    uint16_t rv[3 * ORACLE_MAX_HEAD_DIM];
    uint16_t row[2 * ORACLE_MAX_HEAD_DIM];
    for (int64_t t = t_begin; t < t_end; t++) {
        for (int l = 0; l < L; l++) {
            const int64_t slot = slot_of(in, t, l);
            if (slot < 0)
                continue; /* padding: not written */
            for (int h = 0; h < H; h++) {
                int32_t na = 0;
                rc = dspark_oracle_row(in, t, l, h, row, rd, rv, &na);
                if (rc != ORACLE_OK)
                    return rc;
                int64_t dst = dspark_oracle_dest_row(slot, h, H, in->block_size, in->num_blocks);
                uint8_t *layer = (uint8_t *)caches[l];
                memcpy(layer + (size_t)(dst * row_elems) * esz, row, (size_t)row_elems * esz);
                for (int j = 0; j < na; j++) {
                    if (total_alt < alt_cap) {
                        alt_layer[total_alt] = l;
                        alt_elem[total_alt] = dst * row_elems + rd[j];
                        alt_val[total_alt] = rv[j];
                    }
                    total_alt++;
                }
            }
        }
    }
    if (n_alt)
        *n_alt = total_alt;
    return total_alt > alt_cap ? ORACLE_ERR_ALT_CAP : ORACLE_OK;
}

/* The same write split over n host threads by token ranges (for timing
 * the oracle on every host core): each thread runs dspark_oracle_write on
 * its own range with its own alternate buffers, which it discards; valid
 * slots are distinct, so the threads write disjoint cache rows.  Nothing of
 * the arithmetic changes.  Returns the first failing thread's status. */
typedef struct {
    const dspark_oracle_inputs *in;
    void *const *caches;
    int64_t t_begin, t_end, cap;
    int rc;
} oracle_range;

static void *oracle_range_run(void *arg)
{
    oracle_range *r = (oracle_range *)arg;
    int32_t *al = (int32_t *)malloc((size_t)r->cap * sizeof(int32_t));
    int64_t *ae = (int64_t *)malloc((size_t)r->cap * sizeof(int64_t));
    uint16_t *av = (uint16_t *)malloc((size_t)r->cap * sizeof(uint16_t));
    int64_t n = 0;
    r->rc = (al && ae && av) ? dspark_oracle_write(r->in, r->caches, r->t_begin, r->t_end, al, ae, av, r->cap, &n)
                             : ORACLE_ERR_NOMEM;
    if (r->rc == ORACLE_ERR_ALT_CAP)
        r->rc = ORACLE_OK; /* the caches are complete; only the discarded alternates overflowed */
    free(al);
    free(ae);
    free(av);
    return NULL;
}

int dspark_oracle_write_threads(const dspark_oracle_inputs *in, void *const *caches, int64_t t_begin,
                                int64_t t_end, int32_t nthreads)
{
    if (nthreads < 1 || nthreads > 1024 || t_begin < 0 || t_begin > t_end)
        return ORACLE_ERR_ARG;
    oracle_range *r = (oracle_range *)calloc((size_t)nthreads, sizeof(oracle_range));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!r || !th) {
        free(r);
        free(th);
        return ORACLE_ERR_NOMEM;
    }
    const int64_t n = t_end - t_begin;
    int started = 0, rc = ORACLE_OK;
    for (int i = 0; i < nthreads; i++) {
        r[i].in = in;
        r[i].caches = caches;
        r[i].t_begin = t_begin + n * i / nthreads;
        r[i].t_end = t_begin + n * (i + 1) / nthreads;
        r[i].cap = 1 << 16;
        if (pthread_create(&th[i], NULL, oracle_range_run, &r[i]) != 0) {
            rc = ORACLE_ERR_NOMEM;
            break;
        }
        started++;
    }
    for (int i = 0; i < started; i++) {
        pthread_join(th[i], NULL);
        if (rc == ORACLE_OK && r[i].rc != ORACLE_OK)
            rc = r[i].rc;
    }
    free(r);
    free(th);
    return rc;
}

/* Rows (t, l, h) given as flat indices (t * L + l) * H + h, whatever their
 * slot: out is [n][2D] stored elements; alternates as (index into the row
 * list, dim, value). */
int dspark_oracle_rows(const dspark_oracle_inputs *in, const int64_t *row_ids, int64_t n,
                       void *out, int64_t *alt_row, int32_t *alt_dim, uint16_t *alt_val,
                       int64_t alt_cap, int64_t *n_alt)
{
    const int L = in->num_layers, H = in->num_kv_heads;
    const size_t esz = in->kv_dtype == ORACLE_KV_FP8_E4M3 ? 1 : 2;
    const int64_t row_elems = 2 * (int64_t)head_dim_of(in);
    int64_t total_alt = 0;
    int32_t rd[3 * ORACLE_MAX_HEAD_DIM];
    uint16_t rv[3 * ORACLE_MAX_HEAD_DIM];
    for (int64_t i = 0; i < n; i++) {
        int64_t id = row_ids[i];
        if (id < 0 || id >= in->num_ctx * L * H)
            return ORACLE_ERR_ARG;
        int64_t t = id / ((int64_t)L * H);
        int32_t l = (int32_t)((id / H) % L);
        int32_t h = (int32_t)(id % H);
        int32_t na = 0;
        int rc = dspark_oracle_row(in, t, l, h, (uint8_t *)out + (size_t)(i * row_elems) * esz,
                                   rd, rv, &na);
        if (rc != ORACLE_OK)
            return rc;
        for (int j = 0; j < na; j++) {
            if (total_alt < alt_cap) {
                alt_row[total_alt] = i;
                alt_dim[total_alt] = rd[j];
                alt_val[total_alt] = rv[j];
            }
            total_alt++;
        }
    }
    if (n_alt)
        *n_alt = total_alt;
    return total_alt > alt_cap ? ORACLE_ERR_ALT_CAP : ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* The fused context-KV projection's output (DSpark draft model page,
 * precompute_and_store_context_kv: all_kv = _project_context_kv_token_major
 * (context_states, ...), "the fused projection output all_kv [num_ctx, L, 2,
 * nkv, 128]" of the context-KV writer page): every element is the exact dot
 * product of a context-state row and a weight row (computed by the caller in
 * fp64), rounded once to bf16.  n values in, n bf16 codes out. */
void dspark_oracle_bf16_rne_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = dspark_oracle_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------ */
/* The hidden-state Gemma RMSNorm (DSpark draft model page: hidden_norm =
 * _gemma_rms_norm(hidden_size, eps), applied to the context states by
 * _normalize_context_states; "an fp32 1 + w weight"): for each of `rows`
 * rows of n bf16 values, y = x * rsqrt(mean(x^2) + eps) * (1 + w) rounded
 * to bf16, evaluated here in fp64.  y_alt as for the K norm: the other bf16
 * neighbour where the exact value lies within 2^-18 of a rounding midpoint
 * (else y).  Returns the number of such elements. */
int64_t dspark_oracle_gemma_norm_rows(const uint16_t *x, const uint16_t *w, int64_t rows, int64_t n, float eps,
                                      uint16_t *y, uint16_t *y_alt)
{
    int64_t amb = 0;
    for (int64_t r = 0; r < rows; r++) {
        const uint16_t *xr = x + r * n;
        double ss = 0.0;
        for (int64_t d = 0; d < n; d++) {
            double v = dspark_oracle_bf16_decode(xr[d]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / (double)n + (double)eps);
        for (int64_t d = 0; d < n; d++) {
            double v = dspark_oracle_bf16_decode(xr[d]) * inv * (1.0 + dspark_oracle_bf16_decode(w[d]));
            uint16_t dn = dspark_oracle_bf16_rne(v * (1.0 - ORACLE_TIE_REL));
            uint16_t up = dspark_oracle_bf16_rne(v * (1.0 + ORACLE_TIE_REL));
            uint16_t yy = dspark_oracle_bf16_rne(v);
            y[r * n + d] = yy;
            y_alt[r * n + d] = yy;
            if (dn != up) {
                y_alt[r * n + d] = yy == dn ? up : dn;
                amb++;
            }
        }
    }
    return amb;
}
