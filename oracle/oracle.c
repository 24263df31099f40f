/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the MoE routing +
 * FP8 quantisation path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the package smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library, and includes nothing from it.
 *
 * Compile: cc -O2 -ffp-contract=off -fPIC -shared oracle.c -o liboracle.so -lm
 * (no fast-math; -ffp-contract=off so every float operation written below is
 * rounded on its own, exactly as written).
 *
 * Sources it follows (page title and section):
 *  - "DeepSeek open-sources TileKernels" (itsolotime.com), section 2.1
 *    "Top-K Gating": pick the k highest expert scores per token, ties going to
 *    the lower expert index.
 *  - same page, the routing chain at the top of section 2 ("Top-K Gating ->
 *    Group Counting -> Token-Expert Mapping -> Fused Expand/Reduce -> Weight
 *    Normalization"), whose weight formula the page leaves open: read here as
 *    the softmax over the k selected scores.
 *  - "CuTeDSL at Perplexity", MoE dispatch/combine (TP=1 local kernel): count
 *    tokens per expert and give each routed copy a unique index in its
 *    expert's list; combine accumulates the weighted copies back per token.
 *  - TileKernels page, section 3.1 (CastOutputConfig: clamp_min_value 1e-4 for
 *    E4M3), section 3.2 (per_token_cast: group absmax -> scale -> multiply by
 *    the inverse scale), section 2.2 (expand_to_fused: copy each token and
 *    its scales to the rows given by pos, pos < 0 meaning "no copy"),
 *    section 3.3 (SwiGLU: val_l / (1 + exp(-val_l)) * val_r in fp32, then the
 *    same per-group cast).
 *  - E4M3FN itself (sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *    infinities, S.1111.111 = NaN, largest finite 448) comes from the OCP 8-bit
 *    floating point specification, which the pages name but do not print.
 *
 * Return codes of every entry: 0 = ok, 1 = invalid argument, 2 = non-finite or
 * out-of-range input that the method leaves undefined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 and E4M3FN as plain number formats                                   */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening is exact. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* The non-negative finite E4M3FN value of a 7-bit magnitude code (0..126).
 * Exponent field 0: subnormal m * 2^-9.  Otherwise (1 + m/8) * 2^(e-7). */
double oracle_e4m3_value(int code)
{
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    if (e == 0)
        return ldexp((double)m, -9);
    return ldexp(1.0 + m / 8.0, e - 7);
}

/* Decode any byte; NaN codes (0x7F, 0xFF) give NaN. */
double oracle_e4m3_decode(uint8_t c)
{
    int mag = c & 0x7F;
    double v;
    if (mag == 0x7F)
        return NAN;
    v = oracle_e4m3_value(mag);
    return (c & 0x80) ? -v : v;
}

static double g_e4m3_table[127];
static int g_e4m3_table_ready = 0;

static void e4m3_table_init(void)
{
    int c;
    if (g_e4m3_table_ready)
        return;
    for (c = 0; c < 127; ++c)
        g_e4m3_table[c] = oracle_e4m3_value(c);
    g_e4m3_table_ready = 1;
}

/* Round v to the nearest E4M3FN value, ties to the even code, and saturate
 * magnitudes at or beyond 448 (including infinity) to 448 ("satfinite").
 * The sign bit of v is kept, so -0.0 and negative values that round to zero
 * give 0x80.  NaN gives the NaN code with v's sign. */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a;
    int lo, hi, c;
    double mid;

    e4m3_table_init();
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    a = fabs((double)v);
    if (a >= g_e4m3_table[126])
        return (uint8_t)(sign | 126);
    /* largest c with table[c] <= a (table is increasing; table[0] = 0) */
    lo = 0;
    hi = 126;
    while (hi - lo > 1) {
        int m = (lo + hi) / 2;
        if (g_e4m3_table[m] <= a)
            lo = m;
        else
            hi = m;
    }
    c = lo;
    /* a lies in [table[c], table[c+1]) */
    mid = 0.5 * (g_e4m3_table[c] + g_e4m3_table[c + 1]); /* exact: dyadic */
    if (a < mid)
        return (uint8_t)(sign | c);
    if (a > mid)
        return (uint8_t)(sign | (c + 1));
    return (uint8_t)(sign | ((c % 2 == 0) ? c : c + 1));
}

void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even,
 * directly from the double (no intermediate float, so no double rounding).
 * Returns the 16 bf16 bits. */
uint16_t oracle_bf16_from_double(double x)
{
    double a, q, r, val;
    int ex;
    float f;
    uint32_t u;
    uint16_t sign = signbit(x) ? 0x8000 : 0;

    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0);
    a = fabs(x);
    if (a == 0.0)
        return sign;
    frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
    if (ex - 1 < -126)
        q = ldexp(1.0, -133); /* subnormal spacing of bf16 */
    else
        q = ldexp(1.0, ex - 1 - 7);
    r = nearbyint(a / q); /* default rounding mode: to nearest, ties even */
    val = r * q;
    if (val >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80); /* overflow to infinity */
    f = (float)val; /* exact: val has at most 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* ------------------------------------------------------------------------ */
/* Step 1: top-k gate and top-k weights                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    float score;
    int32_t expert;
} scored_expert_t;

/* Descending score; among equal scores the lower expert index first. */
static int by_score_then_index(const void *pa, const void *pb)
{
    const scored_expert_t *a = (const scored_expert_t *)pa;
    const scored_expert_t *b = (const scored_expert_t *)pb;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    return (a->expert < b->expert) ? -1 : (a->expert > b->expert);
}

/* TileKernels page, section 2.1: for each token the k experts with the
 * largest scores, in descending score order, ties to the lower index.  Written
 * as its plain definition: sort all E (score, index) pairs and keep k.
 *
 * weights (nullable): softmax over the k selected scores,
 *   w_j = exp(s_j - s_0) / sum_i exp(s_i - s_0),
 * evaluated in double and rounded once to fp32.
 * Scores must not be NaN (rc 2); weights also need finite selected scores. */
int oracle_topk_gate(const float *scores, int64_t T, int32_t E, int32_t k,
                     int32_t *topk_idx, float *topk_weights)
{
    scored_expert_t *row;
    int64_t t;
    int32_t e, j;

    if (T < 0 || E < 1 || k < 1 || k > E)
        return 1;
    if (T == 0)
        return 0;
    row = (scored_expert_t *)malloc(sizeof(scored_expert_t) * (size_t)E);
    if (!row)
        return 1;
    for (t = 0; t < T; ++t) {
        for (e = 0; e < E; ++e) {
            float s = scores[t * E + e];
            if (isnan(s)) {
                free(row);
                return 2;
            }
            row[e].score = s;
            row[e].expert = e;
        }
        qsort(row, (size_t)E, sizeof(scored_expert_t), by_score_then_index);
        for (j = 0; j < k; ++j)
            topk_idx[t * k + j] = row[j].expert;
        if (topk_weights) {
            double s0 = (double)row[0].score;
            double sum = 0.0;
            for (j = 0; j < k; ++j) {
                if (!isfinite(row[j].score)) {
                    free(row);
                    return 2;
                }
                sum += exp((double)row[j].score - s0);
            }
            for (j = 0; j < k; ++j)
                topk_weights[t * k + j] =
                    (float)(exp((double)row[j].score - s0) / sum);
        }
    }
    free(row);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: token -> expert mapping                                           */
/* ------------------------------------------------------------------------ */

/* "CuTeDSL at Perplexity", local dispatch: count the routed copies of each
 * expert, then give every copy a unique slot in its expert's list.  Here the
 * list order is made stable: copies are visited in (token, slot) row-major
 * order and each takes the next free slot of its expert, so
 *   counts[e]      = #{(t,j) : idx[t,j] = e}
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   pos[t,j]       = offsets[e] + #{(t',j') before (t,j) : idx[t',j'] = e}
 *   sorted_src[pos[t,j]] = t*k + j.
 * An index outside [0, E) is rc 2. */
int oracle_route_map(const int32_t *topk_idx, int64_t T, int32_t E, int32_t k,
                     int32_t *counts, int32_t *offsets, int32_t *pos,
                     int32_t *sorted_src)
{
    int64_t R, p;
    int32_t e;
    int64_t *cursor;

    if (T < 0 || E < 1 || k < 1)
        return 1;
    R = T * (int64_t)k;
    for (e = 0; e < E; ++e)
        counts[e] = 0;
    for (p = 0; p < R; ++p) {
        int32_t x = topk_idx[p];
        if (x < 0 || x >= E)
            return 2;
        counts[x] += 1;
    }
    offsets[0] = 0;
    for (e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    cursor = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!cursor)
        return 1;
    for (p = 0; p < R; ++p) {
        int32_t x = topk_idx[p];
        int64_t slot = offsets[x] + cursor[x];
        cursor[x] += 1;
        pos[p] = (int32_t)slot;
        sorted_src[slot] = (int32_t)p;
    }
    free(cursor);
    return 0;
}

/* Padded expert layout ("CuTeDSL at Perplexity", dispatch: tokens are
 * optionally copied into padded buffers for the MoE GEMM; TileKernels page,
 * section 2.2: expand_to_fused zero-fills the rows no token lands on).  Each
 * expert's segment is rounded up to a multiple of `align` rows:
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + align * ceil(counts[e] / align)
 * pos[t,j] = offsets[e] + (copies of e before (t,j) in row-major order), and
 * sorted_src[r] = t*k + j for r = pos[t,j], -1 for every other row in
 * [0, num_rows).  num_rows < offsets[E] is rc 1; an index outside [0, E) is
 * rc 2.  align = 1 is oracle_route_map with the -1 tail. */
int oracle_route_map_aligned(const int32_t *topk_idx, int64_t T, int32_t E, int32_t k,
                             int32_t align, int64_t num_rows, int32_t *counts,
                             int32_t *offsets, int32_t *pos, int32_t *sorted_src)
{
    int64_t R, p, r;
    int32_t e;
    int64_t *cursor;

    if (T < 0 || E < 1 || k < 1 || align < 1 || num_rows < 0)
        return 1;
    R = T * (int64_t)k;
    for (e = 0; e < E; ++e)
        counts[e] = 0;
    for (p = 0; p < R; ++p) {
        int32_t x = topk_idx[p];
        if (x < 0 || x >= E)
            return 2;
        counts[x] += 1;
    }
    offsets[0] = 0;
    for (e = 0; e < E; ++e) {
        int64_t padded = ((int64_t)counts[e] + align - 1) / align * align;
        offsets[e + 1] = (int32_t)(offsets[e] + padded);
    }
    if (num_rows < offsets[E])
        return 1;
    for (r = 0; r < num_rows; ++r)
        sorted_src[r] = -1;
    cursor = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!cursor)
        return 1;
    for (p = 0; p < R; ++p) {
        int32_t x = topk_idx[p];
        int64_t slot = offsets[x] + cursor[x];
        cursor[x] += 1;
        pos[p] = (int32_t)slot;
        sorted_src[slot] = (int32_t)p;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The per-group FP8 cast (TileKernels page, sections 3.1 and 3.2)            */
/* ------------------------------------------------------------------------ */

/* Cast one group of n fp32 values: amax = max |v|; sf = max(amax, 1e-4)/448
 * in fp32; sf_inv = 1/sf in fp32; q_i = E4M3(v_i * sf_inv).  Returns sf. */
static float cast_group(const float *v, int n, uint8_t *q)
{
    float amax = 0.0f;
    float clamped, sf, sf_inv;
    int i;

    for (i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    clamped = (amax < 1e-4f) ? 1e-4f : amax;
    sf = clamped / 448.0f;
    sf_inv = 1.0f / sf;
    for (i = 0; i < n; ++i) {
        float scaled = v[i] * sf_inv;
        q[i] = oracle_e4m3_encode(scaled);
    }
    return sf;
}

/* ---- cast options (TileKernels page, section 3.1: CastOutputConfig's
 * round_sf and packed UE8M0; section 2.2: the TMA-aligned column-major scale
 * layout expand_to_fused can write).  Flags:
 *   ORACLE_SF_COLMAJOR (1): scales stored transposed, [G][ld] (ld >= rows)
 *   ORACLE_SF_POW2     (2): round_sf: the scale is the smallest power of two
 *                           >= fl32(max(amax, 1e-4) / 448)
 *   ORACLE_SF_UE8M0    (4): store the (power-of-two) scale as its biased
 *                           exponent byte (UE8M0: value 2^(byte - 127));
 *                           row-major [rows][G] bytes, or with COLMAJOR four
 *                           consecutive groups of a row packed in one 32-bit
 *                           word (group 4i + j in byte j), [ceil(G/4)][ld]. */
#define ORACLE_SF_COLMAJOR 1
#define ORACLE_SF_POW2 2
#define ORACLE_SF_UE8M0 4

/* The power of two >= s (s positive, finite), by its definition. */
static float pow2_at_least(float s)
{
    float p = 1.0f;
    while (p < s)
        p *= 2.0f;
    while (p / 2.0f >= s)
        p /= 2.0f;
    return p;
}

/* Cast one group with the options: returns the scale (f32) actually used. */
static float cast_group_opts(const float *v, int n, int flags, uint8_t *q)
{
    float amax = 0.0f;
    float clamped, sf, sf_inv;
    int i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    clamped = (amax < 1e-4f) ? 1e-4f : amax;
    sf = clamped / 448.0f;
    if (flags & (ORACLE_SF_POW2 | ORACLE_SF_UE8M0))
        sf = pow2_at_least(sf);
    sf_inv = 1.0f / sf;
    for (i = 0; i < n; ++i) {
        float scaled = v[i] * sf_inv;
        q[i] = oracle_e4m3_encode(scaled);
    }
    return sf;
}

/* Write scale `sf` of (row r, group g) in the layout the flags name. */
static void store_scale(void *out_sf, int flags, int64_t ld, int32_t G, int64_t r, int32_t g,
                        float sf)
{
    if (flags & ORACLE_SF_UE8M0) {
        int ex;
        uint8_t byte;
        frexp((double)sf, &ex);  /* sf = 0.5 * 2^ex exactly: log2(sf) = ex - 1 */
        byte = (uint8_t)(ex - 1 + 127);
        if (flags & ORACLE_SF_COLMAJOR)
            ((uint8_t *)out_sf)[((int64_t)(g / 4) * ld + r) * 4 + (g % 4)] = byte;
        else
            ((uint8_t *)out_sf)[r * G + g] = byte;
    } else {
        if (flags & ORACLE_SF_COLMAJOR)
            ((float *)out_sf)[(int64_t)g * ld + r] = sf;
        else
            ((float *)out_sf)[r * G + g] = sf;
    }
}

/* Expand + cast with scale options, optionally zero-filling (codes and
 * scales: 0.0f, or byte 0 for UE8M0) the rows with sorted_src[r] < 0
 * (sorted_src may be NULL).  Rows no pos names and no zero-fill covers are
 * left untouched. */
int oracle_expand_cast_fp8_ex(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                              const int32_t *pos, const int32_t *sorted_src, int64_t num_rows,
                              int32_t group, int32_t flags, int64_t ld, uint8_t *out,
                              void *out_sf)
{
    int64_t t, r;
    int32_t j, g, i, G;
    float *buf, *sfs;
    uint8_t *qrow;

    if (T < 0 || k < 1 || group < 1 || H < group || H % group != 0 || num_rows < 0)
        return 1;
    if ((flags & ORACLE_SF_COLMAJOR) && ld < num_rows)
        return 1;
    G = H / group;
    if (sorted_src) {
        for (r = 0; r < num_rows; ++r) {
            if (sorted_src[r] >= 0)
                continue;
            memset(out + r * H, 0, (size_t)H);
            for (g = 0; g < G; ++g) {
                if (flags & ORACLE_SF_UE8M0) {
                    if (flags & ORACLE_SF_COLMAJOR)
                        ((uint8_t *)out_sf)[((int64_t)(g / 4) * ld + r) * 4 + (g % 4)] = 0;
                    else
                        ((uint8_t *)out_sf)[r * G + g] = 0;
                } else {
                    store_scale(out_sf, flags, ld, G, r, g, 0.0f);
                }
            }
        }
    }
    buf = (float *)malloc(sizeof(float) * (size_t)group);
    sfs = (float *)malloc(sizeof(float) * (size_t)G);
    qrow = (uint8_t *)malloc((size_t)H);
    if (!buf || !sfs || !qrow) {
        free(buf); free(sfs); free(qrow);
        return 1;
    }
    for (t = 0; t < T; ++t) {
        for (g = 0; g < G; ++g) {
            for (i = 0; i < group; ++i)
                buf[i] = bf16_bits_to_float(x[t * H + (int64_t)g * group + i]);
            sfs[g] = cast_group_opts(buf, group, flags, qrow + (int64_t)g * group);
        }
        for (j = 0; j < k; ++j) {
            int32_t rr = pos[t * k + j];
            if (rr < 0)
                continue;
            if (rr >= num_rows) {
                free(buf); free(sfs); free(qrow);
                return 2;
            }
            memcpy(out + (int64_t)rr * H, qrow, (size_t)H);
            for (g = 0; g < G; ++g)
                store_scale(out_sf, flags, ld, G, rr, g, sfs[g]);
        }
    }
    free(buf); free(sfs); free(qrow);
    return 0;
}

/* per_token_cast: x [T, H] bf16 bits -> q [T, H] E4M3 bytes and
 * sf [T, H/group] fp32, row-major. */
int oracle_per_token_cast(const uint16_t *x, int64_t T, int32_t H,
                          int32_t group, uint8_t *q, float *sf)
{
    int64_t t;
    int32_t g, i, G;
    float *buf;

    if (T < 0 || group < 1 || H < group || H % group != 0)
        return 1;
    G = H / group;
    buf = (float *)malloc(sizeof(float) * (size_t)group);
    if (!buf)
        return 1;
    for (t = 0; t < T; ++t) {
        for (g = 0; g < G; ++g) {
            const uint16_t *src = x + t * H + (int64_t)g * group;
            for (i = 0; i < group; ++i)
                buf[i] = bf16_bits_to_float(src[i]);
            sf[t * G + g] = cast_group(buf, group, q + t * H + (int64_t)g * group);
        }
    }
    free(buf);
    return 0;
}

/* Step 3 as the page sequences it: per_token_cast of each token row, then
 * expand_to_fused copies the row's bytes and scales to every row pos[t,j]
 * (pos < 0: that copy is dropped).  Rows of out that no pos names are left
 * untouched.  pos >= num_rows is rc 2. */
int oracle_expand_cast_fp8(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                           const int32_t *pos, int64_t num_rows, int32_t group,
                           uint8_t *out, float *out_sf)
{
    int64_t t;
    int32_t j, G;
    uint8_t *qrow;
    float *sfrow;
    int rc;

    if (T < 0 || k < 1 || group < 1 || H < group || H % group != 0 || num_rows < 0)
        return 1;
    G = H / group;
    qrow = (uint8_t *)malloc((size_t)H);
    sfrow = (float *)malloc(sizeof(float) * (size_t)G);
    if (!qrow || !sfrow) {
        free(qrow);
        free(sfrow);
        return 1;
    }
    for (t = 0; t < T; ++t) {
        rc = oracle_per_token_cast(x + t * H, 1, H, group, qrow, sfrow);
        if (rc) {
            free(qrow);
            free(sfrow);
            return rc;
        }
        for (j = 0; j < k; ++j) {
            int32_t r = pos[t * k + j];
            if (r < 0)
                continue;
            if (r >= num_rows) {
                free(qrow);
                free(sfrow);
                return 2;
            }
            memcpy(out + (int64_t)r * H, qrow, (size_t)H);
            memcpy(out_sf + (int64_t)r * G, sfrow, sizeof(float) * (size_t)G);
        }
    }
    free(qrow);
    free(sfrow);
    return 0;
}

/* Expand into a padded layout in one pass (TileKernels page, section 2.2:
 * the same launch copies the valid rows and zero-fills the invalid ones):
 * every row r of [0, num_rows) with sorted_src[r] < 0 becomes all-zero codes
 * and all-zero scales; the other rows are written as oracle_expand_cast_fp8
 * writes them. */
int oracle_expand_cast_fp8_padded(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                                  const int32_t *pos, const int32_t *sorted_src,
                                  int64_t num_rows, int32_t group, uint8_t *out,
                                  float *out_sf)
{
    int64_t r;
    int32_t G;
    if (T < 0 || k < 1 || group < 1 || H < group || H % group != 0 || num_rows < 0)
        return 1;
    G = H / group;
    for (r = 0; r < num_rows; ++r) {
        if (sorted_src[r] < 0) {
            memset(out + r * H, 0, (size_t)H);
            memset(out_sf + r * G, 0, sizeof(float) * (size_t)G);
        }
    }
    return oracle_expand_cast_fp8(x, T, H, k, pos, num_rows, group, out, out_sf);
}

/* ------------------------------------------------------------------------ */
/* Step 4: SwiGLU + cast (TileKernels page, section 3.3, plain form)          */
/* ------------------------------------------------------------------------ */

/* v[r, c] = g / (1 + exp(-g)) * u with g = x[r, c] (left half, "val_l") and
 * u = x[r, N + c] (right half, "val_r"), each step rounded to fp32 in the
 * order written; exp is the host C library's expf. */
int oracle_swiglu_values(const uint16_t *x, int64_t M, int32_t N, float *v)
{
    int64_t r;
    int32_t c;
    if (M < 0 || N < 1)
        return 1;
    for (r = 0; r < M; ++r) {
        const uint16_t *row = x + r * 2 * (int64_t)N;
        for (c = 0; c < N; ++c) {
            float g = bf16_bits_to_float(row[c]);
            float u = bf16_bits_to_float(row[N + c]);
            float e = expf(-g);
            float den = 1.0f + e;
            float silu = g / den;
            v[r * N + c] = silu * u;
        }
    }
    return 0;
}

/* x [M, 2N] bf16 -> q [M, N] E4M3 + sf [M, N/group] fp32. */
int oracle_swiglu_cast_fp8(const uint16_t *x, int64_t M, int32_t N,
                           int32_t group, uint8_t *q, float *sf)
{
    int64_t r;
    int32_t g, G;
    float *v;

    if (M < 0 || group < 1 || N < group || N % group != 0)
        return 1;
    G = N / group;
    v = (float *)malloc(sizeof(float) * (size_t)N);
    if (!v)
        return 1;
    for (r = 0; r < M; ++r) {
        oracle_swiglu_values(x + r * 2 * (int64_t)N, 1, N, v);
        for (g = 0; g < G; ++g)
            sf[r * G + g] = cast_group(v + (int64_t)g * group, group,
                                       q + r * N + (int64_t)g * group);
    }
    free(v);
    return 0;
}

/* SwiGLU variants (TileKernels page, section 3.3): optional clamp (the gate
 * clamped from above, val_l = min(val_l, c); the up value clamped to [-c, c])
 * and optional per-row top-k weight (v = g / (1 + exp(-g)) * u * w[r]), then
 * the per-group cast with the scale options above.  clamp_count (nullable)
 * receives the number of inputs the clamp changed (gate values > c plus up
 * values with |u| > c), added to its current value.  has_clamp = 0: no clamp. */
int oracle_swiglu_cast_fp8_ex(const uint16_t *x, int64_t M, int32_t N, int32_t group,
                              int32_t has_clamp, float clamp, const float *weights,
                              int32_t flags, int64_t ld, uint8_t *q, void *out_sf,
                              uint64_t *clamp_count)
{
    int64_t r;
    int32_t c, g, G;
    float *v;
    uint64_t count = 0;

    if (M < 0 || group < 1 || N < group || N % group != 0)
        return 1;
    if ((flags & ORACLE_SF_COLMAJOR) && ld < M)
        return 1;
    G = N / group;
    v = (float *)malloc(sizeof(float) * (size_t)N);
    if (!v)
        return 1;
    for (r = 0; r < M; ++r) {
        const uint16_t *row = x + r * 2 * (int64_t)N;
        for (c = 0; c < N; ++c) {
            float gt = bf16_bits_to_float(row[c]);
            float u = bf16_bits_to_float(row[N + c]);
            float e, den, silu, val;
            if (has_clamp) {
                if (gt > clamp) {
                    gt = clamp;
                    count += 1;
                }
                if (u > clamp) {
                    u = clamp;
                    count += 1;
                } else if (u < -clamp) {
                    u = -clamp;
                    count += 1;
                }
            }
            e = expf(-gt);
            den = 1.0f + e;
            silu = gt / den;
            val = silu * u;
            if (weights)
                val = val * weights[r];
            v[c] = val;
        }
        for (g = 0; g < G; ++g) {
            float sf = cast_group_opts(v + (int64_t)g * group, group, flags,
                                       q + r * N + (int64_t)g * group);
            store_scale(out_sf, flags, ld, G, r, g, sf);
        }
    }
    free(v);
    if (clamp_count)
        *clamp_count += count;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP4 E2M1 cast (TileKernels page, section 3.1: CastOutputConfig's           */
/* clamp_min_value for float4_e2m1fn is max_value * 2^-126; section 3.2:      */
/* per-group absmax -> scale -> multiply by the inverse scale, at a group size */
/* the config chooses, num_per_channels)                                      */
/* ------------------------------------------------------------------------ */

/* E2M1 (the FP4 element type of the OCP Microscaling Formats specification):
 * sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0; no infinity or
 * NaN.  Exponent field 0: subnormal m * 0.5.  Otherwise (1 + m/2) * 2^(e-1).
 * Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_value(int code)
{
    int mag = code & 7;
    int e = mag >> 1, m = mag & 1;
    double v = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return (code & 8) ? -v : v;
}

/* Round to nearest, ties to the even code (mantissa bit 0), saturating at
 * +-6; the sign is kept, also for a result of zero.  NaN -> 0xFF (no E2M1
 * encoding; an error marker).  The nearest code is found by comparing the
 * magnitude with every code value in double, which is exact for fp32 inputs. */
uint8_t oracle_e2m1_encode(float v)
{
    double a;
    int c, best = 0;
    uint8_t sign;

    if (v != v)
        return 0xFF;
    sign = signbit(v) ? 8 : 0;
    a = fabs((double)v);
    if (a >= 6.0)
        return (uint8_t)(sign | 7);
    for (c = 1; c < 8; ++c) {
        double dc = fabs(a - oracle_e2m1_value(c));
        double db = fabs(a - oracle_e2m1_value(best));
        if (dc < db || (dc == db && (c & 1) == 0))
            best = c;
    }
    return (uint8_t)(sign | best);
}

void oracle_e2m1_encode_array(const float *v, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_e2m1_encode(v[i]);
}

/* Cast one group of n fp32 values to E2M1: amax = max |v|;
 * sf = fl32(max(amax, 6 * 2^-126) / 6) (6 = the largest E2M1 value, the
 * floor its clamp_min_value), rounded up to a power of two under the POW2 /
 * UE8M0 options; sf_inv = fl32(1 / sf); code_i = E2M1(fl32(v_i * sf_inv)).
 * Returns sf. */
static float cast_group_fp4(const float *v, int n, int flags, uint8_t *codes)
{
    const float floor_v = ldexpf(6.0f, -126);
    float amax = 0.0f;
    float clamped, sf, sf_inv;
    int i;

    for (i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    clamped = (amax < floor_v) ? floor_v : amax;
    sf = clamped / 6.0f;
    if (flags & (ORACLE_SF_POW2 | ORACLE_SF_UE8M0))
        sf = pow2_at_least(sf);
    sf_inv = 1.0f / sf;
    for (i = 0; i < n; ++i) {
        float scaled = v[i] * sf_inv;
        codes[i] = oracle_e2m1_encode(scaled);
    }
    return sf;
}

/* Two E2M1 codes per byte: element 2i in the low nibble, 2i + 1 in the high
 * nibble (the order of the element pairs in memory). */
static void pack_e2m1(const uint8_t *codes, int n, uint8_t *out)
{
    int i;
    for (i = 0; i < n; i += 2)
        out[i / 2] = (uint8_t)((codes[i] & 0xF) | ((codes[i + 1] & 0xF) << 4));
}

/* Expand + FP4 cast: each token's row x[t] cast per group of `group`
 * channels (scales in the layout `flags` names, as the FP8 options), and
 * its packed codes [H/2] and scales copied to the rows pos[t, j] >= 0 of
 * out [num_rows][H/2] and out_sf.  Rows with sorted_src[r] < 0 (sorted_src
 * may be NULL) get zero codes and zero scales (byte 0 for UE8M0); other rows
 * no pos names are left untouched.  group: a divisor of H, even. */
int oracle_expand_cast_fp4(const uint16_t *x, int64_t T, int32_t H, int32_t k,
                           const int32_t *pos, const int32_t *sorted_src, int64_t num_rows,
                           int32_t group, int32_t flags, int64_t ld, uint8_t *out,
                           void *out_sf)
{
    int64_t t, r;
    int32_t j, g, i, G;
    float *buf, *sfs;
    uint8_t *codes, *qrow;

    if (T < 0 || k < 1 || group < 2 || group % 2 != 0 || H < group || H % group != 0 ||
        num_rows < 0)
        return 1;
    if ((flags & ORACLE_SF_COLMAJOR) && ld < num_rows)
        return 1;
    G = H / group;
    if (sorted_src) {
        for (r = 0; r < num_rows; ++r) {
            if (sorted_src[r] >= 0)
                continue;
            memset(out + r * (H / 2), 0, (size_t)(H / 2));
            for (g = 0; g < G; ++g) {
                if (flags & ORACLE_SF_UE8M0) {
                    if (flags & ORACLE_SF_COLMAJOR)
                        ((uint8_t *)out_sf)[((int64_t)(g / 4) * ld + r) * 4 + (g % 4)] = 0;
                    else
                        ((uint8_t *)out_sf)[r * G + g] = 0;
                } else {
                    store_scale(out_sf, flags, ld, G, r, g, 0.0f);
                }
            }
        }
    }
    buf = (float *)malloc(sizeof(float) * (size_t)group);
    sfs = (float *)malloc(sizeof(float) * (size_t)G);
    codes = (uint8_t *)malloc((size_t)H);
    qrow = (uint8_t *)malloc((size_t)(H / 2));
    if (!buf || !sfs || !codes || !qrow) {
        free(buf); free(sfs); free(codes); free(qrow);
        return 1;
    }
    for (t = 0; t < T; ++t) {
        for (g = 0; g < G; ++g) {
            for (i = 0; i < group; ++i)
                buf[i] = bf16_bits_to_float(x[t * H + (int64_t)g * group + i]);
            sfs[g] = cast_group_fp4(buf, group, flags, codes + (int64_t)g * group);
        }
        pack_e2m1(codes, H, qrow);
        for (j = 0; j < k; ++j) {
            int32_t rr = pos[t * k + j];
            if (rr < 0)
                continue;
            if (rr >= num_rows) {
                free(buf); free(sfs); free(codes); free(qrow);
                return 2;
            }
            memcpy(out + (int64_t)rr * (H / 2), qrow, (size_t)(H / 2));
            for (g = 0; g < G; ++g)
                store_scale(out_sf, flags, ld, G, rr, g, sfs[g]);
        }
    }
    free(buf); free(sfs); free(codes); free(qrow);
    return 0;
}

/* SwiGLU + FP4 E2M1 cast: the SwiGLU values of oracle_swiglu_cast_fp8_ex
 * (same clamp, weight and clamp count), cast per group of `group` channels
 * with cast_group_fp4 (max 6, clamp_min 6 * 2^-126); codes packed two per
 * byte, element 2i in the low nibble: q [M][N/2].  Scales as the options
 * name them. */
int oracle_swiglu_cast_fp4(const uint16_t *x, int64_t M, int32_t N, int32_t group,
                           int32_t has_clamp, float clamp, const float *weights, int32_t flags,
                           int64_t ld, uint8_t *q, void *out_sf, uint64_t *clamp_count)
{
    int64_t r;
    int32_t c, g, G;
    float *v;
    uint8_t *codes;
    uint64_t count = 0;

    if (M < 0 || group < 2 || group % 2 != 0 || N < group || N % group != 0)
        return 1;
    if ((flags & ORACLE_SF_COLMAJOR) && ld < M)
        return 1;
    G = N / group;
    v = (float *)malloc(sizeof(float) * (size_t)N);
    codes = (uint8_t *)malloc((size_t)N);
    if (!v || !codes) {
        free(v); free(codes);
        return 1;
    }
    for (r = 0; r < M; ++r) {
        const uint16_t *row = x + r * 2 * (int64_t)N;
        for (c = 0; c < N; ++c) {
            float gt = bf16_bits_to_float(row[c]);
            float u = bf16_bits_to_float(row[N + c]);
            float e, den, silu, val;
            if (has_clamp) {
                if (gt > clamp) {
                    gt = clamp;
                    count += 1;
                }
                if (u > clamp) {
                    u = clamp;
                    count += 1;
                } else if (u < -clamp) {
                    u = -clamp;
                    count += 1;
                }
            }
            e = expf(-gt);
            den = 1.0f + e;
            silu = gt / den;
            val = silu * u;
            if (weights)
                val = val * weights[r];
            v[c] = val;
        }
        for (g = 0; g < G; ++g) {
            float sf = cast_group_fp4(v + (int64_t)g * group, group, flags,
                                      codes + (int64_t)g * group);
            store_scale(out_sf, flags, ld, G, r, g, sf);
        }
        pack_e2m1(codes, N, q + r * (N / 2));
    }
    free(v); free(codes);
    if (clamp_count)
        *clamp_count += count;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 5: weighted combine ("CuTeDSL at Perplexity", combine kernel)         */
/* ------------------------------------------------------------------------ */

/* out[t, c] = sum_j w[t,j] * y[pos[t,j], c], summed in double (each product
 * of an fp32 and a bf16 is exact in double), then rounded once: to fp32 into
 * out_f32 and, directly from the double, to bf16 into out_bf16 (either may be
 * NULL).  pos < 0 drops that copy; pos >= num_rows is rc 2.
 * abs_sum (nullable) receives sum_j |w y| per element, the scale of the
 * rounding error any fp32 accumulation can make. */
int oracle_combine(const uint16_t *y, const float *w, const int32_t *pos,
                   int64_t T, int32_t H, int32_t k, int64_t num_rows,
                   float *out_f32, uint16_t *out_bf16, float *abs_sum)
{
    int64_t t;
    int32_t c, j;
    if (T < 0 || H < 1 || k < 1 || num_rows < 0)
        return 1;
    for (t = 0; t < T; ++t) {
        for (j = 0; j < k; ++j) {
            int32_t r = pos[t * k + j];
            if (r >= num_rows)
                return 2;
        }
        for (c = 0; c < H; ++c) {
            double acc = 0.0, mag = 0.0;
            for (j = 0; j < k; ++j) {
                int32_t r = pos[t * k + j];
                double term;
                if (r < 0)
                    continue;
                term = (double)w[t * k + j] *
                       (double)bf16_bits_to_float(y[(int64_t)r * H + c]);
                acc += term;
                mag += fabs(term);
            }
            if (out_f32)
                out_f32[t * H + c] = (float)acc;
            if (out_bf16)
                out_bf16[t * H + c] = oracle_bf16_from_double(acc);
            if (abs_sum)
                abs_sum[t * H + c] = (float)mag;
        }
    }
    return 0;
}
