/*
 * nvfp4_oracle.c -- CPU oracle for the NVFP4 (W4A4) MoE expert forward.
 *
 * TEST INFRASTRUCTURE.  This is the slow, plain reference that the CUDA path is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never loads it.
 *
 * Source of every rule below: the page "Gemma 4 NVFP4 MoE 空输出"
 * (taking-lying-flat.github.io, a write-up of vLLM issue #51525), cited as
 * [page, section / figure].  Where the page is silent the reading taken is
 * stated beside the code.
 *
 * Conventions
 *   - Floating-point steps that the method performs in FP32 are written as
 *     single IEEE float operations, one rounding each, in the order the method
 *     states them (compile with -ffp-contract=off so no FMA is formed).
 *   - Everything after the block quantisation is fp64 (the GEMM is exact in
 *     int64 before the final global-scale multiply).
 *   - NaN activations are outside the contract of every function here.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* threads: a plain parallel-for over [0, n)                                  */
/* ------------------------------------------------------------------------ */

typedef void (*range_fn)(int64_t lo, int64_t hi, void *ctx);

typedef struct {
    range_fn fn;
    void *ctx;
    int64_t lo, hi;
} range_job;

static void *range_job_run(void *p)
{
    range_job *j = (range_job *)p;
    j->fn(j->lo, j->hi, j->ctx);
    return NULL;
}

int orc_default_threads(void)
{
    const char *env = getenv("ORACLE_THREADS");
    if (env && atoi(env) > 0) return atoi(env);
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx)
{
    if (nthreads <= 0) nthreads = orc_default_threads();
    if (nthreads > 256) nthreads = 256;
    if (n < nthreads) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads <= 1) {
        fn(0, n, ctx);
        return;
    }
    pthread_t tid[256];
    range_job job[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t lo = (int64_t)t * chunk, hi = lo + chunk;
        if (lo >= n) break;
        if (hi > n) hi = n;
        job[t].fn = fn;
        job[t].ctx = ctx;
        job[t].lo = lo;
        job[t].hi = hi;
        if (pthread_create(&tid[t], NULL, range_job_run, &job[t]) != 0) {
            fn(lo, hi, ctx); /* could not start a thread: do the range here */
            job[t].fn = NULL;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (job[t].fn) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* FP4 E2M1                                                                   */
/* ------------------------------------------------------------------------ */

/* Magnitudes of codes 0..7 from the page's 16-entry E2M1 code table
 * [page, §NVFP4, E2M1 code table]; codes 8..15 carry the sign bit (1xxx) and
 * the same magnitudes, so 1000 is -0.0 and 1111 is -6.0. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code)
{
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Nearest E2M1 code to v.
 * [page, §NVFP4, text after the conversion listing]: round to nearest with
 * ties to even, and values beyond the largest finite magnitude (6) saturate to
 * it.  "Even" is the code whose lowest (mantissa) bit is 0.
 * Reading: the sign of v is kept even when the magnitude rounds to 0, as IEEE
 * conversions do, so -0.1 encodes as 1000 (-0.0).
 * Beyond the largest magnitude the value saturates; below it every distance
 * |a - m| is exact in double (a FP32 value and a 3-bit binary fraction below 8
 * need far fewer than 53 bits), so ties are detected exactly. */
int orc_e2m1_encode(float v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (a >= E2M1_MAG[7]) return sign | 7; /* saturate (also +-inf) */
    int best = 0;
    double bestd = fabs(a - E2M1_MAG[0]);
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return sign | best;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 (the block-scale format)                                          */
/* ------------------------------------------------------------------------ */

/* Value of an E4M3 byte.  [page, §NVFP4, two-level scale paragraph]: the block
 * scale is FP8 E4M3 with largest finite value 448.  Reading: the OCP "E4M3FN"
 * layout (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals,
 * no infinities, S.1111.111 is NaN), the only E4M3 layout whose maximum is 448. */
double orc_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Nearest finite E4M3 byte to t: round to nearest, ties to the even code,
 * saturating at +-448 (the scale is produced with the same round-to-nearest,
 * saturating conversion as the FP4 data [page, §NVFP4, runtime-order figure:
 * "generate and round to an FP8 E4M3 block scale"]).  Codes 0x00..0x7E are
 * ordered by value, so the scan below visits neighbours in order.  At or above
 * 448 the result saturates; below it the distances are exact in double. */
int orc_e4m3_encode(float t)
{
    int sign = signbit(t) ? 0x80 : 0;
    double a = fabs((double)t);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double bestd = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(a - orc_e4m3_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return sign | best;
}

/* Array forms of the two encoders (for exhaustive and randomised pins). */
typedef struct {
    const float *v;
    uint8_t *out;
    int which;
} enc_ctx;

static void enc_range(int64_t lo, int64_t hi, void *p)
{
    enc_ctx *c = (enc_ctx *)p;
    for (int64_t i = lo; i < hi; ++i)
        c->out[i] = (uint8_t)(c->which == 0 ? orc_e2m1_encode(c->v[i]) : orc_e4m3_encode(c->v[i]));
}

void orc_e2m1_encode_array(const float *v, int64_t n, uint8_t *out, int nthreads)
{
    enc_ctx c = {v, out, 0};
    parallel_for(n, nthreads, enc_range, &c);
}

void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out, int nthreads)
{
    enc_ctx c = {v, out, 1};
    parallel_for(n, nthreads, enc_range, &c);
}

/* ------------------------------------------------------------------------ */
/* Two-level block quantisation of one 16-element micro-block                  */
/* ------------------------------------------------------------------------ */

/* [page, §NVFP4, runtime-order figure] in the order the figure gives:
 *   1. amax of the 16 values;
 *   2. combine the global scale g (SFScaleVal, = 1/input_scale) with amax and
 *      the E2M1 maximum 6:  t = fl( fl(g * amax) / 6 )   (reading: the
 *      left-to-right FP32 order of "e4m3(g*amax/6)");
 *   3. round t to the E4M3 block scale sb, s = value(sb);
 *   4. normalise each value by the block scale and round to E2M1:
 *      q_i = e2m1( fl( fl(x_i * g) / s ) );
 * Reading for s == 0 (the figure is silent): every code is 0000.
 * Returns the scale byte; writes 16 codes (one per byte, 0..15). */
int orc_quant_block16(const float *x, float g, uint8_t *codes16)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float ga = g * amax;
    float t = ga / 6.0f;
    int sb = orc_e4m3_encode(t);
    double sv = orc_e4m3_value(sb);
    if (sv == 0.0) {
        memset(codes16, 0, 16);
        return sb;
    }
    float s = (float)sv; /* exact: every E4M3 value is a float */
    for (int i = 0; i < 16; ++i) {
        float y = x[i] * g;
        float q = y / s;
        codes16[i] = (uint8_t)orc_e2m1_encode(q);
    }
    return sb;
}

/* ------------------------------------------------------------------------ */
/* UE8M0 block scales (the variant the quantiser's UE8M0_SF flag selects)     */
/* ------------------------------------------------------------------------ */

/* [page, MoE section: the expert quantiser is a template with a UE8M0_SF
 * flag] -- the page names the flag and nothing more.  Reading: UE8M0 is the
 * MX-style scale byte, an unsigned biased exponent: byte b in 0..254 has value
 * 2^(b - 127) and 255 is NaN. */
double orc_ue8m0_value(int byte)
{
    if (byte == 255) return NAN;
    return ldexp(1.0, byte - 127);
}

/* Reading for the encoding: the block scale is the same t as in the E4M3 path,
 * rounded up to a power of two, so that the block's largest element, divided
 * by the scale, stays at or below 6 and does not saturate; t = 0 and values
 * below the range take the smallest byte (2^-127), values above it the largest
 * finite one (2^127).  The scan visits the bytes in value order. */
int orc_ue8m0_encode(float t)
{
    double a = (double)t;
    for (int b = 0; b < 255; ++b)
        if (ldexp(1.0, b - 127) >= a) return b;
    return 254;
}

/* orc_quant_block16 with a UE8M0 scale: steps 1, 2 and 4 as there, step 3
 * rounds t up to the UE8M0 scale s.  s is a power of two, so fl(y / s) is
 * the exact quotient rounded once.  Returns the scale byte. */
int orc_quant_block16_ue8m0(const float *x, float g, uint8_t *codes16)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float ga = g * amax;
    float t = ga / 6.0f;
    int sb = orc_ue8m0_encode(t);
    double s = orc_ue8m0_value(sb);
    for (int i = 0; i < 16; ++i) {
        float y = x[i] * g;
        float q = (float)((double)y / s); /* the quotient is exact in double */
        codes16[i] = (uint8_t)orc_e2m1_encode(q);
    }
    return sb;
}

/* Packing [page, §NVFP4, conversion listing and glossary "Packing"]: two E2M1
 * values per byte.  Reading of the listing's operand order under the PTX
 * definition of the x2 conversion (first source to the upper half): element
 * 2i goes to the low nibble of byte i and element 2i+1 to the high nibble. */
static uint8_t pack2(uint8_t lo_code, uint8_t hi_code)
{
    return (uint8_t)((lo_code & 15) | ((hi_code & 15) << 4));
}

typedef struct {
    const float *x;
    int64_t K;
    const float *g_row;
    uint8_t *q, *sf;
    int ue8m0;
} quant_ctx;

static void quant_range(int64_t lo, int64_t hi, void *p)
{
    quant_ctx *c = (quant_ctx *)p;
    uint8_t codes[16];
    for (int64_t r = lo; r < hi; ++r) {
        const float *xr = c->x + r * c->K;
        for (int64_t b = 0; b < c->K / 16; ++b) {
            c->sf[r * (c->K / 16) + b] =
                (uint8_t)(c->ue8m0 ? orc_quant_block16_ue8m0(xr + 16 * b, c->g_row[r], codes)
                                   : orc_quant_block16(xr + 16 * b, c->g_row[r], codes));
            for (int i = 0; i < 8; ++i)
                c->q[r * (c->K / 2) + 8 * b + i] = pack2(codes[2 * i], codes[2 * i + 1]);
        }
    }
}

/* Quantise `rows` rows of K values (K a multiple of 16), row r with global
 * scale g_row[r].  Outputs: q [rows, K/2] packed E2M1, sf [rows, K/16] E4M3
 * bytes, both row-major. */
void orc_quant_rows(const float *x, int64_t rows, int64_t K, const float *g_row, uint8_t *q,
                    uint8_t *sf, int nthreads)
{
    quant_ctx c = {x, K, g_row, q, sf, 0};
    parallel_for(rows, nthreads, quant_range, &c);
}

/* orc_quant_rows with UE8M0 block scales (sf holds UE8M0 bytes). */
void orc_quant_rows_ue8m0(const float *x, int64_t rows, int64_t K, const float *g_row, uint8_t *q,
                          uint8_t *sf, int nthreads)
{
    quant_ctx c = {x, K, g_row, q, sf, 1};
    parallel_for(rows, nthreads, quant_range, &c);
}

/* ------------------------------------------------------------------------ */
/* Scale validation                                                           */
/* ------------------------------------------------------------------------ */

/* [page, ROOT CAUSE]: the per-expert input scales are allocated uninitialised
 * and only the slots present in the checkpoint are overwritten; the reciprocal
 * is then taken with no completeness check, so a missing slot turns into an
 * inf / NaN / garbage global scale.  The check that was missing: every slot is
 * written, finite, positive and normal, and its FP32 reciprocal is finite and
 * normal.  `written` (nullable) holds one byte per slot, 0 = never written.
 * Returns the number of bad slots; *first_bad = lowest bad index or -1. */
int64_t orc_validate_scales(const float *s, const uint8_t *written, int64_t n, int64_t *first_bad)
{
    int64_t bad = 0;
    *first_bad = -1;
    for (int64_t i = 0; i < n; ++i) {
        float x = s[i];
        int ok = 1;
        if (written && written[i] == 0) ok = 0;
        if (!(x > 0.0f) || !isfinite(x) || !isnormal(x)) ok = 0;
        if (ok) {
            float r = 1.0f / x;
            if (!isfinite(r) || !isnormal(r)) ok = 0;
        }
        if (!ok) {
            if (*first_bad < 0) *first_bad = i;
            ++bad;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Token reorder (permutation)                                                */
/* ------------------------------------------------------------------------ */

/* [page, §矩阵融合 "MoE FFN" and the pipeline figure under it]: rows are
 * reordered by expert so that each expert's rows are contiguous and all
 * experts' GEMMs run as one grouped GEMM.  Reading (the page does not fix the
 * order inside an expert): expert-major, and within an expert ascending flat
 * index f = t*k + j, which makes the permutation unique.
 * Outputs: offsets[E+1] (offsets[e] = first permuted row of expert e,
 * offsets[E] = T*k) and perm[T*k] (permuted row -> flat index).
 * Returns 0, or -1 if an id is outside [0, E). */
int orc_route(const int32_t *ids, int64_t T, int32_t k, int32_t E, int32_t *offsets, int32_t *perm)
{
    int64_t R = T * (int64_t)k;
    for (int64_t f = 0; f < R; ++f)
        if (ids[f] < 0 || ids[f] >= E) return -1;
    memset(offsets, 0, sizeof(int32_t) * (size_t)(E + 1));
    for (int64_t f = 0; f < R; ++f) offsets[ids[f] + 1] += 1;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (!cursor) return -2;
    memcpy(cursor, offsets, sizeof(int32_t) * (size_t)E);
    for (int64_t f = 0; f < R; ++f) perm[cursor[ids[f]]++] = (int32_t)f;
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Router: softmax over the experts, top-k, renormalised                      */
/* ------------------------------------------------------------------------ */

/* [page "Gemma 4 NVFP4 MoE 空输出", §矩阵融合 "MoE FFN": the routing result
 * decides which experts a token visits, and the expert outputs are summed with
 * the routing weights; page "genesis-vllm-patches" (mlqm.cn), §3.3 patch P31:
 * the router's softmax and top-k run on logits upcast to FP32].  Per token,
 * from FP32 logits l[0..E):
 *   1. p_e = exp(l_e) / sum_e' exp(l_e')     softmax, fp64 (shifted by max l)
 *   2. the k experts of largest p, largest first, ties to the lower index
 *   3. w_j = p_ids[j] / sum_i p_ids[i]        renormalised over the k, stored FP32
 * Reading for step 3: the pages do not say whether the k weights are
 * renormalised; renormalising over the selected k (weights sum to 1) is the
 * reading taken.  Reading for step 2: softmax is strictly increasing in the
 * logit, so the exact probability order is the order of the FP32 logits; the
 * selection compares the logits themselves (an fp64 probability can tie where
 * two logits differ by less than its rounding).  Ties between equal logits go
 * to the lower index.  Returns 0, -1 for a bad shape, -2 if out of memory. */
int orc_router(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *ids, float *w)
{
    if (E < 1 || k < 1 || k > E) return -1;
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    uint8_t *taken = (uint8_t *)malloc((size_t)E);
    if (!p || !taken) {
        free(p);
        free(taken);
        return -2;
    }
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        double lmax = l[0];
        for (int32_t e = 1; e < E; ++e)
            if (l[e] > lmax) lmax = l[e];
        double z = 0.0;
        for (int32_t e = 0; e < E; ++e) {
            p[e] = exp((double)l[e] - lmax);
            z += p[e];
        }
        for (int32_t e = 0; e < E; ++e) p[e] /= z;
        memset(taken, 0, (size_t)E);
        double zk = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
            taken[best] = 1;
            ids[t * k + j] = best;
            zk += p[best];
        }
        for (int32_t j = 0; j < k; ++j) w[t * k + j] = (float)(p[ids[t * k + j]] / zk);
    }
    free(p);
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Block-scaled FP4 GEMM, exact                                               */
/* ------------------------------------------------------------------------ */

/* Dequantised values as integers: every E2M1 value is c/2 (|c| <= 12) and
 * every E4M3 value is m * 2^-9 (|m| <= 229376), so code value * scale value
 * * 2^10 is an integer. */
static int32_t deq_int(uint8_t code, uint8_t sfb)
{
    double v = orc_e2m1_value(code) * 2.0 * orc_e4m3_value(sfb) * 512.0;
    return (int32_t)llround(v);
}

typedef struct {
    const uint8_t *aq, *asf;
    const float *ga;
    const int32_t *wint; /* [N, K] */
    float gw;
    int64_t N, K;
    double *y;
} gemm_ctx;

static void gemm_range(int64_t lo, int64_t hi, void *p)
{
    gemm_ctx *c = (gemm_ctx *)p;
    int64_t K = c->K;
    int32_t *arow = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
    if (!arow) return;
    for (int64_t m = lo; m < hi; ++m) {
        for (int64_t kk = 0; kk < K; ++kk) {
            uint8_t byte = c->aq[m * (K / 2) + kk / 2];
            uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 15);
            arow[kk] = deq_int(code, c->asf[m * (K / 16) + kk / 16]);
        }
        double alpha = 1.0 / ((double)c->ga[m] * (double)c->gw);
        for (int64_t n = 0; n < c->N; ++n) {
            const int32_t *wr = c->wint + n * K;
            int64_t acc = 0;
            for (int64_t kk = 0; kk < K; ++kk) acc += (int64_t)arow[kk] * (int64_t)wr[kk];
            c->y[m * c->N + n] = (double)acc * 0x1p-20 * alpha;
        }
    }
    free(arow);
}

typedef struct {
    const uint8_t *wq, *wsf;
    int64_t K;
    int32_t *wint;
} deq_ctx;

static void deq_range(int64_t lo, int64_t hi, void *p)
{
    deq_ctx *c = (deq_ctx *)p;
    int64_t K = c->K;
    for (int64_t n = lo; n < hi; ++n)
        for (int64_t kk = 0; kk < K; ++kk) {
            uint8_t byte = c->wq[n * (K / 2) + kk / 2];
            uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 15);
            c->wint[n * K + kk] = deq_int(code, c->wsf[n * (K / 16) + kk / 16]);
        }
}

/* y[M, N] = dequant(A) . dequant(W)^T, both operands NVFP4 with K-major rows.
 * [page, §NVFP4, runtime-order figure, last two steps]: the FP4 data and FP8
 * block scales enter the GEMM, and the GEMM's output scaling folds in the FP32
 * activation and weight global scales.  Dequantised A = code * s / g_a and
 * dequantised W = code * s / g_w (the inverse of the quantisation map), so
 *     y = (sum_k qa*sa*qw*sw) / (g_a * g_w).
 * The sum is accumulated exactly in int64 (each product is an integer multiple
 * of 2^-20 below 2^43; K <= 2^12 terms stay below 2^55); the only rounding is
 * the final conversion and the multiply by 1/(g_a*g_w) in fp64.
 * ga[M] is the global scale of each A row; gw the one of W. */
int orc_gemm_nvfp4(const uint8_t *aq, const uint8_t *asf, const float *ga, int64_t M,
                   const uint8_t *wq, const uint8_t *wsf, float gw, int64_t N, int64_t K, double *y,
                   int nthreads)
{
    if (K % 16 != 0) return -1;
    int32_t *wint = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N * K > 0 ? N * K : 1));
    if (!wint) return -2;
    deq_ctx dc = {wq, wsf, K, wint};
    parallel_for(N, nthreads, deq_range, &dc);
    gemm_ctx gc = {aq, asf, ga, wint, gw, N, K, y};
    parallel_for(M, nthreads, gemm_range, &gc);
    free(wint);
    return 0;
}

/* y[M, N] = dequant(A) . dequant(W)^T with UE8M0 block scales on both
 * operands [page, MoE section: the expert quantiser's UE8M0_SF flag].
 * Reading: the variant keeps the GEMM above, y = (sum_k qa*sa*qw*sw) /
 * (g_a * g_w), with every block scale s = 2^(byte - 127).  A term
 * code * 2^e is exact in fp64 (an E2M1 value has two significant bits and
 * e lies in [-127, 127]), so is each product of two terms; the sum runs in
 * fp64 in k order, and the result takes one multiply by 1/(g_a * g_w). */
typedef struct {
    const uint8_t *aq, *asf;
    const float *ga;
    const double *wd; /* [N, K] dequantised weights, code * scale */
    float gw;
    int64_t N, K;
    double *y;
} gemm_ue_ctx;

static double deq_ue8m0(uint8_t code, uint8_t sfb) { return orc_e2m1_value(code) * orc_ue8m0_value(sfb); }

static void gemm_ue_range(int64_t lo, int64_t hi, void *p)
{
    gemm_ue_ctx *c = (gemm_ue_ctx *)p;
    int64_t K = c->K;
    double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!arow) return;
    for (int64_t m = lo; m < hi; ++m) {
        for (int64_t kk = 0; kk < K; ++kk) {
            uint8_t byte = c->aq[m * (K / 2) + kk / 2];
            uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 15);
            arow[kk] = deq_ue8m0(code, c->asf[m * (K / 16) + kk / 16]);
        }
        double alpha = 1.0 / ((double)c->ga[m] * (double)c->gw);
        for (int64_t n = 0; n < c->N; ++n) {
            const double *wr = c->wd + n * K;
            double acc = 0.0;
            for (int64_t kk = 0; kk < K; ++kk) acc += arow[kk] * wr[kk];
            c->y[m * c->N + n] = acc * alpha;
        }
    }
    free(arow);
}

typedef struct {
    const uint8_t *wq, *wsf;
    int64_t K;
    double *wd;
} deq_ue_ctx;

static void deq_ue_range(int64_t lo, int64_t hi, void *p)
{
    deq_ue_ctx *c = (deq_ue_ctx *)p;
    int64_t K = c->K;
    for (int64_t n = lo; n < hi; ++n)
        for (int64_t kk = 0; kk < K; ++kk) {
            uint8_t byte = c->wq[n * (K / 2) + kk / 2];
            uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 15);
            c->wd[n * K + kk] = deq_ue8m0(code, c->wsf[n * (K / 16) + kk / 16]);
        }
}

int orc_gemm_nvfp4_ue8m0(const uint8_t *aq, const uint8_t *asf, const float *ga, int64_t M, const uint8_t *wq,
                         const uint8_t *wsf, float gw, int64_t N, int64_t K, double *y, int nthreads)
{
    if (K % 16 != 0) return -1;
    double *wd = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!wd) return -2;
    deq_ue_ctx dc = {wq, wsf, K, wd};
    parallel_for(N, nthreads, deq_ue_range, &dc);
    gemm_ue_ctx gc = {aq, asf, ga, wd, gw, N, K, y};
    parallel_for(M, nthreads, gemm_ue_range, &gc);
    free(wd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Gated activation                                                           */
/* ------------------------------------------------------------------------ */

/* [page, §矩阵融合 "Gated FFN"]: gate and up share the input and are computed
 * by one fused GEMM (w13); the activation is act(gate) * up, with act = SiLU
 * for this FFN.  Reading: the fused output holds the I gate columns first and
 * the I up columns after them; the activation is evaluated in fp64 from the
 * fp64 GEMM output, silu(z) = z / (1 + exp(-z)), and the result is rounded to
 * FP32 (the intermediate that the second quantisation consumes).
 * y1 [M, 2I] -> h [M, I]. */
void orc_silu_mul(const double *y1, int64_t M, int64_t I, float *h)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < I; ++i) {
            double gate = y1[m * 2 * I + i];
            double up = y1[m * 2 * I + I + i];
            double silu = gate / (1.0 + exp(-gate));
            h[m * I + i] = (float)(silu * up);
        }
}

/* ------------------------------------------------------------------------ */
/* Residual + RMSNorm between stacked layers                                  */
/* ------------------------------------------------------------------------ */

/* Nearest BF16 (8 significant bits) to a double, ties to even; finite normal
 * range only (the normalised activations here are O(1)). */
static uint16_t bf16_nearest(double d)
{
    if (d == 0.0) return signbit(d) ? 0x8000 : 0x0000;
    int e;
    double m = frexp(fabs(d), &e);      /* |d| = m * 2^e, m in [0.5, 1) */
    double scaled = ldexp(m, 8);        /* in [128, 256): 8 significant bits */
    double lo = floor(scaled), frac = scaled - lo;
    double pick = lo;
    if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0)) pick = lo + 1.0;
    float f = (float)ldexp(pick, e - 8); /* exact: 9 bits at most */
    if (d < 0) f = -f;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* W4A16 activation step [page, backend figure: the MARLIN path executes the
 * checkpoint as W4A16, so the activations stay 16-bit].  Reading: the
 * intermediate h = SiLU(gate) * up is formed from the fp64 gate/up of the
 * first GEMM and rounded once to BF16, the second GEMM's input.  y1 is
 * [M, 2I] (gate columns then up columns); h [M, I] BF16 bits. */
void orc_silu_mul_bf16(const double *y1, int64_t M, int64_t I, uint16_t *h)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < I; ++i) {
            double gate = y1[m * 2 * I + i];
            double up = y1[m * 2 * I + I + i];
            double silu = gate / (1.0 + exp(-gate));
            h[m * I + i] = bf16_nearest(silu * up);
        }
}

/* Between stacked layers (not on the page; the stacked-layer workload adds it):
 *   r = x + out,  x' = bf16( r / sqrt(mean(r^2) + eps) ),  gamma = 1,
 * in fp64.  x is BF16 bits [T, H], out is FP32 [T, H]. */
void orc_residual_rmsnorm(const uint16_t *x, const float *out, int64_t T, int64_t H, double eps,
                          uint16_t *xn)
{
    double *r = (double *)malloc(sizeof(double) * (size_t)H);
    if (!r) return;
    for (int64_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int64_t i = 0; i < H; ++i) {
            uint32_t u = (uint32_t)x[t * H + i] << 16;
            float xf;
            memcpy(&xf, &u, 4);
            r[i] = (double)xf + (double)out[t * H + i];
            ss += r[i] * r[i];
        }
        double inv = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t i = 0; i < H; ++i) xn[t * H + i] = bf16_nearest(r[i] * inv);
    }
    free(r);
}
