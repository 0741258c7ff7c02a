/*
 * oracle.c - plain CPU oracle of the Engram per-layer forward step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): loaded by the tests, the smoke
 * check and the benchmark's CPU-baseline leg, never by the product.  Slow on
 * purpose: every step is the definition written out, in fp64 wherever the
 * method computes in floating point, with no blocking, fusion or reordering.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32->64 bit     */
/* multiplies with a Weyl-sequence key schedule.                            */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += weyl0;
            k1 += weyl1;
        }
        uint64_t p0 = (uint64_t)mul0 * x0;
        uint64_t p1 = (uint64_t)mul1 * x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* 16-bit lane `lane` (0..7) of the Philox output for a counter. */
static uint32_t philox_lane16(uint64_t seed, const uint32_t ctr[4], uint32_t lane)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return (out[lane / 2] >> (16 * (lane % 2))) & 0xFFFFu;
}

/* ------------------------------------------------------------------------ */
/* Table contents (build convention; the pages fix only that the table is   */
/* MXFP8: E4M3 codes with one E8M0 scale per 32 values, P1 "第二步").        */
/* Data: counter (row_lo, row_hi, col/8, 0), lane col%8, code uniform over  */
/* the 254 finite E4M3 codes (0x7F and 0xFF are never produced).            */
/* Scale: counter (row_lo, row_hi, 0, 1), lane = group, E8M0 exponent       */
/* uniform over 119..127, i.e. scales 2^-8 .. 2^0.                          */
/* ------------------------------------------------------------------------ */
uint8_t orc_table_code(uint64_t seed, uint64_t row, uint32_t col)
{
    uint32_t ctr[4] = {(uint32_t)row, (uint32_t)(row >> 32), col / 8u, 0u};
    uint32_t r = philox_lane16(seed, ctr, col % 8u);
    uint32_t idx = (r * 254u) >> 16; /* 0 .. 253 */
    return (uint8_t)(idx < 127u ? idx : idx + 1u);
}

uint8_t orc_table_scale(uint64_t seed, uint64_t row, uint32_t group)
{
    uint32_t ctr[4] = {(uint32_t)row, (uint32_t)(row >> 32), 0u, 1u};
    uint32_t r = philox_lane16(seed, ctr, group);
    return (uint8_t)(119u + ((r * 9u) >> 16));
}

void orc_table_row(uint64_t seed, uint64_t row, uint32_t row_dim, uint8_t* codes, uint8_t* scales)
{
    for (uint32_t c = 0; c < row_dim; ++c) codes[c] = orc_table_code(seed, row, c);
    for (uint32_t g = 0; g < row_dim / 32u; ++g) scales[g] = orc_table_scale(seed, row, g);
}

/* ------------------------------------------------------------------------ */
/* OCP MX element formats.                                                   */
/* E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is     */
/* subnormal; S.1111.111 is NaN; no infinity; largest finite 448.           */
/* E8M0: 2^(e-127); 0xFF is NaN.                                             */
/* ------------------------------------------------------------------------ */
double orc_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double orc_e8m0_value(uint8_t e)
{
    if (e == 0xFF) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* Round a double to BF16 (8 significant bits, exponent range of fp32) with
 * one round-to-nearest-even step, and return the BF16 bit pattern. */
uint16_t orc_bf16_from_double(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
    if (x == 0.0) return sign;
    double a = fabs(x);
    int e;
    frexp(a, &e);            /* a in [2^(e-1), 2^e)                   */
    int q = e - 8;           /* quantum of 8 significant bits         */
    if (q < -133) q = -133;  /* BF16 subnormal quantum is 2^-133      */
    double r = ldexp(nearbyint(ldexp(a, -q)), q); /* ties to even     */
    const double bf16_max = ldexp(255.0, 120);    /* (2 - 2^-7) 2^127 */
    if (r > bf16_max) return (uint16_t)(sign | 0x7F80u);
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | ((bits >> 16) & 0x7FFFu));
}

double orc_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Primes (P4 "동작 방식": each (order, head) pair indexes its own           */
/* prime-sized bucket range; P2: engram_vocab_size 16,000,000 and the row   */
/* counts 384,006,168 / 384,016,682 are the sums of consecutive primes).    */
/* ------------------------------------------------------------------------ */
int orc_is_prime(uint64_t n)
{
    if (n < 2) return 0;
    if (n % 2 == 0) return n == 2;
    for (uint64_t d = 3; d * d <= n; d += 2)
        if (n % d == 0) return 0;
    return 1;
}

void orc_primes_above(uint64_t base, int count, uint64_t* out)
{
    uint64_t c = base;
    for (int i = 0; i < count; ++i) {
        do { ++c; } while (!orc_is_prime(c));
        out[i] = c;
    }
}

/* Multiplier j of a layer (build convention, see oracle.h): Philox keyed by
 * the layer seed, counter (j, 0, 0, 2); an odd value below
 * floor((2^64-1)/vc), so a product with any compressed id cannot wrap. */
static uint64_t orc_multiplier(uint64_t seed, uint32_t j, uint32_t vc)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {j, 0u, 0u, 2u};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint64_t r = (uint64_t)out[0] | ((uint64_t)out[1] << 32);
    uint64_t bound = UINT64_MAX / (uint64_t)vc;
    uint64_t half = bound / 2u;
    if (half == 0) half = 1;
    return 2u * (r % half) + 1u;
}

int orc_layer_params(const orc_geom* g, int nlayers, const uint64_t* seeds,
                     const uint64_t* bucket_bases, int layer,
                     uint64_t* mult, uint64_t* prime, uint64_t* offset, uint64_t* rows)
{
    if (g->min_n < 1 || g->max_n < g->min_n || g->max_n > 4 || g->heads < 1 || g->vc < 1)
        return -1;
    if (nlayers < 1 || layer < 0 || layer >= nlayers) return -1;
    int nb = (int)((g->max_n - g->min_n + 1) * g->heads);
    uint64_t* used = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)nb * (size_t)(layer + 1));
    if (!used) return -1;
    int nused = 0;
    for (int l = 0; l <= layer; ++l) {
        uint64_t c = bucket_bases[l];
        uint64_t sum = 0;
        for (int b = 0; b < nb; ++b) {
            for (;;) {
                ++c;
                if (!orc_is_prime(c)) continue;
                int taken = 0;
                for (int u = 0; u < nused; ++u)
                    if (used[u] == c) taken = 1;
                if (!taken) break;
            }
            used[nused++] = c;
            if (l == layer) {
                prime[b] = c;
                offset[b] = sum;
            }
            sum += c;
        }
        if (l == layer) {
            *rows = sum;
            for (int b = 0; b < nb; ++b)
                for (uint32_t j = 0; j < 4; ++j)
                    mult[b * 4 + (int)j] = j < g->max_n ? orc_multiplier(seeds[l], j, g->vc) : 0u;
        }
    }
    free(used);
    return *rows <= 0xFFFFFFFFull ? 0 : -2;
}

/* ------------------------------------------------------------------------ */
/* Windows (P1 "第一步" and "第四步"): position t sees its own compressed id  */
/* and those of the three most recent positions of the same history; slots  */
/* before the start of history hold pad_cid; image positions hold DEAD.     */
/* ------------------------------------------------------------------------ */
int orc_windows(const orc_geom* g, const uint32_t* token_map, const int32_t* tokens,
                const uint8_t* is_image, int64_t n, uint32_t* windows)
{
    for (int64_t t = 0; t < n; ++t)
        if (!is_image[t] && (tokens[t] < 0 || (uint32_t)tokens[t] >= g->vocab)) return -1;
    for (int64_t t = 0; t < n; ++t) {
        for (int64_t j = 0; j < 4; ++j) {
            int64_t p = t - j;
            uint32_t c;
            if (p < 0)
                c = g->pad_cid;
            else if (is_image[p])
                c = ORC_DEAD;
            else
                c = token_map[tokens[p]];
            windows[t * 4 + j] = c;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Hash (P1 "第一步", P4 "동작 방식"): for order n and head k the suffix      */
/* n-gram (c_t .. c_{t-n+1}) is mixed by multiplying each id by its         */
/* multiplier and XOR-ing the products (wrapping 64-bit arithmetic); the    */
/* row is the bucket offset plus the mix modulo the bucket's prime.  An     */
/* n-gram containing DEAD is masked for all of its heads.                   */
/* ------------------------------------------------------------------------ */
void orc_hash(const orc_geom* g, const uint64_t* mult, const uint64_t* prime,
              const uint64_t* offset, const uint32_t window[4], uint32_t* rows)
{
    for (uint32_t n = g->min_n; n <= g->max_n; ++n) {
        int masked = 0;
        for (uint32_t j = 0; j < n; ++j)
            if (window[j] == ORC_DEAD) masked = 1;
        for (uint32_t k = 0; k < g->heads; ++k) {
            uint32_t b = (n - g->min_n) * g->heads + k;
            if (masked) {
                rows[b] = ORC_MASKED;
                continue;
            }
            uint64_t x = 0;
            for (uint32_t j = 0; j < n; ++j) x ^= (uint64_t)window[j] * mult[b * 4 + j];
            rows[b] = (uint32_t)(offset[b] + x % prime[b]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Gather and dequantise (P1 "第二步", P2): value = E4M3(code) * 2^(E8M0-127) */
/* with one scale per 32 values, rounded to BF16; rows are concatenated in  */
/* bucket order (order-major, then head); a masked row contributes zeros.   */
/* ------------------------------------------------------------------------ */
void orc_gather(const orc_geom* g, uint64_t seed, const uint32_t* rows, uint16_t* e)
{
    uint32_t nb = (g->max_n - g->min_n + 1) * g->heads;
    for (uint32_t b = 0; b < nb; ++b) {
        for (uint32_t i = 0; i < g->row_dim; ++i) {
            uint16_t out = 0;
            if (rows[b] != ORC_MASKED) {
                double v = orc_e4m3_value(orc_table_code(seed, rows[b], i)) *
                           orc_e8m0_value(orc_table_scale(seed, rows[b], i / 32u));
                out = orc_bf16_from_double(v);
            }
            e[b * g->row_dim + i] = out;
        }
    }
}

/* The same gather from a table held in memory (codes [nrows][row_dim],
 * scales [nrows][row_dim/32]) rather than the generated contents.  Returns -1,
 * leaving e unspecified, if an unmasked row index is >= nrows (the pages define
 * no row outside the table). */
int orc_gather_table(const orc_geom* g, const uint8_t* codes, const uint8_t* scales,
                     uint64_t nrows, const uint32_t* rows, uint16_t* e)
{
    uint32_t nb = (g->max_n - g->min_n + 1) * g->heads;
    uint32_t groups = g->row_dim / 32u;
    for (uint32_t b = 0; b < nb; ++b) {
        if (rows[b] != ORC_MASKED && rows[b] >= nrows) return -1;
        for (uint32_t i = 0; i < g->row_dim; ++i) {
            uint16_t out = 0;
            if (rows[b] != ORC_MASKED) {
                uint64_t r = rows[b];
                double v = orc_e4m3_value(codes[r * g->row_dim + i]) *
                           orc_e8m0_value(scales[r * groups + i / 32u]);
                out = orc_bf16_from_double(v);
            }
            e[b * g->row_dim + i] = out;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* wkv projection (P1 "第二步"): kv = W e with W of shape [(hc+1) d][K].     */
/* ------------------------------------------------------------------------ */
void orc_project(const orc_geom* g, const uint16_t* w, const uint16_t* e, double* kv)
{
    uint64_t K = (uint64_t)(g->max_n - g->min_n + 1) * g->heads * g->row_dim;
    uint64_t N = (uint64_t)(g->hc + 1) * g->d;
    for (uint64_t o = 0; o < N; ++o) {
        double acc = 0.0;
        for (uint64_t i = 0; i < K; ++i) acc += orc_bf16_value(w[o * K + i]) * orc_bf16_value(e[i]);
        kv[o] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* Gate (P1 "第三步", P4 "동작 방식"): for branch b, key = kv[b d .. (b+1) d), */
/* value = the last d entries of kv.  Hidden and key are RMS-normalised     */
/* separately and weighted elementwise by the pre-multiplied q / k weights; */
/* dot = <n(h) w_q, n(k) w_k> / sqrt(d);                                    */
/* gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot));                   */
/* hidden += gate * value.  An image row passes through unchanged.          */
/* ------------------------------------------------------------------------ */
void orc_gate(const orc_geom* g, const double* kv, uint32_t c_t, const uint16_t* h_in,
              const float* wq, const float* wk, double* h_out, uint16_t* h_out_bf16, double* gates)
{
    uint32_t d = g->d;
    const double* v = kv + (uint64_t)g->hc * d;
    for (uint32_t b = 0; b < g->hc; ++b) {
        const uint16_t* h = h_in + (uint64_t)b * d;
        if (c_t == ORC_DEAD) {
            for (uint32_t i = 0; i < d; ++i) {
                if (h_out) h_out[(uint64_t)b * d + i] = orc_bf16_value(h[i]);
                h_out_bf16[(uint64_t)b * d + i] = h[i];
            }
            gates[b] = 0.0;
            continue;
        }
        const double* k = kv + (uint64_t)b * d;
        double sum_h2 = 0.0, sum_k2 = 0.0;
        for (uint32_t i = 0; i < d; ++i) {
            double hi = orc_bf16_value(h[i]);
            sum_h2 += hi * hi;
            sum_k2 += k[i] * k[i];
        }
        double rh = 1.0 / sqrt(sum_h2 / d + g->eps);
        double rk = 1.0 / sqrt(sum_k2 / d + g->eps);
        double dot = 0.0;
        for (uint32_t i = 0; i < d; ++i) {
            double nh = orc_bf16_value(h[i]) * rh * (double)wq[(uint64_t)b * d + i];
            double nk = k[i] * rk * (double)wk[(uint64_t)b * d + i];
            dot += nh * nk;
        }
        dot /= sqrt((double)d);
        double s = copysign(sqrt(fmax(fabs(dot), 1e-6)), dot);
        double gate = 1.0 / (1.0 + exp(-s));
        gates[b] = gate;
        for (uint32_t i = 0; i < d; ++i) {
            double out = orc_bf16_value(h[i]) + gate * v[i];
            if (h_out) h_out[(uint64_t)b * d + i] = out;
            h_out_bf16[(uint64_t)b * d + i] = orc_bf16_from_double(out);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* The whole step on sampled positions, threads over positions.             */
/* ------------------------------------------------------------------------ */
typedef struct fwd_job {
    const orc_geom* g;
    uint64_t seed;
    const uint64_t *mult, *prime, *offset;
    const uint16_t* w;
    const float *wq, *wk;
    const uint32_t* windows;
    const uint16_t* hidden;
    const int64_t* idx;
    const uint8_t *codes, *scales; /* explicit table, or NULL: generated contents */
    uint64_t nrows;
    int64_t begin, end;
    uint32_t* rows_out;
    uint16_t* e_out;
    double* kv_out;
    double* gates_out;
    double* h_out;
    uint16_t* h_bf16_out;
    int status;
} fwd_job;

static void* fwd_worker(void* arg)
{
    fwd_job* j = (fwd_job*)arg;
    const orc_geom* g = j->g;
    uint64_t nb = (uint64_t)(g->max_n - g->min_n + 1) * g->heads;
    uint64_t K = nb * g->row_dim;
    uint64_t N = (uint64_t)(g->hc + 1) * g->d;
    uint64_t HD = (uint64_t)g->hc * g->d;
    uint16_t* e = (uint16_t*)malloc(sizeof(uint16_t) * K);
    double* kv = (double*)malloc(sizeof(double) * N);
    if (!e || !kv) {
        free(e);
        free(kv);
        j->status = -1;
        return NULL;
    }
    for (int64_t s = j->begin; s < j->end; ++s) {
        int64_t t = j->idx[s];
        const uint32_t* win = j->windows + t * 4;
        uint32_t* rows = j->rows_out + (uint64_t)s * nb;
        orc_hash(g, j->mult, j->prime, j->offset, win, rows);
        if (!j->codes)
            orc_gather(g, j->seed, rows, e);
        else if (orc_gather_table(g, j->codes, j->scales, j->nrows, rows, e) != 0) {
            free(e);
            free(kv);
            j->status = -1;
            return NULL;
        }
        orc_project(g, j->w, e, kv);
        orc_gate(g, kv, win[0], j->hidden + (uint64_t)t * HD, j->wq, j->wk,
                 j->h_out ? j->h_out + (uint64_t)s * HD : NULL, j->h_bf16_out + (uint64_t)s * HD,
                 j->gates_out + (uint64_t)s * g->hc);
        if (j->e_out) memcpy(j->e_out + (uint64_t)s * K, e, sizeof(uint16_t) * K);
        if (j->kv_out) memcpy(j->kv_out + (uint64_t)s * N, kv, sizeof(double) * N);
    }
    free(e);
    free(kv);
    j->status = 0;
    return NULL;
}

static int forward_impl(const orc_geom* g, uint64_t seed, const uint8_t* codes,
                        const uint8_t* scales, uint64_t nrows, const uint64_t* mult,
                        const uint64_t* prime, const uint64_t* offset, const uint16_t* w,
                        const float* wq, const float* wk, const uint32_t* windows,
                        const uint16_t* hidden, const int64_t* idx, int64_t nidx, int nthreads,
                        uint32_t* rows_out, uint16_t* e_out, double* kv_out, double* gates_out,
                        double* h_out, uint16_t* h_bf16_out)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nidx) nthreads = nidx > 0 ? (int)nidx : 1;
    fwd_job* jobs = (fwd_job*)calloc((size_t)nthreads, sizeof(fwd_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int i = 0; i < nthreads; ++i) {
        fwd_job* j = &jobs[i];
        j->g = g; j->seed = seed; j->mult = mult; j->prime = prime; j->offset = offset;
        j->w = w; j->wq = wq; j->wk = wk; j->windows = windows; j->hidden = hidden;
        j->idx = idx;
        j->codes = codes; j->scales = scales; j->nrows = nrows;
        j->begin = nidx * i / nthreads;
        j->end = nidx * (i + 1) / nthreads;
        j->rows_out = rows_out; j->e_out = e_out; j->kv_out = kv_out;
        j->gates_out = gates_out; j->h_out = h_out; j->h_bf16_out = h_bf16_out;
        j->status = -1;
    }
    int rc = 0;
    int* created = (int*)calloc((size_t)nthreads, sizeof(int));
    if (!created) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int i = 1; i < nthreads; ++i)
        created[i] = pthread_create(&th[i], NULL, fwd_worker, &jobs[i]) == 0;
    fwd_worker(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) {
        if (created[i])
            pthread_join(th[i], NULL);
        else
            fwd_worker(&jobs[i]);
    }
    free(created);
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].status != 0) rc = -1;
    free(jobs);
    free(th);
    return rc;
}

int orc_forward(const orc_geom* g, uint64_t seed, const uint64_t* mult, const uint64_t* prime,
                const uint64_t* offset, const uint16_t* w, const float* wq, const float* wk,
                const uint32_t* windows, const uint16_t* hidden, const int64_t* idx, int64_t nidx,
                int nthreads, uint32_t* rows_out, uint16_t* e_out, double* kv_out,
                double* gates_out, double* h_out, uint16_t* h_bf16_out)
{
    return forward_impl(g, seed, NULL, NULL, 0, mult, prime, offset, w, wq, wk, windows, hidden,
                        idx, nidx, nthreads, rows_out, e_out, kv_out, gates_out, h_out,
                        h_bf16_out);
}

int orc_forward_table(const orc_geom* g, const uint8_t* codes, const uint8_t* scales,
                      uint64_t nrows, const uint64_t* mult, const uint64_t* prime,
                      const uint64_t* offset, const uint16_t* w, const float* wq, const float* wk,
                      const uint32_t* windows, const uint16_t* hidden, const int64_t* idx,
                      int64_t nidx, int nthreads, uint32_t* rows_out, uint16_t* e_out,
                      double* kv_out, double* gates_out, double* h_out, uint16_t* h_bf16_out)
{
    return forward_impl(g, 0, codes, scales, nrows, mult, prime, offset, w, wq, wk, windows,
                        hidden, idx, nidx, nthreads, rows_out, e_out, kv_out, gates_out, h_out,
                        h_bf16_out);
}
