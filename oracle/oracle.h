/*
 * oracle.h - plain CPU oracle of the Engram per-layer forward step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The product (libengram.so
 * and its Python binding) never links, loads or calls it, and the two share no
 * code, header, table or helper.  Everything here is written from the pages'
 * statement of the method, in the order the pages give it, with fp64
 * arithmetic wherever the method computes in floating point.
 *
 * Sources, by page title and section:
 *  [P1] "DeepSeek V4.1 Flash 的 Engram" (zhuai.tech): sections
 *       "把知识变成可寻址的向量" (geometry: 2/3/4-gram x 8 heads x 256 = 6,144),
 *       "第一步" (token -> compressed id -> current token and the three most
 *       recent positions -> 24 hashes -> 24 row numbers),
 *       "第二步" (MXFP8 rows: E4M3 data + one E8M0 scale per 32 values; wkv
 *       25,600 x 6,144 BF16), "第三步" (the gate formula), "第四步" (history
 *       appended once per token; fork/reset; DEAD markers for image spans).
 *  [P2] "3.84 亿行 Embedding 的存法大揭秘" (lqnn.cn): per-layer row counts
 *       384,006,168 / 384,016,682, engram_vocab_size 16,000,000, the value
 *       is the last 5,120 rows of wkv.
 *  [P3] FlagScale Engram plugin article, section 5: engram_pad_id = 0,
 *       engram_seed.
 *  [P4] vLLM "Engram" feature wiki, section "동작 방식 (How it works)":
 *       per (order, head) multiply-XOR hash into its own prime-sized bucket
 *       range; one key per hyper-connection branch and one shared value;
 *       sigmoid gate on the normalised dot; masked positions pass through.
 *
 * Readings taken where the pages are silent, each with the passage it rests on:
 *  - primes [P4 "동작 방식", P2 row counts]: strictly increasing primes >
 *    bucket_base, bucket order b = (n - min_n) * heads + head, layers in
 *    order, no prime reused by a later layer; offsets are prefix sums of the
 *    primes.  With bucket_base 16,000,000 this gives the row counts P2 prints.
 *  - multipliers [P4 "동작 방식", P1 "第一步"]: a build convention
 *    (Philox4x32-10 keyed by the layer seed, one odd multiplier per n-gram
 *    position shared by all buckets of the layer, bounded so that no product
 *    with a compressed id wraps).  PARITY UNPINNED against the real model:
 *    the pages print no multiplier.  orc_hash itself takes a general table
 *    and is pinned to hand-worked values (tests/golden/hash_worked.txt).
 *  - table contents [P1 "第二步"]: a build convention, a Philox4x32-10
 *    function of (seed, row, column).  PARITY UNPINNED against the real model
 *    (no row is printed); pinned to the published Philox known-answer vectors.
 *  - history before the first token holds pad_cid [P3: engram_pad_id = 0].
 *  - an n-gram containing DEAD yields a masked (all-zero) row for each of its
 *    heads; a row whose own token is DEAD (an image row) is not gated
 *    [P1 "第四步", P4 "동작 방식"].
 *  - RMS-norm epsilon = 1e-6, inside the square root [P1 "第三步" prints no
 *    epsilon; 1e-6 is the gate's own floor constant].
 */
#ifndef ENGRAM_ORACLE_H
#define ENGRAM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_DEAD   0xFFFFFFFFu /* compressed-id marker of an image position */
#define ORC_MASKED 0xFFFFFFFFu /* row index of a masked (n-gram, head)      */

typedef struct orc_geom {
    uint32_t vocab;    /* tokenizer vocabulary V                       */
    uint32_t vc;       /* compressed vocabulary size                   */
    uint32_t min_n;    /* smallest n-gram order (2)                    */
    uint32_t max_n;    /* largest n-gram order (4), at most 4          */
    uint32_t heads;    /* hash heads per order (8)                     */
    uint32_t row_dim;  /* values per table row (256)                   */
    uint32_t hc;       /* hyper-connection branches (4)                */
    uint32_t d;        /* hidden size per branch (5,120)               */
    uint32_t pad_cid;  /* compressed id before the start of history    */
    uint32_t reserved;
    double eps;        /* RMS-norm epsilon                             */
} orc_geom;

/* Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Table contents of a layer with the given seed (build convention). */
uint8_t orc_table_code(uint64_t seed, uint64_t row, uint32_t col);
uint8_t orc_table_scale(uint64_t seed, uint64_t row, uint32_t group);
void    orc_table_row(uint64_t seed, uint64_t row, uint32_t row_dim,
                      uint8_t* codes /*[row_dim]*/, uint8_t* scales /*[row_dim/32]*/);

/* OCP MX element decodes and BF16 round-to-nearest-even. */
double   orc_e4m3_value(uint8_t code);
double   orc_e8m0_value(uint8_t e);
uint16_t orc_bf16_from_double(double x);
double   orc_bf16_value(uint16_t bits);

/* Primality by trial division and the primes strictly above a base. */
int  orc_is_prime(uint64_t n);
void orc_primes_above(uint64_t base, int count, uint64_t* out);

/* Hash parameters of layer `layer` of a model whose layers have the given
 * seeds and bucket bases (layers are assigned primes in order).
 * mult [nb][4], prime [nb], offset [nb]; *rows = sum of the primes. */
int orc_layer_params(const orc_geom* g, int nlayers, const uint64_t* seeds,
                     const uint64_t* bucket_bases, int layer,
                     uint64_t* mult, uint64_t* prime, uint64_t* offset, uint64_t* rows);

/* Windows (c_t, c_{t-1}, c_{t-2}, c_{t-3}) of a token sequence appended to an
 * empty history.  Returns 0, or -1 if a token is outside [0, vocab). */
int orc_windows(const orc_geom* g, const uint32_t* token_map, const int32_t* tokens,
                const uint8_t* is_image, int64_t n, uint32_t* windows /*[n][4]*/);

/* The 24 (in general nb) row indices of one window. */
void orc_hash(const orc_geom* g, const uint64_t* mult, const uint64_t* prime,
              const uint64_t* offset, const uint32_t window[4], uint32_t* rows /*[nb]*/);

/* The concatenated dequantised vector (BF16 bits) of one token's rows. */
void orc_gather(const orc_geom* g, uint64_t seed, const uint32_t* rows /*[nb]*/,
                uint16_t* e /*[K]*/);

/* The same from a table held in memory: codes [nrows][row_dim] (E4M3),
 * scales [nrows][row_dim/32] (E8M0).  Returns -1 if an unmasked index is
 * >= nrows, else 0. */
int orc_gather_table(const orc_geom* g, const uint8_t* codes, const uint8_t* scales,
                     uint64_t nrows, const uint32_t* rows /*[nb]*/, uint16_t* e /*[K]*/);

/* kv[o] = sum_i W[o][i] * e[i] in fp64.  W is BF16 [N][K]. */
void orc_project(const orc_geom* g, const uint16_t* w /*[N][K]*/, const uint16_t* e /*[K]*/,
                 double* kv /*[N]*/);

/* Gate of one token: h_in BF16 [hc][d], wq/wk fp32 [hc][d]. Outputs the fp64
 * updated hidden, its BF16 rounding and the hc gates (0 for an image row). */
void orc_gate(const orc_geom* g, const double* kv, uint32_t c_t, const uint16_t* h_in,
              const float* wq, const float* wk, double* h_out /*[hc][d] or NULL*/,
              uint16_t* h_out_bf16 /*[hc][d]*/, double* gates /*[hc]*/);

/* Full step on a list of token positions, split over `nthreads` threads.
 * Per sampled position i (token idx[i]):
 *   rows_out [i][nb], e_out [i][K] (or NULL), kv_out [i][N] (or NULL),
 *   gates_out [i][hc], h_out [i][hc][d] (or NULL), h_bf16_out [i][hc][d]. */
int orc_forward(const orc_geom* g, uint64_t seed, const uint64_t* mult,
                const uint64_t* prime, const uint64_t* offset, const uint16_t* w,
                const float* wq, const float* wk, const uint32_t* windows,
                const uint16_t* hidden, const int64_t* idx, int64_t nidx, int nthreads,
                uint32_t* rows_out, uint16_t* e_out, double* kv_out, double* gates_out,
                double* h_out, uint16_t* h_bf16_out);

/* orc_forward with the rows read from a table held in memory (as
 * orc_gather_table) instead of the generated contents.  Returns -1 if a row
 * index falls outside the table. */
int orc_forward_table(const orc_geom* g, const uint8_t* codes, const uint8_t* scales,
                      uint64_t nrows, const uint64_t* mult, const uint64_t* prime,
                      const uint64_t* offset, const uint16_t* w, const float* wq,
                      const float* wk, const uint32_t* windows, const uint16_t* hidden,
                      const int64_t* idx, int64_t nidx, int nthreads, uint32_t* rows_out,
                      uint16_t* e_out, double* kv_out, double* gates_out, double* h_out,
                      uint16_t* h_bf16_out);

#ifdef __cplusplus
}
#endif
#endif
