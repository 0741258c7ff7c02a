/*
 * engram.h - C ABI of the Engram per-layer forward step on one GB300 GPU.
 *
 * The Engram layer (conditional memory of DeepSeek V4.1 Flash) injects, at the
 * entry of layers 1 and 14, a gated value read from a huge n-gram table:
 *
 *   tokens --append--> windows (c_t, c_{t-1}, c_{t-2}, c_{t-3})
 *          --hash----> 24 row numbers (2/3/4-gram x 8 heads, each head its own
 *                      prime-sized bucket range of the layer table)
 *          --gather--> 24 MXFP8 rows of 256 values (E4M3 + one E8M0 per 32),
 *                      dequantised to BF16 and concatenated: a 6,144-vector
 *          --project-> kv = wkv e, wkv BF16 [25,600 x 6,144]: one 5,120-wide
 *                      key per hyper-connection branch and one shared value
 *          --gate----> per branch: hidden += sigmoid(copysign(sqrt(max(|dot|,
 *                      1e-6)), dot)) * value, dot = <n(h) w_q, n(k) w_k>/sqrt(d)
 *
 * Sources (page title, section):
 *   "DeepSeek V4.1 Flash 的 Engram" (zhuai.tech): "把知识变成可寻址的向量"
 *     (geometry), "第一步" (token map, windows, 24 hashes), "第二步" (MXFP8
 *     rows, wkv), "第三步" (gate), "第四步" (append once; fork/reset; DEAD).
 *   "3.84 亿行 Embedding 的存法大揭秘" (lqnn.cn): row counts, group-32 UE8M0
 *     scales, the value is the last 5,120 rows of wkv.
 *   vLLM "Engram" feature wiki, "동작 방식 (How it works)": multiply-XOR hash
 *     per (order, head) into its own prime bucket range; one key per branch
 *     and a shared value; masked positions pass through.
 *
 * Conventions for every call:
 *  - Every call returns an engram_status.  Arguments are validated before any
 *    launch; on an error nothing is launched and no state changes.
 *    engram_last_error() returns a thread-local message for the last error.
 *  - The caller owns every device and pinned-host buffer and every stream and
 *    the library never frees them.  The library owns engram_ctx, the sessions,
 *    the per-layer hash parameters, a 16-byte device word per context (error
 *    word and bind-time scan results, allocated at the first
 *    engram_layer_bind), per bound layer the elementwise product of w_q and
 *    w_k (hc x d x 4 bytes) and, on the FP16 operand path, an FP16 copy of
 *    wkv (N x K x 2 bytes), allocated by engram_layer_bind and freed by a
 *    rebind (the FP16 copy) or engram_ctx_destroy.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Device calls are asynchronous on that stream.  Faults found by a kernel
 *    (a row index outside the table, a wait that ran out) set the context's
 *    device error word; engram_sync() synchronises the stream, reads and
 *    clears that word and reports it.  The library never aborts, traps or
 *    prints.
 *  - BF16 values are passed as uint16_t bit patterns.
 *  - Layout of the per-layer tensors (T tokens, nb = (max_n-min_n+1) * heads
 *    buckets, K = nb * row_dim, N = (hc + 1) * d):
 *      windows   uint32 [T][4]         (c_t, c_{t-1}, c_{t-2}, c_{t-3})
 *      rows      uint32 [T][nb]        bucket b = (n - min_n) * heads + head
 *      emb       bf16   [T][K]         bucket-major concatenation
 *      kv        fp32   [T][N]         rows [b d, (b+1) d) key b; last d: value
 *      hidden    bf16   [T][hc][d]     updated in place
 *      gates     fp32   [T][hc]        0 for an image row
 *      table     uint8  [rows][row_dim]       E4M3 codes
 *      scales    uint8  [rows][row_dim / 32]  E8M0 exponents
 *      wkv       bf16   [N][K]         row-major
 *      wq, wk    fp32   [hc][d]        pre-multiplied norm weights
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENGRAM_DEAD   0xFFFFFFFFu /* compressed id of an image position (window slot) */
#define ENGRAM_MASKED 0xFFFFFFFFu /* row index of an n-gram that touches DEAD          */

typedef enum engram_status {
    ENGRAM_OK = 0,
    ENGRAM_EINVAL = 1,      /* bad argument: null pointer, size, layer, token, alignment   */
    ENGRAM_ENOMEM = 2,      /* host or device allocation failed                            */
    ENGRAM_ECUDA = 3,       /* a CUDA runtime call failed (launch or asynchronous error)   */
    ENGRAM_ESTATE = 4,      /* object in the wrong state (layer not bound, bad session)    */
    ENGRAM_ETIMEOUT = 5,    /* a kernel gave up a bounded wait and returned                */
    ENGRAM_EUNSUPPORTED = 6,/* geometry or device the kernels do not support               */
    ENGRAM_EBOUNDS = 7      /* a kernel met a row index outside the table (row zero-filled)*/
} engram_status;

typedef struct engram_ctx engram_ctx;
typedef struct engram_session engram_session;

/* Model geometry and per-layer hash configuration.
 * Source: "把知识变成可寻址的向量" (2/3/4-gram, 8 heads, 256 values per row),
 * "第一步" (129,280-entry token map; multipliers, primes, bucket offsets
 * expanded per layer), FlagScale config fields engram_pad_id / engram_seed. */
typedef struct engram_ctx_desc {
    uint32_t vocab;                /* tokenizer vocabulary V (129,280)                 */
    uint32_t vc;                   /* compressed vocabulary size (every map value < vc) */
    uint32_t min_n;                /* smallest n-gram order (2), >= 1                  */
    uint32_t max_n;                /* largest n-gram order (4), <= 4                   */
    uint32_t heads;                /* hash heads per order (8), 1..8                   */
    uint32_t row_dim;              /* values per row: 32, 64, 128 or 256               */
    uint32_t hc;                   /* hyper-connection branches (4), 1..8              */
    uint32_t d;                    /* hidden size per branch (5,120)                   */
    uint32_t pad_cid;              /* compressed id before the start of history, < vc  */
    uint32_t n_layers;             /* Engram layers of the model, 1..16                */
    double eps;                    /* RMS-norm epsilon (1e-6)                          */
    const uint64_t* layer_seeds;   /* [n_layers] hash seed of each layer               */
    const uint64_t* bucket_bases;  /* [n_layers] primes of a layer are > its base      */
} engram_ctx_desc;

/* Weights of one layer.  table/scales: device memory, or pinned host memory
 * mapped into the device address space (read through UVA, vLLM "CPU 오프로드").
 * The scale array must be readable up to its size rounded up to 16 bytes.
 * wkv must be 16-byte aligned.  The table's contents are scanned at bind
 * (the E8M0 exponent range, see engram_layer_info): bind again after
 * rewriting a table. */
#define ENGRAM_BIND_BF16_OPERANDS 1u /* flags: fused kernels decode to BF16 only */
/* flags: the table holds BF16 rows [rows][row_dim] (2 x row_dim bytes each,
 * the already dequantised values) and no scales (scales may be NULL): the
 * second storage format of the pages ([zhuai], the w8a8 repository's BF16
 * table).  The gathers copy the rows; the operands are BF16.  Such a layer
 * runs through engram_gather_dequant, engram_forward_staged and its two
 * steps; engram_forward, engram_forward_noalloc and engram_project_windows,
 * whose kernels decode MXFP8 rows while they gather, return
 * ENGRAM_EUNSUPPORTED. */
#define ENGRAM_BIND_TABLE_BF16 2u
typedef struct engram_layer_weights {
    const uint8_t* table;   /* [rows][row_dim] E4M3 codes (BF16 table: bf16 [rows][row_dim]) */
    const uint8_t* scales;  /* [rows][row_dim / 32] E8M0 exponents (BF16 table: unused) */
    uint64_t rows;          /* must equal the layer's row count (engram_layer_params) */
    const uint16_t* wkv;    /* bf16 [N][K], device                            */
    const float* wq;        /* fp32 [hc][d], device                           */
    const float* wk;        /* fp32 [hc][d], device                           */
    uint32_t flags;         /* 0, ENGRAM_BIND_BF16_OPERANDS, ENGRAM_BIND_TABLE_BF16 */
} engram_layer_weights;

/* How a bound layer runs.  The fused kernels feed the tensor cores FP16
 * operands that hold the BF16 values exactly (fp16_operands = 1) when the
 * table's E8M0 exponents span at most 23 values: each decoded value is the
 * exact product code x 2^(e - 127 + a_exp_shift), and wkv is held as an FP16
 * copy scaled by 2^wkv_exp (exact for every weight above 2^-28 of the largest;
 * smaller ones round to a multiple of 2^-(24 + wkv_exp)); the accumulator is
 * scaled back by 2^-(a_exp_shift + wkv_exp).  Otherwise (fp16_operands = 0)
 * they decode to BF16 through fp32 and multiply the caller's BF16 wkv. */
typedef struct engram_layer_info_t {
    uint64_t rows;
    int32_t bound;
    int32_t fp16_operands;
    uint32_t scale_min, scale_max;  /* E8M0 exponent range of the table       */
    int32_t wkv_exp;
    int32_t a_exp_shift;
    int32_t bucket_gather;          /* 1: each 256-wide table row is loaded whole,
                                       once per output tile (FP16 path, row_dim
                                       256); 0: 64-column slices per k-block     */
    int32_t table_bf16;             /* 1: bound with ENGRAM_BIND_TABLE_BF16        */
} engram_layer_info_t;
engram_status engram_layer_info(const engram_ctx* ctx, int layer, engram_layer_info_t* out);

/* Create a context.  token_map: host uint32 [vocab] compressed id of each
 * token (all < vc), copied.  No CUDA call is made. */
engram_status engram_ctx_create(const engram_ctx_desc* desc, const uint32_t* token_map,
                                engram_ctx** out);
engram_status engram_ctx_destroy(engram_ctx* ctx);

/* Hash parameters of a layer (host outputs, each may be NULL):
 * mult [nb][4] uint64 (the multiplier of window slot j for bucket b),
 * prime [nb], offset [nb] (prefix sums of the primes), rows = sum of primes.
 * Primes: strictly increasing primes above the layer's bucket base, no prime
 * reused by an earlier layer (vLLM wiki "동작 방식"; the row counts on the
 * lqnn.cn page are sums of such primes).  Multipliers: odd, below
 * floor((2^64-1)/vc), one per window slot shared by the layer's buckets,
 * drawn from Philox4x32-10 keyed by the layer seed. */
engram_status engram_layer_params(const engram_ctx* ctx, int layer, uint64_t* mult,
                                  uint64_t* prime, uint64_t* offset, uint64_t* rows);

/* Replace a layer's multiplier table with a general one (host [nb][4]),
 * e.g. independent multipliers per head.  Applies to later calls. */
engram_status engram_layer_set_multipliers(engram_ctx* ctx, int layer, const uint64_t* mult);

/* Bind a layer's weights (pointers are kept, not copied).  Needs a GPU: it
 * allocates the context's device word at first use, scans the table's scale
 * exponents and wkv's magnitude, builds the FP16 copy of wkv when the FP16
 * operand path applies (engram_layer_info), keeps the product w_q w_k (the
 * gate uses the two only through it: bind again after changing them) and
 * encodes the TMA descriptors.  It synchronises the device. */
engram_status engram_layer_bind(engram_ctx* ctx, int layer, const engram_layer_weights* w);

/* Fill rows [row_begin, row_end) of a table with its deterministic contents:
 * code(row, col) and scale(row, group) are a Philox4x32-10 function of
 * (seed, row, column) - uniform over the 254 finite E4M3 codes and over
 * E8M0 exponents 119..127.  data/scale may be device or mapped pinned host. */
engram_status engram_table_fill(const engram_ctx* ctx, uint64_t seed, uint8_t* data,
                                uint8_t* scale, uint64_t row_begin, uint64_t row_end,
                                void* stream);
/* The same rows for a BF16-table layer: data bf16 [rows][row_dim] (16-byte
 * aligned), value = E4M3(code) x 2^(scale - 127) of engram_table_fill's code
 * and scale for the same (seed, row, column), which BF16 holds exactly.  A
 * layer bound to this table computes the same forward as one bound to the
 * MXFP8 table of the same seed. */
engram_status engram_table_fill_bf16(const engram_ctx* ctx, uint64_t seed, uint16_t* data,
                                     uint64_t row_begin, uint64_t row_end, void* stream);

/* Host memory for a table read through UVA (vLLM "Engram" wiki, "CPU 오프로드":
 * the table in pinned host memory, read by the GPU).  bytes of an anonymous
 * mapping that starts on a transparent-huge-page boundary, advised to use
 * huge pages where the kernel offers them, zeroed (every page touched, in
 * parallel) and registered with CUDA, mapped into the device address space;
 * *out is both its host and its device address.  Random row reads from a
 * table this large are bound by address translation, which huge pages
 * reduce: on GB300 (64 KB base pages, 512 MB huge pages), gathering 8,192
 * tokens x 24 rows from a 101 GB table took 12.8 ms from cudaHostAlloc
 * memory and 5.3-5.4 ms from this (how much of the table huge pages cover
 * depends on the host's free memory; with little of it covered the same
 * gather took 37.6 ms).  The caller owns the
 * memory and releases it with engram_host_table_free(p, bytes) once no layer
 * is bound to it. */
engram_status engram_host_table_alloc(uint64_t bytes, void** out);
engram_status engram_host_table_free(void* p, uint64_t bytes);

/* Sessions: a hash history (the last three compressed ids and a count).
 * "第四步": every token enters the history exactly once; prefill appends a
 * span, decode appends one token; fork copies the history; reset empties it.
 * Layers never append: they consume the windows an append returned. */
engram_status engram_session_create(engram_ctx* ctx, engram_session** out);
engram_status engram_session_fork(const engram_session* s, engram_session** out);
engram_status engram_session_reset(engram_session* s);
engram_status engram_session_destroy(engram_session* s);
/* Append n tokens (host int32 [n]; is_image host uint8 [n] or NULL) and write
 * their windows (host uint32 [n][4]).  An image position appends DEAD (its
 * token value is ignored).  A text token outside [0, vocab) is EINVAL and
 * nothing is appended. */
engram_status engram_session_append(engram_session* s, const int32_t* tokens,
                                    const uint8_t* is_image, int64_t n, uint32_t* windows_out);
/* Decode: append one token to each of n sessions (in array order). */
engram_status engram_batch_append(engram_session* const* sessions, const int32_t* tokens,
                                  const uint8_t* is_image, int64_t n, uint32_t* windows_out);

/* Bytes of device workspace engram_forward needs for T tokens on the current
 * device.  A batch too small to fill the GPU (fewer than two output tiles of
 * 128 tokens x 256 outputs per SM) is run with K split over up to 8 CTAs per
 * tile, and the workspace then also holds the parked fp32 partial tiles:
 * 128 KB per (128-token block, 256-output tile, split), e.g. 79 MB for 256
 * tokens at N = 25,600.  Ask again after switching to a device with another
 * SM count. */
size_t engram_workspace_bytes(const engram_ctx* ctx, int64_t T);

/* The n-gram hash.  "DeepSeek V4.1 Flash 的 Engram", section "第一步": the
 * 2-, 3- and 4-gram suffixes of (c_t, c_{t-1}, c_{t-2}, c_{t-3}) each get one
 * hash per head; vLLM "Engram" wiki, section "동작 방식": per (order, head),
 * the ids are multiplied by that pair's multipliers, the products XORed
 * (wrapping 64-bit) and reduced modulo the pair's prime, inside its own bucket
 * range: row = offset[b] + x mod prime[b].  An n-gram holding DEAD gives
 * ENGRAM_MASKED for every head of its order.
 * d_windows: device uint32 [T][4], 16-byte aligned; d_rows: device uint32
 * [T][nb], written.  The layer need not be bound. */
engram_status engram_hash(const engram_ctx* ctx, int layer, const uint32_t* d_windows, int64_t T,
                          uint32_t* d_rows, void* stream);
/* Gather and dequantise.  "DeepSeek V4.1 Flash 的 Engram", section "第二步",
 * and "3.84 亿行 Embedding 的存法大揭秘": each row holds 256 E4M3 codes and
 * one E8M0 scale per 32 of them; value = E4M3(code) x 2^(scale - 127), exact
 * in BF16; the 24 rows of a token are concatenated in bucket order into its
 * 6,144-vector.  d_rows: device uint32 [T][nb]; d_emb: device bf16 [T][K],
 * 16-byte aligned, written.  A masked row gives zeros; an index >= rows gives
 * zeros and sets the error word (ENGRAM_EBOUNDS at the next engram_sync). */
engram_status engram_gather_dequant(const engram_ctx* ctx, int layer, const uint32_t* d_rows,
                                    int64_t T, uint16_t* d_emb, void* stream);
/* The wkv projection.  "DeepSeek V4.1 Flash 的 Engram", section "第二步": the
 * 6,144-vector is multiplied by wkv [25,600 x 6,144] (BF16) into one 5,120-wide
 * key per hyper-connection branch and one shared value (the last 5,120 rows,
 * "3.84 亿行 Embedding 的存法大揭秘").  kv = emb wkv^T accumulated in fp32.
 * d_emb: device bf16 [T][K], 16-byte aligned; d_kv: device fp32 [T][N],
 * written. */
engram_status engram_project(const engram_ctx* ctx, int layer, const uint16_t* d_emb, int64_t T,
                             float* d_kv, void* stream);
/* The gate.  "DeepSeek V4.1 Flash 的 Engram", section "第三步", and vLLM
 * "Engram" wiki, section "동작 방식": per branch b, hidden and key b are
 * RMS-normalised, weighted by the pre-multiplied w_q / w_k,
 * dot = <n(h) w_q, n(k) w_k> / sqrt(d), gate = sigmoid(copysign(sqrt(max(
 * |dot|, 1e-6)), dot)), hidden_b += gate value, rounded once to BF16.  Image
 * rows (window slot 0 == DEAD, section "第四步") pass through with gate 0.
 * d_kv: device fp32 [T][N]; d_windows: device uint32 [T][4]; d_hidden: device
 * bf16 [T][hc][d], updated in place; all 16-byte aligned; d_gates: device
 * fp32 [T][hc] or NULL. */
engram_status engram_gate(const engram_ctx* ctx, int layer, const float* d_kv,
                          const uint32_t* d_windows, int64_t T, uint16_t* d_hidden,
                          float* d_gates, void* stream);
/* The whole step of the pages ("DeepSeek V4.1 Flash 的 Engram", sections
 * "第一步" to "第三步"; vLLM "Engram" wiki, "동작 방식") in one kernel:
 * hash, gather and dequantise into the GEMM's
 * shared-memory operand tiles, the tcgen05 projection and the gate as the
 * GEMM epilogue.  Neither the 6,144-vector nor the kv reaches HBM (except,
 * for a small batch run with split K, the partial kv tiles that the splits of
 * a tile hand to the last of them, through L2).  The result does not depend
 * on the order in which the splits finish.
 * d_workspace: engram_workspace_bytes(ctx, T) bytes of device memory. */
engram_status engram_forward(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                             int64_t T, uint16_t* d_hidden, void* d_workspace,
                             float* d_gates, void* stream);

/* The same step, staged: the same result as engram_forward in two kernels.  Step 1
 * gathers and dequantises every (token, bucket) row once into a scratch
 * matrix e [T][K] in d_workspace; step 2 is the forward GEMM with its A
 * operand read from e by TMA and the same gate epilogue (kv stays on chip).
 * Unlike engram_forward, the 6,144-vectors pass through device memory (an
 * L2-resident scratch of 12 KB per token); in exchange each table row is
 * read once per call instead of once per output tile.  A batch longer than
 * about 4,864 tokens (on 152 SMs) runs in chunks of that many on the same
 * workspace, so that each chunk's e stays in L2, and each chunk's GEMM runs
 * only its 256-token units that hold a text row.  A batch whose output tiles
 * (128 tokens x 256 outputs) do not fill the GPU twice (decode) runs step 2
 * with stream K: the tiles left after whole waves of one tile per CTA pair
 * have their (tile, stage) sequence cut into one contiguous range per pair,
 * each pair runs its range and then its whole tiles, and a tile that two
 * ranges share is summed, in k order, by the range that holds its first
 * stage.  Its epilogue stores the gate's partial sums of the key tiles and
 * the value v [T][d] (fp32, in the workspace); a third kernel turns the sums
 * into gates and updates hidden.  The result is deterministic on a given
 * device (the ranges depend on its SM count).
 * d_workspace: engram_forward_staged_workspace_bytes(ctx, T) bytes. */
size_t engram_forward_staged_workspace_bytes(const engram_ctx* ctx, int64_t T);
engram_status engram_forward_staged(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                    int64_t T, uint16_t* d_hidden, void* d_workspace,
                                    float* d_gates, void* stream);

/* The two steps of engram_forward_staged as separate calls, so that a caller
 * can gather the rows of the next step while the current step's GEMM runs:
 * the host-table pipeline (the vLLM page, CPU offload: rows read from pinned
 * host memory through UVA cross the host link, while the GEMM reads HBM).
 * engram_stage_rows hashes the windows and gathers and dequantises the rows
 * into the operand matrix e at the start of d_workspace
 * (engram_forward_staged_workspace_bytes(ctx, T) bytes, 16-byte aligned).
 * engram_forward_staged_rows then runs the GEMM and the gate on that
 * workspace; it must see the same layer, windows and T, ordered after the
 * staging (same stream, or an event).  Keep one workspace per step in flight:
 * staging step i+1 into the workspace of step i races with step i's GEMM. */
engram_status engram_stage_rows(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                int64_t T, void* d_workspace, void* stream);
engram_status engram_forward_staged_rows(const engram_ctx* ctx, int layer,
                                         const uint32_t* d_windows, int64_t T, uint16_t* d_hidden,
                                         void* d_workspace, float* d_gates, void* stream);

/* A table sharded over data-parallel ranks by bucket (vLLM "Engram" wiki,
 * section "데이터 병렬 토폴로지": with embedding_across_dp the hash heads are
 * spread over the co-located replicas; each replica looks up the rows of its
 * own heads for the ids every replica sends it and returns them, an
 * all-to-all that replaces an all-reduce, as in the FlagScale plugin's
 * decoupled parallelism).  Rank r owns a contiguous range of buckets, hence a
 * contiguous range of the layer's table rows, and holds only those.  Per
 * step: every rank hashes its own windows bucket-major
 * (engram_hash_by_bucket), sends each owner the ids of the owner's buckets
 * (the caller's collective), the owner gathers the raw rows of the ids it
 * received (engram_shard_gather_raw), the requester receives them back in
 * bucket order and decodes them into its staged operand
 * (engram_stage_raw_rows); engram_forward_staged_rows then runs the GEMM and
 * the gate on its own tokens.  The collectives themselves are the caller's
 * (the package's sharded.py runs them with torch.distributed). */

/* Bind a layer to a shard of its table: table/scales hold rows
 * [row_lo, row_lo + w->rows) of the layer's table (w->rows may be 0, with null
 * table and scales, for a rank that owns no bucket); wkv, wq, wk are whole.
 * scale_min..scale_max is the E8M0 exponent span of the WHOLE table (the
 * ranks combine their shards' spans), which picks the operand encoding as
 * engram_layer_bind's scan does.  MXFP8 tables only (a BF16-table flag is
 * ENGRAM_EUNSUPPORTED).  A layer bound this way serves
 * engram_shard_gather_raw, engram_stage_raw_rows, engram_forward_staged_rows,
 * engram_project and engram_gate; the calls that index the table with global
 * row numbers (engram_gather_dequant, engram_forward, engram_forward_noalloc,
 * engram_forward_staged, engram_stage_rows, engram_project_windows,
 * engram_prepass) return ENGRAM_ESTATE. */
engram_status engram_layer_bind_shard(engram_ctx* ctx, int layer, const engram_layer_weights* w,
                                      uint64_t row_lo, uint32_t scale_min, uint32_t scale_max);
/* The smallest and largest of n E8M0 bytes (device or mapped pinned host
 * memory): a shard's span, for the ranks to combine before
 * engram_layer_bind_shard.  n = 0 gives 255 and 0.  Synchronises the device.
 * To fill a shard that holds rows [row_lo, row_hi) with engram_table_fill,
 * which writes row r at data + r row_dim and its scales at scale + r row_dim /
 * 32, pass data - row_lo row_dim and scale - row_lo row_dim / 32 with that
 * row range: only rows inside the shard are written. */
engram_status engram_scale_range(engram_ctx* ctx, const uint8_t* scales, uint64_t n,
                                 uint32_t* scale_min, uint32_t* scale_max);
/* engram_hash with the row indices bucket-major: d_rows_bm [nb][T], so that
 * the ids of a range of buckets are one contiguous block per owner. */
engram_status engram_hash_by_bucket(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                    int64_t T, uint32_t* d_rows_bm, void* stream);
/* Bytes of one raw row: row_dim E4M3 codes, row_dim / 32 E8M0 scale bytes,
 * zero padding to row_dim + 16 (272 at row_dim 256). */
size_t engram_raw_row_bytes(const engram_ctx* ctx);
/* Owner side: d_raw [n][engram_raw_row_bytes] (device, 16-byte aligned) gets
 * the raw rows of the n global row ids d_ids (device uint32), read from the
 * rows this layer is bound to (a shard, or the whole table).  A masked id
 * gives a zero row; an id outside the bound rows gives a zero row and sets
 * the error word (ENGRAM_EBOUNDS at the next engram_sync). */
engram_status engram_shard_gather_raw(const engram_ctx* ctx, int layer, const uint32_t* d_ids,
                                      int64_t n, uint8_t* d_raw, void* stream);
/* Requester side: decode raw rows, bucket-major d_raw_bm [nb][T][raw row]
 * (16-byte aligned), into the staged operand at the start of d_workspace
 * (engram_forward_staged_workspace_bytes(ctx, T) bytes), as engram_stage_rows
 * would from the table; d_rows_bm [nb][T] are this rank's own row indices
 * (engram_hash_by_bucket), which mark the masked rows.  A raw scale outside
 * the bound exponent span gives zeros and sets the error word.  Then call
 * engram_forward_staged_rows on the same workspace. */
engram_status engram_stage_raw_rows(const engram_ctx* ctx, int layer, const uint32_t* d_rows_bm,
                                    const uint8_t* d_raw_bm, int64_t T, void* d_workspace,
                                    void* stream);

/* engram_forward for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment variant.  A serving engine that
 * reserves the GPU's memory for its own pools, or a plugin host that forbids
 * its plugins to allocate, can pass only the buffers it already owns; this
 * call needs no workspace argument because its scratch (the gate sums and gates) lives
 * in an 8 MiB buffer inside the library's device image, held on every GPU
 * that loads the library until the process exits.  It makes no cudaMalloc or
 * cudaFree call.  T is limited to what 8 MiB holds (8,592 tokens at hc 4,
 * d 5,120); a larger T returns ENGRAM_EINVAL with the limit in the message.
 * K is never split here (the partial tiles would not fit), so a small batch
 * runs on fewer SMs than engram_forward would give it.
 * The first call on a device looks up the buffer's device address (once per
 * device, with that device current) and keeps it until the process exits;
 * make that first call before any stream capture.  A cudaDeviceReset unloads
 * the library's device image and invalidates that address, as it does every
 * context bound on the device: do not call this after a reset.  The size check
 * comes after the same argument checks as engram_forward.  All calls share the
 * buffer: calls whose kernels may overlap on the GPU (other streams, other
 * threads) race on it - keep them on one stream. */
engram_status engram_forward_noalloc(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                     int64_t T, uint16_t* d_hidden, float* d_gates, void* stream);

/* Hash, gather and projection fused: the part of the step that does not depend on hidden
 * ("DeepSeek V4.1 Flash 的 Engram", section "提前投影": hashing, gather and
 * projection depend only on the tokens and can run ahead of the layer):
 * windows (device [T][4]) -> kv fp32 (device [T][N]); the 6,144-vector stays
 * in shared memory.  engram_gate then finishes the step at the layer entry. */
engram_status engram_project_windows(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                     int64_t T, float* d_kv, void* stream);

/* The same pre-pass through the staged path ("DeepSeek V4.1 Flash 的 Engram",
 * section "提前投影"): every (token, bucket) row is gathered and dequantised
 * once into the operand matrix e at the start of d_workspace, then the
 * tcgen05 projection (CTA pairs; stream K for a batch whose output tiles do
 * not fill the GPU twice, as in engram_forward_staged) stores kv [T][N] in
 * d_kv, either as fp32 (ENGRAM_KV_F32, the same values as engram_project
 * up to accumulation order) or rounded once to BF16 (ENGRAM_KV_BF16, half
 * the bytes to keep until the layer entry; every kv value then carries a
 * relative error of at most 2^-9, which is not the plain reading of the
 * step, so the BF16 form is an explicit choice of the caller).
 * d_workspace: engram_forward_staged_workspace_bytes(ctx, T) bytes, 16-byte
 * aligned; d_kv 16-byte aligned.  Works for every bound layer, BF16 tables
 * included.  engram_gate (fp32) or engram_gate_bf16kv then finishes the step. */
#define ENGRAM_KV_F32 0
#define ENGRAM_KV_BF16 1
engram_status engram_prepass(const engram_ctx* ctx, int layer, const uint32_t* d_windows, int64_t T,
                             void* d_kv, int kv_format, void* d_workspace, void* stream);
/* The gate (as engram_gate, "第三步") on a BF16 kv [T][N] (engram_prepass
 * with ENGRAM_KV_BF16); otherwise as engram_gate. */
engram_status engram_gate_bf16kv(const engram_ctx* ctx, int layer, const uint16_t* d_kv,
                                 const uint32_t* d_windows, int64_t T, uint16_t* d_hidden,
                                 float* d_gates, void* stream);

/* Synchronise `stream`, then read and clear the context's device error word:
 * ENGRAM_EBOUNDS / ENGRAM_ETIMEOUT if a kernel reported one, ENGRAM_ECUDA on
 * an asynchronous CUDA error. */
engram_status engram_sync(const engram_ctx* ctx, void* stream);

/* Upper bound, in nanoseconds, of every wait inside a kernel launched from
 * this context (default 4 s).  A wait that runs out makes the kernel raise
 * an abort flag, leave its loops, free its tensor memory and return; the next
 * engram_sync reports ENGRAM_ETIMEOUT and the context stays usable. */
engram_status engram_ctx_set_wait_limit(engram_ctx* ctx, int64_t ns);
/* Test hook for the bounded waits: while on, the GEMM kernels issue no wkv
 * loads, so the tensor-core issuer's wait for them runs out (after the wait
 * limit) and the call ends with ENGRAM_ETIMEOUT.  Nothing faults or hangs. */
engram_status engram_debug_starve_operand(engram_ctx* ctx, int on);

/* Message of the calling thread's last error ("" if none). */
const char* engram_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
