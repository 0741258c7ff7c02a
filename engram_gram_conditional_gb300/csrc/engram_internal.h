// Internal declarations shared by the host API (engram_api.cpp) and the CUDA
// kernels (kernels_misc.cu, kernels_mma.cu) of libengram.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace engram {

constexpr uint32_t kDead = 0xFFFFFFFFu;
constexpr uint32_t kMasked = 0xFFFFFFFFu;
constexpr int kMaxBuckets = 32;  // (max_n - min_n + 1) <= 4 orders x heads <= 8

// Device error word bits.
constexpr uint32_t kErrBounds = 1u;   // a row index >= rows was met
constexpr uint32_t kErrTimeout = 2u;  // a bounded wait gave up

// Hash parameters of one layer, passed to kernels by value.
struct HashParams {
    uint64_t mult[kMaxBuckets][4];
    uint64_t prime[kMaxBuckets];
    uint64_t offset[kMaxBuckets];
    int nb;
    int heads;
    int min_n;
    int pad_;
};

// Layer geometry as the kernels see it.
struct Geometry {
    int nb, heads, min_n, row_dim;
    int K, N, hc, d;
    float eps;
};

// Tile shape of the tcgen05 kernels.
constexpr int kBM = 128;  // tokens per tile (TMEM lanes)
constexpr int kBN = 256;  // outputs per tile (TMEM columns per accumulator)
constexpr int kBK = 64;   // reduction slice per pipeline stage (128-byte rows)

enum EpilogueMode : int {
    kEpiStoreKv = 0,   // write kv fp32
    kEpiForward = 3,   // the gate: key tiles publish per-(token, branch, tile) sums
                       // and the last key tile of each M block quadrant turns them
                       // into gates; value tiles wait for those, then hidden += g v
    kEpiForwardSk = 4,  // stream K (a batch too small to fill the GPU), the gate's
                        // first half: the piece that finishes a key tile (after
                        // adding the later ranges' parked pieces) publishes its
                        // sums, one that finishes a value tile stores v [T][d];
                        // nothing waits for gates, and launch_gate_sums then
                        // turns the sums into gates and updates hidden
    kEpiForwardCompact = 5  // kEpiForward over the M units that hold a text row
                            // only (MmaArgs::block_text); a separate instantiation,
                            // so that kEpiForward's code is untouched by it
};

struct MmaArgs {
    int64_t T;
    int K;
    int n_tile_begin;  // first N tile (of kBN) of this launch
    int n_tiles;       // N tiles of this launch
    int m_blocks;      // ceil(T / kBM)
    int group_m;       // tile rasterisation: M blocks (pair units) per group
    int key_tiles;     // kEpiForward: N tiles of the keys, ordered before the value tiles (else 0)
    int key_tail;      // kEpiForward, one group of M units: the last key_tail key tiles and
                       // the value tiles run M-major (0: all N-major)
    int k_splits;      // split-K factor (>= 1); the tile list holds every (tile, split)
    int b_tiled;       // wkv map over 128 x 64 tiles (the FP16 copy), else row-major [N][K]
    int a_tiled;       // TMA-fed A in 128 x 64 tiles (the staged FP16 operand), else [T][K]
    int64_t kv_split_stride;  // kEpiStoreKv: floats between the kv buffers of two splits
    int hc, d;
    float eps;
    uint32_t* err;
    long long wait_limit_ns;
    int starve_b;          // test hook: the TMA producer issues no wkv loads
    // fused operand A
    const uint4* windows;
    const uint8_t* table;
    const uint8_t* scales;
    uint64_t rows;
    int row_dim;
    int row_dim_log2;
    int a_exp_shift;       // FP16 operands: decoded value x 2^(scale - 127 + a_exp_shift)
    float out_scale;       // accumulator x out_scale = kv (undoes the operand scaling)
    // epilogue
    float* kv;             // kEpiStoreKv: [T][ldkv] fp32, or BF16 when kv_bf16
    int kv_bf16;           // kEpiStoreKv: store kv rounded once to BF16 (no split buffers)
    int64_t ldkv;
    uint16_t* hidden;      // [T][hc][d]
    const float* wqk;      // [hc][d] w_q * w_k (the gate's pre-multiplied weights, product)
    float* partials;       // [T][hc][d / kBN][epi_groups][3]
    int epi_groups;        // kEpiForward: epilogue warps per TMEM quadrant (1, or 2 TMA-fed)
    float* gbuf;           // [T][hc] gates of the call
    // kEpiForward, per (M block, TMEM quadrant): finished key tiles, then a
    // gates-ready flag (zeroed per call)
    uint32_t* counters;
    // kEpiForward with k_splits > 1: one 128 x 256 fp32 slot per (M block, N tile,
    // split), and per (M block, N tile, TMEM quadrant) two counters, arrivals and
    // partials ready (zeroed per call)
    float* split_partials;
    uint32_t* split_counters;
    float* gates;          // [T][hc] or null
    // kEpiStoreKv with stream K, and kEpiForwardSk (k_splits == 1): the (tile, stage) sequence of the
    // launch is cut into one contiguous range per CTA (or pair); a tile that two
    // ranges share is finished by the range holding its first stage, which adds
    // the parked partials of the later ranges in order.  One 128 x 256 fp32 slot
    // and sixteen ready flags (one per epilogue warp) per CTA, flags zeroed per
    // call.
    int stream_k;
    float* sk_slots;
    uint32_t* sk_flags;
    // kEpiForward on a TMA-fed operand without splits: per 128-token block,
    // nonzero when it holds a text row (written by the staging kernel); the
    // items of an M unit whose blocks hold only image rows are skipped by every
    // role (those rows pass through; their gates are written as 0).  Null: no
    // skipping.
    const uint32_t* block_text;
    HashParams hp;
};

// kernels_misc.cu
cudaError_t launch_table_fill(uint64_t seed, uint8_t* data, uint8_t* scale, uint64_t row_begin,
                              uint64_t row_end, int row_dim, cudaStream_t s);
// The same rows stored as BF16 values (the dequantised MXFP8 values, exact).
cudaError_t launch_table_fill_bf16(uint64_t seed, uint16_t* data, uint64_t row_begin,
                                   uint64_t row_end, int row_dim, cudaStream_t s);
// rows [T][nb], or with bucket_major [nb][T]
cudaError_t launch_hash(const HashParams& hp, const uint4* windows, int64_t T, uint32_t* rows,
                        bool bucket_major, cudaStream_t s);
// A table sharded over ranks by bucket.  Owner side: the raw rows (row_dim
// codes, row_dim / 32 scale bytes, zeros to row_dim + 16 bytes) of n global
// row ids from a shard holding rows [row_lo, row_lo + nrows).  Requester side:
// those rows, bucket-major [nb][T], decoded into the staged operand e as
// launch_gather_stage writes it (rows_bm [nb][T]: the requester's row indices,
// for the masked rows; n_clear words at `clear` zeroed as there).
cudaError_t launch_shard_gather_raw(const uint32_t* ids, int64_t n, uint64_t row_lo, uint64_t nrows,
                                    int row_dim, const uint8_t* table, const uint8_t* scales,
                                    uint8_t* raw, uint32_t* err, cudaStream_t s);
// (block_text, may be null: set to 1 for every block - raw rows carry no
// image marks, so nothing is skipped)
cudaError_t launch_stage_raw(const HashParams& hp, const uint32_t* rows_bm, const uint8_t* raw,
                             int64_t T, int row_dim, bool f16, int exp_shift, uint16_t* e,
                             uint32_t* err, uint32_t* clear, int n_clear, uint32_t* block_text,
                             cudaStream_t s);
// table_bf16: BF16 rows [R][row_dim] without scales (scales unused).
cudaError_t launch_gather(const Geometry& g, const uint32_t* rows, int64_t T,
                          const uint8_t* table, const uint8_t* scales, uint64_t nrows,
                          bool table_bf16, uint16_t* emb, uint32_t* err, cudaStream_t s);
// kv: fp32 [T][N], possibly the sum of nsplit (<= 8) partial buffers
// split_stride floats apart, added in split order; or BF16 [T][N] (kv_bf16,
// nsplit 1).  wqk: [hc][d] w_q * w_k.  kv, hidden and wqk 16-byte aligned.
cudaError_t launch_gate(const Geometry& g, const void* kv, bool kv_bf16, int nsplit,
                        int64_t split_stride, const uint4* windows, int64_t T, uint16_t* hidden,
                        const float* wqk, float* gates, cudaStream_t s);
// The gate's second half after a kEpiForwardSk GEMM: per token, the gates from
// the key tiles' sums partials [T][hc][d / 256][groups][3] (added in (tile,
// group) order), then hidden_b += g_b v with v [T][d] fp32; image rows pass
// through with gate 0.  hidden and v 16-byte aligned; gates [T][hc] or null.
cudaError_t launch_gate_sums(const Geometry& g, const float* partials, int groups, const float* v,
                             const uint4* windows, int64_t T, uint16_t* hidden, float* gates,
                             cudaStream_t s);
// out = a * b elementwise (fp32, n values).
cudaError_t launch_mul_f32(const float* a, const float* b, float* out, int64_t n, cudaStream_t s);
// Bind-time scans: out[0] = min, out[1] = max of n E8M0 bytes (out preset by
// the caller to 255 / 0); out[2] = largest |x| of n BF16 values as its bit
// pattern without the sign (out[2] preset to 0).
cudaError_t launch_scale_range(const uint8_t* scales, uint64_t n, uint32_t* out, cudaStream_t s);
cudaError_t launch_absmax_bf16(const uint16_t* x, uint64_t n, uint32_t* out, cudaStream_t s);
// Staged forward, step 1: windows -> operand rows e: FP16 in 128 x 64 tiles
// (element (t, k) at ((t / 128) (K / 64) + k / 64) 8192 + (t % 128) 64 + k % 64;
// rows of the last 128-token block past T are not written), or BF16 row-major
// [T][K].  Also zeroes n_clear words at `clear` (may be null with 0), once the
// kernel before it in the stream has finished.
// block_text (may be null): per 128-token block, 1 when it holds a text row,
// else 0 (written after the kernel before it has finished).
cudaError_t launch_gather_stage(const HashParams& hp, const uint4* windows, int64_t T, int row_dim,
                                const uint8_t* table, const uint8_t* scales, uint64_t nrows,
                                bool table_bf16, bool f16, int exp_shift, uint16_t* e,
                                uint32_t* err, uint32_t* clear, int n_clear, uint32_t* block_text,
                                cudaStream_t s);
// FP16 copy of the BF16 wkv [N][K] (N % 128 == 0, K % 64 == 0), values x
// scale rounded to nearest even, stored as 128 x 64 tiles: element (n, k) at
// ((n / 128) (K / 64) + k / 64) 8192 + (n % 128) 64 + k % 64.
cudaError_t launch_wkv_to_f16_tiles(const uint16_t* src, uint16_t* dst, uint64_t N, uint64_t K,
                                   float scale, cudaStream_t s);

// kernels_mma.cu
// Host-side TMA descriptor for a row-major 16-bit (BF16 or FP16) matrix
// [rows][cols] with a (kBK x box_rows) box and 128-byte swizzle.
cudaError_t make_tma_16bit(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, bool f16);
cudaError_t launch_project(const MmaArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           cudaStream_t s);
cudaError_t launch_forward_phase(const MmaArgs& a, int mode, bool f16, bool bucket,
                                 const CUtensorMap& tmB, cudaStream_t s);
// The projection with a TMA-fed A operand (the staged operand e) and the
// kv-store epilogue: kv fp32 or BF16 (a.kv_bf16), whole tiles or, with
// a.stream_k, stream-K pieces (the staged forward of a small batch, whose gate
// runs after it, and engram_prepass).
cudaError_t launch_project_tma(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, cudaStream_t s);
// The same GEMMs on CTA pairs (clusters of two SMs, tcgen05 cta_group::2):
// each pair computes 256-token x 256-output tiles, each CTA holding half of the
// wkv tile, so tmB_half is a wkv tensor map with 128-row boxes.
cudaError_t launch_project_tma_pair(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                                    const CUtensorMap& tmB_half, cudaStream_t s);
cudaError_t launch_forward_tma_pair(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                                   const CUtensorMap& tmB_half, cudaStream_t s);
// Staged forward, step 2: the whole forward GEMM with a TMA-fed A operand.
cudaError_t launch_forward_tma(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, cudaStream_t s);
// The same forward GEMM of a small batch with stream K (a.stream_k = 1, the
// gate epilogue on the pieces that finish tiles), on CTA pairs or single CTAs.
cudaError_t launch_forward_sk(const MmaArgs& a, bool f16, bool pairs, const CUtensorMap& tmA,
                              const CUtensorMap& tmB, cudaStream_t s);
int device_sm_count();

}  // namespace engram
