// Host side of libengram.so: the C ABI declared in include/engram.h.
//
// Holds the context (geometry, token map, per-layer hash parameters and bound
// weights), the sessions (hash history), argument validation and the launch
// of the kernels.  No compute of the forward step happens here: every step of
// the path runs in the CUDA kernels of kernels_misc.cu and kernels_mma.cu.
#include <cuda_runtime.h>
#include <string.h>
#include <sys/mman.h>
#include <unistd.h>

#include <cstdio>

#include <math.h>

#include <algorithm>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "../../include/engram.h"
#include "engram_internal.h"

using namespace engram;

namespace {

thread_local std::string g_last_error;

engram_status fail(engram_status st, const std::string& msg) {
    g_last_error = msg;
    return st;
}
engram_status ok() {
    g_last_error.clear();
    return ENGRAM_OK;
}
engram_status cuda_fail(cudaError_t e, const char* what) {
    return fail(ENGRAM_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

constexpr uint32_t kSessionMagic = 0x53474E45u;  // "ENGS"

}  // namespace

namespace engram {
// Message for engram_last_error() from the library's other translation units.
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace engram

namespace {

// ---- hash parameters (setup) -------------------------------------------------------
// Deterministic Miller-Rabin for 64-bit n (bases 2..37).
uint64_t mulmod(uint64_t a, uint64_t b, uint64_t m) {
    return (uint64_t)((unsigned __int128)a * b % m);
}
uint64_t powmod(uint64_t a, uint64_t e, uint64_t m) {
    uint64_t r = 1;
    a %= m;
    while (e) {
        if (e & 1) r = mulmod(r, a, m);
        a = mulmod(a, a, m);
        e >>= 1;
    }
    return r;
}
bool prime64(uint64_t n) {
    if (n < 2) return false;
    static const uint64_t small[] = {2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37};
    for (uint64_t p : small) {
        if (n % p == 0) return n == p;
    }
    uint64_t d = n - 1;
    int s = 0;
    while ((d & 1) == 0) {
        d >>= 1;
        ++s;
    }
    for (uint64_t a : small) {
        uint64_t x = powmod(a, d, n);
        if (x == 1 || x == n - 1) continue;
        bool comp = true;
        for (int r = 1; r < s; ++r) {
            x = mulmod(x, x, n);
            if (x == n - 1) {
                comp = false;
                break;
            }
        }
        if (comp) return false;
    }
    return true;
}

// Philox4x32-10 (Salmon et al., SC'11), host copy for the multiplier draw.
void philox(uint32_t c[4], uint32_t k0, uint32_t k1) {
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
        c[1] = (uint32_t)p1;
        c[3] = (uint32_t)p0;
        c[0] = n0;
        c[2] = n2;
    }
}

uint64_t layer_multiplier(uint64_t seed, uint32_t j, uint32_t vc) {
    uint32_t c[4] = {j, 0u, 0u, 2u};
    philox(c, (uint32_t)seed, (uint32_t)(seed >> 32));
    const uint64_t r = (uint64_t)c[0] | ((uint64_t)c[1] << 32);
    uint64_t half = (UINT64_MAX / vc) / 2;
    if (half == 0) half = 1;
    return 2 * (r % half) + 1;
}

}  // namespace

struct LayerState {
    std::vector<uint64_t> mult;    // [nb][4]
    std::vector<uint64_t> prime;   // [nb]
    std::vector<uint64_t> offset;  // [nb]
    uint64_t rows = 0;
    bool bound = false;
    engram_layer_weights w{};
    CUtensorMap tm_wkv{};          // the caller's BF16 wkv
    CUtensorMap tm_wkv_half{};     // the same with 128-row boxes (CTA-pair kernels)
    // FP16 operand path of the fused kernels (see engram_layer_info)
    bool f16 = false;
    uint16_t* wkv_f16 = nullptr;   // library-owned copy, wkv x 2^wkv_exp
    float* wqk = nullptr;          // library-owned w_q * w_k [hc][d], made at bind
    CUtensorMap tm_wkv_f16{};
    CUtensorMap tm_wkv_f16_2k{};   // the tiled FP16 copy with 256-row boxes (2 k-blocks)
    int wkv_exp = 0;
    int a_exp_shift = 0;
    uint32_t scale_min = 0, scale_max = 0;
    bool bucket_gather = false;    // whole 256-wide rows gathered once per tile and bucket
    bool table_bf16 = false;       // BF16 rows without scales (ENGRAM_BIND_TABLE_BF16)
    // bound to a shard of the table (engram_layer_bind_shard): rows
    // [row_lo, row_lo + shard_rows) of the layer's table
    bool shard = false;
    uint64_t row_lo = 0, shard_rows = 0;
};

struct engram_ctx {
    engram_ctx_desc desc{};
    std::vector<uint64_t> seeds, bases;
    std::vector<uint32_t> map;
    int nb = 0, K = 0, N = 0;
    std::vector<LayerState> layers;
    uint32_t* d_err = nullptr;  // [0] error word, [1..3] bind-time scan results
    int device = -1;
    long long wait_limit_ns = 4000000000LL;
    int starve_b = 0;
};

struct engram_session {
    const engram_ctx* ctx;
    uint32_t hist[3];  // c_{t-1}, c_{t-2}, c_{t-3} of the next position
    uint64_t count;
    uint32_t magic;
};

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

engram_status check_layer(const engram_ctx* ctx, int layer, bool need_bound) {
    if (!ctx) return fail(ENGRAM_EINVAL, "null context");
    if (layer < 0 || layer >= (int)ctx->layers.size()) return fail(ENGRAM_EINVAL, "layer out of range");
    if (need_bound && !ctx->layers[layer].bound)
        return fail(ENGRAM_ESTATE, "layer weights not bound (engram_layer_bind)");
    return ENGRAM_OK;
}

// Calls that index the layer's table with global row numbers need all of it.
engram_status check_full_table(const engram_ctx* ctx, int layer) {
    if (ctx->layers[layer].shard)
        return fail(ENGRAM_ESTATE, "layer bound to a table shard: its rows come through "
                                   "engram_shard_gather_raw and engram_stage_raw_rows");
    return ENGRAM_OK;
}

engram_status check_T(int64_t T) {
    if (T < 0 || T > (int64_t)1 << 24) return fail(ENGRAM_EINVAL, "T must be in [0, 2^24]");
    return ENGRAM_OK;
}

HashParams hash_params(const engram_ctx* ctx, int layer) {
    HashParams hp{};
    const LayerState& L = ctx->layers[layer];
    for (int b = 0; b < ctx->nb; ++b) {
        for (int j = 0; j < 4; ++j) hp.mult[b][j] = L.mult[b * 4 + j];
        hp.prime[b] = L.prime[b];
        hp.offset[b] = L.offset[b];
    }
    hp.nb = ctx->nb;
    hp.heads = (int)ctx->desc.heads;
    hp.min_n = (int)ctx->desc.min_n;
    return hp;
}

Geometry geometry(const engram_ctx* ctx) {
    Geometry g{};
    g.nb = ctx->nb;
    g.heads = (int)ctx->desc.heads;
    g.min_n = (int)ctx->desc.min_n;
    g.row_dim = (int)ctx->desc.row_dim;
    g.K = ctx->K;
    g.N = ctx->N;
    g.hc = (int)ctx->desc.hc;
    g.d = (int)ctx->desc.d;
    g.eps = (float)ctx->desc.eps;
    return g;
}

MmaArgs mma_args(const engram_ctx* ctx, int layer, int64_t T) {
    MmaArgs a{};
    const LayerState& L = ctx->layers[layer];
    a.T = T;
    a.K = ctx->K;
    a.m_blocks = (int)((T + kBM - 1) / kBM);
    a.group_m = 16;
    a.key_tiles = 0;
    a.k_splits = 1;
    a.kv_split_stride = 0;
    a.b_tiled = L.f16 ? 1 : 0;  // the FP16 wkv copy is tiled, the caller's BF16 wkv is not
    a.a_tiled = 0;
    a.hc = (int)ctx->desc.hc;
    a.d = (int)ctx->desc.d;
    a.eps = (float)ctx->desc.eps;
    a.err = ctx->d_err;
    a.wait_limit_ns = ctx->wait_limit_ns;
    a.starve_b = ctx->starve_b;
    a.table = L.w.table;
    a.scales = L.w.scales;
    a.rows = L.rows;
    a.row_dim = (int)ctx->desc.row_dim;
    a.row_dim_log2 = 31 - __builtin_clz(ctx->desc.row_dim);
    a.a_exp_shift = 0;
    a.out_scale = 1.0f;
    a.wqk = L.wqk;
    a.hp = hash_params(ctx, layer);
    return a;
}

}  // namespace

namespace engram {

// Split-K factor of the forward for T tokens on this device: 1 while the
// output tiles fill the GPU twice over.  A smaller batch (decode) would leave
// SMs idle while wkv streams, so K is split until there are about four waves
// of (tile, split) work items: the largest s <= that (at most 8, at least 8
// k-blocks per split) that divides the k-blocks - and, for 256-wide rows, the
// buckets, since the fused gather splits on bucket boundaries.
int forward_k_splits(const engram_ctx* ctx, int64_t T, int max_splits) {
    const int64_t tiles = (T + kBM - 1) / kBM * (ctx->N / kBN);
    const int sms = device_sm_count();
    if (max_splits <= 1 || tiles >= 2 * (int64_t)sms) return 1;
    int want = (int)((4 * (int64_t)sms + tiles / 2) / tiles);
    want = std::max(2, std::min({want, 8, max_splits}));
    const int KB = ctx->K / kBK;
    const int nb = ctx->K / (int)ctx->desc.row_dim;
    for (int s = want; s > 1; --s) {
        if (KB % s != 0 || KB / s < 8) continue;
        if (ctx->desc.row_dim == 256 && nb % s != 0) continue;
        return s;
    }
    return 1;
}

// Workspace of the forward epilogue, in order: the gate sums
// [T][hc][d/kBN][groups][3] (groups: the epilogue warps per TMEM quadrant);
// the gates [T][hc]; the counters, zeroed by each call (per (M block, TMEM
// quadrant) finished key tiles and a gates-ready flag, then with split K per
// (M block, N tile, quadrant) arrivals and partials ready); with split K the
// parked partial accumulators, one 128 x 256 fp32 slot per (M block, N tile,
// split).  Each part starts on a 256-byte boundary.
struct ForwardWs {
    int splits;
    size_t part, gbuf, counters, counter_words, slots;
    size_t total() const { return part + gbuf + counters + slots; }
};

ForwardWs forward_ws(const engram_ctx* ctx, int64_t T, int max_splits, int groups) {
    ForwardWs w{};
    const size_t P = ctx->desc.d / kBN * (size_t)groups;
    const size_t mb = ((size_t)T + kBM - 1) / kBM, nt = ctx->N / kBN;
    w.splits = forward_k_splits(ctx, T, max_splits);
    w.part = ((size_t)T * ctx->desc.hc * P * 3 * sizeof(float) + 255) & ~(size_t)255;
    w.gbuf = ((size_t)T * ctx->desc.hc * sizeof(float) + 255) & ~(size_t)255;
    w.counter_words = mb * 8 + (w.splits > 1 ? mb * nt * 8 : 0);
    w.counters = (w.counter_words * sizeof(uint32_t) + 255) & ~(size_t)255;
    w.slots = w.splits > 1 ? mb * nt * w.splits * (size_t)(kBM * kBN) * sizeof(float) : 0;
    return w;
}

size_t forward_workspace_bytes_groups(const engram_ctx* ctx, int64_t T, int max_splits,
                                      int groups) {
    if (!ctx || T <= 0) return 0;
    return forward_ws(ctx, T, max_splits, groups).total();
}
// The fused kernels: one epilogue warp per TMEM quadrant.
size_t forward_workspace_bytes(const engram_ctx* ctx, int64_t T, int max_splits) {
    return forward_workspace_bytes_groups(ctx, T, max_splits, 1);
}

// Points the forward epilogue's fields of `a` into the workspace and zeroes
// its counters on `s` (unless zero is false: the staging kernel before the
// GEMM zeroed them, so that no memset stands between the two launches).
cudaError_t forward_bind_ws(const engram_ctx* ctx, int64_t T, int max_splits, int groups,
                            void* ws, MmaArgs& a, cudaStream_t s, bool zero) {
    const ForwardWs w = forward_ws(ctx, T, max_splits, groups);
    a.epi_groups = groups;
    char* base = static_cast<char*>(ws);
    a.partials = reinterpret_cast<float*>(base);
    a.gbuf = reinterpret_cast<float*>(base + w.part);
    // tile order: the key tiles of every group of 16 M blocks (pair units)
    // before any value tile, so that a value tile does not wait for gates of
    // key tiles that run after it (with one group this is the plain order)
    a.key_tiles = (int)(ctx->desc.hc * ctx->desc.d / kBN);
    a.counters = reinterpret_cast<uint32_t*>(base + w.part + w.gbuf);
    a.k_splits = w.splits;
    if (w.splits > 1) {
        a.split_counters = a.counters + 8 * (size_t)a.m_blocks;
        a.split_partials = reinterpret_cast<float*>(base + w.part + w.gbuf + w.counters);
    }
    return zero ? cudaMemsetAsync(a.counters, 0, w.counter_words * sizeof(uint32_t), s)
                : cudaSuccess;
}

}  // namespace engram

namespace engram {

// The argument checks every fused forward makes before it looks at its buffers.
engram_status check_forward_call(const engram_ctx* ctx, int layer, int64_t T) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T)) || (st = check_full_table(ctx, layer))) return st;
    return ENGRAM_OK;
}

// engram_forward with the split-K factor capped at max_splits; the workspace
// is forward_workspace_bytes(ctx, T, max_splits) bytes.
engram_status forward_fused(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                            int64_t T, uint16_t* d_hidden, void* d_workspace, float* d_gates,
                            void* stream, int max_splits) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T)) || (st = check_full_table(ctx, layer))) return st;
    if (T == 0) return ok();
    if (!d_windows || !d_hidden || !d_workspace || !aligned16(d_windows) || !aligned16(d_hidden) ||
        !aligned16(d_workspace))
        return fail(ENGRAM_EINVAL, "windows / hidden / workspace (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    if (L.table_bf16)
        return fail(ENGRAM_EUNSUPPORTED, "BF16-table layers run through engram_forward_staged");
    MmaArgs a = mma_args(ctx, layer, T);
    a.windows = reinterpret_cast<const uint4*>(d_windows);
    a.hidden = d_hidden;
    a.gates = d_gates;
    if (L.f16) {
        a.a_exp_shift = L.a_exp_shift;
        a.out_scale = ldexpf(1.0f, -(L.a_exp_shift + L.wkv_exp));
    }
    const CUtensorMap& tmB = L.f16 ? L.tm_wkv_f16 : L.tm_wkv;
    a.n_tile_begin = 0;
    a.n_tiles = ctx->N / kBN;
    // one launch: key tiles publish their sums and count in per M block; a
    // value tile's epilogue waits for its block's count before gating
    cudaError_t e =
        forward_bind_ws(ctx, T, max_splits, 1, d_workspace, a, (cudaStream_t)stream, true);
    if (e != cudaSuccess) return cuda_fail(e, "forward counters");
    e = launch_forward_phase(a, kEpiForward, L.f16, L.bucket_gather, tmB, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return ok();
}

}  // namespace engram

extern "C" {

engram_status engram_ctx_create(const engram_ctx_desc* desc, const uint32_t* token_map,
                                engram_ctx** out) {
    if (!desc || !token_map || !out) return fail(ENGRAM_EINVAL, "null argument");
    *out = nullptr;
    const engram_ctx_desc& d = *desc;
    if (d.vocab == 0 || d.vc == 0 || d.vc == 0xFFFFFFFFu) return fail(ENGRAM_EINVAL, "vocab / vc");
    if (d.min_n < 1 || d.max_n < d.min_n || d.max_n > 4) return fail(ENGRAM_EINVAL, "n-gram orders");
    if (d.heads < 1 || d.heads > 8) return fail(ENGRAM_EINVAL, "heads must be 1..8");
    if (!(d.row_dim == 32 || d.row_dim == 64 || d.row_dim == 128 || d.row_dim == 256))
        return fail(ENGRAM_EINVAL, "row_dim must be 32, 64, 128 or 256");
    if (d.hc < 1 || d.hc > 8) return fail(ENGRAM_EINVAL, "hc must be 1..8");
    if (d.d == 0 || d.d % kBN != 0) return fail(ENGRAM_EINVAL, "d must be a positive multiple of 256");
    if (d.pad_cid >= d.vc) return fail(ENGRAM_EINVAL, "pad_cid must be < vc");
    if (d.n_layers < 1 || d.n_layers > 16 || !d.layer_seeds || !d.bucket_bases)
        return fail(ENGRAM_EINVAL, "n_layers must be 1..16 with seeds and bucket bases");
    if (!(d.eps >= 0.0)) return fail(ENGRAM_EINVAL, "eps");
    const int nb = (int)((d.max_n - d.min_n + 1) * d.heads);
    const int K = nb * (int)d.row_dim;
    if (K % kBK != 0) return fail(ENGRAM_EINVAL, "nb * row_dim must be a multiple of 64");
    for (uint32_t v = 0; v < d.vocab; ++v)
        if (token_map[v] >= d.vc) return fail(ENGRAM_EINVAL, "token map value >= vc");

    engram_ctx* ctx = new (std::nothrow) engram_ctx;
    if (!ctx) return fail(ENGRAM_ENOMEM, "host allocation");
    try {
        ctx->desc = d;
        ctx->desc.layer_seeds = nullptr;
        ctx->desc.bucket_bases = nullptr;
        ctx->seeds.assign(d.layer_seeds, d.layer_seeds + d.n_layers);
        ctx->bases.assign(d.bucket_bases, d.bucket_bases + d.n_layers);
        ctx->map.assign(token_map, token_map + d.vocab);
        ctx->nb = nb;
        ctx->K = K;
        ctx->N = (int)((d.hc + 1) * d.d);
        ctx->layers.resize(d.n_layers);
        // primes: layer by layer, bucket by bucket, strictly increasing above
        // the layer's base and never reused by a later layer
        std::vector<uint64_t> used;
        for (uint32_t l = 0; l < d.n_layers; ++l) {
            LayerState& L = ctx->layers[l];
            L.mult.resize((size_t)nb * 4);
            L.prime.resize(nb);
            L.offset.resize(nb);
            uint64_t cand = ctx->bases[l], sum = 0;
            for (int b = 0; b < nb; ++b) {
                do {
                    ++cand;
                } while (!prime64(cand) || std::find(used.begin(), used.end(), cand) != used.end());
                used.push_back(cand);
                L.prime[b] = cand;
                L.offset[b] = sum;
                sum += cand;
            }
            L.rows = sum;
            if (sum > 0xFFFFFFFFull) {
                delete ctx;
                return fail(ENGRAM_EUNSUPPORTED, "layer table above 2^32 - 1 rows");
            }
            for (int b = 0; b < nb; ++b)
                for (uint32_t j = 0; j < 4; ++j)
                    L.mult[(size_t)b * 4 + j] = j < d.max_n ? layer_multiplier(ctx->seeds[l], j, d.vc) : 0;
        }
    } catch (...) {
        delete ctx;
        return fail(ENGRAM_ENOMEM, "host allocation");
    }
    *out = ctx;
    return ok();
}

engram_status engram_ctx_destroy(engram_ctx* ctx) {
    if (!ctx) return fail(ENGRAM_EINVAL, "null context");
    if (ctx->d_err) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (ctx->device >= 0) cudaSetDevice(ctx->device);
        for (LayerState& L : ctx->layers) {
            if (L.wkv_f16) cudaFree(L.wkv_f16);
            if (L.wqk) cudaFree(L.wqk);
        }
        cudaFree(ctx->d_err);
        if (cur >= 0) cudaSetDevice(cur);
    }
    delete ctx;
    return ok();
}

engram_status engram_layer_params(const engram_ctx* ctx, int layer, uint64_t* mult,
                                  uint64_t* prime, uint64_t* offset, uint64_t* rows) {
    engram_status st = check_layer(ctx, layer, false);
    if (st) return st;
    const LayerState& L = ctx->layers[layer];
    if (mult) memcpy(mult, L.mult.data(), L.mult.size() * sizeof(uint64_t));
    if (prime) memcpy(prime, L.prime.data(), L.prime.size() * sizeof(uint64_t));
    if (offset) memcpy(offset, L.offset.data(), L.offset.size() * sizeof(uint64_t));
    if (rows) *rows = L.rows;
    return ok();
}

engram_status engram_layer_set_multipliers(engram_ctx* ctx, int layer, const uint64_t* mult) {
    engram_status st = check_layer(ctx, layer, false);
    if (st) return st;
    if (!mult) return fail(ENGRAM_EINVAL, "null multiplier table");
    std::copy(mult, mult + ctx->nb * 4, ctx->layers[layer].mult.begin());
    return ok();
}

namespace {
// The context's device word (error word and scan results), allocated at the
// first bind or scan on device dev.
engram_status ensure_device_word(engram_ctx* ctx, int dev) {
    if (ctx->d_err) return ENGRAM_OK;
    cudaError_t e = cudaMalloc(&ctx->d_err, 4 * sizeof(uint32_t));
    if (e != cudaSuccess) {
        ctx->d_err = nullptr;
        return fail(ENGRAM_ENOMEM, "cudaMalloc of the error word");
    }
    e = cudaMemset(ctx->d_err, 0, 4 * sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
    ctx->device = dev;
    return ENGRAM_OK;
}
}  // namespace

engram_status engram_scale_range(engram_ctx* ctx, const uint8_t* scales, uint64_t n,
                                 uint32_t* scale_min, uint32_t* scale_max) {
    if (!ctx || !scale_min || !scale_max || (n > 0 && !scales))
        return fail(ENGRAM_EINVAL, "null argument");
    *scale_min = 255u;
    *scale_max = 0u;
    if (n == 0) return ok();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (ctx->device >= 0 && ctx->device != dev)
        return fail(ENGRAM_ESTATE, "context already bound on another device");
    const uint8_t* p = scales;
    cudaPointerAttributes attr{};
    e = cudaPointerGetAttributes(&attr, scales);
    if (e != cudaSuccess || (attr.type == cudaMemoryTypeHost && !attr.devicePointer) ||
        attr.type == cudaMemoryTypeUnregistered) {
        cudaGetLastError();
        return fail(ENGRAM_EINVAL, "scales must be device or mapped pinned host memory");
    }
    if (attr.type == cudaMemoryTypeHost) p = static_cast<const uint8_t*>(attr.devicePointer);
    engram_status st = ensure_device_word(ctx, dev);
    if (st) return st;
    const uint32_t init[2] = {255u, 0u};
    e = cudaMemcpy(ctx->d_err + 1, init, sizeof init, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = launch_scale_range(p, n, ctx->d_err + 1, 0);
    uint32_t res[2] = {255u, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(res, ctx->d_err + 1, sizeof res, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "scale scan");
    *scale_min = res[0];
    *scale_max = res[1];
    return ok();
}

namespace {
// A table shard: rows [row_lo, row_lo + w->rows) of the layer's table, and the
// E8M0 exponent span of the whole table (the shard cannot scan the others).
struct ShardSpec {
    uint64_t row_lo;
    uint32_t scale_min, scale_max;
};

engram_status bind_impl(engram_ctx* ctx, int layer, const engram_layer_weights* w,
                        const ShardSpec* sh);
}  // namespace

engram_status engram_layer_bind(engram_ctx* ctx, int layer, const engram_layer_weights* w) {
    return bind_impl(ctx, layer, w, nullptr);
}

engram_status engram_layer_bind_shard(engram_ctx* ctx, int layer, const engram_layer_weights* w,
                                      uint64_t row_lo, uint32_t scale_min, uint32_t scale_max) {
    if (w && (w->flags & ENGRAM_BIND_TABLE_BF16))
        return fail(ENGRAM_EUNSUPPORTED, "a table shard holds MXFP8 rows");
    if (scale_min > scale_max || scale_max > 254u)
        return fail(ENGRAM_EINVAL, "scale span: scale_min <= scale_max <= 254");
    const ShardSpec sh{row_lo, scale_min, scale_max};
    return bind_impl(ctx, layer, w, &sh);
}

namespace {
engram_status bind_impl(engram_ctx* ctx, int layer, const engram_layer_weights* w,
                        const ShardSpec* sh) {
    engram_status st = check_layer(ctx, layer, false);
    if (st) return st;
    const bool tbf16 = w && (w->flags & ENGRAM_BIND_TABLE_BF16);
    // a shard of no rows (a rank that owns no bucket) needs no table
    const bool no_rows = sh && w && w->rows == 0;
    if (!w || (!no_rows && (!w->table || (!tbf16 && !w->scales))) || !w->wkv || !w->wq || !w->wk)
        return fail(ENGRAM_EINVAL, "null weight pointer");
    if (w->flags & ~(ENGRAM_BIND_BF16_OPERANDS | ENGRAM_BIND_TABLE_BF16))
        return fail(ENGRAM_EINVAL, "unknown bind flag");
    LayerState& L = ctx->layers[layer];
    if (!sh && w->rows != L.rows)
        return fail(ENGRAM_EINVAL, "table rows differ from the layer's row count");
    if (sh && (w->rows > L.rows || sh->row_lo > L.rows - w->rows))
        return fail(ENGRAM_EINVAL, "shard rows outside the layer's table");
    if ((w->table && !aligned16(w->table)) || (!tbf16 && w->scales && !aligned16(w->scales)) ||
        !aligned16(w->wkv) || !aligned16(w->wq) || !aligned16(w->wk))
        return fail(ENGRAM_EINVAL, "weights must be 16-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (ctx->device >= 0 && ctx->device != dev)
        return fail(ENGRAM_ESTATE, "context already bound on another device");
    // The table may live in pinned host memory read through UVA.
    engram_layer_weights bw = *w;
    bool host_table = false;
    if (tbf16) bw.scales = nullptr;  // BF16 rows carry no scales
    for (const uint8_t** p : {&bw.table, &bw.scales}) {
        if (!*p) continue;
        cudaPointerAttributes attr{};
        e = cudaPointerGetAttributes(&attr, *p);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(ENGRAM_EINVAL, "table pointer is neither device nor registered host memory");
        }
        if (attr.type == cudaMemoryTypeHost) {
            if (!attr.devicePointer)
                return fail(ENGRAM_EUNSUPPORTED, "host table not mapped into the device address space");
            *p = static_cast<const uint8_t*>(attr.devicePointer);
            host_table = true;
        } else if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) {
            return fail(ENGRAM_EINVAL, "table pointer must be device or pinned host memory");
        }
    }
    if ((st = ensure_device_word(ctx, dev))) return st;
    CUtensorMap tm, tm_half;
    e = make_tma_16bit(&tm, w->wkv, (uint64_t)ctx->N, (uint64_t)ctx->K, kBN, false);
    if (e == cudaSuccess)
        e = make_tma_16bit(&tm_half, w->wkv, (uint64_t)ctx->N, (uint64_t)ctx->K, kBN / 2, false);
    if (e != cudaSuccess) return cuda_fail(e, "wkv tensor map");

    // Operand path of the fused kernels.  FP16 operands hold the same values
    // exactly when (a) every E8M0 exponent of the table lies in a window of 23
    // values, so code x 2^(s - 127 + shift) is exact in FP16 for one shift,
    // and (b) wkv, scaled by 2^wkv_exp so that max |w| <= 2^15, is exact in
    // FP16 for every weight above max|w| 2^-28 (smaller ones round to a
    // multiple of 2^-(24 + wkv_exp)).  Otherwise the fused kernels decode to
    // BF16 through fp32.
    const uint32_t init[3] = {255u, 0u, 0u};
    e = cudaMemcpy(ctx->d_err + 1, init, sizeof init, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "bind scan init");
    const uint64_t nscale = L.rows * (ctx->desc.row_dim / 32);
    if (!tbf16 && !sh) e = launch_scale_range(bw.scales, nscale, ctx->d_err + 1, 0);
    if (e == cudaSuccess)
        e = launch_absmax_bf16(w->wkv, (uint64_t)ctx->N * ctx->K, ctx->d_err + 3, 0);
    uint32_t res[3] = {0, 0, 0};
    if (e == cudaSuccess) e = cudaMemcpy(res, ctx->d_err + 1, sizeof res, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "bind scans");
    // a shard takes the whole table's exponent span from the caller
    const uint32_t smin = sh ? sh->scale_min : res[0], smax = sh ? sh->scale_max : res[1];
    const uint32_t wabs = res[2];
    // BF16 table rows are copied into BF16 operands (the fused kernels, which
    // decode MXFP8 in their producers, do not take them)
    const bool want_f16 = !(w->flags & ENGRAM_BIND_BF16_OPERANDS) && !tbf16;
    const bool scales_fit = smax != 255u && smax >= smin && smax - smin <= 22u;
    const bool w_finite = wabs < 0x7F80u;
    // the gate's pre-multiplied weights enter only as the product w_q w_k:
    // kept once per layer (read from the caller's arrays here, at bind)
    const int64_t nqk = (int64_t)ctx->desc.hc * ctx->desc.d;
    if (!L.wqk) {
        e = cudaMalloc(&L.wqk, nqk * sizeof(float));
        if (e != cudaSuccess) {
            L.wqk = nullptr;
            return fail(ENGRAM_ENOMEM, "cudaMalloc of the w_q w_k product");
        }
    }
    e = launch_mul_f32(w->wq, w->wk, L.wqk, nqk, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "w_q w_k product");
    if (L.wkv_f16) {
        cudaFree(L.wkv_f16);
        L.wkv_f16 = nullptr;
    }
    L.f16 = false;
    if (want_f16 && scales_fit && w_finite) {
        // exponent shift: all decoded values FP16-normal when the span allows
        const int shift = (smax - smin <= 12u) ? 122 - (int)smin : 112 - (int)smin;
        int wexp = 0;
        if (wabs) {
            uint32_t fb = wabs << 16;
            float maxabs;
            memcpy(&maxabs, &fb, sizeof maxabs);
            int ex;
            frexpf(maxabs, &ex);  // maxabs < 2^ex
            wexp = 15 - ex;
        }
        const size_t bytes = (size_t)ctx->N * ctx->K * sizeof(uint16_t);
        e = cudaMalloc(&L.wkv_f16, bytes);
        if (e != cudaSuccess) {
            L.wkv_f16 = nullptr;
            return fail(ENGRAM_ENOMEM, "cudaMalloc of the FP16 wkv copy");
        }
        // the copy is stored as 128 x 64 tiles, each 16 KB contiguous: one
        // tensor map over them, viewed as [N K / 64][64] with 128-row boxes,
        // feeds both the single-CTA (two boxes per stage) and the pair kernels
        e = launch_wkv_to_f16_tiles(w->wkv, L.wkv_f16, (uint64_t)ctx->N, (uint64_t)ctx->K,
                                    ldexpf(1.0f, wexp), 0);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e == cudaSuccess)
            e = make_tma_16bit(&L.tm_wkv_f16, L.wkv_f16, (uint64_t)ctx->N * ctx->K / kBK, kBK,
                               kBN / 2, true);
        if (e == cudaSuccess)
            e = make_tma_16bit(&L.tm_wkv_f16_2k, L.wkv_f16, (uint64_t)ctx->N * ctx->K / kBK, kBK,
                               kBN, true);
        if (e != cudaSuccess) {
            cudaFree(L.wkv_f16);
            L.wkv_f16 = nullptr;
            return cuda_fail(e, "FP16 wkv copy");
        }
        L.f16 = true;
        L.wkv_exp = wexp;
        L.a_exp_shift = shift;
    }
    // 256-wide rows are gathered whole, once per tile and bucket; other widths
    // per 64-column k-block.
    L.bucket_gather = L.f16 && ctx->desc.row_dim == 256;
    L.table_bf16 = tbf16;
    (void)host_table;
    L.scale_min = smin;
    L.scale_max = smax;
    L.w = bw;
    L.tm_wkv = tm;
    L.tm_wkv_half = tm_half;
    L.shard = sh != nullptr;
    L.row_lo = sh ? sh->row_lo : 0;
    L.shard_rows = sh ? w->rows : L.rows;
    L.bound = true;
    return ok();
}
}  // namespace

engram_status engram_layer_info(const engram_ctx* ctx, int layer, engram_layer_info_t* out) {
    engram_status st = check_layer(ctx, layer, false);
    if (st) return st;
    if (!out) return fail(ENGRAM_EINVAL, "null argument");
    const LayerState& L = ctx->layers[layer];
    out->rows = L.rows;
    out->bound = L.bound ? 1 : 0;
    out->fp16_operands = L.f16 ? 1 : 0;
    out->scale_min = L.scale_min;
    out->scale_max = L.scale_max;
    out->wkv_exp = L.wkv_exp;
    out->a_exp_shift = L.a_exp_shift;
    out->bucket_gather = L.bucket_gather ? 1 : 0;
    out->table_bf16 = L.table_bf16 ? 1 : 0;
    return ok();
}

engram_status engram_table_fill(const engram_ctx* ctx, uint64_t seed, uint8_t* data,
                                uint8_t* scale, uint64_t row_begin, uint64_t row_end,
                                void* stream) {
    if (!ctx || !data || !scale) return fail(ENGRAM_EINVAL, "null argument");
    if (row_end < row_begin) return fail(ENGRAM_EINVAL, "row_end < row_begin");
    if (!aligned16(data)) return fail(ENGRAM_EINVAL, "data must be 16-byte aligned");
    cudaError_t e = launch_table_fill(seed, data, scale, row_begin, row_end,
                                      (int)ctx->desc.row_dim, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "table fill launch");
    return ok();
}

engram_status engram_table_fill_bf16(const engram_ctx* ctx, uint64_t seed, uint16_t* data,
                                     uint64_t row_begin, uint64_t row_end, void* stream) {
    if (!ctx || !data) return fail(ENGRAM_EINVAL, "null argument");
    if (row_end < row_begin) return fail(ENGRAM_EINVAL, "row_end < row_begin");
    if (!aligned16(data)) return fail(ENGRAM_EINVAL, "data must be 16-byte aligned");
    cudaError_t e = launch_table_fill_bf16(seed, data, row_begin, row_end,
                                           (int)ctx->desc.row_dim, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "table fill launch");
    return ok();
}

// ---- host memory for a table read through UVA ----------------------------------------------

engram_status engram_host_table_alloc(uint64_t bytes, void** out) {
    if (!out || bytes == 0) return fail(ENGRAM_EINVAL, "bytes > 0 and an output pointer");
    *out = nullptr;
    // The mapping starts on a huge-page boundary (the transparent huge page
    // size the kernel reports, else 2 MB), so that every whole huge page of
    // the table can be one: the GPU translates random rows of a 100 GB table
    // far faster through huge pages.
    uint64_t huge = 2ull << 20;
    if (FILE* f = fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long v = 0;
        if (fscanf(f, "%llu", &v) == 1 && v >= 4096 && (v & (v - 1)) == 0 && v <= (1ull << 30))
            huge = v;
        fclose(f);
    }
    void* raw = mmap(nullptr, bytes + huge, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS,
                     -1, 0);
    if (raw == MAP_FAILED) return fail(ENGRAM_ENOMEM, "mmap of the host table");
    const uint64_t r0 = reinterpret_cast<uint64_t>(raw);
    const uint64_t a0 = (r0 + huge - 1) & ~(huge - 1);
    if (a0 > r0) munmap(raw, a0 - r0);
    const uint64_t page = (uint64_t)sysconf(_SC_PAGESIZE);
    const uint64_t tail = (a0 + bytes + page - 1) & ~(page - 1);  // first page past the table
    if (r0 + bytes + huge > tail) munmap(reinterpret_cast<void*>(tail), r0 + bytes + huge - tail);
    void* p = reinterpret_cast<void*>(a0);
    // a hint: the kernel may back the mapping with transparent huge pages
    // (ignored where it offers none)
    (void)madvise(p, bytes, MADV_HUGEPAGE);
    // touch every page, in parallel, before the registration pins them
    {
        const unsigned nt = std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
        const uint64_t chunk = (bytes + nt - 1) / nt;
        std::vector<std::thread> th;
        for (unsigned i = 0; i < nt; ++i) {
            const uint64_t lo = std::min<uint64_t>(bytes, i * chunk);
            const uint64_t hi = std::min<uint64_t>(bytes, lo + chunk);
            if (hi > lo)
                th.emplace_back([p, lo, hi] { memset(static_cast<char*>(p) + lo, 0, hi - lo); });
        }
        for (auto& t : th) t.join();
    }
    cudaError_t e = cudaHostRegister(p, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (e != cudaSuccess) {
        cudaGetLastError();
        munmap(p, bytes);
        return cuda_fail(e, "cudaHostRegister of the host table");
    }
    *out = p;
    return ok();
}

engram_status engram_host_table_free(void* p, uint64_t bytes) {
    if (!p) return ok();
    cudaError_t e = cudaHostUnregister(p);
    munmap(p, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostUnregister of the host table");
    return ok();
}

// ---- sessions ---------------------------------------------------------------------------

engram_status engram_session_create(engram_ctx* ctx, engram_session** out) {
    if (!ctx || !out) return fail(ENGRAM_EINVAL, "null argument");
    engram_session* s = new (std::nothrow) engram_session;
    if (!s) return fail(ENGRAM_ENOMEM, "host allocation");
    s->ctx = ctx;
    s->hist[0] = s->hist[1] = s->hist[2] = ctx->desc.pad_cid;
    s->count = 0;
    s->magic = kSessionMagic;
    *out = s;
    return ok();
}

static engram_status check_session(const engram_session* s) {
    if (!s) return fail(ENGRAM_EINVAL, "null session");
    if (s->magic != kSessionMagic) return fail(ENGRAM_ESTATE, "destroyed or invalid session");
    return ENGRAM_OK;
}

engram_status engram_session_fork(const engram_session* s, engram_session** out) {
    engram_status st = check_session(s);
    if (st) return st;
    if (!out) return fail(ENGRAM_EINVAL, "null argument");
    engram_session* c = new (std::nothrow) engram_session(*s);
    if (!c) return fail(ENGRAM_ENOMEM, "host allocation");
    *out = c;
    return ok();
}

engram_status engram_session_reset(engram_session* s) {
    engram_status st = check_session(s);
    if (st) return st;
    s->hist[0] = s->hist[1] = s->hist[2] = s->ctx->desc.pad_cid;
    s->count = 0;
    return ok();
}

engram_status engram_session_destroy(engram_session* s) {
    engram_status st = check_session(s);
    if (st) return st;
    s->magic = 0;
    delete s;
    return ok();
}

static inline void push(engram_session* s, uint32_t c, uint32_t* w) {
    w[0] = c;
    w[1] = s->hist[0];
    w[2] = s->hist[1];
    w[3] = s->hist[2];
    s->hist[2] = s->hist[1];
    s->hist[1] = s->hist[0];
    s->hist[0] = c;
    ++s->count;
}

engram_status engram_session_append(engram_session* s, const int32_t* tokens,
                                    const uint8_t* is_image, int64_t n, uint32_t* windows_out) {
    engram_status st = check_session(s);
    if (st) return st;
    if (n < 0) return fail(ENGRAM_EINVAL, "n < 0");
    if (n == 0) return ok();
    if (!tokens || !windows_out) return fail(ENGRAM_EINVAL, "null argument");
    const engram_ctx* ctx = s->ctx;
    for (int64_t i = 0; i < n; ++i) {
        if (is_image && is_image[i]) continue;
        if (tokens[i] < 0 || (uint32_t)tokens[i] >= ctx->desc.vocab)
            return fail(ENGRAM_EINVAL, "token id outside [0, vocab) at position " + std::to_string(i));
    }
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t c = (is_image && is_image[i]) ? ENGRAM_DEAD : ctx->map[(uint32_t)tokens[i]];
        push(s, c, windows_out + 4 * i);
    }
    return ok();
}

engram_status engram_batch_append(engram_session* const* sessions, const int32_t* tokens,
                                  const uint8_t* is_image, int64_t n, uint32_t* windows_out) {
    if (n < 0) return fail(ENGRAM_EINVAL, "n < 0");
    if (n == 0) return ok();
    if (!sessions || !tokens || !windows_out) return fail(ENGRAM_EINVAL, "null argument");
    for (int64_t i = 0; i < n; ++i) {
        engram_status st = check_session(sessions[i]);
        if (st) return st;
        if (i > 0 && sessions[i]->ctx != sessions[0]->ctx)
            return fail(ENGRAM_EINVAL, "sessions of different contexts");
        if (is_image && is_image[i]) continue;
        if (tokens[i] < 0 || (uint32_t)tokens[i] >= sessions[i]->ctx->desc.vocab)
            return fail(ENGRAM_EINVAL, "token id outside [0, vocab) at position " + std::to_string(i));
    }
    for (int64_t i = 0; i < n; ++i) {
        const engram_ctx* ctx = sessions[i]->ctx;
        const uint32_t c = (is_image && is_image[i]) ? ENGRAM_DEAD : ctx->map[(uint32_t)tokens[i]];
        push(sessions[i], c, windows_out + 4 * i);
    }
    return ok();
}

// ---- device steps ---------------------------------------------------------------------


size_t engram_workspace_bytes(const engram_ctx* ctx, int64_t T) {
    return forward_workspace_bytes(ctx, T, 8);
}

static engram_status hash_impl(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                               int64_t T, uint32_t* d_rows, bool bucket_major, void* stream) {
    engram_status st = check_layer(ctx, layer, false);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_windows || !d_rows || !aligned16(d_windows) || !aligned4(d_rows))
        return fail(ENGRAM_EINVAL, "windows (16-byte aligned) / rows (4-byte aligned)");
    cudaError_t e = launch_hash(hash_params(ctx, layer), reinterpret_cast<const uint4*>(d_windows), T,
                                d_rows, bucket_major, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "hash launch");
    return ok();
}

engram_status engram_hash(const engram_ctx* ctx, int layer, const uint32_t* d_windows, int64_t T,
                          uint32_t* d_rows, void* stream) {
    return hash_impl(ctx, layer, d_windows, T, d_rows, false, stream);
}

engram_status engram_hash_by_bucket(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                    int64_t T, uint32_t* d_rows_bm, void* stream) {
    return hash_impl(ctx, layer, d_windows, T, d_rows_bm, true, stream);
}

size_t engram_raw_row_bytes(const engram_ctx* ctx) {
    return ctx ? (size_t)ctx->desc.row_dim + 16 : 0;
}

engram_status engram_shard_gather_raw(const engram_ctx* ctx, int layer, const uint32_t* d_ids,
                                      int64_t n, uint8_t* d_raw, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st) return st;
    if (n < 0 || n > ((int64_t)1 << 31)) return fail(ENGRAM_EINVAL, "n must be in [0, 2^31]");
    if (n == 0) return ok();
    if (!d_ids || !d_raw || !aligned4(d_ids) || !aligned16(d_raw))
        return fail(ENGRAM_EINVAL, "ids (4-byte aligned) / raw (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    if (L.table_bf16) return fail(ENGRAM_EUNSUPPORTED, "raw rows are MXFP8 rows");
    if (L.shard_rows > 0 && !L.w.table) return fail(ENGRAM_ESTATE, "no table bound");
    cudaError_t e = launch_shard_gather_raw(d_ids, n, L.row_lo, L.shard_rows,
                                            (int)ctx->desc.row_dim, L.w.table, L.w.scales, d_raw,
                                            ctx->d_err, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "shard gather launch");
    return ok();
}

engram_status engram_gather_dequant(const engram_ctx* ctx, int layer, const uint32_t* d_rows,
                                    int64_t T, uint16_t* d_emb, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T)) || (st = check_full_table(ctx, layer))) return st;
    if (T == 0) return ok();
    if (!d_rows || !d_emb || !aligned4(d_rows) || !aligned16(d_emb))
        return fail(ENGRAM_EINVAL, "rows (4-byte aligned) / emb (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    cudaError_t e = launch_gather(geometry(ctx), d_rows, T, L.w.table, L.w.scales, L.rows,
                                  L.table_bf16, d_emb,
                                  ctx->d_err, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    return ok();
}

engram_status engram_project(const engram_ctx* ctx, int layer, const uint16_t* d_emb, int64_t T,
                             float* d_kv, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_emb || !d_kv || !aligned16(d_emb) || !aligned16(d_kv)) return fail(ENGRAM_EINVAL, "emb / kv");
    CUtensorMap tmA;
    cudaError_t e = make_tma_16bit(&tmA, d_emb, (uint64_t)T, (uint64_t)ctx->K, kBM, false);
    if (e != cudaSuccess) return cuda_fail(e, "emb tensor map");
    MmaArgs a = mma_args(ctx, layer, T);
    a.n_tile_begin = 0;
    a.n_tiles = ctx->N / kBN;
    a.kv = d_kv;
    a.ldkv = ctx->N;
    a.b_tiled = 0;  // the caller's BF16 wkv, row-major
    e = launch_project(a, tmA, ctx->layers[layer].tm_wkv, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "project launch");
    return ok();
}

engram_status engram_gate(const engram_ctx* ctx, int layer, const float* d_kv,
                          const uint32_t* d_windows, int64_t T, uint16_t* d_hidden,
                          float* d_gates, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_kv || !d_windows || !d_hidden || !aligned16(d_kv) || !aligned16(d_windows) ||
        !aligned16(d_hidden))
        return fail(ENGRAM_EINVAL, "kv / windows / hidden (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    cudaError_t e = launch_gate(geometry(ctx), d_kv, false, 1, 0,
                                reinterpret_cast<const uint4*>(d_windows), T, d_hidden, L.wqk,
                                d_gates, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "gate launch");
    return ok();
}


engram_status engram_forward(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                             int64_t T, uint16_t* d_hidden, void* d_workspace, float* d_gates,
                             void* stream) {
    return forward_fused(ctx, layer, d_windows, T, d_hidden, d_workspace, d_gates, stream, 8);
}

// A batch whose output tiles (128 tokens x 256 outputs) do not fill the GPU
// twice runs the staged GEMM with stream K: the launch's (tile, stage)
// sequence is cut into one contiguous range per CTA (or pair).  The pieces
// that finish key tiles publish the gate's sums and those that finish value
// tiles store v (kEpiForwardSk); a light kernel then makes the gates and
// updates hidden.  Nothing in the GEMM waits for gates: a value tile that
// waited for every key tile stalled its range's later MMAs (0.147 ms per
// decode step against 0.080 ms).
static bool staged_stream_k(const engram_ctx* ctx, int64_t T) {
    const int64_t tiles = (T + kBM - 1) / kBM * (ctx->N / kBN);
    return tiles < 2 * (int64_t)device_sm_count();
}

// Stream-K workspace after e: the gate sums f32 [T][hc][d/kBN][2][3]; v f32
// [T][d]; one 128 x 256 fp32 slot per CTA for the parked pieces; sixteen
// ready flags per CTA (one per epilogue warp), zeroed before every call.  The
// pre-pass (kv-store epilogue, kv in the caller's buffer) uses the slots and
// the flags only.
struct StreamKWs {
    size_t part, v, slots, flags;
    size_t total() const { return part + v + slots + flags; }
};
static StreamKWs stream_k_ws(const engram_ctx* ctx, int64_t T) {
    const size_t ctas = (size_t)device_sm_count();
    StreamKWs w;
    w.part = ((size_t)T * ctx->desc.hc * (ctx->desc.d / kBN) * 2 * 3 * sizeof(float) + 255) &
             ~(size_t)255;
    w.v = ((size_t)T * ctx->desc.d * sizeof(float) + 255) & ~(size_t)255;
    w.slots = ctas * kBM * kBN * sizeof(float);
    w.flags = (ctas * 16 * sizeof(uint32_t) + 255) & ~(size_t)255;
    return w;
}


// Bytes of the staged operand matrix e: whole 128-token blocks (the FP16
// operand is stored in 128 x 64 tiles).
static size_t staged_e_bytes(const engram_ctx* ctx, int64_t T) {
    const size_t rows = ((size_t)T + kBM - 1) / kBM * kBM;
    return (rows * ctx->K * sizeof(uint16_t) + 255) & ~(size_t)255;
}

size_t engram_forward_staged_workspace_bytes(const engram_ctx* ctx, int64_t T) {
    if (!ctx || T <= 0) return 0;
    const size_t e = staged_e_bytes(ctx, T);
    if (staged_stream_k(ctx, T)) return e + stream_k_ws(ctx, T).total();
    // the TMA-fed kernels run two epilogue warps per TMEM quadrant; then one
    // has-text flag per 128-token block
    return e + forward_workspace_bytes_groups(ctx, T, 8, 2) +
           ((((size_t)T + kBM - 1) / kBM * sizeof(uint32_t) + 255) & ~(size_t)255);
}

// The has-text flags of a large batch's blocks in its staged workspace (null
// for a small batch, whose stream-K GEMM skips nothing).
static uint32_t* staged_block_text(const engram_ctx* ctx, int64_t T, void* d_workspace) {
    if (staged_stream_k(ctx, T)) return nullptr;
    return reinterpret_cast<uint32_t*>(static_cast<char*>(d_workspace) + staged_e_bytes(ctx, T) +
                                       forward_workspace_bytes_groups(ctx, T, 8, 2));
}

// The stream-K flags a small batch's staging zeroes (null, 0 for a large one).
static void staged_clear(const engram_ctx* ctx, int64_t T, void* d_workspace, uint32_t*& clear,
                         int& n_clear) {
    clear = nullptr;
    n_clear = 0;
    char* const rest = static_cast<char*>(d_workspace) + staged_e_bytes(ctx, T);
    if (staged_stream_k(ctx, T)) {
        const StreamKWs w = stream_k_ws(ctx, T);
        clear = reinterpret_cast<uint32_t*>(rest + w.part + w.v + w.slots);
        n_clear = (int)(w.flags / sizeof(uint32_t));
    } else {  // the forward epilogue's counters
        const ForwardWs w = forward_ws(ctx, T, 8, 2);
        clear = reinterpret_cast<uint32_t*>(rest + w.part + w.gbuf);
        n_clear = (int)w.counter_words;
    }
}

engram_status engram_stage_raw_rows(const engram_ctx* ctx, int layer, const uint32_t* d_rows_bm,
                                    const uint8_t* d_raw_bm, int64_t T, void* d_workspace,
                                    void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_rows_bm || !d_raw_bm || !d_workspace || !aligned4(d_rows_bm) || !aligned16(d_raw_bm) ||
        !aligned16(d_workspace))
        return fail(ENGRAM_EINVAL, "rows / raw rows / workspace (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    if (L.table_bf16) return fail(ENGRAM_EUNSUPPORTED, "raw rows are MXFP8 rows");
    uint32_t* clear;
    int n_clear;
    staged_clear(ctx, T, d_workspace, clear, n_clear);
    cudaError_t e = launch_stage_raw(hash_params(ctx, layer), d_rows_bm, d_raw_bm, T,
                                     (int)ctx->desc.row_dim, L.f16, L.a_exp_shift,
                                     static_cast<uint16_t*>(d_workspace), ctx->d_err, clear,
                                     n_clear, nullptr, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "raw staging launch");
    return ok();
}

// Step 1 of the staged forward; flags: also write which 128-token blocks hold
// a text row, for a GEMM that compacts its units (the chunks of a long batch).
static engram_status stage_impl(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                int64_t T, void* d_workspace, void* stream, bool flags) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T)) || (st = check_full_table(ctx, layer))) return st;
    if (T == 0) return ok();
    if (!d_windows || !d_workspace || !aligned16(d_windows) || !aligned16(d_workspace))
        return fail(ENGRAM_EINVAL, "windows / workspace (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    // gather and dequantise every (token, bucket) row once into e; for a small
    // batch the same kernel zeroes the stream-K flags of the GEMM after it
    uint32_t* clear;
    int n_clear;
    staged_clear(ctx, T, d_workspace, clear, n_clear);
    cudaError_t e = launch_gather_stage(hash_params(ctx, layer),
                                        reinterpret_cast<const uint4*>(d_windows), T,
                                        (int)ctx->desc.row_dim, L.w.table, L.w.scales, L.rows,
                                        L.table_bf16, L.f16, L.a_exp_shift,
                                        static_cast<uint16_t*>(d_workspace), ctx->d_err, clear,
                                        n_clear,
                                        flags ? staged_block_text(ctx, T, d_workspace) : nullptr,
                                        (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "staged gather launch");
    return ok();
}

engram_status engram_stage_rows(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                int64_t T, void* d_workspace, void* stream) {
    return stage_impl(ctx, layer, d_windows, T, d_workspace, stream, false);
}

// The GEMM of the staged entry reading e through TMA: `a` with the layer's
// operand scaling, the A tensor map over e and the wkv map.  FP16: e is tiled;
// on CTA pairs each TMA box holds two k-blocks, otherwise one; BF16: e is
// row-major [T][K]; pairs from two 128-token blocks on (a single 128-token
// block runs on one CTA per tile: half of a pair would idle).
static cudaError_t staged_gemm(const engram_ctx* ctx, int layer, int64_t T, void* d_workspace,
                               MmaArgs& a, CUtensorMap& tmA, const CUtensorMap*& tmB,
                               bool& pairs) {
    const LayerState& L = ctx->layers[layer];
    uint16_t* e_scratch = static_cast<uint16_t*>(d_workspace);
    a = mma_args(ctx, layer, T);
    if (L.f16) {
        a.a_exp_shift = L.a_exp_shift;
        a.out_scale = ldexpf(1.0f, -(L.a_exp_shift + L.wkv_exp));
    }
    a.n_tile_begin = 0;
    a.n_tiles = ctx->N / kBN;
    const int KB = ctx->K / kBK;
    const bool two_k = L.f16 && a.m_blocks >= 2 && KB % 2 == 0;
    cudaError_t e;
    if (L.f16) {
        a.a_tiled = 1;
        e = make_tma_16bit(&tmA, e_scratch, (uint64_t)a.m_blocks * KB * kBM, kBK,
                           two_k ? 2 * kBM : kBM, true);
    } else {
        e = make_tma_16bit(&tmA, e_scratch, (uint64_t)T, (uint64_t)ctx->K, kBM, false);
    }
    // wkv: FP16 tiled (2-k-block boxes for pairs), or the caller's BF16
    pairs = L.f16 ? two_k : a.m_blocks >= 2;
    tmB = L.f16 ? (pairs ? &L.tm_wkv_f16_2k : &L.tm_wkv_f16) : (pairs ? &L.tm_wkv_half : &L.tm_wkv);
    return e;
}


// Step 2 of the staged forward; flags_clear: the stream-K flags of the
// workspace were zeroed earlier on the stream (else this call zeroes them);
// compact: the staging wrote the block flags, and the GEMM of a large batch
// runs only the M units that hold text.
static engram_status staged_rows(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                 int64_t T, uint16_t* d_hidden, void* d_workspace, float* d_gates,
                                 void* stream, bool flags_clear, bool compact);

engram_status engram_forward_staged_rows(const engram_ctx* ctx, int layer,
                                         const uint32_t* d_windows, int64_t T, uint16_t* d_hidden,
                                         void* d_workspace, float* d_gates, void* stream) {
    return staged_rows(ctx, layer, d_windows, T, d_hidden, d_workspace, d_gates, stream, false,
                       false);
}

static engram_status staged_rows(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                 int64_t T, uint16_t* d_hidden, void* d_workspace, float* d_gates,
                                 void* stream, bool flags_clear, bool compact) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_windows || !d_hidden || !d_workspace || !aligned16(d_windows) || !aligned16(d_hidden) ||
        !aligned16(d_workspace))
        return fail(ENGRAM_EINVAL, "windows / hidden / workspace (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    char* rest = static_cast<char*>(d_workspace) + staged_e_bytes(ctx, T);
    MmaArgs a;
    CUtensorMap tmA;
    const CUtensorMap* tmBp = nullptr;
    bool pairs = false;
    cudaError_t e = staged_gemm(ctx, layer, T, d_workspace, a, tmA, tmBp, pairs);
    if (e != cudaSuccess) return cuda_fail(e, "e tensor map");
    const CUtensorMap& tmB = *tmBp;
    a.windows = reinterpret_cast<const uint4*>(d_windows);
    a.hidden = d_hidden;
    a.gates = d_gates;
    cudaStream_t s = (cudaStream_t)stream;
    const bool small = staged_stream_k(ctx, T);
    if (small) {
        // small batch: stream K; key tiles publish the gate's sums, value tiles
        // store v; then the gates and hidden += g v
        const StreamKWs w = stream_k_ws(ctx, T);
        a.k_splits = 1;
        a.stream_k = 1;
        a.epi_groups = 2;
        a.key_tiles = (int)(ctx->desc.hc * ctx->desc.d / kBN);
        a.key_tail = 0;
        a.partials = reinterpret_cast<float*>(rest);
        a.kv = reinterpret_cast<float*>(rest + w.part);
        a.ldkv = ctx->desc.d;
        a.kv_bf16 = 0;
        a.kv_split_stride = 0;
        a.sk_slots = reinterpret_cast<float*>(rest + w.part + w.v);
        a.sk_flags = reinterpret_cast<uint32_t*>(rest + w.part + w.v + w.slots);
        if (!flags_clear) {
            e = cudaMemsetAsync(a.sk_flags, 0, w.flags, s);
            if (e != cudaSuccess) return cuda_fail(e, "stream-K flags");
        }
        e = launch_forward_sk(a, L.f16, pairs, tmA, tmB, s);
        if (e != cudaSuccess) return cuda_fail(e, "stream-K forward launch");
        e = launch_gate_sums(geometry(ctx), a.partials, 2, a.kv, a.windows, T, d_hidden, d_gates,
                             s);
        if (e != cudaSuccess) return cuda_fail(e, "gate launch");
        return ok();
    }
    e = forward_bind_ws(ctx, T, 8, 2, rest, a, s, !flags_clear);
    // the staging wrote which blocks hold text: the GEMM runs only the units
    // that hold some (a unit of image rows only passes through)
    a.block_text = compact ? staged_block_text(ctx, T, d_workspace) : nullptr;
    // the pair kernel finishes the key tiles M unit by M unit: a unit's value
    // tiles then find their gates ready (2,048 tokens: 0.417 -> 0.399 ms);
    // the fused kernel keeps the N-major order, which suits it better
    a.key_tail = 8;
    if (e != cudaSuccess) return cuda_fail(e, "forward counters");
    e = pairs ? launch_forward_tma_pair(a, L.f16, tmA, tmB, s)
              : launch_forward_tma(a, L.f16, tmA, tmB, s);
    if (e != cudaSuccess) return cuda_fail(e, "staged forward launch");
    return ok();
}

// Chunk of a long staged batch: a multiple of 256 tokens (a CTA-pair unit)
// from 3,072 to 6,144 (e of 36 to 72 MB, inside the 126 MB L2 beside the wkv
// stream), the one whose output tiles (units x N / 256) leave the least of a
// last wave idle on this device's CTA pairs; the smallest such on a tie.  On
// 152 SMs: 4,864 tokens, 19 units x 100 tiles = 25 waves of 76 pairs exactly
// (4,096 tokens gave 21 waves and 4 tiles).
static int64_t staged_chunk_tokens(const engram_ctx* ctx) {
    const int64_t pairs = std::max(1, device_sm_count() / 2);
    const int64_t nt = ctx->N / kBN;
    int64_t best = 4096, best_idle = -1;
    for (int64_t units = 12; units <= 24; ++units) {
        const int64_t tiles = units * nt;
        const int64_t idle = (pairs - tiles % pairs) % pairs;  // empty slots of the last wave
        // per tile of work, so that larger chunks are not favoured by size alone
        if (best_idle < 0 || idle * best / 256 < best_idle * units) {
            best = units * 256;
            best_idle = idle;
        }
    }
    return best;
}

engram_status engram_forward_staged(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                    int64_t T, uint16_t* d_hidden, void* d_workspace,
                                    float* d_gates, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_windows || !d_hidden || !d_workspace || !aligned16(d_windows) || !aligned16(d_hidden) ||
        !aligned16(d_workspace))
        return fail(ENGRAM_EINVAL, "windows / hidden / workspace (16-byte aligned)");
    // A long batch runs in chunks on the same workspace, so that each chunk's
    // operand matrix e (12 KB a token) stays in L2 between the gather that
    // writes it and the GEMM that reads it, instead of going through HBM; a
    // chunk's gather waits for the GEMM before it (as two calls in a row do)
    // before it overwrites e.
    // The chunks of a long batch also run only their M units that hold text
    // (units of image rows only pass through): their GEMMs wait for the
    // staging before loading wkv, which costs a few microseconds a chunk
    // against the whole units a long image span saves.  A batch of one chunk
    // (the 2,048-token prefill) keeps the early wkv loads.
    const int64_t chunk = staged_chunk_tokens(ctx);
    const bool compact = T > chunk;
    for (int64_t t0 = 0; t0 < T; t0 += chunk) {
        const int64_t n = std::min(chunk, T - t0);
        const uint32_t* w = d_windows + t0 * 4;
        uint16_t* h = d_hidden + t0 * (int64_t)ctx->desc.hc * ctx->desc.d;
        float* g = d_gates ? d_gates + t0 * (int64_t)ctx->desc.hc : nullptr;
        // the gather zeroes a small batch's stream-K flags, so that nothing stands
        // between the gather and the GEMM that it hands its rows to
        st = stage_impl(ctx, layer, w, n, d_workspace, stream, compact);
        if (st) return st;
        st = staged_rows(ctx, layer, w, n, h, d_workspace, g, stream, true, compact);
        if (st) return st;
    }
    return ok();
}

engram_status engram_prepass(const engram_ctx* ctx, int layer, const uint32_t* d_windows, int64_t T,
                             void* d_kv, int kv_format, void* d_workspace, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (kv_format != ENGRAM_KV_F32 && kv_format != ENGRAM_KV_BF16)
        return fail(ENGRAM_EINVAL, "kv_format must be ENGRAM_KV_F32 or ENGRAM_KV_BF16");
    if (T == 0) return ok();
    if (!d_windows || !d_kv || !d_workspace || !aligned16(d_windows) || !aligned16(d_kv) ||
        !aligned16(d_workspace))
        return fail(ENGRAM_EINVAL, "windows / kv / workspace (16-byte aligned)");
    cudaStream_t s = (cudaStream_t)stream;
    const bool small = staged_stream_k(ctx, T);
    cudaError_t e;
    // (the gather zeroes the stream-K flags, as in engram_forward_staged)
    st = engram_stage_rows(ctx, layer, d_windows, T, d_workspace, stream);
    if (st) return st;
    const LayerState& L = ctx->layers[layer];
    MmaArgs a;
    CUtensorMap tmA;
    const CUtensorMap* tmB = nullptr;
    bool pairs = false;
    e = staged_gemm(ctx, layer, T, d_workspace, a, tmA, tmB, pairs);
    if (e != cudaSuccess) return cuda_fail(e, "e tensor map");
    a.windows = reinterpret_cast<const uint4*>(d_windows);
    a.kv = static_cast<float*>(d_kv);
    a.ldkv = ctx->N;
    a.kv_bf16 = kv_format == ENGRAM_KV_BF16 ? 1 : 0;
    a.k_splits = 1;
    a.kv_split_stride = 0;
    if (small) {
        const StreamKWs w = stream_k_ws(ctx, T);
        char* rest = static_cast<char*>(d_workspace) + staged_e_bytes(ctx, T);
        a.stream_k = 1;
        a.sk_slots = reinterpret_cast<float*>(rest + w.part + w.v);
        a.sk_flags = reinterpret_cast<uint32_t*>(rest + w.part + w.v + w.slots);
    }
    e = pairs ? launch_project_tma_pair(a, L.f16, tmA, *tmB, s)
              : launch_project_tma(a, L.f16, tmA, *tmB, s);
    if (e != cudaSuccess) return cuda_fail(e, "pre-pass projection launch");
    return ok();
}

engram_status engram_gate_bf16kv(const engram_ctx* ctx, int layer, const uint16_t* d_kv,
                                 const uint32_t* d_windows, int64_t T, uint16_t* d_hidden,
                                 float* d_gates, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T))) return st;
    if (T == 0) return ok();
    if (!d_kv || !d_windows || !d_hidden || !aligned16(d_kv) || !aligned16(d_windows) ||
        !aligned16(d_hidden))
        return fail(ENGRAM_EINVAL, "kv / windows / hidden (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    cudaError_t e = launch_gate(geometry(ctx), d_kv, true, 1, 0,
                                reinterpret_cast<const uint4*>(d_windows), T, d_hidden, L.wqk,
                                d_gates, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "gate launch");
    return ok();
}

engram_status engram_project_windows(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                                     int64_t T, float* d_kv, void* stream) {
    engram_status st = check_layer(ctx, layer, true);
    if (st || (st = check_T(T)) || (st = check_full_table(ctx, layer))) return st;
    if (T == 0) return ok();
    if (!d_windows || !d_kv || !aligned16(d_windows) || !aligned16(d_kv))
        return fail(ENGRAM_EINVAL, "windows / kv (16-byte aligned)");
    const LayerState& L = ctx->layers[layer];
    if (L.table_bf16)
        return fail(ENGRAM_EUNSUPPORTED, "BF16-table layers: engram_gather_dequant + engram_project");
    MmaArgs a = mma_args(ctx, layer, T);
    a.windows = reinterpret_cast<const uint4*>(d_windows);
    a.kv = d_kv;
    a.ldkv = ctx->N;
    a.n_tile_begin = 0;
    a.n_tiles = ctx->N / kBN;
    if (L.f16) {
        a.a_exp_shift = L.a_exp_shift;
        a.out_scale = ldexpf(1.0f, -(L.a_exp_shift + L.wkv_exp));
    }
    cudaError_t e = launch_forward_phase(a, kEpiStoreKv, L.f16, L.bucket_gather,
                                         L.f16 ? L.tm_wkv_f16 : L.tm_wkv, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "fused projection launch");
    return ok();
}

engram_status engram_sync(const engram_ctx* ctx, void* stream) {
    if (!ctx) return fail(ENGRAM_EINVAL, "null context");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "asynchronous error");
    if (ctx->d_err) {
        uint32_t w = 0;
        e = cudaMemcpy(&w, ctx->d_err, sizeof w, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "error word read");
        if (w) {
            cudaMemset(ctx->d_err, 0, sizeof(uint32_t));
            if (w & kErrTimeout) return fail(ENGRAM_ETIMEOUT, "a kernel gave up a bounded wait");
            return fail(ENGRAM_EBOUNDS, "a kernel met a row index outside the table");
        }
    }
    return ok();
}

engram_status engram_ctx_set_wait_limit(engram_ctx* ctx, int64_t ns) {
    if (!ctx || ns < 1000) return fail(ENGRAM_EINVAL, "wait limit must be >= 1 us");
    ctx->wait_limit_ns = ns;
    return ok();
}

engram_status engram_debug_starve_operand(engram_ctx* ctx, int on) {
    if (!ctx) return fail(ENGRAM_EINVAL, "null context");
    ctx->starve_b = on ? 1 : 0;
    return ok();
}

const char* engram_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
