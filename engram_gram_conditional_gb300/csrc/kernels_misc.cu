// Table fill, hash, gather-dequant and the standalone gate (sm_103a).
//
// All four are bound by memory or latency, not arithmetic: grids are sized in
// multiples of the SM count with grid-stride loops, loads and stores are 8- or
// 16-byte vectors, and consecutive threads touch consecutive bytes.
#include <algorithm>

#include "device_common.cuh"

namespace engram {

namespace {

int g_sm_count = 0;

// SMs of the current device (of the first one asked about); 152, a GB300's
// count, when no device answers.
int sm_count() {
    if (g_sm_count == 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            g_sm_count = n;
        else
            return 152;
    }
    return g_sm_count;
}

int grid_for(int64_t items, int threads, int per_sm) {
    int64_t want = (items + threads - 1) / threads;
    int64_t cap = (int64_t)sm_count() * per_sm;
    return (int)std::max<int64_t>(1, std::min(want, cap));
}

// Philox4x32-10 (Salmon et al., SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

__device__ __forceinline__ uint32_t lane16(const uint4& o, int lane) {
    const uint32_t w = (lane >> 1) == 0 ? o.x : (lane >> 1) == 1 ? o.y : (lane >> 1) == 2 ? o.z : o.w;
    return (lane & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Table contents: code(row, col) from Philox counter (row, col / 8, 0) lane
// col % 8, uniform over the 254 finite E4M3 codes; scale(row, g) from counter
// (row, 0, 1) lane g, E8M0 exponent uniform over 119..127.
// One thread per (row, 8-column chunk); chunk 0 also writes the row's scales.
__global__ void k_table_fill(uint64_t seed, uint8_t* __restrict__ data,
                             uint8_t* __restrict__ scale, uint64_t row_begin, uint64_t nrows,
                             int row_dim) {
    const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    const int cpr = row_dim / 8;
    const int groups = row_dim / 32;
    const uint64_t items = nrows * (uint64_t)cpr;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < items;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t row = row_begin + i / cpr;
        const uint32_t chunk = (uint32_t)(i % cpr);
        const uint4 o = philox4x32_10(make_uint4((uint32_t)row, (uint32_t)(row >> 32), chunk, 0u),
                                      k0, k1);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int l = 0; l < 8; ++l) {
            const uint32_t idx = (lane16(o, l) * 254u) >> 16;
            const uint32_t code = idx < 127u ? idx : idx + 1u;
            w[l >> 2] |= code << (8 * (l & 3));
        }
        *reinterpret_cast<uint2*>(data + row * (uint64_t)row_dim + chunk * 8u) = make_uint2(w[0], w[1]);
        if (chunk == 0) {
            const uint4 s = philox4x32_10(make_uint4((uint32_t)row, (uint32_t)(row >> 32), 0u, 1u),
                                          k0, k1);
            uint8_t* dst = scale + row * (uint64_t)groups;
            for (int g = 0; g < groups; ++g) dst[g] = (uint8_t)(119u + ((lane16(s, g) * 9u) >> 16));
        }
    }
}

// The same table stored as BF16 rows without scales: every value is the
// dequantised MXFP8 value E4M3(code) x 2^(scale - 127), which BF16 holds
// exactly, so a BF16-table layer computes the same forward as the MXFP8 one.
__global__ void k_table_fill_bf16(uint64_t seed, uint16_t* __restrict__ data, uint64_t row_begin,
                                  uint64_t nrows, int row_dim) {
    const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    const int cpr = row_dim / 8;
    const uint64_t items = nrows * (uint64_t)cpr;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < items;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t row = row_begin + i / cpr;
        const uint32_t chunk = (uint32_t)(i % cpr);
        const uint4 o = philox4x32_10(make_uint4((uint32_t)row, (uint32_t)(row >> 32), chunk, 0u),
                                      k0, k1);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int l = 0; l < 8; ++l) {
            const uint32_t idx = (lane16(o, l) * 254u) >> 16;
            const uint32_t code = idx < 127u ? idx : idx + 1u;
            w[l >> 2] |= code << (8 * (l & 3));
        }
        const uint4 sv = philox4x32_10(make_uint4((uint32_t)row, (uint32_t)(row >> 32), 0u, 1u),
                                       k0, k1);
        const uint32_t se = 119u + ((lane16(sv, (int)(chunk / 4)) * 9u) >> 16);
        *reinterpret_cast<uint4*>(data + row * (uint64_t)row_dim + chunk * 8u) =
            decode8(w[0], w[1], e8m0_to_f32(se));
    }
}

// a2: one thread per (token, bucket).
__global__ void k_hash(const __grid_constant__ HashParams hp, const uint4* __restrict__ windows,
                       int64_t T, uint32_t* __restrict__ rows, int bucket_major) {
    const int64_t items = T * hp.nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / hp.nb;
        const int b = (int)(i - t * hp.nb);
        rows[bucket_major ? b * T + t : i] = hash_bucket(hp, windows[t], b);
    }
}

// Owner side of a table sharded over ranks by bucket: the raw MXFP8 rows of
// the n global row ids a rank received.  A raw row is row_dim + 16 bytes: the
// row_dim E4M3 codes, then its row_dim / 32 E8M0 scale bytes, zero-padded to
// 16.  One thread per 16-byte chunk.  The shard holds rows [row_lo, row_lo +
// nrows); a masked id gives a zero row; an id outside the shard gives a zero
// row and sets the error word.
__global__ void k_shard_gather_raw(const uint32_t* __restrict__ ids, int64_t n, uint64_t row_lo,
                                   uint64_t nrows, int row_dim, const uint8_t* __restrict__ table,
                                   const uint8_t* __restrict__ scales, uint8_t* __restrict__ raw,
                                   uint32_t* err) {
    const int cpr = row_dim / 16;  // code chunks; chunk cpr holds the scales
    const int64_t items = n * (int64_t)(cpr + 1);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / (cpr + 1);
        const int j = (int)(i - r * (cpr + 1));
        const uint32_t id = ids[r];
        bool ok = id != kMasked;
        const uint64_t local = (uint64_t)id - row_lo;
        if (ok && ((uint64_t)id < row_lo || local >= nrows)) {
            if (j == 0) atomicOr(err, kErrBounds);
            ok = false;
        }
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ok && j < cpr) {
            v = __ldg(reinterpret_cast<const uint4*>(table + local * row_dim) + j);
        } else if (ok) {
            uint32_t w[4] = {0, 0, 0, 0};
            const uint8_t* s = scales + local * (row_dim / 32);
            for (int k = 0; k < row_dim / 32; ++k) w[k >> 2] |= (uint32_t)__ldg(s + k) << (8 * (k & 3));
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        reinterpret_cast<uint4*>(raw + r * (int64_t)(row_dim + 16))[j] = v;
    }
}

// a3: one thread per 16 columns of one (token, bucket) row: a 16-byte load of
// codes, one scale byte, two 16-byte stores of BF16.
// With table_bf16 the table holds BF16 rows (row_dim x 2 bytes, no scales)
// and the decode is a copy.
__global__ void k_gather(const uint32_t* __restrict__ rows, int64_t T, int nb, int row_dim,
                         const uint8_t* __restrict__ table, const uint8_t* __restrict__ scales,
                         uint64_t nrows, int table_bf16, uint16_t* __restrict__ emb,
                         uint32_t* err) {
    const int cpr = row_dim / 16;
    const int groups = row_dim / 32;
    const int64_t items = T * nb * (int64_t)cpr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tb = i / cpr;  // token * nb + bucket
        const int chunk = (int)(i - tb * cpr);
        uint32_t row = rows[tb];
        uint4 out0 = make_uint4(0, 0, 0, 0), out1 = out0;
        if (row != kMasked && row >= nrows) {
            atomicOr(err, kErrBounds);
            row = kMasked;
        }
        if (row != kMasked && table_bf16) {
            const uint4* src = reinterpret_cast<const uint4*>(table + (uint64_t)row * row_dim * 2) + chunk * 2;
            out0 = __ldg(src);
            out1 = __ldg(src + 1);
        } else if (row != kMasked) {
            const uint4 c = __ldg(reinterpret_cast<const uint4*>(table + (uint64_t)row * row_dim) + chunk);
            const float sf = e8m0_to_f32(__ldg(scales + (uint64_t)row * groups + chunk / 2));
            out0 = decode8(c.x, c.y, sf);
            out1 = decode8(c.z, c.w, sf);
        }
        uint4* dst = reinterpret_cast<uint4*>(emb + tb * (int64_t)row_dim) + chunk * 2;
        dst[0] = out0;
        dst[1] = out1;
    }
}

// Staged forward, step 1: windows -> dequantised operand rows in a scratch
// matrix e (FP16 scaled by 2^(s - 127 + exp_shift) in 128 x 64 tiles, or BF16
// row-major [T][K]).  Each table
// row is read whole: row_dim / 16 lanes per row, 16 codes and their scale per
// lane; the first lane of a row hashes its (token, bucket) pair.
// Launched as a programmatic dependent: the hashing and the row loads (of
// windows and table, which no kernel of the stream writes) may overlap the
// kernel before; every thread waits for it (pdl_wait) before its first store,
// since e may still be read by the GEMM of the previous call.  Block 0 then
// also zeroes n_clear words at `clear` (the stream-K flags of the GEMM after).
// kRaw: the rows come not from the table but from raw MXFP8 rows that the
// ranks owning their buckets returned (k_shard_gather_raw), bucket-major:
// row (t, b) at raw + (b T + t) (row_dim + 16); rows_bm [nb][T] are the
// requester's own row indices, which mark the masked rows.  A raw scale that
// the FP16 operand cannot take (outside the layer's bound exponent span)
// gives a zero row and sets the error word.
template <bool kF16, bool kRaw>
__global__ void k_gather_stage(const __grid_constant__ HashParams hp, const uint4* __restrict__ windows,
                               int64_t T, int row_dim, const uint8_t* __restrict__ table,
                               const uint8_t* __restrict__ scales, uint64_t nrows, int exp_shift,
                               int table_bf16, uint16_t* __restrict__ e, uint32_t* err,
                               uint32_t* __restrict__ clear, int n_clear,
                               const uint32_t* __restrict__ rows_bm, const uint8_t* __restrict__ raw,
                               uint32_t* __restrict__ block_text) {
    // the GEMM that reads e may start its prologue as soon as every CTA of
    // this grid runs (it waits for this grid's end before reading e)
    pdl_launch_dependents();
    if (blockIdx.x == 0 && n_clear > 0) {
        pdl_wait();
        for (int i = threadIdx.x; i < n_clear; i += blockDim.x) clear[i] = 0u;
    }
    bool waited = false;
    const int lpr = row_dim / 16;              // lanes per row
    const int rpw = 32 / lpr;                  // rows per warp pass
    const int lane = threadIdx.x & 31;
    const int sub = lane / lpr, chunk = lane % lpr;
    const int K = hp.nb * row_dim;
    const int64_t items = T * hp.nb;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp0 * rpw; base < items; base += nwarps * rpw) {
        const int64_t item = base + sub;
        const bool live_item = item < items;
        const int64_t t = live_item ? item / hp.nb : 0;
        const int b = live_item ? (int)(item - t * hp.nb) : 0;
        uint32_t row = kMasked;
        if (live_item && chunk == 0) {
            if (kRaw) {
                row = rows_bm[b * T + t];
            } else {
                row = hash_bucket(hp, windows[t], b);
                if (row != kMasked && (uint64_t)row >= nrows) {
                    atomicOr(err, kErrBounds);
                    row = kMasked;
                }
            }
        }
        row = __shfl_sync(0xFFFFFFFFu, row, sub * lpr);
        if (!live_item) continue;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (row != kMasked && !kF16 && !kRaw && table_bf16) {  // BF16 rows: a copy
            const uint4* src = reinterpret_cast<const uint4*>(table + (uint64_t)row * row_dim * 2) + chunk * 2;
            lo = __ldg(src);
            hi = __ldg(src + 1);
        } else if (row != kMasked) {
            uint4 c;
            uint32_t se;
            if (kRaw) {
                const uint8_t* rr = raw + (b * T + t) * (int64_t)(row_dim + 16);
                c = __ldg(reinterpret_cast<const uint4*>(rr) + chunk);
                se = __ldg(rr + row_dim + chunk / 2);
            } else {
                c = __ldg(reinterpret_cast<const uint4*>(table + (uint64_t)row * row_dim) + chunk);
                se = __ldg(scales + (uint64_t)row * (row_dim / 32) + chunk / 2);
            }
            int ex = (int)se - 127 + exp_shift;  // in [-24, 15] for a bound table (its scan)
            if (kF16 && kRaw && (ex < -24 || ex > 15)) {
                atomicOr(err, kErrBounds);
                c = make_uint4(0, 0, 0, 0);
                ex = 0;
            }
            if (kF16) {
                const uint32_t h = ex >= -14 ? (uint32_t)(ex + 15) << 10 : 1u << (ex + 24);
                const uint32_t sc2 = h | (h << 16);
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
                uint32_t o[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    asm("{\n\t.reg .b16 l, h;\n\t.reg .b32 a, b;\n\tmov.b32 {l, h}, %2;\n\t"
                        "cvt.rn.f16x2.e4m3x2 a, l;\n\tcvt.rn.f16x2.e4m3x2 b, h;\n\t"
                        "mul.rn.f16x2 %0, a, %3;\n\tmul.rn.f16x2 %1, b, %3;\n\t}"
                        : "=r"(o[2 * q]), "=r"(o[2 * q + 1])
                        : "r"(w[q]), "r"(sc2));
                }
                lo = make_uint4(o[0], o[1], o[2], o[3]);
                hi = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
                const float sf = e8m0_to_f32(se);
                lo = decode8(c.x, c.y, sf);
                hi = decode8(c.z, c.w, sf);
            }
        }
        if (!waited) {
            pdl_wait();
            waited = true;
        }
        // column k of row t: row-major, or (kF16) in 128 x 64 tiles, tile
        // (t / 128) (K / 64) + k / 64, so that two k-blocks of a 128-token
        // block are 32 contiguous KB (one TMA box)
        const int64_t k = (int64_t)b * row_dim + 16 * chunk;
        const int64_t off = kF16 ? ((((t >> 7) * (K >> 6) + (k >> 6)) << 7) + (t & 127)) * 64 + (k & 63)
                                 : t * (int64_t)K + k;
        uint4* dst = reinterpret_cast<uint4*>(e + off);
        dst[0] = lo;
        dst[1] = hi;
    }
    // Per 128-token block: does it hold a text row?  The GEMM after this skips
    // the units whose blocks hold only image rows.  Raw rows carry no image
    // marks: every block counts as text.  (Written after the wait: the GEMM
    // before may still read the flags.)
    if (block_text) {
        if (!waited) pdl_wait();
        const int64_t nblk = (T + 127) / 128;
        for (int64_t mb = warp0; mb < nblk; mb += nwarps) {
            bool text = kRaw;
            if (!kRaw)
                for (int r = lane; r < 128; r += 32) {
                    const int64_t t = mb * 128 + r;
                    if (t < T && windows[t].x != kDead) text = true;
                }
            text = __any_sync(0xFFFFFFFFu, text);
            if (lane == 0) block_text[mb] = text ? 1u : 0u;
        }
    }
}

// a5 standalone.  kv may be the sum of nsplit partial buffers split_stride
// floats apart (a projection split over K), added in split order.
constexpr int kGateMaxSplits = 8;

__device__ __forceinline__ float4 kv_sum4(const float4* p, int nsplit, int64_t stride4) {
    float4 x = __ldcg(p);
#pragma unroll
    for (int sp = 1; sp < kGateMaxSplits; ++sp)
        if (sp < nsplit) {
            const float4 y = __ldcg(p + sp * stride4);
            x.x += y.x;
            x.y += y.y;
            x.z += y.z;
            x.w += y.w;
        }
    return x;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Four kv values at float4 index i of a row: fp32 (the sum of nsplit split
// buffers, stride4 float4 apart), or BF16 (a single buffer).
template <bool kBf16>
__device__ __forceinline__ float4 kv_load4(const void* row, int64_t i, int nsplit, int64_t stride4) {
    if constexpr (kBf16) {
        const uint2 u = __ldcg(reinterpret_cast<const uint2*>(row) + i);
        return make_float4(bf16_bits_to_f32(u.x & 0xFFFFu), bf16_bits_to_f32(u.x >> 16),
                           bf16_bits_to_f32(u.y & 0xFFFFu), bf16_bits_to_f32(u.y >> 16));
    } else {
        return kv_sum4(reinterpret_cast<const float4*>(row) + i, nsplit, stride4);
    }
}

// One CTA per (token, branch b).  Pass 1 reduces sum k^2, sum h^2 and
// sum h w_q w_k k over the branch's d columns (float4 loads, then a
// fixed-order block reduction) into the gate;
// pass 2 applies h_b += g_b v with one BF16 rounding.  The branches of a token
// are separate CTAs (each reads v itself), so no pass waits on another branch
// and a batch of T tokens gives T hc CTAs of two short passes each.  Image
// rows (c_t == DEAD) are left untouched.
constexpr int kGateBranchThreads = 256;

// The gate's second half after the stream-K GEMM whose key tiles published
// their sums (Σk², Σh², Σh w_q w_k k per (token, branch, column tile, epilogue
// group)) and whose value tiles stored v [T][d].  CTA (t, part) takes
// kGateSumsCols float4 columns of token t for every branch: it turns the
// branch sums into gates (added in (tile, group) order, as the whole-tile gate
// epilogue adds them), then hidden_b += g_b v with one BF16 rounding, v read
// once for all branches.  Image rows pass through.  Every load is issued at
// once: the thread's v and hidden columns, and all of the token's sums
// (hc x d / 256 x groups x 3 floats, staged in shared memory by the whole CTA)
// before the gates are added up, so the kernel waits for memory about once.
// Small CTAs of two float4 columns a thread: a decode batch (256 tokens, d =
// 5,120) is 1,280 CTAs, all resident at once (nine per SM).  kMaxHc bounds
// hc, so that a thread holds registers for the branches there are.
constexpr int kGateSumsThreads = 128;
constexpr int kGateSumsPer = 2;  // float4 columns a thread
constexpr int kGateSumsCols = kGateSumsThreads * kGateSumsPer;
template <int kMaxHc>
__global__ void __launch_bounds__(kGateSumsThreads, 9)
k_gate_sums(const float* __restrict__ partials, int groups, const float* __restrict__ v,
            const uint4* __restrict__ windows, int hc, int d, float eps, int parts,
            uint16_t* __restrict__ hidden, float* __restrict__ gates) {
    extern __shared__ float sums[];  // [hc][P][3] of this token
    __shared__ float gsh[8];
    pdl_wait();  // launched to overlap the end of the GEMM that writes the sums and v
    pdl_launch_dependents();
    const int64_t t = blockIdx.x / parts;
    const int part = (int)(blockIdx.x - t * parts);
    if (windows[t].x == kDead) {
        if (gates && part == 0 && (int)threadIdx.x < hc) gates[t * hc + threadIdx.x] = 0.0f;
        return;
    }
    const int n4 = d / 4;
    uint2* const ht = reinterpret_cast<uint2*>(hidden + t * hc * (int64_t)d);
    const float4* const vt = reinterpret_cast<const float4*>(v + t * (int64_t)d);
    float4 vi[kGateSumsPer];
    uint2 h2[kGateSumsPer][kMaxHc];
#pragma unroll
    for (int c = 0; c < kGateSumsPer; ++c) {
        const int i = part * kGateSumsCols + c * kGateSumsThreads + (int)threadIdx.x;
        if (i < n4) {
            vi[c] = __ldcg(vt + i);
#pragma unroll
            for (int b = 0; b < kMaxHc; ++b)
                if (b < hc) h2[c][b] = ht[(int64_t)b * n4 + i];
        }
    }
    const int P = d / 256 * groups;
    const int nsum = hc * P * 3;
    const float* pt = partials + t * (int64_t)nsum;
    for (int k = threadIdx.x; k < nsum; k += kGateSumsThreads) sums[k] = __ldcg(pt + k);
    __syncthreads();
    if ((int)threadIdx.x < hc) {  // (column tile, group) order, as the whole-tile epilogue adds them
        const float* pp = sums + threadIdx.x * P * 3;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f;
        for (int p = 0; p < P; ++p) {
            s0 += pp[3 * p];
            s1 += pp[3 * p + 1];
            s2 += pp[3 * p + 2];
        }
        const float g = gate_from_sums(s0, s1, s2, d, eps);
        gsh[threadIdx.x] = g;
        if (gates && part == 0) gates[t * hc + threadIdx.x] = g;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kGateSumsPer; ++c) {
        const int i = part * kGateSumsCols + c * kGateSumsThreads + (int)threadIdx.x;
        if (i >= n4) continue;
#pragma unroll
        for (int b = 0; b < kMaxHc; ++b)
            if (b < hc) {
                const float g = gsh[b];
                const float o0 = fmaf(g, vi[c].x, bf16_bits_to_f32(h2[c][b].x & 0xFFFFu));
                const float o1 = fmaf(g, vi[c].y, bf16_bits_to_f32(h2[c][b].x >> 16));
                const float o2 = fmaf(g, vi[c].z, bf16_bits_to_f32(h2[c][b].y & 0xFFFFu));
                const float o3 = fmaf(g, vi[c].w, bf16_bits_to_f32(h2[c][b].y >> 16));
                ht[(int64_t)b * n4 + i] = make_uint2(bf16x2_pack_rn(o0, o1), bf16x2_pack_rn(o2, o3));
            }
    }
}

// Thirty-two registers a thread (eight CTAs per SM): latency is hidden by
// resident CTAs rather than by loads in flight per thread.  kv is fp32, or
// BF16 (kBf16Kv: the pre-pass's rounded kv).
template <bool kBf16Kv>
__global__ void __launch_bounds__(kGateBranchThreads, 8)
k_gate_branch(const void* __restrict__ kv, int nsplit, int64_t split_stride,
              const uint4* __restrict__ windows, int hc, int d, float eps,
              uint16_t* __restrict__ hidden, const float* __restrict__ wqk,
              float* __restrict__ gates) {
    __shared__ float red[kGateBranchThreads / 32][3];
    __shared__ float gsh;
    pdl_wait();  // launched to overlap the end of the projection that writes kv
    // the next call's gather may start hashing and loading rows meanwhile
    pdl_launch_dependents();
    const int64_t t = blockIdx.x / hc;
    const int b = (int)(blockIdx.x - t * hc);
    if (windows[t].x == kDead) {
        if (gates && threadIdx.x == 0) gates[t * hc + b] = 0.0f;
        return;
    }
    const int n4 = d / 4;
    const int64_t stride4 = split_stride / 4;
    const size_t kv_elem = kBf16Kv ? 2 : 4;
    const char* kvt = static_cast<const char*>(kv) + t * (int64_t)(hc + 1) * d * kv_elem;
    const char* kb = kvt + (int64_t)b * d * kv_elem;
    const char* vb = kvt + (int64_t)hc * d * kv_elem;
    uint2* hb = reinterpret_cast<uint2*>(hidden + (t * hc + b) * (int64_t)d);
    const float4* qkb = reinterpret_cast<const float4*>(wqk + (int64_t)b * d);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float skk = 0.f, shh = 0.f, shk = 0.f;
#pragma unroll 1
    for (int i = threadIdx.x; i < n4; i += kGateBranchThreads) {
        const float4 k = kv_load4<kBf16Kv>(kb, i, nsplit, stride4);
        const uint2 h2 = hb[i];
        const float4 qk = __ldg(qkb + i);
        const float h[4] = {bf16_bits_to_f32(h2.x & 0xFFFFu), bf16_bits_to_f32(h2.x >> 16),
                            bf16_bits_to_f32(h2.y & 0xFFFFu), bf16_bits_to_f32(h2.y >> 16)};
        const float kk[4] = {k.x, k.y, k.z, k.w};
        const float qw[4] = {qk.x, qk.y, qk.z, qk.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            skk += kk[e] * kk[e];
            shh += h[e] * h[e];
            shk += h[e] * qw[e] * kk[e];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        skk += __shfl_xor_sync(0xFFFFFFFFu, skk, o);
        shh += __shfl_xor_sync(0xFFFFFFFFu, shh, o);
        shk += __shfl_xor_sync(0xFFFFFFFFu, shk, o);
    }
    if (lane == 0) {
        red[warp][0] = skk;
        red[warp][1] = shh;
        red[warp][2] = shk;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f;
        for (int w = 0; w < kGateBranchThreads / 32; ++w) {
            a0 += red[w][0];
            a1 += red[w][1];
            a2 += red[w][2];
        }
        const float g = gate_from_sums(a0, a1, a2, d, eps);
        gsh = g;
        if (gates) gates[t * hc + b] = g;
    }
    __syncthreads();
    const float g = gsh;
#pragma unroll 1
    for (int i = threadIdx.x; i < n4; i += kGateBranchThreads) {
        const float4 vi = kv_load4<kBf16Kv>(vb, i, nsplit, stride4);
        const uint2 h2 = hb[i];
        const float o0 = fmaf(g, vi.x, bf16_bits_to_f32(h2.x & 0xFFFFu));
        const float o1 = fmaf(g, vi.y, bf16_bits_to_f32(h2.x >> 16));
        const float o2 = fmaf(g, vi.z, bf16_bits_to_f32(h2.y & 0xFFFFu));
        const float o3 = fmaf(g, vi.w, bf16_bits_to_f32(h2.y >> 16));
        hb[i] = make_uint2(bf16x2_pack_rn(o0, o1), bf16x2_pack_rn(o2, o3));
    }
}

// Bind-time scans and the FP16 copy of wkv.
__global__ void k_scale_range(const uint8_t* __restrict__ s, uint64_t n, uint32_t* out) {
    uint32_t lo = 255u, hi = 0u;
    const uint64_t tid = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    // bytes up to the first 16-byte boundary one by one, then 16 at a time,
    // then the tail one by one (s may start anywhere)
    const uint64_t head = min(n, (uint64_t)((16u - ((uintptr_t)s & 15u)) & 15u));
    for (uint64_t i = tid; i < head; i += stride) {
        lo = min(lo, (uint32_t)s[i]);
        hi = max(hi, (uint32_t)s[i]);
    }
    const uint64_t nv = (n - head) / 16;
    const uint4* sv = reinterpret_cast<const uint4*>(s + head);
    for (uint64_t i = tid; i < nv; i += stride) {
        const uint4 v = __ldg(sv + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t b = (w[k >> 2] >> (8 * (k & 3))) & 0xFFu;
            lo = min(lo, b);
            hi = max(hi, b);
        }
    }
    for (uint64_t i = head + nv * 16 + tid; i < n; i += stride) {
        lo = min(lo, (uint32_t)s[i]);
        hi = max(hi, (uint32_t)s[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicMin(out, lo);
        atomicMax(out + 1, hi);
    }
}

__global__ void k_absmax_bf16(const uint16_t* __restrict__ x, uint64_t n, uint32_t* out) {
    uint32_t m = 0;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x)
        m = max(m, (uint32_t)(x[i] & 0x7FFFu));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}

// FP16 copy of wkv [N][K] in 128 x 64 tiles: the tile of rows [128 nb, 128 nb
// + 128) and columns [64 kb, 64 kb + 64) is 16 KB of contiguous row-major
// memory at tile index nb (K / 64) + kb.  A TMA box of one tile then reads
// 16 contiguous KB instead of 128 rows of 128 bytes spread over 1.5 MB.
__global__ void k_wkv_to_f16_tiles(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                   uint64_t N, uint64_t K, float scale) {
    const uint64_t n_el = N * K, KB = K / 64;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n_el;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t n = i / K, k = i - n * K;
        const uint64_t o = (((n >> 7) * KB + (k >> 6)) * 128 + (n & 127)) * 64 + (k & 63);
        const float v = __uint_as_float((uint32_t)src[i] << 16) * scale;
        dst[o] = __half_as_ushort(__float2half_rn(v));
    }
}

}  // namespace

cudaError_t launch_table_fill_bf16(uint64_t seed, uint16_t* data, uint64_t row_begin,
                                   uint64_t row_end, int row_dim, cudaStream_t s) {
    const uint64_t nrows = row_end - row_begin;
    if (nrows == 0) return cudaSuccess;
    const int threads = 256;
    const int grid = grid_for((int64_t)std::min<uint64_t>(nrows * (row_dim / 8), 1ull << 40),
                              threads, 16);
    k_table_fill_bf16<<<grid, threads, 0, s>>>(seed, data, row_begin, nrows, row_dim);
    return cudaGetLastError();
}

cudaError_t launch_table_fill(uint64_t seed, uint8_t* data, uint8_t* scale, uint64_t row_begin,
                              uint64_t row_end, int row_dim, cudaStream_t s) {
    const uint64_t nrows = row_end - row_begin;
    if (nrows == 0) return cudaSuccess;
    const int threads = 256;
    const int grid = grid_for((int64_t)std::min<uint64_t>(nrows * (row_dim / 8), 1ull << 40),
                              threads, 16);
    k_table_fill<<<grid, threads, 0, s>>>(seed, data, scale, row_begin, nrows, row_dim);
    return cudaGetLastError();
}

cudaError_t launch_hash(const HashParams& hp, const uint4* windows, int64_t T, uint32_t* rows,
                        bool bucket_major, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    k_hash<<<grid_for(T * hp.nb, threads, 8), threads, 0, s>>>(hp, windows, T, rows,
                                                               bucket_major ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_gather(const Geometry& g, const uint32_t* rows, int64_t T,
                          const uint8_t* table, const uint8_t* scales, uint64_t nrows,
                          bool table_bf16, uint16_t* emb, uint32_t* err, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t items = T * g.nb * (int64_t)(g.row_dim / 16);
    k_gather<<<grid_for(items, threads, 16), threads, 0, s>>>(rows, T, g.nb, g.row_dim, table,
                                                              scales, nrows, table_bf16 ? 1 : 0,
                                                              emb, err);
    return cudaGetLastError();
}

cudaError_t launch_gate(const Geometry& g, const void* kv, bool kv_bf16, int nsplit,
                        int64_t split_stride, const uint4* windows, int64_t T, uint16_t* hidden,
                        const float* wqk, float* gates, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (nsplit < 1 || nsplit > kGateMaxSplits || g.d % 4 != 0 || g.hc > 8 || (kv_bf16 && nsplit != 1))
        return cudaErrorInvalidValue;
    if (T * g.hc > INT32_MAX) return cudaErrorInvalidValue;
    // programmatic dependent launch: the CTAs are scheduled while the kernel
    // before them drains, and wait for it in pdl_wait
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(T * g.hc));
    cfg.blockDim = dim3(kGateBranchThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (kv_bf16)
        return cudaLaunchKernelEx(&cfg, k_gate_branch<true>, kv, nsplit, split_stride, windows,
                                  g.hc, g.d, g.eps, hidden, wqk, gates);
    return cudaLaunchKernelEx(&cfg, k_gate_branch<false>, kv, nsplit, split_stride, windows, g.hc,
                              g.d, g.eps, hidden, wqk, gates);
}

// out = a * b elementwise in fp32 (bind: the gate's w_q w_k product).
__global__ void k_mul_f32(const float* __restrict__ a, const float* __restrict__ b,
                          float* __restrict__ out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = a[i] * b[i];
}

cudaError_t launch_gate_sums(const Geometry& g, const float* partials, int groups, const float* v,
                             const uint4* windows, int64_t T, uint16_t* hidden, float* gates,
                             cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (g.hc > 8 || g.d % kBN != 0 || groups < 1) return cudaErrorInvalidValue;
    const int parts = (g.d / 4 + kGateSumsCols - 1) / kGateSumsCols;
    if (T * parts > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = (size_t)g.hc * (g.d / kBN) * groups * 3 * sizeof(float);
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(T * parts));
    cfg.blockDim = dim3(kGateSumsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (g.hc <= 4)
        return cudaLaunchKernelEx(&cfg, k_gate_sums<4>, partials, groups, v, windows, g.hc, g.d,
                                  g.eps, parts, hidden, gates);
    return cudaLaunchKernelEx(&cfg, k_gate_sums<8>, partials, groups, v, windows, g.hc, g.d, g.eps,
                              parts, hidden, gates);
}

cudaError_t launch_mul_f32(const float* a, const float* b, float* out, int64_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    k_mul_f32<<<grid_for(n, 256, 8), 256, 0, s>>>(a, b, out, n);
    return cudaGetLastError();
}

cudaError_t launch_scale_range(const uint8_t* scales, uint64_t n, uint32_t* out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    k_scale_range<<<grid_for((int64_t)std::min<uint64_t>(n / 16 + 1, 1ull << 40), 256, 8), 256, 0,
                    s>>>(scales, n, out);
    return cudaGetLastError();
}

cudaError_t launch_absmax_bf16(const uint16_t* x, uint64_t n, uint32_t* out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    k_absmax_bf16<<<grid_for((int64_t)n, 256, 8), 256, 0, s>>>(x, n, out);
    return cudaGetLastError();
}

cudaError_t launch_wkv_to_f16_tiles(const uint16_t* src, uint16_t* dst, uint64_t N, uint64_t K,
                                   float scale, cudaStream_t s) {
    if (N == 0 || K == 0 || N % 128 != 0 || K % 64 != 0) return cudaErrorInvalidValue;
    k_wkv_to_f16_tiles<<<grid_for((int64_t)(N * K), 256, 8), 256, 0, s>>>(src, dst, N, K, scale);
    return cudaGetLastError();
}

cudaError_t launch_gather_stage(const HashParams& hp, const uint4* windows, int64_t T, int row_dim,
                                const uint8_t* table, const uint8_t* scales, uint64_t nrows,
                                bool table_bf16, bool f16, int exp_shift, uint16_t* e,
                                uint32_t* err, uint32_t* clear, int n_clear, uint32_t* block_text,
                                cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (table_bf16 && f16) return cudaErrorInvalidValue;  // BF16 rows feed BF16 operands
    const int threads = 256;
    const int64_t rows_per_warp = 32 / (row_dim / 16);
    const int64_t warps = (T * hp.nb + rows_per_warp - 1) / rows_per_warp;
    // programmatic dependent launch (see the kernel)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid_for(warps * 32, threads, 8));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint32_t* no_rows = nullptr;
    const uint8_t* no_raw = nullptr;
    if (f16)
        return cudaLaunchKernelEx(&cfg, k_gather_stage<true, false>, hp, windows, T, row_dim, table,
                                  scales, nrows, exp_shift, 0, e, err, clear, n_clear, no_rows,
                                  no_raw, block_text);
    return cudaLaunchKernelEx(&cfg, k_gather_stage<false, false>, hp, windows, T, row_dim, table,
                              scales, nrows, exp_shift, table_bf16 ? 1 : 0, e, err, clear, n_clear,
                              no_rows, no_raw, block_text);
}

cudaError_t launch_stage_raw(const HashParams& hp, const uint32_t* rows_bm, const uint8_t* raw,
                             int64_t T, int row_dim, bool f16, int exp_shift, uint16_t* e,
                             uint32_t* err, uint32_t* clear, int n_clear, uint32_t* block_text,
                             cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t rows_per_warp = 32 / (row_dim / 16);
    const int64_t warps = (T * hp.nb + rows_per_warp - 1) / rows_per_warp;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid_for(warps * 32, threads, 8));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint4* no_windows = nullptr;
    const uint8_t* no_table = nullptr;
    if (f16)
        return cudaLaunchKernelEx(&cfg, k_gather_stage<true, true>, hp, no_windows, T, row_dim,
                                  no_table, no_table, (uint64_t)0, exp_shift, 0, e, err, clear,
                                  n_clear, rows_bm, raw, block_text);
    return cudaLaunchKernelEx(&cfg, k_gather_stage<false, true>, hp, no_windows, T, row_dim,
                              no_table, no_table, (uint64_t)0, exp_shift, 0, e, err, clear, n_clear,
                              rows_bm, raw, block_text);
}

cudaError_t launch_shard_gather_raw(const uint32_t* ids, int64_t n, uint64_t row_lo, uint64_t nrows,
                                    int row_dim, const uint8_t* table, const uint8_t* scales,
                                    uint8_t* raw, uint32_t* err, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    k_shard_gather_raw<<<grid_for(n * (row_dim / 16 + 1), threads, 16), threads, 0, s>>>(
        ids, n, row_lo, nrows, row_dim, table, scales, raw, err);
    return cudaGetLastError();
}

int device_sm_count() { return sm_count(); }

}  // namespace engram
