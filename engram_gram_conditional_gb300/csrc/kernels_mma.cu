// The wkv projection on the 5th-generation tensor cores (tcgen05 + TMEM), and
// the fused Engram forward built on it (sm_103a).
//
// One persistent CTA per SM (320 threads, ~223 KB of shared memory) walks a
// list of 128 x 256 output tiles.  Warp roles:
//   warp 0      TMA producer: wkv tiles (and, unfused, the emb tiles) into a
//               4-stage ring of 128-byte-swizzled K-major shared-memory tiles
//   warp 1      MMA issuer: one thread issues tcgen05.mma kind::f16 (BF16 x
//               BF16 -> F32) into one of two TMEM accumulators of 256 columns;
//               the warp owns the TMEM allocation
//   warps 2..5  (fused only) A-operand producers, one thread per token row:
//               hash the token's window in registers, copy the selected MXFP8
//               row slice and its E8M0 scales into a private cp.async ring,
//               decode E4M3 x 2^E8M0 -> BF16 and write it straight into the
//               swizzled A tile - the 6,144-vector never reaches HBM
//   warps 6..9  epilogue: tcgen05.ld of the accumulator, then
//               store kv (unfused projection), or per-(token, branch, tile)
//               sums of k^2, h^2 and h w_q w_k k (key tiles), or gates from
//               those sums and hidden += g v (value tiles) - kv never reaches
//               HBM in the fused forward.
// Every mbarrier wait is bounded: on time-out the kernel raises an abort flag,
// sets the error word and all roles leave their loops and free TMEM.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "device_common.cuh"

namespace engram {

namespace {

constexpr int kThreads = 320;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpProd = 2, kWarpEpi = 6;
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBK * 2;  // 16 KB
constexpr int kBStage = kBN * kBK * 2;  // 32 KB
constexpr int kRawDepth = 3;            // k-blocks of raw MXFP8 in flight per producer
constexpr int kRawRow = 80;             // 64 code bytes + 2 scale words + shifts
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAStage;
constexpr int kOffRaw = kOffB + kStages * kBStage;
constexpr int kOffBar = kOffRaw + kRawDepth * kBM * kRawRow;
constexpr int kNumBars = 2 * kStages + 4;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kOffFlag = kOffTmem + 4;
constexpr int kSmemUsed = kOffFlag + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
constexpr int kTmemCols = 2 * kBN;
static_assert(kSmemBytes <= 232448, "shared memory above the sm_100 per-block limit");
static_assert(kOffB % 1024 == 0 && kAStage % 1024 == 0 && kBStage % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");

// Instruction descriptor, kind::f16: F32 accumulate (bits 4-5 = 1), A and B
// BF16 (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at 24.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for the phase of parity `parity`; false on time-out or abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 31u) == 0u) {
            if (*abort_flag) return false;
            if ((long long)(globaltimer() - t0) > limit_ns) return false;
        }
    }
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// ---- TMA, cp.async, proxies ------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ---- tcgen05 -------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// Shared-memory matrix descriptor: K-major operand in 128-byte swizzled rows,
// 8-row groups 1024 bytes apart (SBO); LBO unused for this layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i gets row (lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Tile order: groups of `group_m` M blocks; inside a group, N-major so the
// CTAs in flight share wkv tiles in L2 while the group's gathered rows stay
// L2-resident.
__device__ __forceinline__ void tile_coords(const MmaArgs& a, int tile, int& mb, int& nt) {
    const int per_group = a.group_m * a.n_tiles;
    const int g = tile / per_group;
    const int first_m = g * a.group_m;
    const int gm = min(a.group_m, a.m_blocks - first_m);
    const int r = tile - g * per_group;
    nt = r / gm;
    mb = first_m + (r - nt * gm);
}

// ---- fused A producer ------------------------------------------------------------
struct RowCache {
    int b;
    uint32_t row;
};

__device__ __forceinline__ uint32_t row_of(const MmaArgs& a, uint4 w, int b, RowCache& rc) {
    if (b != rc.b) {
        rc.b = b;
        uint32_t r = hash_bucket(a.hp, w, b);
        if (r != kMasked && (uint64_t)r >= a.rows) {
            atomicOr(a.err, kErrBounds);
            r = kMasked;
        }
        rc.row = r;
    }
    return rc.row;
}

// Copy k-block kb (64 columns) of one token's concatenated rows into its raw
// slot: 64 code bytes at +0, the aligned 4-byte scale words at +64/+68, the
// byte offsets of the scales inside those words at +72.  A masked row gets
// zero codes and scale exponent 127, which decode to +0.
__device__ __forceinline__ void issue_kblock(const MmaArgs& a, uint4 w, int kb, uint32_t slot,
                                             RowCache& rc) {
    const int sub = a.row_dim < 64 ? a.row_dim : 64;
    const int nsub = 64 / sub;
    uint32_t shifts = 0;
    for (int j = 0; j < nsub; ++j) {
        const int col = kb * 64 + j * sub;
        const int b = col / a.row_dim;
        const int c0 = col - b * a.row_dim;
        const uint32_t row = row_of(a, w, b, rc);
        const uint32_t dst = slot + (uint32_t)(j * sub);
        if (row == kMasked) {
            for (int q = 0; q < sub / 16; ++q) st_shared_v4(dst + q * 16, make_uint4(0, 0, 0, 0));
            st_shared_u32(slot + 64 + 4 * j, 0x7F7F7F7Fu);
        } else {
            const uint8_t* src = a.table + (uint64_t)row * a.row_dim + c0;
            for (int q = 0; q < sub / 16; ++q) cp_async16(dst + q * 16, src + q * 16);
            const uint64_t sidx = (uint64_t)row * (a.row_dim / 32) + c0 / 32;
            cp_async4(slot + 64 + 4 * j, a.scales + (sidx & ~3ull));
            shifts |= (uint32_t)(sidx & 3ull) << (8 * j);
        }
    }
    st_shared_u32(slot + 72, shifts);
}

// Decode a raw slot into row m of a swizzled A stage (128-byte rows; 16-byte
// chunk q of row m lives at chunk q ^ (m % 8)).
__device__ __forceinline__ void decode_kblock(uint32_t slot, uint32_t a_stage, int m, int row_dim) {
    uint4 c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = ld_shared_v4(slot + 16 * q);
    const uint32_t sw0 = ld_shared_u32(slot + 64);
    const uint32_t sw1 = ld_shared_u32(slot + 68);
    const uint32_t sh = ld_shared_u32(slot + 72);
    float sf0, sf1;
    if (row_dim >= 64) {
        const uint32_t s0 = (sh & 0xFFu) * 8u;
        sf0 = e8m0_to_f32((sw0 >> s0) & 0xFFu);
        sf1 = e8m0_to_f32((sw0 >> (s0 + 8u)) & 0xFFu);
    } else {
        sf0 = e8m0_to_f32((sw0 >> ((sh & 0xFFu) * 8u)) & 0xFFu);
        sf1 = e8m0_to_f32((sw1 >> (((sh >> 8) & 0xFFu) * 8u)) & 0xFFu);
    }
    const uint32_t rowbase = a_stage + (uint32_t)m * 128u;
    const uint32_t sw = (uint32_t)(m & 7);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint4& cc = c[q >> 1];
        const uint32_t w0 = (q & 1) ? cc.z : cc.x;
        const uint32_t w1 = (q & 1) ? cc.w : cc.y;
        const uint4 o = decode8(w0, w1, q < 4 ? sf0 : sf1);
        st_shared_v4(rowbase + (((uint32_t)q ^ sw) << 4), o);
    }
}

// ---- the kernel ---------------------------------------------------------------------
template <bool kFusedA, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
k_mma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
      const __grid_constant__ MmaArgs a) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = sbase + kOffBar;
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(kStages + s); };
    auto tfull = [&](int acc) { return bar0 + 8u * (uint32_t)(2 * kStages + acc); };
    auto tempty = [&](int acc) { return bar0 + 8u * (uint32_t)(2 * kStages + 2 + acc); };
    auto a_stage = [&](int s) { return sbase + kOffA + (uint32_t)(s * kAStage); };
    auto b_stage = [&](int s) { return sbase + kOffB + (uint32_t)(s * kBStage); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffFlag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), kFusedA ? 1u + kBM : 1u);
            mbar_init(empty(s), 1u);
        }
        for (int acc = 0; acc < 2; ++acc) {
            mbar_init(tfull(acc), 1u);
            mbar_init(tempty(acc), 4u);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpTma && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
        if (!kFusedA) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
    }
    if (warp == kWarpMma) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int total = a.m_blocks * a.n_tiles;
    const int KB = a.K / kBK;
    const long long lim = a.wait_limit_ns;

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
    };

    if (warp == kWarpTma) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int mb, nt;
                tile_coords(a, tile, mb, nt);
                const int n0 = (a.n_tile_begin + nt) * kBN;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, lim)) {
                        fail();
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full(s), kFusedA ? kBStage : kAStage + kBStage);
                    if (!kFusedA) tma_load_2d(a_stage(s), &tmA, full(s), kb * kBK, mb * kBM);
                    tma_load_2d(b_stage(s), &tmB, full(s), kb * kBK, n0);
                }
            }
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++tc) {
                const int acc = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                if (!mbar_wait(tempty(acc), aph ^ 1u, abort_flag, lim)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(full(s), ph, abort_flag, lim)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_sw128(a_stage(s));
                    const uint64_t bd = sdesc_sw128(b_stage(s));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)  // 16 BF16 = 32 bytes per MMA
                        umma_bf16(d_tmem, ad + 2ull * k, bd + 2ull * k, (kb | k) != 0);
                    umma_commit(empty(s));
                }
                if (ok) umma_commit(tfull(acc));
            }
        }
    } else if (warp < kWarpEpi) {
        if (kFusedA) {
            const int p = threadIdx.x - kWarpProd * 32;  // token row of the tile
            const uint32_t raw = sbase + kOffRaw;
            auto slot = [&](int j) { return raw + (uint32_t)((j * kBM + p) * kRawRow); };
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int mb, nt;
                tile_coords(a, tile, mb, nt);
                const int64_t t = (int64_t)mb * kBM + p;
                const uint4 w = t < a.T ? a.windows[t] : make_uint4(kDead, kDead, kDead, kDead);
                RowCache rc{-1, kMasked};
#pragma unroll
                for (int j = 0; j < kRawDepth; ++j) {
                    if (j < KB) issue_kblock(a, w, j, slot(j), rc);
                    cp_async_commit();
                }
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    cp_async_wait<kRawDepth - 1>();
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, lim)) {
                        fail();
                        ok = false;
                        break;
                    }
                    decode_kblock(slot(kb % kRawDepth), a_stage(s), p, a.row_dim);
                    fence_proxy_async();
                    mbar_arrive(full(s));
                    if (kb + kRawDepth < KB) issue_kblock(a, w, kb + kRawDepth, slot(kb % kRawDepth), rc);
                    cp_async_commit();
                }
            }
            cp_async_wait<0>();
        }
    } else {
        // ---- epilogue ----
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const int m = q * 32 + lane;
        int tc = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tc) {
            int mb, nt;
            tile_coords(a, tile, mb, nt);
            const int acc = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            if (!mbar_wait(tfull(acc), aph, abort_flag, lim)) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
            const int64_t t = (int64_t)mb * kBM + m;
            const int n0 = (a.n_tile_begin + nt) * kBN;
            if (kMode == kEpiStoreKv) {
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)(c * 32), r);
                    tmem_wait_ld();
                    if (t < a.T) {
                        float4* dst = reinterpret_cast<float4*>(a.kv + t * a.ldkv + n0 + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                    }
                }
            } else if (kMode == kEpiKeyPartial) {
                const int branch = n0 / a.d;
                const int col0 = n0 - branch * a.d;
                const bool text = t < a.T && a.windows[t].x != kDead;
                const uint16_t* hrow = a.hidden + (t * a.hc + branch) * (int64_t)a.d + col0;
                const float* wqr = a.wq + (int64_t)branch * a.d + col0;
                const float* wkr = a.wk + (int64_t)branch * a.d + col0;
                float skk = 0.f, shh = 0.f, shk = 0.f;
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)(c * 32), r);
                    uint4 hv[4];
                    if (text) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            hv[i] = __ldg(reinterpret_cast<const uint4*>(hrow + c * 32) + i);
                    }
                    tmem_wait_ld();
                    if (text) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 q0 = __ldg(reinterpret_cast<const float4*>(wqr + c * 32) + 2 * i);
                            const float4 q1 = __ldg(reinterpret_cast<const float4*>(wqr + c * 32) + 2 * i + 1);
                            const float4 k0 = __ldg(reinterpret_cast<const float4*>(wkr + c * 32) + 2 * i);
                            const float4 k1 = __ldg(reinterpret_cast<const float4*>(wkr + c * 32) + 2 * i + 1);
                            const float wqk[8] = {q0.x * k0.x, q0.y * k0.y, q0.z * k0.z, q0.w * k0.w,
                                                  q1.x * k1.x, q1.y * k1.y, q1.z * k1.z, q1.w * k1.w};
                            const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float h = (e & 1) ? bf16_hi(hw[e >> 1]) : bf16_lo(hw[e >> 1]);
                                const float k = __uint_as_float(r[8 * i + e]);
                                skk = fmaf(k, k, skk);
                                shh = fmaf(h, h, shh);
                                shk = fmaf(h * wqk[e], k, shk);
                            }
                        }
                    }
                }
                if (text) {
                    const int P = a.d / kBN;
                    float* pp = a.partials + ((t * a.hc + branch) * P + col0 / kBN) * 3;
                    pp[0] = skk;
                    pp[1] = shh;
                    pp[2] = shk;
                }
            } else {  // kEpiValueUpdate
                const int cv = n0 - a.hc * a.d;
                const bool text = t < a.T && a.windows[t].x != kDead;
                const int P = a.d / kBN;
                float g[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    g[b] = 0.f;
                    if (b < a.hc && text) {
                        const float* pp = a.partials + (t * a.hc + b) * (int64_t)P * 3;
                        float skk = 0.f, shh = 0.f, shk = 0.f;
                        for (int p = 0; p < P; ++p) {
                            skk += pp[3 * p];
                            shh += pp[3 * p + 1];
                            shk += pp[3 * p + 2];
                        }
                        g[b] = gate_from_sums(skk, shh, shk, a.d, a.eps);
                    }
                }
                if (a.gates && nt == 0 && t < a.T) {
                    for (int b = 0; b < a.hc; ++b) a.gates[t * a.hc + b] = text ? g[b] : 0.f;
                }
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)(c * 32), r);
                    tmem_wait_ld();
                    if (text) {
#pragma unroll
                        for (int b = 0; b < 8; ++b) {
                            if (b < a.hc) {
                                uint4* hp = reinterpret_cast<uint4*>(
                                    a.hidden + (t * a.hc + b) * (int64_t)a.d + cv + c * 32);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const uint4 hv = hp[i];
                                    const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
                                    uint32_t o[4];
#pragma unroll
                                    for (int e2 = 0; e2 < 4; ++e2) {
                                        const float v0 = __uint_as_float(r[8 * i + 2 * e2]);
                                        const float v1 = __uint_as_float(r[8 * i + 2 * e2 + 1]);
                                        o[e2] = bf16x2_pack_rn(fmaf(g[b], v0, bf16_lo(hw[e2])),
                                                               fmaf(g[b], v1, bf16_hi(hw[e2])));
                                    }
                                    hp[i] = make_uint4(o[0], o[1], o[2], o[3]);
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
        }
    }

    __syncthreads();
    if (*abort_flag) {
        // let copies and MMAs still in flight land before TMEM is freed
        if (threadIdx.x == 0) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 2000000ull) __nanosleep(1000);
        }
        __syncthreads();
    }
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <bool kFusedA, int kMode>
cudaError_t launch(const MmaArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                   cudaStream_t s) {
    static bool attr_set = false;
    auto kern = k_mma<kFusedA, kMode>;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int total = a.m_blocks * a.n_tiles;
    if (total == 0) return cudaSuccess;
    const int grid = std::min(total, device_sm_count());
    kern<<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t make_tma_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_project(const MmaArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           cudaStream_t s) {
    return launch<false, kEpiStoreKv>(a, tmA, tmB, s);
}

cudaError_t launch_forward_phase(const MmaArgs& a, int mode, const CUtensorMap& tmB,
                                 cudaStream_t s) {
    if (mode == kEpiKeyPartial) return launch<true, kEpiKeyPartial>(a, tmB, tmB, s);
    if (mode == kEpiValueUpdate) return launch<true, kEpiValueUpdate>(a, tmB, tmB, s);
    return launch<true, kEpiStoreKv>(a, tmB, tmB, s);
}

}  // namespace engram
