// The wkv projection on the 5th-generation tensor cores (tcgen05 + TMEM), and
// the fused Engram forward built on it (sm_103a).
//
// One persistent CTA per SM (512 threads) walks a list of 128 x 256 output
// tiles; every tile reduces over K = 6,144 in 64-wide k-blocks.  Operands sit
// in 128-byte-swizzled K-major shared-memory tiles: an A ring (128 tokens x 64)
// and a B ring (256 wkv rows x 64).  Warp roles, by warpgroup (each group
// sets its own register budget with setmaxnreg):
//   warp 12     TMA producer: wkv tiles into the B ring (and, for the unfused
//               projection, the emb tiles into the A ring)
//   warp 13     MMA issuer: one thread issues tcgen05.mma kind::f16 into one
//               of two TMEM accumulators of 256 columns; the warp owns TMEM
//               (warps 12..15: 56 registers each, warps 14 and 15 idle)
//   warps 0..7  fused A producers, 144 registers (16 token rows each): hash each token's
//               window in registers, load the selected MXFP8 rows, decode
//               E4M3 x 2^E8M0 and write the operand straight into the swizzled
//               A tiles - the 6,144-vector never reaches HBM.  Two gathers:
//                 bucket gather (256-wide rows): each table row is loaded whole
//                 (16 lanes x 16 bytes, two rows per instruction) once per
//                 tile and bucket, one bucket ahead in registers, and decoded
//                 into the four A stages of its bucket at once (8-stage A
//                 ring, 3-stage B ring).  Fetching whole rows matters: random
//                 row fetches, not bytes, limit a gather on this GPU (about
//                 0.12 rows per clock per SM whatever their size).
//                 k-block gather (other row widths): per k-block, four lanes
//                 load a row's 64-byte slice (4-stage rings).
//               Operands are FP16 when they hold the values exactly (one
//               e4m3x2->f16x2 conversion and one f16x2 multiply per pair;
//               wkv as an exact FP16 copy scaled by a power of two), else BF16
//               (decode through fp32)
//   warps 8..11 epilogue, 168 registers: tcgen05.ld of the accumulator, then store kv
//               (projection), or per-(token, branch, tile) sums of k^2, h^2
//               and h w_q w_k k (key tiles), or gates from those sums and
//               hidden += g v (value tiles) - kv never reaches HBM in the
//               fused forward.  With a TMA-fed A (no producers) warps 4..11
//               run the epilogue, 216 registers, two per TMEM quadrant on
//               alternate 32-column chunks; warps 0..3 idle.
// Every mbarrier wait is bounded: on time-out the kernel raises an abort flag,
// sets the error word and all roles leave their loops and free TMEM.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "device_common.cuh"

namespace engram {

namespace {

constexpr int kThreads = 512;  // four warpgroups
constexpr int kProdWarps = 8;  // A producers: warps 0..7, 16 token rows each
constexpr int kRowsPerProd = kBM / kProdWarps;
constexpr int kWarpProd = 0, kWarpEpi = 8, kWarpTma = 12, kWarpMma = 13, kWarpTmaA = 14;
// Register split (setmaxnreg): launch budget 512 x 128 = 65,536 registers;
// 128 x (2 x 144 + 168 + 56) = 65,536 - the four shares add up to it exactly
// (and each scheduler holds one warp of each group: 32 x 512 = 16,384).
constexpr int kLaunchRegs = 128;
constexpr int kRegsProd = 144, kRegsEpi = 168, kRegsCtl = 56;
static_assert(kThreads * kLaunchRegs == 128 * (2 * kRegsProd + kRegsEpi + kRegsCtl),
              "setmaxnreg shares must add up to the launch allocation");
// The TMA-fed kernels have no A producers: warps 4..11 all run the epilogue
// with 216 registers each and warps 0..3 idle with 24 (24 + 2 x 216 + 56 =
// 512 per scheduler, as above).
constexpr int kRegsWideEpi = 216, kRegsIdle = 24;
static_assert(kThreads * kLaunchRegs == 128 * (kRegsIdle + 2 * kRegsWideEpi + kRegsCtl),
              "setmaxnreg shares must add up to the launch allocation");
// Ready flags per CTA of a stream-K launch: one per epilogue warp.
constexpr int kSkFlagsPerCta = 16;
constexpr int kAStage = kBM * kBK * 2;  // 16 KB
constexpr int kBStage = kBN * kBK * 2;  // 32 KB
constexpr int kRowStride = kMaxBuckets + 1;  // row-index table stride (odd: no bank conflicts)
constexpr int kPrefetch = 3;   // k-blocks of row slices in flight per lane
constexpr int kTmemCols = 2 * kBN;

// Source of the A operand.
enum ASource : int {
    kASrcTma = 0,           // TMA tiles of a 16-bit operand matrix (unfused projection)
    kASrcGatherKb = 1,      // fused: k-block gather of 64-byte row slices
    kASrcGatherBucket = 2,  // fused: bucket gather of whole 256-byte rows
    kASrcTmaPair = 3,       // TMA tiles, a CTA pair per 256 x 256 tile (cta_group::2)
};

// CTA pair (cluster of two SMs): the pair computes a 256-token x 256-output
// tile with tcgen05.mma.cta_group::2.  Each CTA stages its own 128 tokens of A
// and its own half (128 rows) of the wkv tile, so an SM takes in 32 KB per
// k-block instead of 48 KB; the accumulator rows of each CTA land in its own
// TMEM.  The even CTA issues the MMAs.
constexpr int kBStageHalf = kBStage / 2;  // 16 KB

// k-blocks per pipeline stage.  A TMA copy costs the SM about the same time
// (some 0.2 us of its copy engine) whether it moves 16 or 32 KB, so the
// FP16 pair kernel, whose operands are both stored in 128 x 64 tiles, loads
// two k-blocks of each operand with one 32 KB box per stage.
template <int kASrc, bool kF16>
__host__ __device__ constexpr int k_blocks_per_stage() {
    return kASrc == kASrcTmaPair && kF16 ? 2 : 1;
}

// Epilogue warps per TMEM quadrant: the TMA-fed kernels have no A producers,
// so warps 4..11 all run the epilogue, two per quadrant, each on every other
// 32-column chunk of a tile.
template <int kASrc>
__host__ __device__ constexpr int epilogue_groups() {
    return kASrc == kASrcTma || kASrc == kASrcTmaPair ? 2 : 1;
}

// Shared-memory layout of each variant.  The FP16 pair kernel holds seven or
// six stages of two k-blocks: with the kv-store epilogue (small batches, whose
// launch streams wkv from HBM once) four of them wkv; with the forward
// epilogue (compute-bound batches) three and three.
template <int kASrc, int kKS = 1, int kMode = 0>
struct Layout {
    static constexpr bool kPair = kASrc == kASrcTmaPair;
    // ring stages (each kKS k-blocks)
    static constexpr int kA = kASrc == kASrcGatherBucket ? 8 : kKS == 2 ? 3 : 4;
    static constexpr int kB = kASrc == kASrcGatherBucket ? 3
                              : kKS == 2 ? (kMode == kEpiStoreKv || kMode == kEpiForwardSk ? 4 : 3)
                              : kPair                    ? 8
                                                         : 4;
    static constexpr int kAStageBytes = kAStage * kKS;
    static constexpr int kBStageBytes = (kPair ? kBStageHalf : kBStage) * kKS;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kA * kAStageBytes;
    static constexpr int kOffRows = kOffB + kB * kBStageBytes;
    static constexpr int kRowsBytes = kASrc == kASrcGatherKb ? kBM * kRowStride * 4 : 0;
    static constexpr int kOffBar = kOffRows + kRowsBytes;
    // a_full[kA], a_empty[kA], b_full[kB], b_empty[kB], tfull[2], tempty[2]
    static constexpr int kNumBars = 2 * kA + 2 * kB + 4;
    static constexpr int kOffTmem = kOffBar + kNumBars * 8;
    static constexpr int kOffFlag = kOffTmem + 4;
    static constexpr int kBytes = kOffFlag + 4 + 1024;  // + slack to align the base to 1 KB
    static_assert(kBytes <= 232448, "shared memory above the per-block limit");
    static_assert(kOffB % 1024 == 0 && kOffRows % 1024 == 0, "swizzled tiles need 1 KB alignment");
};

// Instruction descriptor, kind::f16: F32 accumulate (bits 4-5 = 1), A and B
// both BF16 (bits 7-9 = 1, 10-12 = 1) or both FP16 (0, 0), both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24 (M = 128 for one CTA, 256 for a pair).
template <bool kF16, int kM = kBM>
__host__ __device__ constexpr uint32_t idesc() {
    return (1u << 4) | (kF16 ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)(kBN >> 3) << 17) |
           ((uint32_t)(kM >> 4) << 24);
}

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
// CTA-pair form: the completion is signalled on `bar`, a shared::cluster
// address that may lie in the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
// The same two loads with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map,
                                                      uint32_t bar, int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
// A policy that makes the lines it brings into L2 the first to be evicted.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// A policy that keeps the lines it brings into L2 longest.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---- tcgen05 -------------------------------------------------------------------
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
template <int kRegs>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
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
__device__ __forceinline__ void umma_f16kind(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc_bits, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc_bits), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// ---- CTA pair (cluster of two) ------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of both CTAs; orders barrier inits and teardown across the pair.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
// Shared::cluster address of the same shared variable in CTA `rank` of the pair.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait for a barrier that the other CTA of the pair also arrives on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, long long limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((n & 31u) == 0u) {
            if (*abort_flag) return false;
            if ((long long)(globaltimer() - t0) > limit_ns) return false;
        }
    }
}
// TMEM of both CTAs, allocated collectively by one warp of each.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void umma_f16kind_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                  uint32_t idesc_bits, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc_bits), "r"(accumulate)
        : "memory");
}
// Arrives on the barrier at this offset in both CTAs once the issued MMAs finish.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar), "h"((uint16_t)3)
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
// The inverse of tmem_ld32: thread i writes row (lane base + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Starts loading `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// Drops a 128-byte line from L2 without writing it back (its contents become
// undefined): for scratch that nobody reads again.
__device__ __forceinline__ void discard_l2_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Split-K reduction of one TMEM quadrant (32 rows) of an output tile in the
// forward epilogue.  The splits of a tile count their arrivals per quadrant:
// every split but the last parks its accumulator in its fp32 slot; the last
// waits (bounded) until those are written, sums the S partials in split order
// - its own from TMEM - and writes the sum back into TMEM, so the gate
// epilogue that follows sees the full K reduction.  The sum does not depend
// on which split arrives last.  Returns 1 for the warp that holds the sum,
// 0 for a warp that parked its partial, -1 on a time-out.
// Slot layout: [32-column chunk c][float4 i][row]: the 32 rows of a warp for
// one (c, i) are 512 contiguous bytes.
__device__ __forceinline__ int split_k_quadrant(const MmaArgs& a, int mb, int nt, int ks, int q,
                                                int lane, uint32_t taddr,
                                                volatile int* abort_flag, long long lim) {
    const int S = a.k_splits;
    const int64_t tile = (int64_t)mb * a.n_tiles + nt;
    uint32_t* cnt = a.split_counters + (tile * 4 + q) * 2;
    uint32_t order = 0;
    if (lane == 0) order = atomicAdd(cnt, 1u);
    order = __shfl_sync(0xFFFFFFFFu, order, 0);
    float4* const slots = reinterpret_cast<float4*>(a.split_partials) + tile * S * (kBM * kBN / 4);
    const int m = q * 32 + lane;
    if ((int)order < S - 1) {
        float4* dst = slots + (int64_t)ks * (kBM * kBN / 4);
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + (uint32_t)(c * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
                __stcg(dst + (c * 8 + i) * kBM + m,
                       make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                   __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(cnt + 1, 1u);
        return 0;
    }
    int ready = 1;
    if (lane == 0) {
        const uint64_t t0 = globaltimer();
        uint32_t n = 0;
        while (ld_acquire_u32(cnt + 1) < (uint32_t)(S - 1)) {
            if ((++n & 63u) == 0u && ((long long)(globaltimer() - t0) > lim || *abort_flag)) {
                ready = 0;
                break;
            }
        }
    }
    ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
    if (!ready) return -1;
    __threadfence();
#pragma unroll 1
    for (int c = 0; c < kBN / 32; ++c) {
        uint32_t own[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), own);
        tmem_wait_ld();
        float acc[32];
#pragma unroll 1
        for (int k = 0; k < S; ++k) {
            float v[32];
            if (k == ks) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(own[j]);
            } else {
                const float4* src = slots + (int64_t)k * (kBM * kBN / 4) + c * 8 * kBM + m;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 x = __ldcg(src + i * kBM);
                    v[4 * i] = x.x;
                    v[4 * i + 1] = x.y;
                    v[4 * i + 2] = x.z;
                    v[4 * i + 3] = x.w;
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = k == 0 ? v[j] : acc[j] + v[j];
        }
        uint32_t out[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) out[j] = __float_as_uint(acc[j]);
        tmem_st32(taddr + (uint32_t)(c * 32), out);
        // the parked lines of this chunk are read: drop them from L2 unwritten
        __syncwarp();
        for (int k = 0; k < S; ++k)
            if (k != ks)
                discard_l2_line(slots + (int64_t)k * (kBM * kBN / 4) + (c * 8 + (lane >> 2)) * kBM +
                                q * 32 + (lane & 3) * 8);
    }
    tmem_wait_st();
    return 1;
}

// Tile order: groups of `group_m` M blocks (or pair units); inside a group,
// N-major so the CTAs in flight share wkv tiles in L2 while the group's
// gathered rows stay L2-resident.
// With split-K (small M) the order is (N tile, split) outer, M block inner.
__device__ __forceinline__ void tile_coords(const MmaArgs& a, int m_units, int tile, int& mb,
                                            int& nt, int& ks) {
    if (a.k_splits > 1) {
        mb = tile % m_units;
        const int r = tile / m_units;
        ks = r % a.k_splits;
        nt = r / a.k_splits;
        return;
    }
    ks = 0;
    // the forward's key tiles (N tiles [0, key_tiles)) all come before its
    // value tiles, so that a value tile finds its gates long computed
    int base_nt = 0, ntiles = a.n_tiles;
    if (a.key_tiles > 0) {
        const int key_items = m_units * a.key_tiles;
        if (tile < key_items) {
            ntiles = a.key_tiles;
        } else {
            tile -= key_items;
            base_nt = a.key_tiles;
            ntiles = a.n_tiles - a.key_tiles;
        }
    }
    const int per_group = a.group_m * ntiles;
    const int g = tile / per_group;
    const int first_m = g * a.group_m;
    const int gm = min(a.group_m, m_units - first_m);
    const int r = tile - g * per_group;
    if (a.key_tiles > 0 && a.key_tail > 0 && m_units <= a.group_m) {
        // the forward in one group: the last key_tail key tiles and all value
        // tiles run M-major, so that the M units get their gates one after
        // the other and each unit's value tiles come after its gates.  (With
        // several groups the first value tiles are those of group 0, whose
        // gates are long done, and M-major value tiles would spread each wkv
        // value tile over a whole group's worth of time.)
        const int head = base_nt == 0 ? max(ntiles - a.key_tail, 0) : 0;  // N-major part
        if (r >= head * gm) {
            const int tail = ntiles - head;
            const int rr = r - head * gm;
            mb = first_m + rr / tail;
            nt = base_nt + head + rr % tail;
            return;
        }
    }
    nt = base_nt + r / gm;
    mb = first_m + (r - (r / gm) * gm);
}

// Forward epilogue: starts the L2 loads of the hidden slices that row m of
// the tile (M block mb, N tile nt) will read (key tile: its branch's 256 columns; value tile: those
// columns of every branch), so that the epilogue's own loads hit L2.
__device__ __forceinline__ void prefetch_hidden(const MmaArgs& a, int mb, int nt, int m) {
    const int64_t t = (int64_t)mb * kBM + m;
    if (t >= a.T) return;
    const int n0 = (a.n_tile_begin + nt) * kBN;
    const int key_cols = a.hc * a.d;
    if (n0 < key_cols) {
        const int branch = n0 / a.d;
        prefetch_l2(a.hidden + (t * a.hc + branch) * (int64_t)a.d + (n0 - branch * a.d),
                    kBN * 2);
    } else {
        for (int b = 0; b < a.hc; ++b)
            prefetch_l2(a.hidden + (t * a.hc + b) * (int64_t)a.d + (n0 - key_cols), kBN * 2);
    }
}

// Gates of row t (every branch), from the per-(branch, column tile, epilogue
// group) sums the key tiles published, added in (tile, group) order.
__device__ __forceinline__ void row_gates(const MmaArgs& a, int64_t t, int groups, float (&g)[8]) {
    const int P = a.d / kBN * groups;
#pragma unroll
    for (int b = 0; b < 8; ++b) g[b] = 0.f;
    // one branch at a time (its loads all in flight), then the gate into its
    // static register slot
#pragma unroll 1
    for (int b = 0; b < a.hc; ++b) {
        const float* pp = a.partials + (t * a.hc + b) * (int64_t)P * 3;
        float sum[3] = {0.f, 0.f, 0.f};
        const int n4 = 3 * P / 4;
        // rounds of 9 float4 = 12 (k^2, h^2, h w k) triples; 4 x 9 is a multiple
        // of 3, so element 4 j + k of a round adds to sum (4 j + k) % 3
        if (3 * P % 4 == 0) {
#pragma unroll 1
            for (int j0 = 0; j0 < n4; j0 += 9) {
                float4 v[9];
#pragma unroll
                for (int j = 0; j < 9; ++j)
                    if (j0 + j < n4) v[j] = __ldcg(reinterpret_cast<const float4*>(pp) + j0 + j);
#pragma unroll
                for (int j = 0; j < 9; ++j)
                    if (j0 + j < n4) {
                        const float e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) sum[(4 * j + k) % 3] += e[k];
                    }
            }
        } else {
            for (int p = 0; p < P; ++p) {
                sum[0] += __ldcg(pp + 3 * p);
                sum[1] += __ldcg(pp + 3 * p + 1);
                sum[2] += __ldcg(pp + 3 * p + 2);
            }
        }
        const float gb = gate_from_sums(sum[0], sum[1], sum[2], a.d, a.eps);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j == b) g[j] = gb;
    }
}

// ---- fused A producer ------------------------------------------------------------
// Lane l of a producer warp owns the 16-column chunk c = l % 4 of each 64-column
// k-block for the rows rsub + 8 j (j = 0..1, rsub = l / 4) of its 16-row slice:
// the four lanes of a row load its 64 contiguous code bytes, one instruction
// covers eight rows.
struct RawKb {
    uint4 code[kRowsPerProd / 8];      // 16 E4M3 codes per row slot
    uint32_t scale[kRowsPerProd / 8];  // E8M0 exponent of those 16 columns
};

__device__ __forceinline__ void load_kb(const MmaArgs& a, const uint32_t* rows_s, int m0, int c,
                                        int kb, RawKb& o) {
    const int col = kb * kBK + 16 * c;
    const int b = col >> a.row_dim_log2;
    const int c0 = col & (a.row_dim - 1);
    const int groups_log2 = a.row_dim_log2 - 5;
#pragma unroll
    for (int j = 0; j < kRowsPerProd / 8; ++j) {
        const uint32_t row = rows_s[(m0 + 8 * j) * kRowStride + b];
        if (row != kMasked) {
            o.code[j] = __ldg(reinterpret_cast<const uint4*>(a.table + ((uint64_t)row << a.row_dim_log2) + c0));
            o.scale[j] = __ldg(a.scales + ((uint64_t)row << groups_log2) + (c0 >> 5));
        } else {
            o.code[j] = make_uint4(0, 0, 0, 0);
            o.scale[j] = 127u;
        }
    }
}

// 2^e in both halves of an f16x2, e in [-24, 15].
__device__ __forceinline__ uint32_t f16x2_pow2(int e) {
    const uint32_t h = e >= -14 ? (uint32_t)(e + 15) << 10 : 1u << (e + 24);
    return h | (h << 16);
}

// Four E4M3 codes -> four FP16 values times 2^e (two f16x2, low code first).
__device__ __forceinline__ void e4m3x4_f16_scaled(uint32_t w, uint32_t sc2, uint32_t& lo,
                                                  uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\t.reg .b32 a, b;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 a, l;\n\tcvt.rn.f16x2.e4m3x2 b, h;\n\t"
        "mul.rn.f16x2 %0, a, %3;\n\tmul.rn.f16x2 %1, b, %3;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w), "r"(sc2));
}

// Decode one k-block's raw codes into the A stage (row m of a 128-byte
// swizzled K-major tile: 16-byte chunk q lives at chunk q ^ (m % 8)).
template <bool kF16>
__device__ __forceinline__ void store_kb(const RawKb& r, uint32_t a_stage, int m0, int c,
                                         int exp_shift) {
#pragma unroll
    for (int j = 0; j < kRowsPerProd / 8; ++j) {
        const int m = m0 + 8 * j;
        uint32_t o[8];
        if (kF16) {
            const uint32_t sc2 = f16x2_pow2((int)r.scale[j] - 127 + exp_shift);
            e4m3x4_f16_scaled(r.code[j].x, sc2, o[0], o[1]);
            e4m3x4_f16_scaled(r.code[j].y, sc2, o[2], o[3]);
            e4m3x4_f16_scaled(r.code[j].z, sc2, o[4], o[5]);
            e4m3x4_f16_scaled(r.code[j].w, sc2, o[6], o[7]);
        } else {
            const float sf = e8m0_to_f32(r.scale[j]);
            const uint4 lo = decode8(r.code[j].x, r.code[j].y, sf);
            const uint4 hi = decode8(r.code[j].z, r.code[j].w, sf);
            o[0] = lo.x; o[1] = lo.y; o[2] = lo.z; o[3] = lo.w;
            o[4] = hi.x; o[5] = hi.y; o[6] = hi.z; o[7] = hi.w;
        }
        const uint32_t rowbase = a_stage + (uint32_t)m * 128u;
        const uint32_t sw = (uint32_t)(m & 7);
        st_shared_v4(rowbase + (((uint32_t)(2 * c) ^ sw) << 4), make_uint4(o[0], o[1], o[2], o[3]));
        st_shared_v4(rowbase + (((uint32_t)(2 * c + 1) ^ sw) << 4), make_uint4(o[4], o[5], o[6], o[7]));
    }
}


// ---- bucket gather ---------------------------------------------------------------
// Lane l of a producer warp loads 16-byte chunk (l % 16) of rows 2 i + l / 16
// (i = 0..7) of the warp's 16 rows: chunk c holds columns 16 c .. 16 c + 15 of
// the 256-wide row, i.e. k-block c / 4 of the bucket, columns 16 (c % 4) ...
// The row index of each token comes from the lane that hashed it (shuffle).
struct BucketRows {
    uint4 r[kRowsPerProd / 2];
};

__device__ __forceinline__ void load_bucket(const MmaArgs& a, uint32_t own_row, int lane,
                                            BucketRows& o) {
    const int half = lane >> 4, chunk = lane & 15;
#pragma unroll
    for (int i = 0; i < kRowsPerProd / 2; ++i) {
        const uint32_t row = __shfl_sync(0xFFFFFFFFu, own_row, 2 * i + half);
        if (row != kMasked)
            o.r[i] = __ldg(reinterpret_cast<const uint4*>(a.table + ((uint64_t)row << 8)) + chunk);
        else
            o.r[i] = make_uint4(0, 0, 0, 0);
    }
}

// Row of bucket b for this lane's token (bounds-checked) and its 8 scale bytes.
__device__ __forceinline__ uint32_t own_bucket_row(const MmaArgs& a, uint4 w, int b) {
    uint32_t r = hash_bucket(a.hp, w, b);
    if (r != kMasked && (uint64_t)r >= a.rows) {
        atomicOr(a.err, kErrBounds);
        r = kMasked;
    }
    return r;
}
__device__ __forceinline__ uint2 own_scale_word(const MmaArgs& a, uint32_t row) {
    if (row == kMasked) return make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);  // 2^0: zeros stay zeros
    return __ldg(reinterpret_cast<const uint2*>(a.scales + ((uint64_t)row << 3)));
}

// Decode a loaded bucket into its four A stages (base stage index `it`).
// The two 16-byte stores of a lane go to chunks 2 (c % 4) and 2 (c % 4) + 1 of
// its row; odd k-blocks store the odd chunk first, so the eight lanes of a
// shared-memory wavefront always hit eight different bank groups.
template <bool kF16>
__device__ __forceinline__ void decode_bucket(const MmaArgs& a, const BucketRows& br, uint2 sw,
                                              uint32_t a_base, int kA, int it, int pw, int lane) {
    const int half = lane >> 4, chunk = lane & 15;
    const int kbl = chunk >> 2, cp = chunk & 3;
    const int g = chunk >> 1;  // 32-column scale group of the chunk
    const uint32_t stage = a_base + (uint32_t)(((it + kbl) % kA) * kAStage);
    const uint32_t first = (uint32_t)(2 * cp + (kbl & 1));
    const uint32_t second = first ^ 1u;
#pragma unroll
    for (int i = 0; i < kRowsPerProd / 2; ++i) {
        const int tl = 2 * i + half;  // token lane of this slot
        const int m = pw * kRowsPerProd + tl;
        const uint32_t swx = __shfl_sync(0xFFFFFFFFu, sw.x, tl);
        const uint32_t swy = __shfl_sync(0xFFFFFFFFu, sw.y, tl);
        const uint32_t se = ((g < 4 ? swx : swy) >> (8 * (g & 3))) & 0xFFu;
        uint4 lo, hi;  // columns 16 cp .. +7 and +8 .. +15
        if (kF16) {
            const uint32_t sc2 = f16x2_pow2((int)se - 127 + a.a_exp_shift);
            e4m3x4_f16_scaled(br.r[i].x, sc2, lo.x, lo.y);
            e4m3x4_f16_scaled(br.r[i].y, sc2, lo.z, lo.w);
            e4m3x4_f16_scaled(br.r[i].z, sc2, hi.x, hi.y);
            e4m3x4_f16_scaled(br.r[i].w, sc2, hi.z, hi.w);
        } else {
            const float sf = e8m0_to_f32(se);
            lo = decode8(br.r[i].x, br.r[i].y, sf);
            hi = decode8(br.r[i].z, br.r[i].w, sf);
        }
        const uint32_t rowbase = stage + (uint32_t)m * 128u;
        const uint32_t swz = (uint32_t)(m & 7);
        st_shared_v4(rowbase + ((first ^ swz) << 4), (kbl & 1) ? hi : lo);
        st_shared_v4(rowbase + ((second ^ swz) << 4), (kbl & 1) ? lo : hi);
    }
}

// ---- the kernel ---------------------------------------------------------------------
template <int kASrc, bool kF16, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
k_mma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
      const __grid_constant__ MmaArgs a) {
    constexpr int kKS = k_blocks_per_stage<kASrc, kF16>();
    // the whole-tile gate epilogue, plain or over the units that hold text
    constexpr bool kFwdWhole = kMode == kEpiForward || kMode == kEpiForwardCompact;
    using L = Layout<kASrc, kKS, kMode>;
    constexpr int kA = L::kA, kB = L::kB;
    constexpr bool kPair = L::kPair;
    constexpr bool kFusedA = kASrc != kASrcTma && !kPair;
    // without A producers, warps 0..7 join the epilogue
    constexpr int kG = epilogue_groups<kASrc>();
    constexpr bool kWideEpi = kG == 2;
    static_assert(kWideEpi == !kFusedA, "the TMA-fed variants have the wide epilogue");
    constexpr int kEpiWarps = 4 * kG;
    constexpr int kFirstEpi = kWarpEpi - 4 * (kG - 1);  // first epilogue warp
    // in a pair, the even CTA issues the MMAs; the odd one only feeds them
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const bool issuer = rank == 0u;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = sbase + L::kOffBar;
    auto a_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto a_empty = [&](int s) { return bar0 + 8u * (uint32_t)(kA + s); };
    auto b_full = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kA + s); };
    auto b_empty = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kA + kB + s); };
    auto tfull = [&](int acc) { return bar0 + 8u * (uint32_t)(2 * kA + 2 * kB + acc); };
    auto tempty = [&](int acc) { return bar0 + 8u * (uint32_t)(2 * kA + 2 * kB + 2 + acc); };
    const uint32_t a_base = sbase + L::kOffA;
    auto a_stage = [&](int s) { return a_base + (uint32_t)(s * L::kAStageBytes); };
    auto b_stage = [&](int s) { return sbase + L::kOffB + (uint32_t)(s * L::kBStageBytes); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffFlag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmem);

    if (threadIdx.x == 0) {
        // in a pair, the issuer's full barriers take the bytes of both CTAs'
        // copies (the odd CTA's own full barriers stay unused)
        for (int s = 0; s < kA; ++s) {
            mbar_init(a_full(s), kFusedA ? (uint32_t)kProdWarps : 1u);  // producer warps or TMA
            mbar_init(a_empty(s), 1u);
        }
        for (int s = 0; s < kB; ++s) {
            mbar_init(b_full(s), 1u);
            mbar_init(b_empty(s), 1u);
        }
        for (int acc = 0; acc < 2; ++acc) {
            mbar_init(tfull(acc), 1u);
            mbar_init(tempty(acc), (kPair ? 2u : 1u) * kEpiWarps);  // epilogue warps (of both CTAs)
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpTma && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
        if (!kFusedA) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
    }
    if (warp == kWarpMma) {
        if constexpr (kPair)
            tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        else
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Launched as a programmatic dependent, the kernel may start while the
    // kernel before it in the stream (the gather that writes the A operand, or
    // the previous call) still runs.  The roles that touch memory earlier work
    // writes wait for it (pdl_wait) first: the A producer and the epilogue.
    // The wkv producer does not: wkv is written only at bind, so the first wkv
    // stages load while the gather finishes.  The kernel after this one (the
    // gate) may be scheduled as CTAs of this one exit.
    pdl_launch_dependents();

    // work items: (M unit, N tile, split); a CTA pair shares one item sequence
    // and its M unit is two M blocks, this CTA's being 2 mu + rank
    int m_units = kPair ? (a.m_blocks + 1) / 2 : a.m_blocks;
    int total = m_units * a.n_tiles * a.k_splits;
    // Compaction (MmaArgs::block_text): the item sequence covers only the M
    // units that hold a text row; bit u of units_on is unit u.  Set by
    // compact_units() in every role alike, after pdl_wait.
    uint64_t units_on = 0;
    bool compact = false;
    const int item0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int istep = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    auto coords = [&](int tile, int& mb, int& nt, int& ks) {
        tile_coords(a, m_units, tile, mb, nt, ks);
        if (compact) {  // the mb-th unit that holds text (__fns: n-th set bit)
            const uint32_t lo = (uint32_t)units_on, hi = (uint32_t)(units_on >> 32);
            const int nlo = __popc(lo);
            mb = mb < nlo ? (int)__fns(lo, 0, mb + 1) : 32 + (int)__fns(hi, 0, mb - nlo + 1);
        }
        if constexpr (kPair) mb = 2 * mb + (int)rank;
    };
    const int KB = a.K / kBK;
    const long long lim = a.wait_limit_ns;
    // With a TMA-fed A, each N tile walks its k-blocks from its own starting
    // point, so that the CTAs in flight do not all read the same A k-block
    // (the operand matrix of a small batch is shared by every N tile) at the
    // same moment.  Gathered A operands come in order.
    auto k_rotation = [&](int nt, int nkb) { return kFusedA ? 0 : (nt * 13) % nkb; };

    // Work items of this CTA (a pair shares them).  Without stream K: the
    // (tile, split)s item0, item0 + istep, ...  With stream K: first the
    // pieces of this unit's contiguous range [g0, g1) of the (tile, stage)
    // sequence of the launch's first sk_tiles tiles, one piece per tile the
    // range touches; then whole tiles sk_tiles + k istep + unit, k = 0 ..
    // dp_waves - 1.  sk_tiles is what is left of the tiles after whole waves
    // of one tile per unit (all of them when there are fewer tiles than
    // units), so every unit gets the same number of stages, and each unit's
    // last item is a whole tile: the pieces that wait for parked partials
    // finish while the whole tiles' MMAs run, not after the last MMA.
    const int nst_tile = KB / kKS;
    const bool sk = (kMode == kEpiStoreKv && a.stream_k != 0) || kMode == kEpiForwardSk;
    const int tiles_all = m_units * a.n_tiles;
    const int dp_waves = sk ? tiles_all / istep : 0;
    const int sk_tiles = tiles_all - dp_waves * istep;
    const int64_t sk_total = (int64_t)sk_tiles * nst_tile;
    auto sk_start = [&](int u) { return (int64_t)u * sk_total / istep; };
    const int64_t sk_g0 = sk_start(item0), sk_g1 = sk_start(item0 + 1);
    const int sk_j0 = (int)(sk_g0 / nst_tile);
    const int n_sk_items = sk_g1 > sk_g0 ? (int)((sk_g1 - 1) / nst_tile) - sk_j0 + 1 : 0;
    int n_items = sk ? n_sk_items + dp_waves
                     : (item0 < total ? (total - item0 + istep - 1) / istep : 0);
    // item i: output tile (mb, nt), split ks, k-blocks [kb_lo, kb_lo + nkb), and
    // its stage range [st_lo, st_hi) within the tile's nst_tile stages
    auto get_item = [&](int i, int& mb, int& nt, int& ks, int& kb_lo, int& nkb, int& st_lo,
                        int& st_hi) {
        if (sk && i >= n_sk_items) {  // a whole tile
            coords(sk_tiles + (i - n_sk_items) * istep + item0, mb, nt, ks);
            st_lo = 0;
            st_hi = nst_tile;
            kb_lo = 0;
            nkb = KB;
        } else if (sk) {
            const int j = sk_j0 + i;
            coords(j, mb, nt, ks);
            const int64_t base = (int64_t)j * nst_tile;
            st_lo = (int)(max(sk_g0, base) - base);
            st_hi = (int)(min(sk_g1, base + nst_tile) - base);
            kb_lo = st_lo * kKS;
            nkb = (st_hi - st_lo) * kKS;
        } else {
            coords(item0 + i * istep, mb, nt, ks);
            kb_lo = ks * KB / a.k_splits;
            nkb = (ks + 1) * KB / a.k_splits - kb_lo;
            st_lo = 0;
            st_hi = nkb / kKS;
        }
    };

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(a.err, kErrTimeout);
    };

    // Compaction of a batch with long image spans (TMA-fed operand, whole
    // tiles, at most 64 units): the units whose blocks hold only image rows
    // get no items at all, so the work left stays evenly spread over the
    // CTAs; those rows pass through and their gates are written as 0 (the
    // epilogue, below).  Called by all 32 lanes of a warp, after pdl_wait:
    // the staging kernel writes the flags.
    const bool may_compact = kMode == kEpiForwardCompact && !kFusedA && !sk && a.k_splits == 1 &&
                             a.block_text != nullptr && m_units <= 64;
    auto compact_units = [&]() {
        if (!may_compact) return;
        uint64_t on = 0;
        for (int base = 0; base < m_units; base += 32) {
            const int u = base + lane;
            bool text = false;
            if (u < m_units) {
                const int b0 = kPair ? 2 * u : u;
                text = a.block_text[b0] != 0u ||
                       (kPair && b0 + 1 < a.m_blocks && a.block_text[b0 + 1] != 0u);
            }
            on |= (uint64_t)__ballot_sync(0xFFFFFFFFu, text) << base;
        }
        units_on = on;
        compact = true;
        m_units = __popcll((long long)on);
        total = m_units * a.n_tiles * a.k_splits;
        n_items = item0 < total ? (total - item0 + istep - 1) / istep : 0;
    };

    if (warp >= kWarpTma) {
        setmaxnreg_dec<kRegsCtl>();
    }
    if (warp == kWarpTma || (!kFusedA && warp == kWarpTmaA)) {
        // TMA producers: warp 12 loads the wkv tiles, warp 14 the A tiles of
        // the TMA-fed variants, each running ahead on its own ring
        const bool do_b = warp == kWarpTma;
        if (!do_b || may_compact) pdl_wait();
        compact_units();
        // with one M unit every wkv byte is read once per launch: its lines
        // are marked for early eviction, so that they do not push the
        // launch's outputs (the kv of a small batch) out of L2
        const bool wkv_once = m_units == 1;
        const uint64_t policy = l2_evict_first_policy();
        // the operand matrix is read once per N tile: its lines stay in L2
        // before any wkv line is evicted for them
        const uint64_t policy_a = l2_evict_last_policy();
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int i = 0; i < n_items && ok; ++i) {
                int mb, nt, ks, kb_lo, nkb, st_lo, st_hi;
                get_item(i, mb, nt, ks, kb_lo, nkb, st_lo, st_hi);
                const int n0 = (a.n_tile_begin + nt) * kBN;
                // stages of kKS k-blocks (the host keeps every split's range a
                // multiple of kKS); a stream-K piece walks its range in order
                const int nst = nkb / kKS;
                const int rot = sk ? 0 : k_rotation(nt, nst);
                for (int j = 0; j < nst && !a.starve_b; ++j, ++it) {
                    const int kb = kb_lo + ((j + rot) % nst) * kKS;  // first k-block of the stage
                    const int sb = it % kB;
                    if (do_b) {
                        if (!mbar_wait(b_empty(sb), ((uint32_t)(it / kB) & 1u) ^ 1u, abort_flag, lim)) {
                            fail();
                            ok = false;
                            break;
                        }
                        // wkv rows [r, r + 128) of k-block kb: in the tiled FP16 copy,
                        // box row ((r / 128) KB + kb) 128 at column 0 (a box of kKS
                        // tiles holds the stage's kKS k-blocks)
                        auto b_x = [&](int r) { return a.b_tiled ? 0 : kb * kBK; };
                        auto b_y = [&](int r) { return a.b_tiled ? ((r >> 7) * KB + kb) * 128 : r; };
                        if constexpr (kPair) {
                            // each CTA loads its half of the wkv tile (rows n0 + 128
                            // rank) and signals the issuer, who expects both halves
                            const int r = n0 + (int)rank * (kBN / 2);
                            if (issuer) mbar_expect_tx(b_full(sb), 2 * L::kBStageBytes);
                            if (wkv_once)
                                tma_load_2d_pair_hint(b_stage(sb), &tmB, map_rank(b_full(sb), 0),
                                                      b_x(r), b_y(r), policy);
                            else
                                tma_load_2d_pair(b_stage(sb), &tmB, map_rank(b_full(sb), 0), b_x(r),
                                                 b_y(r));
                        } else {
                            mbar_expect_tx(b_full(sb), L::kBStageBytes);
                            auto load = [&](uint32_t dst, int x, int y) {
                                if (wkv_once)
                                    tma_load_2d_hint(dst, &tmB, b_full(sb), x, y, policy);
                                else
                                    tma_load_2d(dst, &tmB, b_full(sb), x, y);
                            };
                            if (a.b_tiled) {  // two 128-row boxes, the second 16 KB further
                                load(b_stage(sb), b_x(n0), b_y(n0));
                                load(b_stage(sb) + kBStageHalf, b_x(n0 + 128), b_y(n0 + 128));
                            } else {
                                load(b_stage(sb), kb * kBK, n0);
                            }
                        }
                    } else {
                        const int sa = it % kA;
                        if (!mbar_wait(a_empty(sa), ((uint32_t)(it / kA) & 1u) ^ 1u, abort_flag, lim)) {
                            fail();
                            ok = false;
                            break;
                        }
                        // the operand of M block mb, k-block kb: row-major [T][K], or
                        // in 128 x 64 tiles at box row (mb KB + kb) 128
                        const int ax = a.a_tiled ? 0 : kb * kBK;
                        const int ay = a.a_tiled ? (mb * KB + kb) * 128 : mb * kBM;
                        if constexpr (kPair) {
                            if (issuer) mbar_expect_tx(a_full(sa), 2 * L::kAStageBytes);
                            tma_load_2d_pair_hint(a_stage(sa), &tmA, map_rank(a_full(sa), 0), ax, ay,
                                                  policy_a);
                        } else {
                            mbar_expect_tx(a_full(sa), L::kAStageBytes);
                            tma_load_2d_hint(a_stage(sa), &tmA, a_full(sa), ax, ay, policy_a);
                        }
                    }
                }
            }
        }
    } else if (warp == kWarpMma) {
        // waits on barriers that the other CTA of a pair arrives on use cluster scope
        auto wait = [&](uint32_t bar, uint32_t parity) {
            return kPair ? mbar_wait_cluster(bar, parity, abort_flag, lim)
                         : mbar_wait(bar, parity, abort_flag, lim);
        };
        if (may_compact) pdl_wait();
        compact_units();
        if (lane == 0 && issuer) {
            int it = 0, tc = 0;
            bool ok = true;
            for (; tc < n_items && ok; ++tc) {
                const int acc = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                if (!wait(tempty(acc), aph ^ 1u)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
                int mb_, nt_, ks, kb_lo, nkb, st_lo, st_hi;
                get_item(tc, mb_, nt_, ks, kb_lo, nkb, st_lo, st_hi);
                const int nst = nkb / kKS;
                for (int j = 0; j < nst; ++j, ++it) {
                    const int sa = it % kA, sb = it % kB;
                    if (!wait(a_full(sa), (uint32_t)(it / kA) & 1u) ||
                        !wait(b_full(sb), (uint32_t)(it / kB) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKS; ++kk) {  // the stage's k-blocks, one tile apart
                        const uint64_t ad = sdesc_sw128(a_stage(sa) + kk * (L::kAStageBytes / kKS));
                        const uint64_t bd = sdesc_sw128(b_stage(sb) + kk * (L::kBStageBytes / kKS));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {  // 16 elements = 32 bytes per MMA
                            const uint32_t accum = (j != 0) || (kk != 0) || (k != 0);
                            if constexpr (kPair)
                                umma_f16kind_pair(d_tmem, ad + 2ull * k, bd + 2ull * k,
                                                  idesc<kF16, 2 * kBM>(), accum);
                            else
                                umma_f16kind(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc<kF16>(),
                                             accum);
                        }
                    }
                    if constexpr (kPair) {  // frees the stage in both CTAs
                        umma_commit_pair(a_empty(sa));
                        umma_commit_pair(b_empty(sb));
                    } else {
                        umma_commit(a_empty(sa));
                        umma_commit(b_empty(sb));
                    }
                }
                if (ok) {
                    if constexpr (kPair)
                        umma_commit_pair(tfull(acc));
                    else
                        umma_commit(tfull(acc));
                }
            }
        }
    } else if (warp >= kWarpTma) {
        // warp 15 (and 14 with a gathered A): idle
    } else if (kWideEpi && warp < kFirstEpi) {
        setmaxnreg_dec<kRegsIdle>();  // warps 0..3 of a TMA-fed kernel: idle
    } else if (warp < kWarpEpi && !kWideEpi) {
        setmaxnreg_inc<kRegsProd>();
        if (kASrc == kASrcGatherBucket) {
            // whole-row gather; rows of this warp: [16 pw, 16 pw + 16); lanes
            // l and l + 16 both hash token 16 pw + (l % 16)
            const int pw = warp - kWarpProd;
            const int nbk = a.hp.nb;
            int it = 0;
            bool ok = true;
            BucketRows R0, R1;
            for (int tile = item0; tile < total && ok; tile += istep) {
                int mb, nt, ks;
                coords(tile, mb, nt, ks);
                // this split's buckets (the host splits K on bucket boundaries)
                const int b_lo = ks * nbk / a.k_splits, b_hi = (ks + 1) * nbk / a.k_splits;
                const int64_t t = (int64_t)mb * kBM + pw * kRowsPerProd + (lane & (kRowsPerProd - 1));
                const uint4 w = t < a.T ? a.windows[t] : make_uint4(kDead, kDead, kDead, kDead);
                uint32_t row0 = own_bucket_row(a, w, b_lo);
                uint2 sw0 = own_scale_word(a, row0);
                load_bucket(a, row0, lane, R0);
                uint2 sw1 = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
                // buckets in pairs so the two register sets keep static names
                auto run = [&](int b, const BucketRows& cur, uint2 cur_sw, BucketRows& nxt,
                               uint2& nxt_sw) -> bool {
                    if (b + 1 < b_hi) {  // the next bucket's loads go out first
                        const uint32_t r = own_bucket_row(a, w, b + 1);
                        nxt_sw = own_scale_word(a, r);
                        load_bucket(a, r, lane, nxt);
                    }
                    int freed = 1;
                    if (lane == 0) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (freed)
                                freed = mbar_wait(a_empty((it + j) % kA),
                                                  ((uint32_t)((it + j) / kA) & 1u) ^ 1u, abort_flag,
                                                  lim);
                    }
                    freed = __shfl_sync(0xFFFFFFFFu, freed, 0);
                    if (!freed) {
                        if (lane == 0) fail();
                        return false;
                    }
                    decode_bucket<kF16>(a, cur, cur_sw, a_base, kA, it, pw, lane);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) mbar_arrive(a_full((it + j) % kA));
                    }
                    it += 4;
                    return true;
                };
                for (int b = b_lo; b < b_hi && ok; b += 2) {
                    ok = run(b, R0, sw0, R1, sw1);
                    if (ok && b + 1 < b_hi) ok = run(b + 1, R1, sw1, R0, sw0);
                }
            }
        } else if (kASrc == kASrcGatherKb) {
            const int pw = warp - kWarpProd;        // rows [16 pw, 16 pw + 16) of the tile
            const int c = lane & 3;                 // 16-column chunk of each k-block
            const int m0 = pw * kRowsPerProd + (lane >> 2);  // this lane's rows: m0 + 8 j
            uint32_t* rows_s = reinterpret_cast<uint32_t*>(smem + L::kOffRows);
            int it = 0;
            bool ok = true;
            for (int tile = item0; tile < total && ok; tile += istep) {
                int mb, nt, ks;
                coords(tile, mb, nt, ks);
                const int kb_lo = ks * KB / a.k_splits, kb_hi = (ks + 1) * KB / a.k_splits;
                {   // hash: lanes l, l + 16 <-> token, every bucket, into the row-index table
                    const int m = pw * kRowsPerProd + (lane & (kRowsPerProd - 1));
                    const int64_t t = (int64_t)mb * kBM + m;
                    const uint4 w = t < a.T ? a.windows[t] : make_uint4(kDead, kDead, kDead, kDead);
                    for (int b = 0; b < a.hp.nb; ++b) {
                        uint32_t r = hash_bucket(a.hp, w, b);
                        if (r != kMasked && (uint64_t)r >= a.rows) {
                            atomicOr(a.err, kErrBounds);
                            r = kMasked;
                        }
                        rows_s[m * kRowStride + b] = r;
                    }
                }
                __syncwarp();
                // Ring of kPrefetch k-blocks of loads in flight.  The loop body
                // is unrolled kPrefetch times so every slot index is static:
                // a register that still awaits its load is never copied (a copy
                // would stall the warp until the load lands).
                RawKb q[kPrefetch];
#pragma unroll
                for (int i = 0; i < kPrefetch; ++i)
                    if (kb_lo + i < kb_hi) load_kb(a, rows_s, m0, c, kb_lo + i, q[i]);
                for (int kb0 = kb_lo; kb0 < kb_hi && ok; kb0 += kPrefetch) {
#pragma unroll
                    for (int u = 0; u < kPrefetch; ++u) {
                        const int kb = kb0 + u;
                        if (kb < kb_hi && ok) {
                            const int s = it % kA;
                            const uint32_t ph = (uint32_t)(it / kA) & 1u;
                            ++it;
                            // one lane waits for the stage to be free, the warp follows
                            int freed = 1;
                            if (lane == 0) freed = mbar_wait(a_empty(s), ph ^ 1u, abort_flag, lim);
                            freed = __shfl_sync(0xFFFFFFFFu, freed, 0);
                            if (!freed) {
                                if (lane == 0) fail();
                                ok = false;
                            } else {
                                store_kb<kF16>(q[u], a_stage(s), m0, c, a.a_exp_shift);
                                // every lane makes its writes visible to the tensor
                                // core's (async) proxy, then one arrival per warp
                                fence_proxy_async();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(a_full(s));
                                if (kb + kPrefetch < kb_hi) load_kb(a, rows_s, m0, c, kb + kPrefetch, q[u]);
                            }
                        }
                    }
                }
                __syncwarp();  // the row-index table is rewritten by the next tile
            }
        }
    } else {
        // ---- epilogue ----
        if constexpr (kWideEpi)
            setmaxnreg_inc<kRegsWideEpi>();
        else
            setmaxnreg_inc<kRegsEpi>();
        pdl_wait();
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        // the warp's group (of kG sharing the quadrant): its 32-column chunks
        // are c_first, c_first + kG, ...; its ready flag in a stream-K launch
        const int grp = (warp - kFirstEpi) >> 2;
        const int c_first = grp;
        constexpr int kCStep = kG;
        const int eslot = kWideEpi ? warp : q;
        const int m = q * 32 + lane;
        compact_units();
        if (compact && a.gates && grp == 0) {
            // units of image rows only (no items): their rows' gates are 0,
            // written by the CTA (pair) that unit index u % istep names
            for (int u = item0; u < (kPair ? (a.m_blocks + 1) / 2 : a.m_blocks); u += istep) {
                if ((units_on >> u) & 1u) continue;
                const int mb = kPair ? 2 * u + (int)rank : u;
                const int64_t t = (int64_t)mb * kBM + m;
                if (mb < a.m_blocks && t < a.T)
                    for (int b = 0; b < a.hc; ++b) a.gates[t * a.hc + b] = 0.0f;
            }
        }
        int tc = 0;
        // The fused kernels start L2 loads of the next tile's hidden slices (one
        // bulk prefetch per row and branch); the TMA-fed kernels do not: there
        // those prefetches share the copy engine with the operand and wkv
        // copies, and the 2,048-token call ran 0.393 ms with them against
        // 0.385 ms without.
        constexpr bool kPrefetchHidden = kFwdWhole && kFusedA;
        if (kPrefetchHidden && item0 < total && grp == 0) {
            int mb, nt, ks;
            coords(item0, mb, nt, ks);
            if (mb < a.m_blocks) prefetch_hidden(a, mb, nt, m);
        }
        for (; tc < n_items; ++tc) {
            const int tile = item0 + tc * istep;  // (without stream K)
            int mb, nt, ks, kb_lo, nkb, st_lo, st_hi;
            get_item(tc, mb, nt, ks, kb_lo, nkb, st_lo, st_hi);
            // the next tile's hidden slices travel to L2 while this one is finished
            if (kPrefetchHidden && tile + istep < total && grp == 0) {
                int mb2, nt2, ks2;
                coords(tile + istep, mb2, nt2, ks2);
                if (mb2 < a.m_blocks) prefetch_hidden(a, mb2, nt2, m);
            }
            const int acc = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            const int64_t t = (int64_t)mb * kBM + m;
            const int n0 = (a.n_tile_begin + nt) * kBN;
            // Stream K, the tile's first piece (this range's last item, or a
            // whole tile): the tile's later stages, if any, lie in the ranges
            // of the next units, each of which holds one of them as its first
            // piece, parked in its slot long before.  Their flags are waited
            // for (bounded), and the first chunk's operands loaded, while the
            // MMAs of this item still run; each later chunk's operands load
            // while the chunk before it is finished.
            constexpr bool kSkEpi = kMode == kEpiStoreKv || kMode == kEpiForwardSk;
            const bool sk_finish = kSkEpi && sk && st_lo == 0 && mb < a.m_blocks;
            int u_last = item0;
            if (sk_finish && st_hi < nst_tile) {
                const int64_t g_end = (int64_t)(sk_j0 + tc) * nst_tile + nst_tile - 1;
                u_last = (int)(((g_end + 1) * istep - 1) / sk_total);
                int ready = 1;
                if (lane == 0) {
                    const uint64_t t0 = globaltimer();
                    for (int u = item0 + 1; u <= u_last && ready; ++u) {
                        if (sk_start(u) == sk_start(u + 1)) continue;  // an empty range
                        const uint32_t* f = a.sk_flags +
                                            (kPair ? 2 * u + (int)rank : u) * kSkFlagsPerCta + eslot;
                        uint32_t n = 0;
                        while (ld_acquire_u32(f) == 0u) {
                            if ((++n & 63u) == 0u &&
                                ((long long)(globaltimer() - t0) > lim || *abort_flag)) {
                                ready = 0;
                                break;
                            }
                        }
                    }
                }
                ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
                if (!ready) {
                    if (lane == 0) fail();
                    break;
                }
                // the warp's later loads of the parked pieces are ordered after
                // lane 0's acquire (a full fence here would first wait for the
                // stores of the item before)
                __syncwarp();
            }
            // The parked pieces to add, in unit order (which is k order): the
            // first (u1; -1 for none) is loaded with the chunk's other operands,
            // any later ones (u_rest .. u_last: ranges shorter than a tile) one
            // after another.
            int u1 = -1, u_rest = u_last + 1;
            for (int u = item0 + 1; u <= u_last; ++u) {
                if (sk_start(u) == sk_start(u + 1)) continue;  // an empty range
                if (u1 < 0) {
                    u1 = u;
                } else {
                    u_rest = u;
                    break;
                }
            }
            auto slot_src = [&](int u, int c) {
                return reinterpret_cast<const float4*>(a.sk_slots) +
                       (int64_t)(kPair ? 2 * u + (int)rank : u) * (kBM * kBN / 4) + q * (kBN / 4) * 32 +
                       c * 8 * 32 + lane;
            };
            // v[0..31] += the parked pieces of chunk c (x1 loaded already)
            auto add_parked = [&](float* v, const float4* x1, int c) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (u1 >= 0) {
                        v[4 * i] += x1[i].x;
                        v[4 * i + 1] += x1[i].y;
                        v[4 * i + 2] += x1[i].z;
                        v[4 * i + 3] += x1[i].w;
                    }
                }
#pragma unroll 1
                for (int u = u_rest; u <= u_last; ++u) {
                    if (sk_start(u) == sk_start(u + 1)) continue;
                    const float4* src = slot_src(u, c);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 x = __ldcg(src + i * 32);
                        v[4 * i] += x.x;
                        v[4 * i + 1] += x.y;
                        v[4 * i + 2] += x.z;
                        v[4 * i + 3] += x.w;
                    }
                }
            };
            // kEpiForwardSk key tile: the rows' hidden slice of this branch
            const bool key_tile = kMode == kEpiForwardSk && n0 < a.hc * a.d;
            const int branch = key_tile ? n0 / a.d : 0;
            const int col0 = n0 - branch * a.d;
            const bool text = key_tile && t < a.T && a.windows[t].x != kDead;
            const uint16_t* hrow = text ? a.hidden + (t * a.hc + branch) * (int64_t)a.d + col0 : nullptr;
            // Operands of chunk c: the hidden slice (key tiles of text rows),
            // w_q w_k of column 32 c + lane (passed round the warp by shuffles)
            // and the parked piece u1.  The first chunk's are loaded before
            // the accumulator is ready, each later chunk's while the chunk
            // before it is finished.
            const float* wqkr = key_tile ? a.wqk + (int64_t)branch * a.d + col0 : nullptr;
            uint4 hv_n[4];
            float wq_n = 0.f;
            float4 x_n[8];
            auto issue = [&](int c) {
                if (key_tile) wq_n = __ldg(wqkr + c * 32 + lane);
                if (text) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) hv_n[i] = __ldg(reinterpret_cast<const uint4*>(hrow + c * 32) + i);
                }
                if (u1 >= 0) {
                    const float4* src = slot_src(u1, c);
#pragma unroll
                    for (int i = 0; i < 8; ++i) x_n[i] = __ldcg(src + i * 32);
                }
            };
            if (sk_finish) issue(c_first);
            int full_ok = 1;
            if (lane == 0) full_ok = mbar_wait(tfull(acc), aph, abort_flag, lim);
            full_ok = __shfl_sync(0xFFFFFFFFu, full_ok, 0);
            if (!full_ok) {
                if (lane == 0) fail();
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(acc * kBN) + ((uint32_t)(q * 32) << 16);
            // an odd pair CTA past the last M block has no rows to write
            int holds_sum = mb < a.m_blocks ? 1 : 0;
            if (holds_sum && kFwdWhole && a.k_splits > 1) {
                holds_sum = split_k_quadrant(a, mb, nt, ks, q, lane, taddr, abort_flag, lim);
                if (holds_sum < 0) {
                    if (lane == 0) fail();
                    break;
                }
            }
            if (!holds_sum) {
                // partial parked for the split that arrives last
            } else if ((kMode == kEpiStoreKv || kMode == kEpiForwardSk) && sk && st_lo > 0) {
                // stream K, a piece after the tile's first: park the raw
                // accumulator in this CTA's slot ([quadrant][chunk][float4][lane],
                // 512 contiguous bytes per warp store) and raise the quadrant's flag
                const int cta = (int)blockIdx.x;
                float4* const slot = reinterpret_cast<float4*>(a.sk_slots) +
                                     (int64_t)cta * (kBM * kBN / 4) + q * (kBN / 4) * 32 + lane;
#pragma unroll 1
                for (int c = c_first; c < kBN / 32; c += kCStep) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)(c * 32), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        __stcg(slot + (c * 8 + i) * 32,
                               make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                           __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_u32(a.sk_flags + cta * kSkFlagsPerCta + eslot, 1u);
            } else if (kSkEpi) {
                // kEpiForwardSk: a key tile publishes its gate sums; a value
                // tile stores its 256 columns of v into kv = v [T][d]
                const int kv_col0 = kMode == kEpiForwardSk ? a.hc * a.d : 0;
                if (key_tile) {
                    float skk = 0.f, shh = 0.f, shk = 0.f;
#pragma unroll 1
                    for (int c = c_first; c < kBN / 32; c += kCStep) {
                        uint4 hv[4];
                        const float wq = wq_n;
#pragma unroll
                        for (int i = 0; i < 4; ++i) hv[i] = hv_n[i];
                        uint32_t r[32];
                        tmem_ld32(taddr + (uint32_t)(c * 32), r);
                        tmem_wait_ld();
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        add_parked(v, x_n, c);
                        if (c + kCStep < kBN / 32) issue(c + kCStep);  // hv_n, x_n are free again
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                // every lane takes part in the shuffle; image rows add nothing
                                const float wqk = __shfl_sync(0xFFFFFFFFu, wq, 8 * i + e);
                                if (text) {
                                    const float h = (e & 1) ? bf16_hi(hw[e >> 1]) : bf16_lo(hw[e >> 1]);
                                    const float k = v[8 * i + e] * a.out_scale;
                                    skk = fmaf(k, k, skk);
                                    shh = fmaf(h, h, shh);
                                    shk = fmaf(h * wqk, k, shk);
                                }
                            }
                        }
                    }
                    if (text) {
                        // [token][branch][column tile][group][3]
                        const int P = a.d / kBN;
                        float* pp =
                            a.partials + (((t * a.hc + branch) * P + col0 / kBN) * kG + grp) * 3;
                        pp[0] = skk;
                        pp[1] = shh;
                        pp[2] = shk;
                    }
                } else {
                // A lane holds 32 columns of its own row.  An 8 x 8 transpose of
                // float4 within each group of 8 lanes (three butterfly rounds of
                // shuffles) gives lane 8 g + j the float4 j of rows 8 g .. 8 g + 7,
                // so that each store writes four whole 128-byte row segments
                // instead of 32 scattered 16-byte pieces.
                const int g8 = lane & ~7, j8 = lane & 7;
                float* const kv0 = a.kv + ks * a.kv_split_stride + (n0 - kv_col0) + j8 * 4;
                const int64_t row0 = (int64_t)mb * kBM + q * 32 + g8;
#pragma unroll 1
                for (int c = c_first; c < kBN / 32; c += kCStep) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)(c * 32), r);
                    tmem_wait_ld();
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    add_parked(v, x_n, c);
                    if (c + kCStep < kBN / 32) issue(c + kCStep);  // x_n is free again
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= a.out_scale;
                    if (a.kv_bf16) {
                        // kv rounded once to BF16: the lane's 64 bytes are four
                        // 16-byte pieces; a 4 x 4 transpose within each group of 4
                        // lanes gives lane 4 g + j piece j of rows 4 g .. 4 g + 3,
                        // so that each store writes eight whole 64-byte segments
                        uint32_t o[4][4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2)
                                o[i][e2] = bf16x2_pack_rn(v[8 * i + 2 * e2], v[8 * i + 2 * e2 + 1]);
#pragma unroll
                        for (int msk = 1; msk < 4; msk <<= 1) {
                            const bool upper = (lane & msk) != 0;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if ((e & msk) == 0) {
#pragma unroll
                                    for (int f = 0; f < 4; ++f) {
                                        const uint32_t out = upper ? o[e][f] : o[e ^ msk][f];
                                        const uint32_t in = __shfl_xor_sync(0xFFFFFFFFu, out, msk);
                                        if (upper)
                                            o[e][f] = in;
                                        else
                                            o[e ^ msk][f] = in;
                                    }
                                }
                            }
                        }
                        const int64_t row4 = (int64_t)mb * kBM + q * 32 + (lane & ~3);
                        uint16_t* const kvb = reinterpret_cast<uint16_t*>(a.kv) + (n0 - kv_col0) + c * 32 +
                                              (lane & 3) * 8;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (row4 + i < a.T)
                                *reinterpret_cast<uint4*>(kvb + (row4 + i) * a.ldkv) =
                                    make_uint4(o[i][0], o[i][1], o[i][2], o[i][3]);
                        continue;
                    }
#pragma unroll
                    for (int msk = 1; msk < 8; msk <<= 1) {
                        const bool upper = (lane & msk) != 0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            if ((e & msk) == 0) {
#pragma unroll
                                for (int f = 0; f < 4; ++f) {
                                    const float out = upper ? v[4 * e + f] : v[4 * (e ^ msk) + f];
                                    const float in = __shfl_xor_sync(0xFFFFFFFFu, out, msk);
                                    if (upper)
                                        v[4 * e + f] = in;
                                    else
                                        v[4 * (e ^ msk) + f] = in;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int64_t tr = row0 + i;
                        if (tr < a.T)
                            *reinterpret_cast<float4*>(kv0 + tr * a.ldkv + c * 32) =
                                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                }
                }  // kv store
            } else if (kFwdWhole && n0 < a.hc * a.d) {
                const int branch = n0 / a.d;
                const int col0 = n0 - branch * a.d;
                const bool text = t < a.T && a.windows[t].x != kDead;
                const uint16_t* hrow = a.hidden + (t * a.hc + branch) * (int64_t)a.d + col0;
                const float* wqkr = a.wqk + (int64_t)branch * a.d + col0;
                float skk = 0.f, shh = 0.f, shk = 0.f;
#pragma unroll 1
                for (int c = c_first; c < kBN / 32; c += kCStep) {
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
                            const float4 p0 = __ldg(reinterpret_cast<const float4*>(wqkr + c * 32) + 2 * i);
                            const float4 p1 = __ldg(reinterpret_cast<const float4*>(wqkr + c * 32) + 2 * i + 1);
                            const float wqk[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                            const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float h = (e & 1) ? bf16_hi(hw[e >> 1]) : bf16_lo(hw[e >> 1]);
                                const float k = __uint_as_float(r[8 * i + e]) * a.out_scale;
                                skk = fmaf(k, k, skk);
                                shh = fmaf(h, h, shh);
                                shk = fmaf(h * wqk[e], k, shk);
                            }
                        }
                    }
                }
                if (text) {
                    // [token][branch][column tile][group][3]
                    const int P = a.d / kBN;
                    float* pp =
                        a.partials + (((t * a.hc + branch) * P + col0 / kBN) * kG + grp) * 3;
                    pp[0] = skk;
                    pp[1] = shh;
                    pp[2] = shk;
                }
                if (kFwdWhole) {
                    // publish the warp's sums and count them in for its quadrant;
                    // the quadrant's last key tile turns the sums into gates and
                    // raises the quadrant's gates-ready flag
                    uint32_t* const cnt = a.counters + 2 * (mb * 4 + q);
                    __threadfence();
                    __syncwarp();
                    uint32_t done = 0;
                    if (lane == 0) done = atomicAdd(cnt, 1u) + 1u;
                    done = __shfl_sync(0xFFFFFFFFu, done, 0);
                    if (done == (uint32_t)(a.hc * a.d / kBN * kG)) {
                        __threadfence();
                        float g[8];
                        if (text) row_gates(a, t, kG, g);
                        if (t < a.T) {
                            for (int b = 0; b < a.hc; ++b) {
                                const float gb = text ? g[b] : 0.f;
                                a.gbuf[t * a.hc + b] = gb;
                                if (a.gates) a.gates[t * a.hc + b] = gb;
                            }
                        }
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) st_release_u32(cnt + 1, 1u);
                    }
                }
            } else {  // value tile
                if (kFwdWhole) {
                    // wait (bounded) for the gates of this M block quadrant
                    if (lane == 0) {
                        const uint64_t t0 = globaltimer();
                        uint32_t n = 0;
                        while (ld_acquire_u32(a.counters + 2 * (mb * 4 + q) + 1) == 0u) {
                            if ((++n & 63u) == 0u &&
                                ((long long)(globaltimer() - t0) > lim || *abort_flag)) {
                                fail();
                                break;
                            }
                        }
                    }
                    __syncwarp();
                    __threadfence();
                }
                const int cv = n0 - a.hc * a.d;
                const bool text = t < a.T && a.windows[t].x != kDead;
                float g[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) g[b] = 0.f;
                if (text) {
                    if (a.hc == 4) {
                        const float4 g4 = __ldcg(reinterpret_cast<const float4*>(a.gbuf + t * 4));
                        g[0] = g4.x;
                        g[1] = g4.y;
                        g[2] = g4.z;
                        g[3] = g4.w;
                    } else {
#pragma unroll
                        for (int b = 0; b < 8; ++b)
                            if (b < a.hc) g[b] = __ldcg(a.gbuf + t * a.hc + b);
                    }
                }
                // hidden += g v, two branches per round: their eight loads go out
                // before any store (a store could alias a later load, so loads
                // issued after it would each wait for memory in turn)
                uint16_t* const hrow = a.hidden + t * a.hc * (int64_t)a.d + cv;
#pragma unroll 1
                for (int c = c_first; c < kBN / 32; c += kCStep) {
                    uint32_t r[32];
                    tmem_ld32(taddr + (uint32_t)(c * 32), r);
                    tmem_wait_ld();
                    if (text) {
#pragma unroll
                        for (int b0 = 0; b0 < 8; b0 += 2) {
                            if (b0 < a.hc) {
                                uint4 hv[2][4];
#pragma unroll
                                for (int bb = 0; bb < 2; ++bb)
                                    if (b0 + bb < a.hc) {
                                        const uint4* hp = reinterpret_cast<const uint4*>(
                                            hrow + (int64_t)(b0 + bb) * a.d + c * 32);
#pragma unroll
                                        for (int i = 0; i < 4; ++i) hv[bb][i] = hp[i];
                                    }
#pragma unroll
                                for (int bb = 0; bb < 2; ++bb)
                                    if (b0 + bb < a.hc) {
                                        uint4* hp = reinterpret_cast<uint4*>(
                                            hrow + (int64_t)(b0 + bb) * a.d + c * 32);
                                        const float gb = g[b0 + bb];
#pragma unroll
                                        for (int i = 0; i < 4; ++i) {
                                            const uint32_t hw[4] = {hv[bb][i].x, hv[bb][i].y,
                                                                    hv[bb][i].z, hv[bb][i].w};
                                            uint32_t o[4];
#pragma unroll
                                            for (int e2 = 0; e2 < 4; ++e2) {
                                                const float v0 = __uint_as_float(r[8 * i + 2 * e2]) * a.out_scale;
                                                const float v1 = __uint_as_float(r[8 * i + 2 * e2 + 1]) * a.out_scale;
                                                o[e2] = bf16x2_pack_rn(fmaf(gb, v0, bf16_lo(hw[e2])),
                                                                       fmaf(gb, v1, bf16_hi(hw[e2])));
                                            }
                                            hp[i] = make_uint4(o[0], o[1], o[2], o[3]);
                                        }
                                    }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (kPair)  // the issuer's barrier counts the epilogue warps of both CTAs
                    mbar_arrive_cluster(map_rank(tempty(acc), 0));
                else
                    mbar_arrive(tempty(acc));
            }
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
    // a pair leaves together: no arrival or multicast may target a CTA that exited
    if constexpr (kPair) cluster_sync();
    if (warp == kWarpMma) {
        tc_fence_after();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <int kASrc, bool kF16, int kMode>
cudaError_t launch(const MmaArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                   cudaStream_t s) {
    static bool attr_set = false;
    auto kern = k_mma<kASrc, kF16, kMode>;
    constexpr int kSmem = Layout<kASrc, k_blocks_per_stage<kASrc, kF16>(), kMode>::kBytes;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // work units: the (tile, split)s, or with stream K the (tile, stage)s
    constexpr int kKS = k_blocks_per_stage<kASrc, kF16>();
    // stream K: the kv-store epilogue, or the gate-sum epilogue of kEpiForwardSk
    // (which always runs it), on a TMA-fed operand, one split
    if ((kMode == kEpiForwardSk) != (a.stream_k && kMode != kEpiStoreKv)) return cudaErrorInvalidValue;
    if (a.stream_k && (kMode == kEpiForward || a.k_splits != 1 || (a.K / kBK) % kKS != 0 ||
                       (kMode == kEpiForwardSk && kASrc != kASrcTma && kASrc != kASrcTmaPair)))
        return cudaErrorInvalidValue;
    if ((kMode == kEpiForward || kMode == kEpiForwardSk || kMode == kEpiForwardCompact) &&
        a.epi_groups != epilogue_groups<kASrc>())
        return cudaErrorInvalidValue;
    const int stages = a.stream_k ? (a.K / kBK) / kKS : a.k_splits;
    if (kASrc == kASrcTmaPair) {
        // clusters of two; no more pairs than can be resident at once, since
        // the forward epilogue's tiles (and stream-K pieces) wait on tiles of
        // other CTAs
        const int units = (a.m_blocks + 1) / 2 * a.n_tiles * stages;
        if (units == 0) return cudaSuccess;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * (device_sm_count() / 2));
        int resident = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (resident < 1) return cudaErrorLaunchOutOfResources;
        cfg.gridDim = dim3(2 * std::min(units, std::min(resident, device_sm_count() / 2)));
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, a);
    }
    const int total = a.m_blocks * a.n_tiles * stages;
    if (total == 0) return cudaSuccess;
    // programmatic dependent launch (see pdl_wait)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(std::min(total, device_sm_count()));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, a);
}

template <int kASrc, bool kF16>
cudaError_t launch_mode(const MmaArgs& a, int mode, const CUtensorMap& tmB, cudaStream_t s) {
    if (mode == kEpiForward) return launch<kASrc, kF16, kEpiForward>(a, tmB, tmB, s);
    return launch<kASrc, kF16, kEpiStoreKv>(a, tmB, tmB, s);
}

}  // namespace
cudaError_t make_tma_16bit(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, bool f16) {
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
    CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_project(const MmaArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           cudaStream_t s) {
    return launch<kASrcTma, false, kEpiStoreKv>(a, tmA, tmB, s);
}


cudaError_t launch_project_tma(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, cudaStream_t s) {
    if (f16) return launch<kASrcTma, true, kEpiStoreKv>(a, tmA, tmB, s);
    return launch<kASrcTma, false, kEpiStoreKv>(a, tmA, tmB, s);
}

cudaError_t launch_project_tma_pair(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                                    const CUtensorMap& tmB_half, cudaStream_t s) {
    if (f16) return launch<kASrcTmaPair, true, kEpiStoreKv>(a, tmA, tmB_half, s);
    return launch<kASrcTmaPair, false, kEpiStoreKv>(a, tmA, tmB_half, s);
}

cudaError_t launch_forward_tma_pair(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                                   const CUtensorMap& tmB_half, cudaStream_t s) {
    if (a.block_text)  // compacted over the units that hold text
        return f16 ? launch<kASrcTmaPair, true, kEpiForwardCompact>(a, tmA, tmB_half, s)
                   : launch<kASrcTmaPair, false, kEpiForwardCompact>(a, tmA, tmB_half, s);
    if (f16) return launch<kASrcTmaPair, true, kEpiForward>(a, tmA, tmB_half, s);
    return launch<kASrcTmaPair, false, kEpiForward>(a, tmA, tmB_half, s);
}

cudaError_t launch_forward_tma(const MmaArgs& a, bool f16, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, cudaStream_t s) {
    if (a.block_text)
        return f16 ? launch<kASrcTma, true, kEpiForwardCompact>(a, tmA, tmB, s)
                   : launch<kASrcTma, false, kEpiForwardCompact>(a, tmA, tmB, s);
    if (f16) return launch<kASrcTma, true, kEpiForward>(a, tmA, tmB, s);
    return launch<kASrcTma, false, kEpiForward>(a, tmA, tmB, s);
}

cudaError_t launch_forward_sk(const MmaArgs& a, bool f16, bool pairs, const CUtensorMap& tmA,
                              const CUtensorMap& tmB, cudaStream_t s) {
    if (pairs)
        return f16 ? launch<kASrcTmaPair, true, kEpiForwardSk>(a, tmA, tmB, s)
                   : launch<kASrcTmaPair, false, kEpiForwardSk>(a, tmA, tmB, s);
    return f16 ? launch<kASrcTma, true, kEpiForwardSk>(a, tmA, tmB, s)
               : launch<kASrcTma, false, kEpiForwardSk>(a, tmA, tmB, s);
}

// Operand paths of the fused kernels: bucket gather (256-wide rows) or k-block
// gather, with FP16 operands; k-block gather with BF16 operands.
cudaError_t launch_forward_phase(const MmaArgs& a, int mode, bool f16, bool bucket,
                                 const CUtensorMap& tmB, cudaStream_t s) {
    if (f16 && bucket) return launch_mode<kASrcGatherBucket, true>(a, mode, tmB, s);
    if (f16) return launch_mode<kASrcGatherKb, true>(a, mode, tmB, s);
    return launch_mode<kASrcGatherKb, false>(a, mode, tmB, s);
}

}  // namespace engram
