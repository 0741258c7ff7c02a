// engram_forward_noalloc: the fused forward for callers that may not allocate
// device memory.
//
// Some hosts of this library own all of the GPU's memory: a serving engine
// that reserves nearly all HBM for its KV-cache pool at start-up and hands
// memory out only through its own allocator, or a plugin framework whose
// plugins are not allowed to allocate.  Such callers can pass the inputs and
// outputs they already own, but cannot hand engram_forward a freshly
// allocated workspace, and a cudaMalloc/cudaFree inside a hot path would also
// synchronise the device.  This entry point keeps the forward's scratch (the
// per-token, per-branch, per-tile gate sums, the gates and the tile counters)
// in a fixed buffer that is part of the library's device image: it is
// reserved on every GPU that loads the library and stays there until the
// process exits.
//
// The buffer is shared by every call in the process.  Each call zeroes its
// counters on its stream and its key tiles write every sum and gate its value
// tiles read, but two calls whose kernels overlap on the GPU - on different
// streams, or from different threads - race on it.  Order such calls on one
// stream, or use engram_forward with a workspace per stream.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/engram.h"

namespace engram {
void set_last_error(const std::string& msg);
// The fused forward with its split-K factor capped at max_splits, and its
// workspace size (engram_api.cpp).
engram_status forward_fused(const engram_ctx* ctx, int layer, const uint32_t* d_windows,
                            int64_t T, uint16_t* d_hidden, void* d_workspace, float* d_gates,
                            void* stream, int max_splits);
size_t forward_workspace_bytes(const engram_ctx* ctx, int64_t T, int max_splits);
engram_status check_forward_call(const engram_ctx* ctx, int layer, int64_t T);
}

namespace {

constexpr size_t kScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_forward_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch buffer on the current device.  The address is
// looked up once per device, with that device current, on the first call made
// on it, and kept until the process exits; host code must not use the symbol
// itself (on the host it names a stand-in object, not device memory).  A
// cudaDeviceReset unloads the library's device image, so the kept address (like
// every context bound on that device) is not valid after one.
engram_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        engram::set_last_error("engram_forward_noalloc: no usable current device");
        return ENGRAM_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_forward_scratch);
        if (e != cudaSuccess || !p) {
            engram::set_last_error(std::string("engram_forward_noalloc: cudaGetSymbolAddress: ") +
                                   cudaGetErrorString(e));
            return ENGRAM_ECUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return ENGRAM_OK;
}

// Largest batch whose scratch fits the buffer: the workspace grows with T,
// so a binary search over [0, 2^24] on the same layout the forward uses.
int64_t max_tokens(const engram_ctx* ctx) {
    int64_t lo = 0, hi = (int64_t)1 << 24;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) / 2;
        if (engram::forward_workspace_bytes(ctx, mid, 1) <= kScratchBytes)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

}  // namespace

extern "C" engram_status engram_forward_noalloc(const engram_ctx* ctx, int layer,
                                                const uint32_t* d_windows, int64_t T,
                                                uint16_t* d_hidden, float* d_gates,
                                                void* stream) {
    // the same checks as engram_forward (context, layer bound, T in range)
    engram_status st = engram::check_forward_call(ctx, layer, T);
    if (st != ENGRAM_OK) return st;
    if (T == 0) return engram_forward(ctx, layer, d_windows, 0, d_hidden, nullptr, d_gates, stream);
    // K is never split here: split-K partials of a small batch would need far
    // more scratch than the gate sums, so such a batch runs on fewer SMs
    const size_t need = engram::forward_workspace_bytes(ctx, T, 1);
    if (need > kScratchBytes) {
        engram::set_last_error(
            "engram_forward_noalloc: " + std::to_string(T) + " tokens need " + std::to_string(need) +
            " bytes of scratch, above the built-in 8 MiB (at most " +
            std::to_string(max_tokens(ctx)) +
            " tokens for this geometry); split the batch or use engram_forward");
        return ENGRAM_EINVAL;
    }
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != ENGRAM_OK) return st;
    return engram::forward_fused(ctx, layer, d_windows, T, d_hidden, scratch, d_gates, stream, 1);
}
