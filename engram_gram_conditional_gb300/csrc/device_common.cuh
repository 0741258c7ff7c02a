// Device helpers shared by the kernels: the multiply-XOR prime-bucket hash and
// the MXFP8 (E4M3 x 2^E8M0) -> BF16 decode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "engram_internal.h"

namespace engram {

// Row of bucket b for window w = (c_t, c_{t-1}, c_{t-2}, c_{t-3}).
// Order n = min_n + b / heads reads the suffix n-gram w[0..n-1]; the mix is
// the XOR of each id times its multiplier (wrapping 64-bit); the row is the
// bucket offset plus the mix modulo the bucket prime; any DEAD in the n-gram
// masks the row (vLLM wiki "동작 방식", zhuai.tech "第一步").
__device__ __forceinline__ uint32_t hash_bucket(const HashParams& hp, uint4 w, int b) {
    const int n = hp.min_n + b / hp.heads;
    const uint32_t c[4] = {w.x, w.y, w.z, w.w};
    uint64_t x = 0;
    bool dead = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j < n) {
            dead |= (c[j] == kDead);
            x ^= (uint64_t)c[j] * hp.mult[b][j];
        }
    }
    if (dead) return kMasked;
    return (uint32_t)(hp.offset[b] + x % hp.prime[b]);
}

// 2^(e - 127) as fp32 for an E8M0 exponent; e = 0 is the subnormal 2^-127,
// e = 255 is NaN (OCP MX).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
    float v = __uint_as_float(e << 23);
    v = (e == 0u) ? __uint_as_float(0x00400000u) : v;
    v = (e == 255u) ? __uint_as_float(0x7FC00000u) : v;
    return v;
}

// Two E4M3 codes (low byte first) -> two BF16 values times the scale, packed
// low-first.  E4M3 -> f16 is exact, f16 -> f32 is exact, the product with a
// power of two is exact unless it leaves fp32's range, and the final rounding
// to BF16 is round-to-nearest-even, so the result is the exact product
// rounded once.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes, float scale) {
    uint32_t h2;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(h2)
        : "r"(two_codes));
    __half2 hh = *reinterpret_cast<__half2*>(&h2);
    float2 f = __half22float2(hh);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<uint32_t*>(&b);
}

// Eight E4M3 codes (two little-endian words) -> eight BF16 values (uint4).
__device__ __forceinline__ uint4 decode8(uint32_t w0, uint32_t w1, float scale) {
    uint4 o;
    o.x = e4m3x2_to_bf16x2(w0 & 0xFFFFu, scale);
    o.y = e4m3x2_to_bf16x2(w0 >> 16, scale);
    o.z = e4m3x2_to_bf16x2(w1 & 0xFFFFu, scale);
    o.w = e4m3x2_to_bf16x2(w1 >> 16, scale);
    return o;
}

__device__ __forceinline__ uint32_t bf16x2_pack_rn(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Programmatic dependent launch.  A kernel launched with the
// programmatic-serialisation attribute may start while the kernel before it in
// the stream is still running, once every CTA of that kernel has called
// pdl_launch_dependents (or exited); pdl_wait then blocks until that kernel
// has finished and its writes are visible.  Every kernel launched this way
// calls pdl_wait before it touches memory that earlier work in the stream
// writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float gate_from_sums(float s_kk, float s_hh, float s_hk, int d,
                                                float eps) {
    // dot = <h rh w_q, k rk w_k> / sqrt(d); gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot))
    const float inv_d = 1.0f / (float)d;
    const float rh = 1.0f / sqrtf(s_hh * inv_d + eps);
    const float rk = 1.0f / sqrtf(s_kk * inv_d + eps);
    const float dot = rh * rk * s_hk / sqrtf((float)d);
    const float s = copysignf(sqrtf(fmaxf(fabsf(dot), 1e-6f)), dot);
    return 1.0f / (1.0f + expf(-s));
}

}  // namespace engram
