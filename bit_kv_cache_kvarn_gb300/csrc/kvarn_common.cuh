// Device helpers shared by the libkvarn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int kTile = 128;                       // tokens per tile = channels per head
constexpr float kInvSqrt128 = 0.08838834764831845f;
constexpr float kDegenerateRel = 1e-5f;          // variance <= 1e-5 * mean square: constant
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMagic = 8388608.0f;             // 2^23: float with an empty 23-bit mantissa
constexpr uint32_t kMagicBits = 0x4B000000u;
constexpr int kYStride = 144;                    // fp32 row stride of the FWHT staging tile

// Bit set in a kernel's device-side error word when a bounded wait gives up.
constexpr unsigned int kErrTmaTimeout = 1u;
constexpr long long kSpinLimit = 1ll << 24;      // try_wait polls before giving up

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
// a * b rounded to nearest and clamped to [0, 1] (one instruction)
__device__ __forceinline__ float mul_sat(float a, float b) {
    float r;
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// ---- number formats (hardware conversions) ----------------------------------------------------
__device__ __forceinline__ uint8_t e4m3_rn(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_value(uint8_t b) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}
// Smallest E4M3 value >= x for 0 <= x <= 448: round to nearest, step up one code if below.
__device__ __forceinline__ uint8_t e4m3_up(float x) {
    uint8_t b = e4m3_rn(x);
    if (e4m3_value(b) < x) b = (uint8_t)(b + 1);
    return b;
}
__device__ __forceinline__ float fp16_value(uint16_t bits) {
    __half_raw h;
    h.x = bits;
    return __half2float(__half(h));
}
__device__ __forceinline__ int ceil_log2(float v) {  // v > 0
    int e;
    float f = frexpf(v, &e);  // v = f * 2^e, f in [0.5, 1)
    return f == 0.5f ? e - 1 : e;
}

// code bits placed in the low mantissa of 2^23: returns code * 2^shift exactly (shift+bits <= 23)
__device__ __forceinline__ float magic_code(uint32_t x, uint32_t mask) {
    return __uint_as_float((x & mask) | kMagicBits);
}

// ---- TMA bulk copies (cp.async.bulk, 1-D) and mbarriers ---------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
// global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for the mbarrier phase with the given parity.  Bounded: gives up after limit_ns of wall time
// (or kSpinLimit polls), sets *err_word and returns false; once *err_word is set by any thread of
// the grid, every later wait returns false at once, so a stuck kernel ends within about a second.
constexpr uint64_t kWaitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned int* err_word,
                                              uint64_t limit_ns) {
    const uint32_t addr = smem_addr(bar);
    uint64_t t0 = 0;
    for (long long i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 255) == 0) {
            if (*reinterpret_cast<volatile unsigned int*>(err_word)) return false;
            const uint64_t t = global_ns();
            if (i == 0) t0 = t;
            else if (t - t0 > limit_ns) break;
        }
    }
    atomicOr(err_word, kErrTmaTimeout);
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err_word) {
    return mbar_wait_for(bar, parity, err_word, kWaitNs);
}

// After a give-up: wait (bounded by time only) for a copy this CTA issued, so it never exits with a
// bulk copy still writing into its shared memory.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = smem_addr(bar);
    const uint64_t t0 = global_ns();
    for (long long i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done || ((i & 255) == 0 && global_ns() - t0 > kWaitNs)) return;
    }
}

// ---- Hadamard butterflies in registers ---------------------------------------------------------
template <int N>
__device__ __forceinline__ void fwht_regs(float (&v)[N]) {
#pragma unroll
    for (int s = 1; s < N; s <<= 1) {
#pragma unroll
        for (int m = 0; m < N; ++m) {
            if ((m & s) == 0) {
                float a = v[m], b = v[m + s];
                v[m] = a + b;
                v[m + s] = a - b;
            }
        }
    }
}

// Walsh-Hadamard butterflies over 2*N2 values held as N2 float2 pairs (element 2p in .x, 2p+1 in
// .y), unnormalised: the stage inside a pair is scalar, the wider stages pair whole float2s, so
// each of them is one FADD2 and one FFMA2 per two butterflies.
template <int N2>
__device__ __forceinline__ void fwht_pairs(float2 (&f)[N2]) {
#pragma unroll
    for (int p = 0; p < N2; ++p) f[p] = make_float2(f[p].x + f[p].y, f[p].x - f[p].y);
#pragma unroll
    for (int s = 1; s < N2; s <<= 1) {
#pragma unroll
        for (int p = 0; p < N2; ++p) {
            if ((p & s) == 0) {
                const float2 a = f[p], b = f[p + s];
                f[p] = fadd2(a, b);
                f[p + s] = ffma2(b, make_float2(-1.f, -1.f), a);
            }
        }
    }
}

// 128-point transform of a vector held 4 values per lane (lane l holds elements 4l..4l+3):
// two stages in registers, five across lanes.  Unnormalised.
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane) {
    fwht_regs<4>(v);
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float o = __shfl_xor_sync(0xffffffffu, v[m], s);
            v[m] = upper ? (o - v[m]) : (v[m] + o);
        }
    }
}

// Rotate four float4 chunks left by rot (0..3) without dynamic register indexing:
// afterwards a[q] holds the chunk that was at (q + rot) & 3.
__device__ __forceinline__ void rotl4(float4& a0, float4& a1, float4& a2, float4& a3, int rot) {
    if (rot & 1) {
        float4 t = a0;
        a0 = a1;
        a1 = a2;
        a2 = a3;
        a3 = t;
    }
    if (rot & 2) {
        float4 t = a0;
        a0 = a2;
        a2 = t;
        t = a1;
        a1 = a3;
        a3 = t;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xffffffffu, v, s);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
    return v;
}

}  // namespace kvarn
