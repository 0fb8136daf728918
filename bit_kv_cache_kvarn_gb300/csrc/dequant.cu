// Dequantisation of packed tiles to float32, both scales applied in one pass
// (paperlayer.ai summary of KVarN, "I KVarN Dequantization Overhead": the second scale s2 is
// fused into the dequantisation kernel so no extra HBM round trip is needed).
//   Yhat[t][j] = g * s2[other] * (S1[group] * code[t][j] + Z[group])   (rotated basis)
//   Xhat = Yhat * H                                                      (original basis)
// One CTA per tile; the optional inverse rotation is the encoder's two-pass transform in reverse
// order (H_8 over channel bits 4..6 in registers, then H_16 over bits 0..3 after a transpose).
#include "kvarn_common.cuh"
#include "kvarn_internal.h"

namespace kvarn {

namespace {

constexpr int kThreads = 256;

template <int BITS, int KIND>
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ params,
               const float* __restrict__ tile_scale, float* __restrict__ out, int original_basis,
               int rotate) {
    extern __shared__ __align__(16) float dsm[];
    float* ys = dsm;                         // [128][kYStride]
    float* s1v = dsm + kTile * kYStride;     // group scale
    float* s2v = s1v + kTile;                // other-axis scale times g
    float* zv = s2v + kTile;                 // zero-point
    constexpr int kCodeBytes = kTile * 16 * BITS;
    constexpr uint32_t kMask = (1u << BITS) - 1u;

    const int64_t tile = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int h = lane & 15;
    const int tg = 2 * (tid >> 5) + (lane >> 4);
    const uint8_t* p = params + tile * KVARN_PARAM_BYTES;
    const float g = tile_scale[tile];
    if (tid < kTile) {
        s1v[tid] = e4m3_value(p[tid]);
        s2v[tid] = e4m3_value(p[128 + tid]) * g;  // g folded into s2
        zv[tid] = fp16_value(reinterpret_cast<const uint16_t*>(p + 256)[tid]);
    }
    __syncthreads();

    const uint8_t* c = codes + tile * kCodeBytes;
    // K rows are tokens (lane h of row t: channels h + 16 i); V rows are channels (lane tg of
    // row j: tokens tg + 16 k).  Thread (tg, h) owns tokens tg + 16 k and channels h + 16 i.
    uint32_t vlanes[8];
    if (KIND == KVARN_KIND_V) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = h + 16 * i;
            vlanes[i] = (BITS == 2) ? reinterpret_cast<const uint16_t*>(c)[j * 16 + tg]
                                    : reinterpret_cast<const uint32_t*>(c)[j * 16 + tg];
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int t = tg + 16 * k;
        uint32_t lanev = 0;
        if (KIND == KVARN_KIND_K)
            lanev = (BITS == 2) ? reinterpret_cast<const uint16_t*>(c)[t * 16 + h]
                                : reinterpret_cast<const uint32_t*>(c)[t * 16 + h];
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = h + 16 * i;
            const uint32_t bits = (KIND == KVARN_KIND_K) ? (lanev >> (BITS * i)) : (vlanes[i] >> (BITS * k));
            const float code = (float)(bits & kMask);
            const int grp = (KIND == KVARN_KIND_K) ? j : t;
            const int oth = (KIND == KVARN_KIND_K) ? t : j;
            v[i] = s2v[oth] * fmaf(s1v[grp], code, zv[grp]);
        }
        if (original_basis && rotate) fwht_regs<8>(v);
#pragma unroll
        for (int i = 0; i < 8; ++i) ys[t * kYStride + h + 16 * i] = v[i];
    }
    __syncthreads();

    float* o = out + tile * kTile * kTile;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + kThreads * it;
        const int t = idx >> 3, cc = idx & 7;
        float v[16];
        const float* src = ys + t * kYStride + 16 * cc;
        {
            // read the 16-byte chunks in a lane-dependent rotation (bank-conflict free), then undo it
            const int rot = (cc >> 1) & 3;
            float4 a0 = *reinterpret_cast<const float4*>(src + 4 * ((0 + rot) & 3));
            float4 a1 = *reinterpret_cast<const float4*>(src + 4 * ((1 + rot) & 3));
            float4 a2 = *reinterpret_cast<const float4*>(src + 4 * ((2 + rot) & 3));
            float4 a3 = *reinterpret_cast<const float4*>(src + 4 * ((3 + rot) & 3));
            rotl4(a0, a1, a2, a3, (4 - rot) & 3);
            const float4 f[4] = {a0, a1, a2, a3};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[4 * q] = f[q].x;
                v[4 * q + 1] = f[q].y;
                v[4 * q + 2] = f[q].z;
                v[4 * q + 3] = f[q].w;
            }
        }
        if (original_basis && rotate) {
            fwht_regs<16>(v);
#pragma unroll
            for (int m = 0; m < 16; ++m) v[m] *= kInvSqrt128;
        }
        float4* dst = reinterpret_cast<float4*>(o + t * kTile + 16 * cc);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
}

}  // namespace

cudaError_t launch_dequant(int bits, int kind, const void* codes, const void* params,
                           const float* tile_scale, int64_t n_tiles, int original_basis,
                           int rotate, float* out, cudaStream_t stream) {
    const uint8_t* c = static_cast<const uint8_t*>(codes);
    const uint8_t* p = static_cast<const uint8_t*>(params);
    const size_t smem = (size_t)(kTile * kYStride + 3 * kTile) * sizeof(float);
    dim3 grid((unsigned)n_tiles);  // the API limits n_tiles to 2^31 - 1
    auto run = [&](auto kern) -> cudaError_t {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = set_smem_limit_once(kern, (int)smem, false, dev);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, stream>>>(c, p, tile_scale, out, original_basis, rotate);
        return cudaGetLastError();
    };
    if (bits == 2 && kind == KVARN_KIND_K) return run(dequant_kernel<2, KVARN_KIND_K>);
    if (bits == 2) return run(dequant_kernel<2, KVARN_KIND_V>);
    if (kind == KVARN_KIND_K) return run(dequant_kernel<4, KVARN_KIND_K>);
    return run(dequant_kernel<4, KVARN_KIND_V>);
}

}  // namespace kvarn
