// Measurement program (not part of libkvarn): the FP32 FMA peak of the GPU, the denominator of the
// encoder's ALU roofline.  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o /tmp/fp32_fma_peak \
//        bit_kv_cache_kvarn_gb300/measure/fp32_fma_peak.cu && /tmp/fp32_fma_peak
// FP32 FMA peak: independent FFMA (or packed FFMA2) chains, full occupancy, timed with CUDA events.
#include <cstdio>
#include <cuda_runtime.h>
template <bool PACKED>
__global__ void __launch_bounds__(256) fma_loop(float* out, int iters, float a, float b) {
    float2 acc[8];
    for (int i = 0; i < 8; ++i) acc[i] = make_float2(threadIdx.x * 1e-3f + i, i * 0.5f);
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (PACKED) acc[i] = __ffma2_rn(acc[i], a2, b2);
            else { acc[i].x = fmaf(acc[i].x, a, b); acc[i].y = fmaf(acc[i].y, a, b); }
        }
    }
    float s = 0.f;
    for (int i = 0; i < 8; ++i) s += acc[i].x + acc[i].y;
    if (s == 1234.5f) out[threadIdx.x] = s;
}
int main() {
    int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    float* out; cudaMalloc(&out, 4096);
    const int iters = 1 << 14, grid = sms * 8, block = 256;
    for (int packed = 0; packed < 2; ++packed) {
        float best = 1e30f;
        for (int rep = 0; rep < 5; ++rep) {
            cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
            cudaEventRecord(e0);
            if (packed) fma_loop<true><<<grid, block>>>(out, iters, 0.999f, 0.001f);
            else fma_loop<false><<<grid, block>>>(out, iters, 0.999f, 0.001f);
            cudaEventRecord(e1); cudaEventSynchronize(e1);
            float ms; cudaEventElapsedTime(&ms, e0, e1); if (ms < best) best = ms;
        }
        const double flops = 2.0 * 16.0 * iters * (double)grid * block;  // 16 fp32 FMAs per iteration per thread
        printf("%s: %.3f ms, %.1f TFLOP/s fp32\n", packed ? "FFMA2" : "FFMA ", best, flops / (best * 1e-3) / 1e12);
    }
    cudaError_t e = cudaGetLastError();
    printf("%s\n", cudaGetErrorString(e));
    return 0;
}
