// Measurement program (not part of libkvarn): can a tcgen05.mma A operand read from shared memory
// with zero core-matrix strides (LBO = SBO = 0) stand for a constant matrix held in one 8 x 8 fp16
// core matrix (128 bytes)?  If so, sums over K such as the decode kernel's zero-point terms could be
// taken by the tensor cores against a block of ones without storing a 128 x 128 operand.
//   nvcc -gencode arch=compute_103a,code=sm_103a -O2 -o /tmp/tcgen05_zero_stride_a \
//        bit_kv_cache_kvarn_gb300/measure/tcgen05_zero_stride_a.cu && /tmp/tcgen05_zero_stride_a
//
// kind::f16, M = 128, N = 16, K = 16, A and B from shared memory (no swizzle), fp32 D in tensor
// memory.  A: one core matrix of fp16 ones (row r of it = 8 K-elements), described with LBO = SBO =
// 0, so every (row block, K block) reads the same 128 bytes.  B: MN-major, element (k, n) =
// (k + 1) * 2^-(n % 4) (exact in fp16).  Expected D[m][n] = sum_k B[k][n] for every row m.  The
// reads stay inside the two shared arrays whatever the strides do.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cuda_fp16.h>

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return ((uint64_t)((saddr & 0x3FFFF) >> 4)) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);
}

__global__ void probe(float* out, int* err) {
    __shared__ __align__(1024) __half a[64];        // one 8 x 8 core matrix of ones
    __shared__ __align__(1024) __half b[16 * 16];   // K = 16 x N = 16, MN-major
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < 64; i += blockDim.x) a[i] = __float2half(1.f);
    for (int i = tid; i < 256; i += blockDim.x) {
        const int k = i >> 4, n = i & 15;
        // MN-major core matrices of 8 K-rows x 8 N-elements: (k>>3)*256 + (n>>3)*128 + (k&7)*16 bytes
        const int off = ((k >> 3) * 256 + (n >> 3) * 128 + (k & 7) * 16) / 2 + (n & 7);
        b[off] = __float2half((float)(k + 1) * ldexpf(1.f, -(n % 4)));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&slot)), "r"(32));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar)), "r"(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t t = slot;
    if (tid == 0) {
        const uint64_t adesc = desc(smem_u32(a), 0, 0);       // K-major A, zero strides
        const uint64_t bdesc = desc(smem_u32(b), 256, 128);   // MN-major B: 256 B along K, 128 B along N
        const uint32_t idesc = (1u << 4) | (1u << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, 0, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                     ::"r"(t), "l"(adesc), "l"(bdesc), "r"(idesc) : "memory");
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
    }
    bool ok = false;
    for (long long i = 0; i < (1ll << 22); ++i) {
        uint32_t done;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                     : "=r"(done) : "r"(smem_u32(&bar)), "r"(0) : "memory");
        if (done) { ok = true; break; }
    }
    if (!ok && tid == 0) *err = 1;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok) {
        uint32_t d[16];
        const uint32_t taddr = t + ((uint32_t)(32 * warp) << 16);
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                     : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
                       "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
                     : "r"(taddr) : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        for (int n = 0; n < 16; ++n) out[tid * 16 + n] = __uint_as_float(d[n]);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(32));
}

int main() {
    float* out;
    int* err;
    cudaMallocManaged(&out, 128 * 16 * sizeof(float));
    cudaMallocManaged(&err, sizeof(int));
    *err = 0;
    probe<<<1, 128>>>(out, err);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess || *err) {
        printf("cuda %s, timeout %d\n", cudaGetErrorString(e), *err);
        return 1;
    }
    int exact = 0;
    double worst = 0.0;
    for (int m = 0; m < 128; ++m)
        for (int n = 0; n < 16; ++n) {
            double ref = 0.0;
            for (int k = 0; k < 16; ++k) ref += (k + 1) * std::ldexp(1.0, -(n % 4));
            if (out[m * 16 + n] == ref) ++exact;
            worst = std::fmax(worst, std::fabs(out[m * 16 + n] - ref) / ref);
        }
    printf("A = ones through zero core-matrix strides: %d of 2048 sums exact, worst relative error %.3e\n", exact, worst);
    printf("row 0: %.4f %.4f %.4f %.4f (expected %.4f %.4f %.4f %.4f); row 127: %.4f\n", out[0], out[1], out[2], out[3],
           136.0, 68.0, 34.0, 17.0, out[127 * 16]);
    return 0;
}
