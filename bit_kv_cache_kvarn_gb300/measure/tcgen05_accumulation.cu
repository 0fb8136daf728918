// Measurement program (not part of libkvarn): which small products survive in a tcgen05.mma
// kind::f16 sum, with a normal and with a subnormal A operand -- the decode kernel holds its codes
// as fp16 subnormals.  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O2 -o /tmp/tcgen05_accumulation \
//        bit_kv_cache_kvarn_gb300/measure/tcgen05_accumulation.cu && /tmp/tcgen05_accumulation
// Probe: accumulation precision of tcgen05.mma kind::f16 (fp16 in, fp32 out), M=128, N=16, K=16.
// A = 1.0 everywhere; column n of B: k = 0 -> 1.0, k = 1..15 -> 2^-(6+n).  Exact D[*, n] = 1 + 15 * 2^-(6+n).
// A second run uses subnormal A (2^-24) with B scaled by 2^14 / 2^(6+n) alike, like the decode kernel.
// A third run has no large product: subnormal A (2^-24) and all sixteen B entries of column n equal to
// 2^-n, so every product is 2^-(24+n) and the exact sum 2^-(20+n): it tells whether small products
// are lost below a fixed size or only next to a much larger product.
#include <cstdio>
#include <cstdint>
#include <cuda_fp16.h>
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__global__ void probe(float* out, int* err, int sub) {
    __shared__ __align__(1024) __half b[16 * 16];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid >> 5;
    // B MN-major: element (k, n) at byte ((k>>3)*256 + (n>>3)*128 + (k&7)*16) + 2*(n&7); 512 bytes total
    for (int i = tid; i < 256; i += blockDim.x) {
        const int k = i >> 4, n = i & 15;
        float v = (k == 0) ? 1.f : ldexpf(1.f, -(6 + n));
        if (sub == 1) v *= 16384.f;  // A is 2^-24 below: keep products in the same range as the decode kernel
        if (sub == 2) v = ldexpf(1.f, -n);
        const int off = ((k >> 3) * 256 + (n >> 3) * 128 + (k & 7) * 16) / 2 + (n & 7);
        b[off] = __float2half_rn(v);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&slot)), "r"(64));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar)), "r"(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t t = slot;
    // A: 8 columns of fp16 pairs per lane
    const uint32_t aw = sub ? 0x00010001u : 0x3C003C00u;  // 2^-24 (subnormal) or 1.0
    {
        const uint32_t taddr = t + ((uint32_t)(32 * warp) << 16);
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(taddr), "r"(aw) : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t sa = smem_u32(b);
        const uint64_t desc = ((uint64_t)((sa & 0x3FFFF) >> 4)) | ((uint64_t)(256 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
        const uint32_t idesc = (1u << 4) | (1u << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, 0, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                     ::"r"(t + 32), "r"(t), "l"(desc), "r"(idesc) : "memory");
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
    uint32_t d[16];
    const uint32_t taddr = t + 32 + ((uint32_t)(32 * warp) << 16);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
                   "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
                 : "r"(taddr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    if (tid == 0) for (int n = 0; n < 16; ++n) out[n] = __uint_as_float(d[n]);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(64));
}
int main() {
    float* out; int* err;
    cudaMallocManaged(&out, 64); cudaMallocManaged(&err, 4); *err = 0;
    for (int sub = 0; sub < 3; ++sub) {
        probe<<<1, 128>>>(out, err, sub);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) { printf("err %s\n", cudaGetErrorString(e)); return 1; }
        printf("%s\n", sub == 2 ? "A = 2^-24 (subnormal), all B of column n = 2^-n" :
                        (sub ? "A = 2^-24 (subnormal), B x 2^14" : "A = 1.0"));
        for (int n = 0; n < 16; ++n) {
            double ex = 1.0 + 15.0 * ldexp(1.0, -(6 + n));
            if (sub == 1) ex = ex * 16384.0 * ldexp(1.0, -24);
            if (sub == 2) ex = 16.0 * ldexp(1.0, -(24 + n));
            // fp16 B for n >= 9 is subnormal (2^-15 and below) in the A = 1.0 run
            printf("  n=%2d small=2^-%2d  got %.10e  exact %.10e  rel err %.2e\n", n, 6 + n, out[n], ex, (out[n] - ex) / ex);
        }
    }
    printf("wait_err=%d\n", *err);
    return *err;
}
