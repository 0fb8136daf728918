// Measurement program (not part of libkvarn): tcgen05.mma kind::f8f6f4 with E4M3 operands, A in
// tensor memory, B in shared memory stored MN-major (N contiguous), M=128, N=16, K=32 per
// instruction.  Checks (1) the operand layouts and (2) that the sums are exact when A holds small
// integers: a byte v < 16 read as E4M3 is exactly v * 2^-9 (exponent field 0 or 1), which is how
// packed 2- and 4-bit codes can be used in place after one mask.
//   nvcc -gencode arch=compute_103a,code=sm_103a -O2 -o /tmp/tcgen05_f8_operands \
//        bit_kv_cache_kvarn_gb300/measure/tcgen05_f8_operands.cu && /tmp/tcgen05_f8_operands
//
// Layouts tested: A row m = TMEM lane m, column c holds K elements 4c..4c+3 (byte j = element
// 4c + j); B element (k, n) at byte (k / 8) * 128 + (k % 8) * 16 + n (core matrices of 8 K-rows x
// 16 bytes, 128 bytes apart along K).  D = sum over K = 128 (four MMAs, accumulating).
#include <cmath>
#include <cstdint>
#include <cstdio>

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__global__ void probe(const uint8_t* a_g, const uint8_t* b_g, float* d_out, int n_mma, int* err) {
    __shared__ __align__(1024) uint8_t b[128 * 16];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < 128 * 16; i += blockDim.x) {
        const int k = i >> 4, n = i & 15;
        b[(k >> 3) * 128 + (k & 7) * 16 + n] = b_g[k * 16 + n];
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
    {
        // thread m writes row m of A: 32 columns of 4 bytes
        uint32_t r[32];
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a_g + tid * 128);
        for (int c = 0; c < 32; ++c) r[c] = src[c];
        const uint32_t taddr = t + ((uint32_t)(32 * warp) << 16);
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
            "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr + 16),
            "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
            "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t sa = smem_u32(b);
        // E4M3 x E4M3 (format fields 0), fp32 D, B MN-major, N = 16, M = 128
        const uint32_t idesc = (1u << 4) | (1u << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
        for (int s = 0; s < n_mma; ++s) {
            const uint32_t bs = sa + s * 512;  // 32 K-rows = 4 core matrices of 128 bytes
            const uint64_t desc = ((uint64_t)((bs & 0x3FFFF) >> 4)) | ((uint64_t)(128 >> 4) << 16) |
                                  ((uint64_t)(256 >> 4) << 32) | (1ull << 46);
            asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}"
                         ::"r"(t + 32), "r"(t + 8 * s), "l"(desc), "r"(idesc), "r"(s) : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
    }
    bool ok = false;
    for (long long i = 0; i < (1ll << 22); ++i) {
        uint32_t done;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                     : "=r"(done) : "r"(smem_u32(&bar)), "r"(0) : "memory");
        if (done) { ok = true; break; }
    }
    if (!ok) atomicOr(err, 1);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok) {
        uint32_t r[16];
        const uint32_t taddr = t + 32 + ((uint32_t)(32 * warp) << 16);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr) : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        for (int n = 0; n < 16; ++n) d_out[tid * 16 + n] = __uint_as_float(r[n]);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(64));
}

// E4M3 code of j * 2^e (1 <= j <= 15, the value a normal E4M3 number): exact.
static uint8_t e4m3_code(int j, int e) {
    int E = 0;
    while ((j >> (E + 1)) > 0) ++E;  // j = 1.m * 2^E
    const int mant = (j << 3 >> E) & 7;  // three fraction bits
    return (uint8_t)(((E + e + 7) << 3) | mant);
}

int main() {
    static uint8_t a[128 * 128], b[128 * 16];
    static double bv[128 * 16];
    static float d[128 * 16];
    for (int m = 0; m < 128; ++m)
        for (int k = 0; k < 128; ++k) a[m * 128 + k] = (uint8_t)((m * 7 + k * 13 + 5) % 16);
    for (int k = 0; k < 128; ++k)
        for (int n = 0; n < 16; ++n) {
            const int j = (k * 3 + n * 5) % 15 + 1, e = (k + n) % 5 - 2;
            b[k * 16 + n] = e4m3_code(j, e);
            bv[k * 16 + n] = std::ldexp((double)j, e);
        }
    uint8_t *a_d, *b_d;
    float* d_d;
    int* err_d;
    cudaMalloc(&a_d, sizeof(a));
    cudaMalloc(&b_d, sizeof(b));
    cudaMalloc(&d_d, sizeof(d));
    cudaMalloc(&err_d, sizeof(int));
    cudaMemcpy(a_d, a, sizeof(a), cudaMemcpyHostToDevice);
    cudaMemcpy(b_d, b, sizeof(b), cudaMemcpyHostToDevice);
    for (int n_mma = 1; n_mma <= 4; n_mma += 3) {
        cudaMemset(err_d, 0, sizeof(int));
        cudaMemset(d_d, 0, sizeof(d));
        probe<<<1, 128>>>(a_d, b_d, d_d, n_mma, err_d);
        cudaError_t e = cudaDeviceSynchronize();
        int err = 0;
        cudaMemcpy(&err, err_d, sizeof(int), cudaMemcpyDeviceToHost);
        cudaMemcpy(d, d_d, sizeof(d), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess || err) {
            printf("n_mma %d: cuda %s, timeout %d\n", n_mma, cudaGetErrorString(e), err);
            return 1;
        }
        int exact = 0, worst_m = -1, worst_n = -1;
        double worst = 0.0;
        for (int m = 0; m < 128; ++m)
            for (int n = 0; n < 16; ++n) {
                double ref = 0.0;
                for (int k = 0; k < 32 * n_mma; ++k) ref += a[m * 128 + k] * std::ldexp(1.0, -9) * bv[k * 16 + n];
                const double got = d[m * 16 + n];
                if (got == ref) ++exact;
                const double rel = std::fabs(got - ref) / std::fmax(std::fabs(ref), 1e-30);
                if (rel > worst) { worst = rel; worst_m = m; worst_n = n; }
            }
        printf("K = %3d (%d MMA): %d of 2048 sums exact, worst relative error %.3e at (%d, %d)\n", 32 * n_mma, n_mma,
               exact, worst, worst_m, worst_n);
        if (worst_m >= 0) {
            double ref = 0.0;
            for (int k = 0; k < 32 * n_mma; ++k) ref += a[worst_m * 128 + k] * std::ldexp(1.0, -9) * bv[k * 16 + worst_n];
            printf("  D = %.9g, expected %.9g\n", d[worst_m * 16 + worst_n], ref);
        }
    }
    return 0;
}
