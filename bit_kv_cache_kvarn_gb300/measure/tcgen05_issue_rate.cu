// Measurement program (not part of libkvarn): how fast tcgen05.mma instructions complete when one
// warp issues them and when several warps do -- the reason the decode kernel spreads each tile's
// MMAs over a worker's four warps.  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O2 -o /tmp/tcgen05_issue_rate \
//        bit_kv_cache_kvarn_gb300/measure/tcgen05_issue_rate.cu && /tmp/tcgen05_issue_rate
// Probe: tcgen05.mma throughput with several issuing warps (which warps, how many) and kind::f16 vs
// kind::f8f6f4 (E4M3 x E4M3).  M=128, N=16, A in TMEM, B in shared memory.
#include <cstdio>
#include <cstdint>

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return ((uint64_t)((saddr & 0x3FFFF) >> 4)) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}
struct Exp { unsigned mask; int n; int f8; const char* name; };
__constant__ Exp c_exps[16];

__global__ void __launch_bounds__(512, 1) probe(int n_exps, long long* out, int* err) {
    __shared__ __align__(1024) unsigned char bsm[16384];
    __shared__ __align__(8) uint64_t bar[16];
    __shared__ uint32_t slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 16384 / 16; i += blockDim.x) reinterpret_cast<uint4*>(bsm)[i] = make_uint4(0x3c003c00u, 0, 0x3c003c00u, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&slot)), "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid < 16) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar[tid])), "r"(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t t = slot;
    uint32_t phase = 0;  // this warp's barrier phase (lane 0)
    for (int e = 0; e < n_exps; ++e) {
        const Exp x = c_exps[e];
        const bool issuer = lane == 0 && ((x.mask >> warp) & 1u);
        // f16: B MN-major (bit 16); f8: B K-major
        const uint32_t idesc = (1u << 4) | ((x.f8 ? 0u : 1u) << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
        long long best = 1ll << 60;
        for (int rep = 0; rep < 12; ++rep) {
            __syncthreads();
            const long long t0 = clock64();
            if (issuer) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dcol = t + 64 + 16u * (uint32_t)warp;  // columns 64 .. 319
                for (int s = 0; s < x.n; ++s) {
                    const uint64_t bdesc = desc(smem_u32(bsm) + (s % 16) * 512, 256, 128);  // <= 16 KB
                    const uint32_t a = t + 8 * (s % 8);                                      // columns 0 .. 63
                    const uint32_t acc = s > 0;
                    if (x.f8)
                        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}"
                                     ::"r"(dcol), "r"(a), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
                    else
                        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                                     ::"r"(dcol), "r"(a), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar[warp])) : "memory");
                bool ok = false;
                for (long long i = 0; i < (1ll << 22); ++i) {
                    uint32_t done;
                    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                                 : "=r"(done) : "r"(smem_u32(&bar[warp])), "r"(phase) : "memory");
                    if (done) { ok = true; break; }
                }
                phase ^= 1;
                if (!ok) atomicExch(err, 1);
            }
            __syncthreads();
            const long long t1 = clock64();
            if (t1 - t0 < best) best = t1 - t0;
        }
        if (tid == 0) out[e] = best;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(512));
}

int main() {
    Exp exps[] = {
        {0x0001u, 8, 0, "f16 warp 0, 8"},          {0x0001u, 32, 0, "f16 warp 0, 32"},
        {0x0011u, 32, 0, "f16 warps 0,4, 32 each"}, {0x1111u, 32, 0, "f16 warps 0,4,8,12"},
        {0x000Fu, 32, 0, "f16 warps 0-3"},          {0x8421u, 32, 0, "f16 warps 0,5,10,15"},
        {0x00FFu, 32, 0, "f16 warps 0-7"},          {0xFFFFu, 32, 0, "f16 warps 0-15"},
        {0x0001u, 8, 1, "f8 warp 0, 8"},            {0x0001u, 32, 1, "f8 warp 0, 32"},
        {0x000Fu, 32, 1, "f8 warps 0-3"},           {0xFFFFu, 32, 1, "f8 warps 0-15"},
    };
    const int n = sizeof(exps) / sizeof(exps[0]);
    cudaMemcpyToSymbol(c_exps, exps, sizeof(exps));
    long long* out; int* err;
    cudaMallocManaged(&out, 16 * 8); cudaMallocManaged(&err, 4); *err = 0;
    probe<<<1, 512>>>(n, out, err);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("err %s\n", cudaGetErrorString(e)); return 1; }
    for (int i = 0; i < n; ++i) printf("%-28s %6lld cycles\n", exps[i].name, out[i]);
    printf("wait_err=%d\n", *err);
    return *err;
}
