// Appending a decode step's tokens to the KVarN cache: the accepted tokens go to the bf16 tail; a
// block they complete is staged and encoded into its pool slot.
//
// Method: the cache holds a quantised body of 128-token blocks and unquantised trailing tokens
// (paperlayer.ai summary, "D Experimental details"); a block is quantised once it is done
// (agihunt.info, pipeline paragraph).  Only the accepted tokens of a step are committed, so a
// speculative step's rejected tokens never reach the cache.
//
// One block of threads per sequence moves the tokens of every kv head (16-byte copies) and, when
// the sequence's block completes, copies it to the staging slot of its (sequence, kv head) and
// records the pool tile it belongs to (-1 for slots with nothing staged); one encoder launch over K
// and V then encodes the staged slots into their pool tiles and skips the others.  Two launches per
// call, whatever number of blocks completes.
#include "kvarn_common.cuh"
#include "kvarn_internal.h"

namespace kvarn {

// Set when a completed block has no slot in the block table (its index >= max_tiles); such a
// sequence is left unchanged.  Read by kvarn_device_error.
__device__ unsigned int g_append_error = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kRowChunks = kTile * 2 / 16;  // 16-byte pieces of a 128-channel bf16 row

__device__ __forceinline__ void copy_rows(__nv_bfloat16* dst, const __nv_bfloat16* src, int rows) {
    uint4* d = reinterpret_cast<uint4*>(dst);
    const uint4* s = reinterpret_cast<const uint4*>(src);
    for (int i = threadIdx.x; i < rows * kRowChunks; i += kThreads) d[i] = s[i];
}

__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
    const int b = blockIdx.x;
    const int len = a.seq_lens[b];
    int acc = a.n_accept != nullptr ? a.n_accept[b] : a.n_new;
    acc = acc < 0 ? 0 : (acc > a.n_new ? a.n_new : acc);
    int t0, blk;
    bool complete;
    if (a.full_tail) {
        // the tail keeps 1..128 tokens: a full block leaves it only when a newer token arrives
        t0 = len > 0 ? ((len - 1) & (kTile - 1)) + 1 : 0;
        blk = len > 0 ? (len - 1) >> 7 : 0;
        complete = t0 + acc > kTile;
    } else {
        t0 = len & (kTile - 1);
        blk = len >> 7;
        complete = t0 + acc >= kTile;
    }
    if (complete && (blk >= a.max_tiles || len < 0)) {
        if (threadIdx.x == 0) atomicOr(&g_append_error, 1u);
        for (int h = threadIdx.x; h < a.Hkv; h += kThreads) a.dest[(size_t)b * a.Hkv + h] = -1;
        return;
    }
    const int need = complete ? kTile - t0 : acc;  // new tokens that go into the current block
    if (!complete)
        for (int h = threadIdx.x; h < a.Hkv; h += kThreads) a.dest[(size_t)b * a.Hkv + h] = -1;
    for (int h = 0; h < a.Hkv; ++h) {
        const size_t u = (size_t)b * a.Hkv + h;
        __nv_bfloat16* kt = a.k_tail + u * kTile * kTile;
        __nv_bfloat16* vt = a.v_tail + u * kTile * kTile;
        const __nv_bfloat16* kn = a.k_new + u * a.n_new * kTile;
        const __nv_bfloat16* vn = a.v_new + u * a.n_new * kTile;
        if (complete) {
            const size_t slot = u;
            __nv_bfloat16* ks = a.k_stage + (size_t)slot * kTile * kTile;
            __nv_bfloat16* vs = a.v_stage + (size_t)slot * kTile * kTile;
            copy_rows(ks, kt, t0);
            copy_rows(vs, vt, t0);
            copy_rows(ks + (size_t)t0 * kTile, kn, need);
            copy_rows(vs + (size_t)t0 * kTile, vn, need);
            if (threadIdx.x == 0) a.dest[slot] = a.block_table[u * a.max_tiles + blk];
            __syncthreads();  // the old tail rows are staged before the new tail overwrites them
            copy_rows(kt, kn + (size_t)need * kTile, acc - need);
            copy_rows(vt, vn + (size_t)need * kTile, acc - need);
        } else {
            copy_rows(kt + (size_t)t0 * kTile, kn, acc);
            copy_rows(vt + (size_t)t0 * kTile, vn, acc);
        }
    }
    if (threadIdx.x == 0) a.seq_lens[b] = len + acc;
}

}  // namespace

size_t append_workspace_bytes(int B, int Hkv) {
    const size_t tiles = (size_t)B * Hkv;
    return 2 * tiles * kTile * kTile * sizeof(__nv_bfloat16) + ((tiles * sizeof(int32_t) + 255) & ~(size_t)255);
}

cudaError_t read_and_clear_append_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_append_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_append_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

cudaError_t launch_append(const AppendArgs& a, int B, int k_bits, int v_bits, int iters, int rotate,
                          int normalize, void* k_codes, void* k_params, float* k_scale, void* v_codes,
                          void* v_params, float* v_scale, cudaStream_t stream) {
    append_kernel<<<B, kThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // encode the staged blocks (dest >= 0) of every (sequence, kv head) slot into their pool tiles
    const int64_t slots = (int64_t)B * a.Hkv;
    return launch_encode_kv(k_bits, v_bits, a.k_stage, slots, k_codes, k_params, k_scale, a.v_stage, slots,
                            v_codes, v_params, v_scale, iters, rotate, normalize, stream, a.dest);
}

}  // namespace kvarn
