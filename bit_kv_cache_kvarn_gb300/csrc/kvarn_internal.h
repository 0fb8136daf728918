// Launchers behind the libkvarn C-ABI (host side, not exported).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace kvarn {

// Launch facts cached per device, so that a call makes no driver query after the first one on a
// device (they cost host time on every call otherwise).
constexpr int kMaxCachedDevices = 64;

// The calling thread's device and its SM count (queried once per device).
cudaError_t current_device(int* dev, int* sms);

// Raise the kernel's dynamic shared-memory limit to bytes (and, with max_carveout, prefer the
// largest shared-memory carveout) unless an earlier call already did so for this kernel (by address)
// on this device with at least bytes.
cudaError_t set_smem_limit_once(const void* kernel, int bytes, bool max_carveout, int dev);
template <typename Kern>
cudaError_t set_smem_limit_once(Kern kern, int bytes, bool max_carveout, int dev) {
    return set_smem_limit_once(reinterpret_cast<const void*>(kern), bytes, max_carveout, dev);
}

size_t encode_smem_bytes();
cudaError_t read_and_clear_device_error(unsigned int* out);
cudaError_t read_and_clear_decode_error(unsigned int* out);
cudaError_t launch_encode(int bits, int kind, const void* x, int64_t n_tiles, void* codes,
                          void* params, float* tile_scale, int iters, int rotate, int normalize,
                          cudaStream_t stream);

// K tiles then V tiles in one grid.  dest (optional, device, [n_k] with n_k == n_v): input tile u of
// either kind goes to output slot dest[u], and is skipped when dest[u] < 0.
cudaError_t launch_encode_kv(int k_bits, int v_bits, const void* k_x, int64_t n_k, void* k_codes,
                             void* k_params, float* k_scale, const void* v_x, int64_t n_v, void* v_codes,
                             void* v_params, float* v_scale, int iters, int rotate, int normalize,
                             cudaStream_t stream, const int32_t* dest = nullptr);

cudaError_t launch_dequant(int bits, int kind, const void* codes, const void* params,
                           const float* tile_scale, int64_t n_tiles, int original_basis,
                           int rotate, float* out, cudaStream_t stream);

// Split-K layout for decode attention: piece granularity P (minimum piece and tiles per partial
// slot block), slot count and workspace size.
struct DecodePlan {
    int piece;
    int splits;
    size_t workspace_bytes;
};
DecodePlan plan_decode(int B, int Hq, int Hkv, int max_tiles);

cudaError_t launch_decode(int k_bits, int v_bits, int group, const void* q, int B, int Hq, int Hkv,
                          const void* k_codes, const void* k_params, const float* k_scale,
                          const void* v_codes, const void* v_params, const float* v_scale,
                          const int32_t* block_table, int max_tiles, const int32_t* seq_lens,
                          const void* k_sink, const void* v_sink, int sink_len, const void* k_tail,
                          const void* v_tail, float softmax_scale, int rotate, int full_tail,
                          void* workspace, const DecodePlan& plan, float* out, cudaStream_t stream);

// Appending tokens: arguments of the append kernel (all device pointers).
struct AppendArgs {
    int Hkv, n_new, max_tiles, full_tail;
    const __nv_bfloat16* k_new;  // [B][Hkv][n_new][128]
    const __nv_bfloat16* v_new;
    const int32_t* n_accept;     // [B] or null (all offered tokens)
    int32_t* seq_lens;           // [B], updated
    __nv_bfloat16* k_tail;       // [B][Hkv][128][128], updated
    __nv_bfloat16* v_tail;
    const int32_t* block_table;  // [B][Hkv][max_tiles]
    __nv_bfloat16* k_stage;      // workspace: [B * Hkv][128][128], slot b * Hkv + h
    __nv_bfloat16* v_stage;
    int32_t* dest;               // workspace: [B * Hkv] pool tile of each staged block, -1 if none
};
size_t append_workspace_bytes(int B, int Hkv);
cudaError_t launch_append(const AppendArgs& a, int B, int k_bits, int v_bits, int iters, int rotate,
                          int normalize, void* k_codes, void* k_params, float* k_scale, void* v_codes,
                          void* v_params, float* v_scale, cudaStream_t stream);
cudaError_t read_and_clear_append_error(unsigned int* out);

// Self-check: one kernel whose bounded mbarrier wait runs out after limit_us (see bounded_wait.cu).
cudaError_t launch_bounded_wait_check(uint32_t limit_us, cudaStream_t stream);
cudaError_t read_and_clear_selftest_error(unsigned int* out);

}  // namespace kvarn
