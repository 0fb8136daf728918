// libkvarn C-ABI: argument validation and kernel launches.  See include/kvarn.h for the contract.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "../../include/kvarn.h"
#include "kvarn_internal.h"

namespace kvarn {

cudaError_t current_device(int* dev, int* sms) {
    static std::atomic<int> sm_count[kMaxCachedDevices] = {};  // 0: not queried yet
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    const bool cached = *dev >= 0 && *dev < kMaxCachedDevices;
    if (cached) {
        const int v = sm_count[*dev].load(std::memory_order_relaxed);
        if (v > 0) {
            *sms = v;
            return cudaSuccess;
        }
    }
    e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev);
    if (e == cudaSuccess && cached) sm_count[*dev].store(*sms, std::memory_order_relaxed);
    return e;
}

cudaError_t set_smem_limit_once(const void* kernel, int bytes, bool max_carveout, int dev) {
    struct Entry {
        const void* kernel;
        int dev, bytes;
    };
    static std::mutex mutex;
    static Entry done[256];  // a few dozen kernels x devices in practice
    static int n_done = 0;
    std::lock_guard<std::mutex> lock(mutex);
    for (int i = 0; i < n_done; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess && n_done < 256) done[n_done++] = Entry{kernel, dev, bytes};
    return e;
}

}  // namespace kvarn

namespace {

thread_local std::string g_last_error;

kvarn_status fail(kvarn_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvarn_status fail(kvarn_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

kvarn_status ok() {
    g_last_error.clear();
    return KVARN_OK;
}

kvarn_status cuda_fail(cudaError_t e, const char* what) {
    cudaGetLastError();  // consume
    return fail(KVARN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

kvarn_status check_cfg(const kvarn_config* cfg) {
    if (!cfg) return fail(KVARN_ERR_INVALID_ARG, "cfg is NULL");
    if (cfg->k_bits != 2 && cfg->k_bits != 4)
        return fail(KVARN_ERR_INVALID_ARG, "k_bits = %d; supported: 2, 4", cfg->k_bits);
    if (cfg->v_bits != 2 && cfg->v_bits != 4)
        return fail(KVARN_ERR_INVALID_ARG, "v_bits = %d; supported: 2, 4", cfg->v_bits);
    if (cfg->sinkhorn_iters < 0 || cfg->sinkhorn_iters > 64)
        return fail(KVARN_ERR_INVALID_ARG, "sinkhorn_iters = %d; allowed 0..64", cfg->sinkhorn_iters);
    if (cfg->flags & ~(KVARN_FLAG_NO_ROTATE | KVARN_FLAG_NO_NORMALIZE | KVARN_FLAG_FULL_TAIL))
        return fail(KVARN_ERR_INVALID_ARG, "unknown flag bits 0x%x", cfg->flags);
    return KVARN_OK;
}

kvarn_status check_ptr(const void* p, size_t align, const char* name) {
    if (!p) return fail(KVARN_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, align)) return fail(KVARN_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
    return KVARN_OK;
}

#define KV_TRY(expr)                     \
    do {                                 \
        kvarn_status _s = (expr);        \
        if (_s != KVARN_OK) return _s;   \
    } while (0)

}  // namespace

extern "C" {

kvarn_status kvarn_config_from_preset(const char* name, kvarn_config* out) {
    if (!name || !out) return fail(KVARN_ERR_INVALID_ARG, "name or out is NULL");
    struct Preset {
        const char* name;
        kvarn_config cfg;
    };
    static const Preset kPresets[] = {
        {"kvarn_k4v2_g128", {4, 2, 8, 0u}},
        {"kvarn_k2v2_g128", {2, 2, 8, 0u}},
        {"kvarn_k4v4_g128", {4, 4, 8, 0u}},
        {"kvarn_k2v4_g128", {2, 4, 8, 0u}},
        {"hadamard_k2v2_g128", {2, 2, 0, KVARN_FLAG_NO_NORMALIZE}},
        {"kivi_k2v2_g128", {2, 2, 0, KVARN_FLAG_NO_ROTATE | KVARN_FLAG_NO_NORMALIZE}},
    };
    for (const Preset& p : kPresets) {
        if (strcmp(name, p.name) == 0) {
            *out = p.cfg;
            return ok();
        }
    }
    return fail(KVARN_ERR_INVALID_ARG,
                "unknown preset '%s' (known: kvarn_k4v2_g128, kvarn_k2v2_g128, kvarn_k4v4_g128, "
                "kvarn_k2v4_g128, hadamard_k2v2_g128, kivi_k2v2_g128)",
                name);
}

size_t kvarn_tile_code_bytes(int bits) {
    return (bits == 2 || bits == 4) ? (size_t)KVARN_TILE_TOKENS * 16 * bits : 0;
}

size_t kvarn_tile_param_bytes(void) { return KVARN_PARAM_BYTES; }

kvarn_status kvarn_encode_blocks(const kvarn_config* cfg, kvarn_kind kind, const void* x_bf16,
                                 int64_t n_tiles, void* codes, void* params, float* tile_scale,
                                 kvarn_stream_t stream) {
    KV_TRY(check_cfg(cfg));
    if (kind != KVARN_KIND_K && kind != KVARN_KIND_V)
        return fail(KVARN_ERR_INVALID_ARG, "kind = %d; expected KVARN_KIND_K or KVARN_KIND_V", (int)kind);
    if (n_tiles < 0) return fail(KVARN_ERR_INVALID_ARG, "n_tiles = %lld < 0", (long long)n_tiles);
    if (n_tiles == 0) return ok();
    KV_TRY(check_ptr(x_bf16, 16, "x_bf16"));
    KV_TRY(check_ptr(codes, 16, "codes"));
    KV_TRY(check_ptr(params, 16, "params"));
    KV_TRY(check_ptr(tile_scale, 4, "tile_scale"));
    const int bits = kind == KVARN_KIND_K ? cfg->k_bits : cfg->v_bits;
    cudaError_t e = kvarn::launch_encode(bits, (int)kind, x_bf16, n_tiles, codes, params, tile_scale,
                                         cfg->sinkhorn_iters, !(cfg->flags & KVARN_FLAG_NO_ROTATE),
                                         !(cfg->flags & KVARN_FLAG_NO_NORMALIZE), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "encode launch");
    return ok();
}

kvarn_status kvarn_encode_kv_blocks(const kvarn_config* cfg, const void* k_bf16, const void* v_bf16,
                                    int64_t n_tiles, void* k_codes, void* k_params, float* k_scale,
                                    void* v_codes, void* v_params, float* v_scale,
                                    kvarn_stream_t stream) {
    KV_TRY(check_cfg(cfg));
    if (n_tiles < 0) return fail(KVARN_ERR_INVALID_ARG, "n_tiles = %lld < 0", (long long)n_tiles);
    if (n_tiles == 0) return ok();
    KV_TRY(check_ptr(k_bf16, 16, "k_bf16"));
    KV_TRY(check_ptr(v_bf16, 16, "v_bf16"));
    KV_TRY(check_ptr(k_codes, 16, "k_codes"));
    KV_TRY(check_ptr(k_params, 16, "k_params"));
    KV_TRY(check_ptr(k_scale, 4, "k_scale"));
    KV_TRY(check_ptr(v_codes, 16, "v_codes"));
    KV_TRY(check_ptr(v_params, 16, "v_params"));
    KV_TRY(check_ptr(v_scale, 4, "v_scale"));
    cudaError_t e = kvarn::launch_encode_kv(cfg->k_bits, cfg->v_bits, k_bf16, n_tiles, k_codes, k_params,
                                            k_scale, v_bf16, n_tiles, v_codes, v_params, v_scale,
                                            cfg->sinkhorn_iters, !(cfg->flags & KVARN_FLAG_NO_ROTATE),
                                            !(cfg->flags & KVARN_FLAG_NO_NORMALIZE), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "encode launch");
    return ok();
}

kvarn_status kvarn_dequant(const kvarn_config* cfg, kvarn_kind kind, const void* codes,
                           const void* params, const float* tile_scale, int64_t n_tiles,
                           int original_basis, float* out, kvarn_stream_t stream) {
    KV_TRY(check_cfg(cfg));
    if (kind != KVARN_KIND_K && kind != KVARN_KIND_V)
        return fail(KVARN_ERR_INVALID_ARG, "kind = %d; expected KVARN_KIND_K or KVARN_KIND_V", (int)kind);
    if (n_tiles < 0 || n_tiles > 0x7fffffffLL)
        return fail(KVARN_ERR_INVALID_ARG, "n_tiles = %lld outside 0..2^31-1", (long long)n_tiles);
    if (original_basis != 0 && original_basis != 1)
        return fail(KVARN_ERR_INVALID_ARG, "original_basis = %d; expected 0 or 1", original_basis);
    if (n_tiles == 0) return ok();
    KV_TRY(check_ptr(codes, 16, "codes"));
    KV_TRY(check_ptr(params, 16, "params"));
    KV_TRY(check_ptr(tile_scale, 4, "tile_scale"));
    KV_TRY(check_ptr(out, 16, "out"));
    const int bits = kind == KVARN_KIND_K ? cfg->k_bits : cfg->v_bits;
    cudaError_t e = kvarn::launch_dequant(bits, (int)kind, codes, params, tile_scale, n_tiles,
                                          original_basis, !(cfg->flags & KVARN_FLAG_NO_ROTATE), out,
                                          (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
    return ok();
}

static kvarn_status check_decode_shape(const kvarn_config* cfg, int B, int Hq, int Hkv, int max_tiles) {
    KV_TRY(check_cfg(cfg));
    if (B < 0 || B > 65535) return fail(KVARN_ERR_INVALID_ARG, "B = %d outside 0..65535", B);
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return fail(KVARN_ERR_INVALID_ARG, "Hq = %d, Hkv = %d: need Hq a positive multiple of Hkv", Hq, Hkv);
    if (Hq > 65535) return fail(KVARN_ERR_INVALID_ARG, "Hq = %d outside 1..65535", Hq);
    if (max_tiles < 0 || max_tiles > (1 << 24))
        return fail(KVARN_ERR_INVALID_ARG, "max_tiles = %d outside 0..2^24", max_tiles);
    return KVARN_OK;
}

size_t kvarn_decode_workspace_size(const kvarn_config* cfg, int B, int Hq, int Hkv, int max_tiles) {
    if (check_decode_shape(cfg, B, Hq, Hkv, max_tiles) != KVARN_OK) return 0;
    return kvarn::plan_decode(B, Hq, Hkv, max_tiles).workspace_bytes;
}

namespace {

kvarn_status decode_impl(const kvarn_config* cfg, const void* q_bf16, int B, int Hq, int Hkv,
                         const void* k_codes, const void* k_params, const float* k_scale,
                         const void* v_codes, const void* v_params, const float* v_scale,
                         const int32_t* block_table, int max_tiles, const int32_t* seq_lens,
                         const int32_t* seq_lens_host, const void* k_sink_bf16, const void* v_sink_bf16,
                         int sink_len, const void* k_tail_bf16, const void* v_tail_bf16,
                         float softmax_scale, void* workspace, size_t workspace_bytes, float* out,
                         kvarn_stream_t stream) {
    KV_TRY(check_decode_shape(cfg, B, Hq, Hkv, max_tiles));
    if (!isfinite(softmax_scale)) return fail(KVARN_ERR_INVALID_ARG, "softmax_scale is not finite");
    if (sink_len < 0 || sink_len > KVARN_TILE_TOKENS)
        return fail(KVARN_ERR_INVALID_ARG, "sink_len = %d outside 0..128", sink_len);
    if (B == 0) return ok();
    KV_TRY(check_ptr(q_bf16, 16, "q_bf16"));
    KV_TRY(check_ptr(seq_lens, 4, "seq_lens"));
    KV_TRY(check_ptr(k_tail_bf16, 16, "k_tail_bf16"));
    KV_TRY(check_ptr(v_tail_bf16, 16, "v_tail_bf16"));
    KV_TRY(check_ptr(out, 16, "out"));
    if (sink_len > 0) {
        KV_TRY(check_ptr(k_sink_bf16, 16, "k_sink_bf16"));
        KV_TRY(check_ptr(v_sink_bf16, 16, "v_sink_bf16"));
    }
    if (max_tiles > 0) {
        KV_TRY(check_ptr(k_codes, 16, "k_codes"));
        KV_TRY(check_ptr(k_params, 16, "k_params"));
        KV_TRY(check_ptr(k_scale, 4, "k_scale"));
        KV_TRY(check_ptr(v_codes, 16, "v_codes"));
        KV_TRY(check_ptr(v_params, 16, "v_params"));
        KV_TRY(check_ptr(v_scale, 4, "v_scale"));
        KV_TRY(check_ptr(block_table, 4, "block_table"));
    }
    if (seq_lens_host) {
        const long long cap = (long long)sink_len + (long long)max_tiles * KVARN_TILE_TOKENS +
                              ((cfg->flags & KVARN_FLAG_FULL_TAIL) ? KVARN_TILE_TOKENS : KVARN_TILE_TOKENS - 1);
        for (int b = 0; b < B; ++b)
            if (seq_lens_host[b] < 0 || seq_lens_host[b] > cap)
                return fail(KVARN_ERR_INVALID_ARG, "seq_lens[%d] = %d outside 0..%lld", b, seq_lens_host[b], cap);
    }
    const kvarn::DecodePlan plan = kvarn::plan_decode(B, Hq, Hkv, max_tiles);
    KV_TRY(check_ptr(workspace, 16, "workspace"));
    if (workspace_bytes < plan.workspace_bytes)
        return fail(KVARN_ERR_WORKSPACE, "workspace_bytes = %zu < required %zu", workspace_bytes,
                    plan.workspace_bytes);
    cudaError_t e = kvarn::launch_decode(cfg->k_bits, cfg->v_bits, Hq / Hkv, q_bf16, B, Hq, Hkv, k_codes,
                                         k_params, k_scale, v_codes, v_params, v_scale, block_table,
                                         max_tiles, seq_lens, k_sink_bf16, v_sink_bf16, sink_len, k_tail_bf16,
                                         v_tail_bf16, softmax_scale, !(cfg->flags & KVARN_FLAG_NO_ROTATE),
                                         (cfg->flags & KVARN_FLAG_FULL_TAIL) != 0, workspace, plan, out,
                                         (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
    return ok();
}

}  // namespace

kvarn_status kvarn_decode_attention(const kvarn_config* cfg, const void* q_bf16, int B, int Hq,
                                    int Hkv, const void* k_codes, const void* k_params,
                                    const float* k_scale, const void* v_codes,
                                    const void* v_params, const float* v_scale,
                                    const int32_t* block_table, int max_tiles,
                                    const int32_t* seq_lens, const int32_t* seq_lens_host,
                                    const void* k_tail_bf16, const void* v_tail_bf16,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    float* out, kvarn_stream_t stream) {
    return decode_impl(cfg, q_bf16, B, Hq, Hkv, k_codes, k_params, k_scale, v_codes, v_params, v_scale,
                       block_table, max_tiles, seq_lens, seq_lens_host, nullptr, nullptr, 0, k_tail_bf16,
                       v_tail_bf16, softmax_scale, workspace, workspace_bytes, out, stream);
}

kvarn_status kvarn_decode_attention_sink(const kvarn_config* cfg, const void* q_bf16, int B, int Hq,
                                         int Hkv, const void* k_codes, const void* k_params,
                                         const float* k_scale, const void* v_codes, const void* v_params,
                                         const float* v_scale, const int32_t* block_table, int max_tiles,
                                         const int32_t* seq_lens, const int32_t* seq_lens_host,
                                         const void* k_sink_bf16, const void* v_sink_bf16, int sink_len,
                                         const void* k_tail_bf16, const void* v_tail_bf16,
                                         float softmax_scale, void* workspace, size_t workspace_bytes,
                                         float* out, kvarn_stream_t stream) {
    return decode_impl(cfg, q_bf16, B, Hq, Hkv, k_codes, k_params, k_scale, v_codes, v_params, v_scale,
                       block_table, max_tiles, seq_lens, seq_lens_host, k_sink_bf16, v_sink_bf16, sink_len,
                       k_tail_bf16, v_tail_bf16, softmax_scale, workspace, workspace_bytes, out, stream);
}

kvarn_status kvarn_device_error(uint32_t* code_out) {
    if (!code_out) return fail(KVARN_ERR_INVALID_ARG, "code_out is NULL");
    unsigned int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
    e = kvarn::read_and_clear_device_error(&v);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    unsigned int w = 0;
    e = kvarn::read_and_clear_decode_error(&w);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    unsigned int x = 0;
    e = kvarn::read_and_clear_append_error(&x);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    unsigned int y = 0;
    e = kvarn::read_and_clear_selftest_error(&y);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    *code_out = v | (w << 1) | (x << 2) | (y << 3);
    if (*code_out & KVARN_DEVICE_TIMEOUT_BITS)
        return fail(KVARN_ERR_TIMEOUT, "a bounded device wait gave up (device error bits 0x%x)", *code_out);
    return ok();
}

kvarn_status kvarn_check_bounded_wait(uint32_t limit_us, kvarn_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000)
        return fail(KVARN_ERR_INVALID_ARG, "limit_us = %u outside 1..1000000", limit_us);
    cudaError_t e = kvarn::launch_bounded_wait_check(limit_us, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "bounded-wait check launch");
    return ok();
}

size_t kvarn_append_workspace_size(int B, int Hkv) {
    if (B < 0 || B > 65535 || Hkv < 1 || Hkv > 1024) return 0;
    return kvarn::append_workspace_bytes(B, Hkv);
}

kvarn_status kvarn_append_tokens(const kvarn_config* cfg, int B, int Hkv, const void* k_new_bf16,
                                 const void* v_new_bf16, int n_new, const int32_t* n_accept,
                                 int32_t* seq_lens, void* k_tail_bf16, void* v_tail_bf16, void* k_codes,
                                 void* k_params, float* k_scale, void* v_codes, void* v_params,
                                 float* v_scale, const int32_t* block_table, int max_tiles, void* workspace,
                                 size_t workspace_bytes, kvarn_stream_t stream) {
    KV_TRY(check_cfg(cfg));
    if (B < 0 || B > 65535) return fail(KVARN_ERR_INVALID_ARG, "B = %d outside 0..65535", B);
    if (Hkv < 1 || Hkv > 1024) return fail(KVARN_ERR_INVALID_ARG, "Hkv = %d outside 1..1024", Hkv);
    if (n_new < 1 || n_new > KVARN_TILE_TOKENS) return fail(KVARN_ERR_INVALID_ARG, "n_new = %d outside 1..128", n_new);
    if (max_tiles < 0 || max_tiles > (1 << 24))
        return fail(KVARN_ERR_INVALID_ARG, "max_tiles = %d outside 0..2^24", max_tiles);
    if (B == 0) return ok();
    KV_TRY(check_ptr(k_new_bf16, 16, "k_new_bf16"));
    KV_TRY(check_ptr(v_new_bf16, 16, "v_new_bf16"));
    if (n_accept) KV_TRY(check_ptr(n_accept, 4, "n_accept"));
    KV_TRY(check_ptr(seq_lens, 4, "seq_lens"));
    KV_TRY(check_ptr(k_tail_bf16, 16, "k_tail_bf16"));
    KV_TRY(check_ptr(v_tail_bf16, 16, "v_tail_bf16"));
    if (max_tiles > 0) {
        KV_TRY(check_ptr(k_codes, 16, "k_codes"));
        KV_TRY(check_ptr(k_params, 16, "k_params"));
        KV_TRY(check_ptr(k_scale, 4, "k_scale"));
        KV_TRY(check_ptr(v_codes, 16, "v_codes"));
        KV_TRY(check_ptr(v_params, 16, "v_params"));
        KV_TRY(check_ptr(v_scale, 4, "v_scale"));
        KV_TRY(check_ptr(block_table, 4, "block_table"));
    }
    KV_TRY(check_ptr(workspace, 256, "workspace"));
    const size_t need = kvarn::append_workspace_bytes(B, Hkv);
    if (workspace_bytes < need)
        return fail(KVARN_ERR_WORKSPACE, "workspace_bytes = %zu < required %zu", workspace_bytes, need);
    kvarn::AppendArgs a;
    a.Hkv = Hkv;
    a.n_new = n_new;
    a.max_tiles = max_tiles;
    a.full_tail = (cfg->flags & KVARN_FLAG_FULL_TAIL) != 0;
    a.k_new = static_cast<const __nv_bfloat16*>(k_new_bf16);
    a.v_new = static_cast<const __nv_bfloat16*>(v_new_bf16);
    a.n_accept = n_accept;
    a.seq_lens = seq_lens;
    a.k_tail = static_cast<__nv_bfloat16*>(k_tail_bf16);
    a.v_tail = static_cast<__nv_bfloat16*>(v_tail_bf16);
    a.block_table = block_table;
    const size_t tiles = (size_t)B * Hkv;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    a.k_stage = reinterpret_cast<__nv_bfloat16*>(w);
    a.v_stage = reinterpret_cast<__nv_bfloat16*>(w + tiles * KVARN_TILE_TOKENS * KVARN_TILE_TOKENS * 2);
    a.dest = reinterpret_cast<int32_t*>(w + 2 * tiles * KVARN_TILE_TOKENS * KVARN_TILE_TOKENS * 2);
    cudaError_t e = kvarn::launch_append(a, B, cfg->k_bits, cfg->v_bits, cfg->sinkhorn_iters,
                                         !(cfg->flags & KVARN_FLAG_NO_ROTATE),
                                         !(cfg->flags & KVARN_FLAG_NO_NORMALIZE), k_codes, k_params, k_scale,
                                         v_codes, v_params, v_scale, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return ok();
}

// ---- decode attention with library-owned scratch (no allocation by the caller or the library) ----
// The split-K partials normally live in a caller-supplied workspace.  This variant keeps them in a
// fixed device array instead, for callers that have no way to obtain device memory at this point.
// Every GPU that loads the library holds the array (KVARN_STATIC_WS_BYTES) until the process exits.
static __device__ __align__(256) unsigned char g_kvarn_static_ws[KVARN_STATIC_WS_BYTES];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_static_ws_mutex;
void* g_static_ws_ptr[kMaxDevices] = {};  // device address of g_kvarn_static_ws, per device
}  // namespace

kvarn_status kvarn_decode_attention_static_ws(
    const kvarn_config* cfg, const void* q_bf16, int B, int Hq, int Hkv, const void* k_codes,
    const void* k_params, const float* k_scale, const void* v_codes, const void* v_params,
    const float* v_scale, const int32_t* block_table, int max_tiles, const int32_t* seq_lens,
    const int32_t* seq_lens_host, const void* k_tail_bf16, const void* v_tail_bf16,
    float softmax_scale, float* out, kvarn_stream_t stream) {
    const size_t need = kvarn_decode_workspace_size(cfg, B, Hq, Hkv, max_tiles);
    if (need > (size_t)KVARN_STATIC_WS_BYTES)
        return fail(KVARN_ERR_WORKSPACE,
                    "this shape needs %zu bytes of split-K scratch; the static scratch holds %zu "
                    "(use kvarn_decode_attention with a caller workspace)",
                    need, (size_t)KVARN_STATIC_WS_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KVARN_ERR_UNSUPPORTED, "device index %d", dev);
    void* ws = nullptr;
    {
        // First call on this device (with it current): look up the array's device address once.
        std::lock_guard<std::mutex> lock(g_static_ws_mutex);
        if (!g_static_ws_ptr[dev]) {
            e = cudaGetSymbolAddress(&g_static_ws_ptr[dev], g_kvarn_static_ws);
            if (e != cudaSuccess) {
                g_static_ws_ptr[dev] = nullptr;
                return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
            }
        }
        ws = g_static_ws_ptr[dev];
    }
    // Every partial the kernels read is written earlier in the same call, so the array needs no
    // clearing between calls.
    return kvarn_decode_attention(cfg, q_bf16, B, Hq, Hkv, k_codes, k_params, k_scale, v_codes,
                                  v_params, v_scale, block_table, max_tiles, seq_lens, seq_lens_host,
                                  k_tail_bf16, v_tail_bf16, softmax_scale, ws,
                                  (size_t)KVARN_STATIC_WS_BYTES, out, stream);
}

const char* kvarn_status_string(kvarn_status status) {
    switch (status) {
        case KVARN_OK: return "KVARN_OK";
        case KVARN_ERR_INVALID_ARG: return "KVARN_ERR_INVALID_ARG: an argument is out of range";
        case KVARN_ERR_UNSUPPORTED: return "KVARN_ERR_UNSUPPORTED: valid but not implemented";
        case KVARN_ERR_CUDA: return "KVARN_ERR_CUDA: a CUDA call or kernel launch failed";
        case KVARN_ERR_WORKSPACE: return "KVARN_ERR_WORKSPACE: workspace too small";
        case KVARN_ERR_TIMEOUT: return "KVARN_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown kvarn_status";
}

const char* kvarn_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
