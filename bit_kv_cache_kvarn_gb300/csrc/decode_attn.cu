// Decode attention over the packed KVarN cache: one query per sequence, grouped-query heads.
//
// Method: the quantised cache is restored at attention read time (dimensionstp.github.io review,
// "4-2 Training strategy"); the query is rotated by the same head-wise Hadamard after RoPE, so
// keys stay in the rotated basis (paperlayer.ai summary, "A Hadamard Transform Arrangement");
// the second scale s2 costs one multiply per element and is fused into the dequantisation
// (paperlayer.ai, "3 Methods" and "I KVarN Dequantization Overhead").  Here both scales are
// folded out of the inner loops entirely:
//   K (groups = channels): s_t = s2_t * g * (sum_j q'_j S1_j code_tj + sum_j q'_j Z_j)
//   V (groups = tokens):   o_j += g * s2_j * (sum_t p_t S1_t code_tj + sum_t p_t Z_t)
//
// Kernel 1 (split): CTA = (split of the context, kv head, sequence); each of its 8 warps owns whole
// tiles and keeps its own online-softmax state.  Codes become floats without int->float
// conversions: OR-ing a code field into the mantissa of 2^23 and subtracting 2^23 gives
// code * 2^shift exactly, and the 2^-shift is folded into the per-channel factors; pairs of
// channels then go through packed FFMA2.  Kernel 2 (merge): one warp per query head merges the
// splits by log-sum-exp, applies the inverse rotation, attends to the unquantised bf16 tail and
// normalises.  No device-side waits anywhere.
#include <math.h>

#include "kvarn_common.cuh"
#include "kvarn_internal.h"
#include "tcgen05.cuh"

namespace kvarn {

// Set when a tensor-core completion wait gives up (bounded); read by kvarn_device_error.
__device__ unsigned int g_decode_error = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kTilesPerSplit = 16;
constexpr int kWsStride = 132;  // floats per (sequence, query head, split): m, l, pad, pad, o[128]

struct DecodeArgs {
    const __nv_bfloat16* q;
    int Hq, Hkv, group;
    const uint8_t* k_codes;
    const uint8_t* k_params;
    const float* k_scale;
    const uint8_t* v_codes;
    const uint8_t* v_params;
    const float* v_scale;
    const int32_t* block_table;
    int max_tiles;
    const int32_t* seq_lens;
    const __nv_bfloat16* k_tail;
    const __nv_bfloat16* v_tail;
    float qscale;  // softmax scale * log2(e): scores are kept in the log2 domain
    int rotate;
    int splits;
    float* ws;
    float* out;
};

__device__ __forceinline__ int clamp_len(int len, int max_tiles) {
    const int cap = max_tiles * kTile + (kTile - 1);
    return len < 0 ? 0 : (len > cap ? cap : len);
}

// ---- tensor-core split kernel -------------------------------------------------------------------
// Per warpgroup and tile: thread r unpacks K row r (token r) to fp16 straight into TMEM (the A
// operand), builds column r of q'' = q' o S1 (channel r) as fp16 hi/lo pieces in shared memory
// (the B operand), and one thread issues D_S[128 tok x 16] = A x B.  Thread r then owns token r's
// scores, runs the online softmax, writes p o S1 for token r as the next B operand, unpacks V row r
// (channel r) into TMEM and D_O[128 ch x 16] = A x B gives channel r of the output.  N = 16 holds
// up to 8 heads x (hi, lo).

constexpr int kWG = 2;                    // warpgroups per CTA
constexpr int kTmemColsPerWG = 128;       // A: 0..63, D_S: 64..79, D_O: 96..111
constexpr uint32_t kBBytes = 16 * 128 * 2;  // one B operand: 16 rows x 128 K fp16
constexpr uint32_t kLbo = 128, kSbo = 2048;  // K-major core-matrix strides of B
constexpr float kWScale = 32.f;          // p * S1 <= 256 -> x32 stays inside fp16

// Byte offset of B element (row n, K index kk) in the K-major no-swizzle layout.
__device__ __forceinline__ uint32_t b_off(int n, int kk) {
    return (uint32_t)((kk >> 3) * kLbo + (n >> 3) * kSbo + (n & 7) * 16 + (kk & 7) * 2);
}

// Position of column c (0..127) of a packed row in the MMA K order, and the power-of-two factor
// the unpacked code carries there (the B element is multiplied by its inverse).
template <int BITS>
__device__ __forceinline__ void k_slot(int c, int& kk, float& inv_pre) {
    const int h = c & 15, i = c >> 4;
    if (BITS == 2) {
        // word h>>1 holds lanes (h even: low half, h odd: high half); pair i -> TMEM column 8w+i
        const int col = 8 * (h >> 1) + i;
        kk = 2 * col + (h & 1);
        inv_pre = ldexpf(1.f, -2 * (i <= 4 ? i : i - 5));
    } else {
        // word h holds codes i at bits 4i; pair (i, i+4) -> TMEM column 4h + (i&3)
        const int ii = i & 3;
        kk = 2 * (4 * h + ii) + (i >> 2);
        inv_pre = ldexpf(1.f, -4 * (ii <= 1 ? ii : ii - 2));
    }
}

__device__ __forceinline__ uint32_t hsub1024(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    v = __hsub2(v, __floats2half2_rn(1024.f, 1024.f));
    return *reinterpret_cast<uint32_t*>(&v);
}

// Unpack one packed row (BITS*4 words) into 64 fp16x2 TMEM columns starting at taddr.
template <int BITS>
__device__ __forceinline__ void unpack_row_to_tmem(const uint4 (&row)[BITS], uint32_t taddr) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&row[0]);
#pragma unroll
    for (int chunk = 0; chunk < 4; ++chunk) {
        uint32_t r[16];
        if (BITS == 2) {
#pragma unroll
            for (int ww = 0; ww < 2; ++ww) {
                const uint32_t x = w[2 * chunk + ww];
                const uint32_t xs = x >> 10;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t u = (i <= 4) ? ((x & (0x00030003u << (2 * i))) | 0x64006400u)
                                                : ((xs & (0x00030003u << (2 * (i - 5)))) | 0x64006400u);
                    r[8 * ww + i] = hsub1024(u);
                }
            }
        } else {
#pragma unroll
            for (int ww = 0; ww < 4; ++ww) {
                const uint32_t x = w[4 * chunk + ww];
                const uint32_t xs = x >> 8;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t u = (i <= 1) ? ((x & (0x000F000Fu << (4 * i))) | 0x64006400u)
                                                : ((xs & (0x000F000Fu << (4 * (i - 2)))) | 0x64006400u);
                    r[4 * ww + i] = hsub1024(u);
                }
            }
        }
        tc::st16(taddr + 16 * chunk, r);
    }
}

__device__ __forceinline__ void split_hi_lo(float x, __half& hi, __half& lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier over n threads that also returns the AND of every thread's flag.
__device__ __forceinline__ bool named_sync_and(int id, int n, bool flag) {
    uint32_t out;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n bar.red.and.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(out)
        : "r"(id), "r"(n), "r"((uint32_t)flag)
        : "memory");
    return out != 0;
}

template <int KB, int VB>
struct TileRegs {
    uint4 k[KB];
    uint4 v[VB];
    float s1k, zk, s2k, s1v, zv, s2v, gk, gv;
};

template <int KB, int VB>
__device__ __forceinline__ void load_tile(TileRegs<KB, VB>& t, const DecodeArgs& a, int64_t tile, int r) {
    const uint4* kc = reinterpret_cast<const uint4*>(a.k_codes + tile * (kTile * 16 * KB) + r * (16 * KB));
    const uint4* vc = reinterpret_cast<const uint4*>(a.v_codes + tile * (kTile * 16 * VB) + r * (16 * VB));
#pragma unroll
    for (int u = 0; u < KB; ++u) t.k[u] = __ldg(kc + u);
#pragma unroll
    for (int u = 0; u < VB; ++u) t.v[u] = __ldg(vc + u);
    const uint8_t* kp = a.k_params + tile * KVARN_PARAM_BYTES;
    const uint8_t* vp = a.v_params + tile * KVARN_PARAM_BYTES;
    t.s1k = e4m3_value(kp[r]);         // K group scale: channel r
    t.s2k = e4m3_value(kp[128 + r]);   // K other-axis scale: token r
    t.zk = fp16_value(reinterpret_cast<const uint16_t*>(kp + 256)[r]);
    t.s1v = e4m3_value(vp[r]);         // V group scale: token r
    t.s2v = e4m3_value(vp[128 + r]);   // V other-axis scale: channel r
    t.zv = fp16_value(reinterpret_cast<const uint16_t*>(vp + 256)[r]);
    t.gk = a.k_scale[tile];
    t.gv = a.v_scale[tile];
}

template <int KB, int VB, int GH>
__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    uint8_t* b_all = dsm;                                                  // [WG][2][kBBytes]
    float* qrs = reinterpret_cast<float*>(dsm + kWG * 2 * kBBytes);        // [GH][128] scaled q'
    float* einv = qrs + GH * kTile;                                        // [GH] 2^-E_h
    float* red = einv + 8;                                                 // [WG][3][4 warps][8]
    float* ms = red + kWG * 3 * 4 * 8;                                     // [WG][GH]
    float* ls = ms + kWG * GH;                                             // [WG][GH]
    float* os = ls + kWG * GH;                                             // [WG][GH][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(os + kWG * GH * kTile);   // [WG]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kWG);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wg = warp >> 2, wq = warp & 3, r = tid & 127;
    const int split = blockIdx.x;
    const int hblocks = a.group / GH;
    const int kvh = blockIdx.y / hblocks;
    const int hq0 = kvh * a.group + (blockIdx.y % hblocks) * GH;
    const int b = blockIdx.z;
    const int len = clamp_len(a.seq_lens[b], a.max_tiles);
    const int n_full = len >> 7;
    const int t_begin = split * kTilesPerSplit;
    const int t_end = min(t_begin + kTilesPerSplit, n_full);

    if (t_begin >= t_end) {  // nothing to read: empty partials
        for (int e = tid; e < GH * kTile; e += kThreads) {
            float* dst = a.ws + (((size_t)b * a.Hq + hq0 + (e >> 7)) * a.splits + split) * kWsStride;
            dst[4 + (e & 127)] = 0.f;
            if ((e & 127) == 0) {
                dst[0] = -INFINITY;
                dst[1] = 0.f;
            }
        }
        return;
    }

    // rotated queries, scaled so that |q'| * 2^E_h <= 2^6 (then q'' = q' S1 <= 2^14 fits fp16)
    if (warp < GH) {
        const __nv_bfloat16* qp = a.q + ((size_t)b * a.Hq + hq0 + warp) * kTile + 4 * lane;
        const uint2 raw = *reinterpret_cast<const uint2*>(qp);
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        float v[4] = {f0.x, f0.y, f1.x, f1.y};
        float sc = a.qscale;
        if (a.rotate) {
            fwht128_warp(v, lane);
            sc *= kInvSqrt128;
        }
        float mx = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            v[m] *= sc;
            mx = fmaxf(mx, fabsf(v[m]));
        }
        mx = warp_max(mx);
        const int e = mx > 0.f ? 6 - ceil_log2(mx) : 0;
        const float s = ldexpf(1.f, e);
#pragma unroll
        for (int m = 0; m < 4; ++m) qrs[warp * kTile + 4 * lane + m] = v[m] * s;
        if (lane == 0) einv[warp] = ldexpf(1.f, -e);
    }
    // B operands: rows 2*GH..15 stay zero
    for (int i = tid; i < (int)(kWG * 2 * kBBytes / 16); i += kThreads)
        reinterpret_cast<uint4*>(b_all)[i] = make_uint4(0, 0, 0, 0);
    if (tid < kWG) mbar_init(&bars[tid], 1);
    if (warp == 0) tc::alloc(tmem_slot, kWG * kTmemColsPerWG);
    fence_mbar_init();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    uint8_t* bk = b_all + wg * 2 * kBBytes;
    uint8_t* bv = bk + kBBytes;
    float* cpart = red + wg * 96;   // [4 warps][8]
    float* mpart = cpart + 32;
    float* zpart = mpart + 32;
    const uint32_t col0 = tmem + wg * kTmemColsPerWG;
    const uint32_t lane_addr = col0 + ((uint32_t)(32 * wq) << 16);  // this thread's TMEM lane
    const uint32_t bk_addr = smem_addr(bk), bv_addr = smem_addr(bv);
    constexpr uint32_t kIdesc = tc::idesc_f16_f32(128, 16);
    const int bar_id = 1 + wg;

    // this thread's slot in the MMA K order: as channel r of a K row, and as token r of a V row
    int kk_k, kk_v;
    float pre_k, pre_v;
    k_slot<KB>(r, kk_k, pre_k);
    k_slot<VB>(r, kk_v, pre_v);

    float m_run[GH], l_part[GH], o[GH];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
        o[h] = 0.f;
    }
    uint32_t phase = 0;
    bool alive = true;
    const int32_t* table = a.block_table + ((size_t)b * a.Hkv + kvh) * a.max_tiles;

    TileRegs<KB, VB> cur, nxt;
    int ti = t_begin + wg;
    if (ti < t_end) load_tile(cur, a, table[ti], r);
    for (; ti < t_end && alive; ti += kWG) {
        if (ti + kWG < t_end) load_tile(nxt, a, table[ti + kWG], r);

        // ---- scores: A = K codes (row r = token r), B = q'' pieces (column r = channel r) ----
        unpack_row_to_tmem<KB>(cur.k, lane_addr);
        {
            const float s1 = cur.s1k * pre_k;
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                __half hi, lo;
                split_hi_lo(qrs[h * kTile + r] * s1, hi, lo);
                *reinterpret_cast<__half*>(bk + b_off(2 * h, kk_k)) = hi;
                *reinterpret_cast<__half*>(bk + b_off(2 * h + 1, kk_k)) = lo;
                const float c = warp_sum(qrs[h * kTile + r] * cur.zk);
                if (lane == 0) cpart[wq * 8 + h] = c;
            }
        }
        fence_proxy_async();
        tc::wait_st();
        tc::fence_before();
        named_sync(bar_id, 128);
        if (r == 0) {
            tc::fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma_f16_ts(col0 + 64, col0 + 8 * s, tc::smem_desc(bk_addr + s * 2 * kLbo, kLbo, kSbo), kIdesc, s > 0);
            tc::commit(&bars[wg]);
        }
        alive = mbar_wait(&bars[wg], phase, &g_decode_error);
        phase ^= 1;
        tc::fence_after();
        uint32_t d[16];
        tc::ld16(lane_addr + 64, d);
        tc::wait_ld();

        // ---- online softmax over this tile's 128 tokens (thread r = token r), log2 domain ----
        float s[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const float c = cpart[h] + cpart[8 + h] + cpart[16 + h] + cpart[24 + h];
            s[h] = (__uint_as_float(d[2 * h]) + __uint_as_float(d[2 * h + 1]) + c) * (einv[h] * cur.gk * cur.s2k);
            const float mx = warp_max(s[h]);
            if (lane == 0) mpart[wq * 8 + h] = mx;
        }
        named_sync(bar_id, 128);
        float alpha[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const float mt = fmaxf(fmaxf(mpart[h], mpart[8 + h]), fmaxf(mpart[16 + h], mpart[24 + h]));
            const float m_new = fmaxf(m_run[h], mt);
            alpha[h] = exp2f(m_run[h] - m_new);
            m_run[h] = m_new;
            const float p = exp2f(s[h] - m_new);
            l_part[h] = fmaf(l_part[h], alpha[h], p);
            __half hi, lo;
            split_hi_lo(p * cur.s1v * (kWScale * pre_v), hi, lo);
            *reinterpret_cast<__half*>(bv + b_off(2 * h, kk_v)) = hi;
            *reinterpret_cast<__half*>(bv + b_off(2 * h + 1, kk_v)) = lo;
            const float z = warp_sum(p * cur.zv);
            if (lane == 0) zpart[wq * 8 + h] = z;
        }

        // ---- PV: A = V codes (row r = channel r), B = p S1 pieces (column r = token r) ----
        unpack_row_to_tmem<VB>(cur.v, lane_addr);
        fence_proxy_async();
        tc::wait_st();
        tc::fence_before();
        named_sync(bar_id, 128);
        if (r == 0) {
            tc::fence_after();
#pragma unroll
            for (int s2 = 0; s2 < 8; ++s2)
                tc::mma_f16_ts(col0 + 96, col0 + 8 * s2, tc::smem_desc(bv_addr + s2 * 2 * kLbo, kLbo, kSbo), kIdesc, s2 > 0);
            tc::commit(&bars[wg]);
        }
        alive = mbar_wait(&bars[wg], phase, &g_decode_error) && alive;
        phase ^= 1;
        tc::fence_after();
        tc::ld16(lane_addr + 96, d);
        tc::wait_ld();
        {
            const float sc = cur.gv * cur.s2v;  // channel r
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float z = zpart[h] + zpart[8 + h] + zpart[16 + h] + zpart[24 + h];
                const float acc = (__uint_as_float(d[2 * h]) + __uint_as_float(d[2 * h + 1])) * (1.f / kWScale) + z;
                o[h] = fmaf(o[h], alpha[h], acc * sc);
            }
        }
        cur = nxt;
        // the scratch (cpart/mpart/zpart, B) of this tile is reused by the next: all threads must
        // be past their reads; the barrier also makes the give-up decision uniform
        tc::fence_before();
        alive = named_sync_and(bar_id, 128, alive);
        tc::fence_after();
    }

    // ---- merge the warpgroups of this CTA ----
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        const float lsum = warp_sum(l_part[h]);
        if (lane == 0) red[wg * 96 + wq * 8 + h] = lsum;
        os[(wg * GH + h) * kTile + r] = o[h];
        if (r == 0) ms[wg * GH + h] = m_run[h];
    }
    tc::fence_before();
    __syncthreads();
    for (int e = tid; e < GH * kTile; e += kThreads) {
        const int h = e >> 7, j = e & 127;
        float mmax = -INFINITY;
#pragma unroll
        for (int g = 0; g < kWG; ++g) mmax = fmaxf(mmax, ms[g * GH + h]);
        float ov = 0.f, l = 0.f;
        if (mmax != -INFINITY) {
#pragma unroll
            for (int g = 0; g < kWG; ++g) {
                const float f = exp2f(ms[g * GH + h] - mmax);
                const float lg = red[g * 96 + h] + red[g * 96 + 8 + h] + red[g * 96 + 16 + h] + red[g * 96 + 24 + h];
                ov = fmaf(os[(g * GH + h) * kTile + j], f, ov);
                l = fmaf(lg, f, l);
            }
        }
        float* dst = a.ws + (((size_t)b * a.Hq + hq0 + h) * a.splits + split) * kWsStride;
        dst[4 + j] = ov;
        if (j == 0) {
            dst[0] = mmax;
            dst[1] = l;
        }
    }
    tc::fence_after();
    if (warp == 0) tc::dealloc(tmem, kWG * kTmemColsPerWG);
}

// One warp per (sequence, query head): merge splits, inverse rotation, bf16 tail, normalise.
__global__ void __launch_bounds__(32) decode_merge_kernel(DecodeArgs a) {
    const int lane = threadIdx.x;
    const int hq = blockIdx.x, b = blockIdx.y;
    const int kvh = hq / a.group;
    const int len = clamp_len(a.seq_lens[b], a.max_tiles);
    const int tail = len & 127;
    const float* base = a.ws + ((size_t)b * a.Hq + hq) * a.splits * kWsStride;

    float mmax = -INFINITY;
    for (int s = lane; s < a.splits; s += 32) mmax = fmaxf(mmax, base[s * kWsStride]);
    mmax = warp_max(mmax);
    float l = 0.f;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    if (mmax != -INFINITY) {
        for (int s = 0; s < a.splits; ++s) {
            const float f = exp2f(base[s * kWsStride] - mmax);
            l = fmaf(base[s * kWsStride + 1], f, l);
            const float4 v = *reinterpret_cast<const float4*>(base + s * kWsStride + 4 + 4 * lane);
            o[0] = fmaf(v.x, f, o[0]);
            o[1] = fmaf(v.y, f, o[1]);
            o[2] = fmaf(v.z, f, o[2]);
            o[3] = fmaf(v.w, f, o[3]);
        }
        if (a.rotate) {
            fwht128_warp(o, lane);
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] *= kInvSqrt128;
        }
    }
    if (tail > 0) {
        const __nv_bfloat16* qp = a.q + ((size_t)b * a.Hq + hq) * kTile + 4 * lane;
        float qv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) qv[m] = __bfloat162float(qp[m]) * a.qscale;
        const size_t tb = ((size_t)b * a.Hkv + kvh) * kTile * kTile;
        for (int t = 0; t < tail; ++t) {
            const __nv_bfloat16* kt = a.k_tail + tb + (size_t)t * kTile + 4 * lane;
            const __nv_bfloat16* vt = a.v_tail + tb + (size_t)t * kTile + 4 * lane;
            float d = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) d = fmaf(qv[m], __bfloat162float(kt[m]), d);
            d = warp_sum(d);
            const float m_new = fmaxf(mmax, d);
            const float al = exp2f(mmax - m_new);
            const float p = exp2f(d - m_new);
            l = fmaf(l, al, p);
#pragma unroll
            for (int m = 0; m < 4; ++m) o[m] = fmaf(o[m], al, p * __bfloat162float(vt[m]));
            mmax = m_new;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float4 r = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
    *reinterpret_cast<float4*>(a.out + ((size_t)b * a.Hq + hq) * kTile + 4 * lane) = r;
}

template <int GH>
size_t split_smem_bytes() {
    size_t bytes = (size_t)kWG * 2 * kBBytes + (size_t)GH * kTile * 4 + 8 * 4 + kWG * 3 * 4 * 8 * 4 +
                   2 * kWG * GH * 4 + (size_t)kWG * GH * kTile * 4 + kWG * 8 + 16;
    // at least 80 KB, so no more than two CTAs (2 x 256 TMEM columns) share an SM
    return bytes < 80 * 1024 ? 80 * 1024 : bytes;
}

template <int KB, int VB, int GH>
cudaError_t run_split(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
    auto kern = decode_split_kernel<KB, VB, GH>;
    const size_t smem = split_smem_bytes<GH>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int KB, int VB>
cudaError_t run_split_g(const DecodeArgs& a, int gh, dim3 grid, cudaStream_t stream) {
    if (gh == 1) return run_split<KB, VB, 1>(a, grid, stream);
    if (gh == 2) return run_split<KB, VB, 2>(a, grid, stream);
    if (gh == 4) return run_split<KB, VB, 4>(a, grid, stream);
    return run_split<KB, VB, 8>(a, grid, stream);
}

}  // namespace

DecodePlan plan_decode(int B, int Hq, int /*Hkv*/, int max_tiles) {
    DecodePlan p;
    p.tiles_per_split = kTilesPerSplit;
    p.splits = max_tiles <= 0 ? 1 : (max_tiles + kTilesPerSplit - 1) / kTilesPerSplit;
    p.workspace_bytes = (size_t)B * Hq * p.splits * kWsStride * sizeof(float);
    return p;
}

cudaError_t read_and_clear_decode_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

cudaError_t launch_decode(int k_bits, int v_bits, int group, const void* q, int B, int Hq, int Hkv,
                          const void* k_codes, const void* k_params, const float* k_scale,
                          const void* v_codes, const void* v_params, const float* v_scale,
                          const int32_t* block_table, int max_tiles, const int32_t* seq_lens,
                          const void* k_tail, const void* v_tail, float softmax_scale, int rotate,
                          void* workspace, const DecodePlan& plan, float* out,
                          cudaStream_t stream) {
    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.group = group;
    a.k_codes = static_cast<const uint8_t*>(k_codes);
    a.k_params = static_cast<const uint8_t*>(k_params);
    a.k_scale = k_scale;
    a.v_codes = static_cast<const uint8_t*>(v_codes);
    a.v_params = static_cast<const uint8_t*>(v_params);
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.max_tiles = max_tiles;
    a.seq_lens = seq_lens;
    a.k_tail = static_cast<const __nv_bfloat16*>(k_tail);
    a.v_tail = static_cast<const __nv_bfloat16*>(v_tail);
    a.qscale = softmax_scale * kLog2e;
    a.rotate = rotate;
    a.splits = plan.splits;
    a.ws = static_cast<float*>(workspace);
    a.out = out;
    const int gh = group;  // up to 8 heads x (hi, lo) fill the 16 MMA columns
    dim3 grid(plan.splits, Hkv * (group / gh), B);
    cudaError_t e;
    if (k_bits == 2 && v_bits == 2) e = run_split_g<2, 2>(a, gh, grid, stream);
    else if (k_bits == 4 && v_bits == 2) e = run_split_g<4, 2>(a, gh, grid, stream);
    else if (k_bits == 2 && v_bits == 4) e = run_split_g<2, 4>(a, gh, grid, stream);
    else e = run_split_g<4, 4>(a, gh, grid, stream);
    if (e != cudaSuccess) return e;
    decode_merge_kernel<<<dim3(Hq, B), 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvarn
