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

namespace kvarn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
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

__device__ __forceinline__ uint32_t word_of(const uint4& v, int c) {
    return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

template <int KB, int VB, int GH>
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t dsm[];
    float* qr = reinterpret_cast<float*>(dsm);                         // [GH][128]
    float2* q2_all = reinterpret_cast<float2*>(qr + GH * kTile);       // [warp][64 pairs][GH]
    float2* wb_all = q2_all + kWarps * 64 * GH;                        // [warp][128 tok][GH]
    float* ms = reinterpret_cast<float*>(wb_all + kWarps * kTile * GH); // [warp][GH]
    float* ls = ms + kWarps * GH;                                      // [warp][GH]
    float* os = ls + kWarps * GH;                                      // [warp][GH][128]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x;
    const int hblocks = a.group / GH;
    const int kvh = blockIdx.y / hblocks;
    const int hq0 = kvh * a.group + (blockIdx.y % hblocks) * GH;  // first query head of the CTA
    const int b = blockIdx.z;

    const int len = clamp_len(a.seq_lens[b], a.max_tiles);
    const int n_full = len >> 7;
    const int t_begin = split * kTilesPerSplit;
    const int t_end = min(t_begin + kTilesPerSplit, n_full);

    // rotated, scaled queries
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
#pragma unroll
        for (int m = 0; m < 4; ++m) qr[warp * kTile + 4 * lane + m] = v[m] * sc;
    }
    __syncthreads();

    float2* q2 = q2_all + warp * 64 * GH;
    float2* wb = wb_all + warp * kTile * GH;
    const int lw = lane & 15, ts = lane >> 4;

    float m_run[GH], l_lane[GH];
    float2 o2[GH][4];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        m_run[h] = -INFINITY;
        l_lane[h] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) o2[h][i] = make_float2(0.f, 0.f);
    }

    const int32_t* table = a.block_table + ((size_t)b * a.Hkv + kvh) * a.max_tiles;
    for (int ti = t_begin + warp; ti < t_end; ti += kWarps) {
        const int64_t tile = table[ti];
        const uint8_t* kp = a.k_params + tile * KVARN_PARAM_BYTES;
        const uint8_t* vp = a.v_params + tile * KVARN_PARAM_BYTES;
        const float gk = a.k_scale[tile];
        const float gv = a.v_scale[tile];
        const uint8_t* kc = a.k_codes + tile * (kTile * 16 * KB);
        const uint8_t* vc = a.v_codes + tile * (kTile * 16 * VB);

        // issue the K code loads first (rows l, l+32, l+64, l+96; 16-byte loads)
        constexpr int kRowU4 = KB;  // uint4 per row: 2 (2-bit), 4 (4-bit)
        uint4 rows[4][kRowU4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int u = 0; u < kRowU4; ++u)
                rows[m][u] = __ldg(reinterpret_cast<const uint4*>(kc + (lane + 32 * m) * (16 * KB)) + u);

        // per-tile query factors: q''_j = q'_j S1_j g 2^-shift(j), paired as the codes are
        float cpart[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) cpart[h] = 0.f;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            const int p = lane + 32 * pp;
            int ja, jb;
            float pre;
            if (KB == 2) {
                const int w = p >> 3, i = p & 7;
                ja = 2 * w + 16 * i;
                jb = ja + 1;
                pre = ldexpf(1.f, -2 * i);
            } else {
                const int w = p >> 2, i = p & 3;
                ja = w + 16 * i;
                jb = ja + 64;
                pre = ldexpf(1.f, -4 * i);
            }
            const float sa = e4m3_value(kp[ja]) * gk, sb = e4m3_value(kp[jb]) * gk;
            const float za = fp16_value(reinterpret_cast<const uint16_t*>(kp + 256)[ja]) * gk;
            const float zb = fp16_value(reinterpret_cast<const uint16_t*>(kp + 256)[jb]) * gk;
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float qa = qr[h * kTile + ja], qb = qr[h * kTile + jb];
                q2[p * GH + h] = make_float2(qa * sa * pre, qb * sb * pre);
                cpart[h] = fmaf(qa, za, fmaf(qb, zb, cpart[h]));
            }
        }
        float cz_k[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) cz_k[h] = warp_sum(cpart[h]);
        __syncwarp();

        // ---- scores for tokens lane + 32 m ----
        float2 acc[4][GH];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int h = 0; h < GH; ++h) acc[m][h] = make_float2(0.f, 0.f);
        const float2 neg_magic = make_float2(-kMagic, -kMagic);
#pragma unroll
        for (int w = 0; w < 4 * KB; ++w) {
            uint32_t x[4], xh[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                x[m] = word_of(rows[m][w >> 2], w & 3);
                xh[m] = x[m] >> 16;
            }
            constexpr int kPairs = (KB == 2) ? 8 : 4;
#pragma unroll
            for (int i = 0; i < kPairs; ++i) {
                const uint32_t mask = (KB == 2) ? (3u << (2 * i)) : (15u << (4 * i));
                const int p = w * kPairs + i;
                float2 qv[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) qv[h] = q2[p * GH + h];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 f = fadd2(make_float2(magic_code(x[m], mask), magic_code(xh[m], mask)), neg_magic);
#pragma unroll
                    for (int h = 0; h < GH; ++h) acc[m][h] = ffma2(f, qv[h], acc[m][h]);
                }
            }
        }
        float s[4][GH];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float s2 = e4m3_value(kp[128 + lane + 32 * m]);
#pragma unroll
            for (int h = 0; h < GH; ++h) s[m][h] = (acc[m][h].x + acc[m][h].y + cz_k[h]) * s2;
        }

        // ---- online softmax (log2 domain), per head ----
        float alpha[GH], czv[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            float mx = fmaxf(fmaxf(s[0][h], s[1][h]), fmaxf(s[2][h], s[3][h]));
            mx = warp_max(mx);
            const float m_new = fmaxf(m_run[h], mx);
            alpha[h] = exp2f(m_run[h] - m_new);
            m_run[h] = m_new;
            float psum = 0.f, zsum = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int t = lane + 32 * m;
                const float p = exp2f(s[m][h] - m_new);
                psum += p;
                zsum = fmaf(p, fp16_value(reinterpret_cast<const uint16_t*>(vp + 256)[t]), zsum);
                const float w = p * e4m3_value(vp[t]);
                wb[t * GH + h] = make_float2(w, w);
            }
            l_lane[h] = fmaf(l_lane[h], alpha[h], psum);
            czv[h] = warp_sum(zsum);
        }
        __syncwarp();

        // ---- V: lane (lw, ts) accumulates channels lw + 16 i over tokens ts + 2 n ----
        float2 a2[GH][4];
#pragma unroll
        for (int h = 0; h < GH; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) a2[h][i] = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int n0 = 0; n0 < 64; n0 += 8) {
            uint32_t xv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = ts + 2 * (n0 + u);
                xv[u] = (VB == 2) ? (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(vc + t * 32) + lw)
                                  : __ldg(reinterpret_cast<const uint32_t*>(vc + t * 64) + lw);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = ts + 2 * (n0 + u);
                float2 wv[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) wv[h] = wb[t * GH + h];
                const uint32_t xhi = xv[u] >> 16;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 f;
                    if (VB == 2)
                        f = make_float2(magic_code(xv[u], 3u << (2 * i)), magic_code(xv[u], 3u << (2 * i + 8)));
                    else
                        f = make_float2(magic_code(xv[u], 15u << (4 * i)), magic_code(xhi, 15u << (4 * i)));
                    f = fadd2(f, neg_magic);
#pragma unroll
                    for (int h = 0; h < GH; ++h) a2[h][i] = ffma2(f, wv[h], a2[h][i]);
                }
            }
        }
        // fold 2^-shift, the zero-point term (once per channel: ts == 0 lanes) and g * s2_j
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ja = lw + 16 * i, jb = ja + 64;
            const float2 sc = make_float2(gv * e4m3_value(vp[128 + ja]), gv * e4m3_value(vp[128 + jb]));
            const float2 pre = (VB == 2) ? make_float2(ldexpf(1.f, -2 * i), ldexpf(1.f, -2 * i - 8))
                                         : make_float2(ldexpf(1.f, -4 * i), ldexpf(1.f, -4 * i));
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float cz = ts == 0 ? czv[h] : 0.f;
                const float2 v = ffma2(a2[h][i], pre, make_float2(cz, cz));
                o2[h][i] = ffma2(o2[h][i], make_float2(alpha[h], alpha[h]), fmul2(v, sc));
            }
        }
        __syncwarp();  // q2 / wb are rewritten by the next tile
    }

    // ---- merge the 8 warps of this CTA ----
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        const float lw_sum = warp_sum(l_lane[h]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o2[h][i].x += __shfl_xor_sync(0xffffffffu, o2[h][i].x, 16);
            o2[h][i].y += __shfl_xor_sync(0xffffffffu, o2[h][i].y, 16);
        }
        if (ts == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                os[(warp * GH + h) * kTile + lw + 16 * i] = o2[h][i].x;
                os[(warp * GH + h) * kTile + lw + 16 * i + 64] = o2[h][i].y;
            }
        }
        if (lane == 0) {
            ms[warp * GH + h] = m_run[h];
            ls[warp * GH + h] = lw_sum;
        }
    }
    __syncthreads();
    for (int e = tid; e < GH * kTile; e += kThreads) {
        const int h = e >> 7, j = e & 127;
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mmax = fmaxf(mmax, ms[w * GH + h]);
        float o = 0.f, l = 0.f;
        if (mmax != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(ms[w * GH + h] - mmax);
                o = fmaf(os[(w * GH + h) * kTile + j], f, o);
                l = fmaf(ls[w * GH + h], f, l);
            }
        }
        float* dst = a.ws + (((size_t)b * a.Hq + hq0 + h) * a.splits + split) * kWsStride;
        dst[4 + j] = o;
        if (j == 0) {
            dst[0] = mmax;
            dst[1] = l;
        }
    }
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
    return (size_t)GH * kTile * 4 + (size_t)kWarps * 64 * GH * 8 + (size_t)kWarps * kTile * GH * 8 +
           (size_t)kWarps * GH * 8 + (size_t)kWarps * GH * kTile * 4;
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
    return run_split<KB, VB, 4>(a, grid, stream);
}

}  // namespace

DecodePlan plan_decode(int B, int Hq, int /*Hkv*/, int max_tiles) {
    DecodePlan p;
    p.tiles_per_split = kTilesPerSplit;
    p.splits = max_tiles <= 0 ? 1 : (max_tiles + kTilesPerSplit - 1) / kTilesPerSplit;
    p.workspace_bytes = (size_t)B * Hq * p.splits * kWsStride * sizeof(float);
    return p;
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
    const int gh = group >= 4 ? 4 : group;
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
