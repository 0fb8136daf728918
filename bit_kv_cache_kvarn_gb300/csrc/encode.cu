// KVarN tile encoder: Hadamard rotation -> dual-axis variance normalisation -> scale split ->
// round-to-nearest -> bit packing, one 128x128 bf16 tile at a time per CTA.
//
// Method: KVarN (arXiv:2606.03458) as summarised on paperlayer.ai ("3 Methods": channel-wise
// Hadamard rotation and online variance scaling across both the channel and the token
// dimension; "D Experimental details": 2-bit codes, two FP8 scales and one FP16 zero-point per
// 128-element group) and agihunt.info (pipeline: rotate, then Sinkhorn-Knopp style alternating
// token/channel variance normalisation, then RTN; normalisation factors absorbed into the
// group scale).
//
// Design (GB300): persistent grid, two CTAs per SM, so that one tile's barriers and dependent
// chains overlap the other's work; the bf16 tile (32 KB, contiguous) arrives by a 1-D TMA bulk copy,
// and the next tile's copy starts as soon as the first rotation pass has consumed the current one.
// The rotation is two register passes around one shared-memory transpose
// (H_128 = (H_8 x I_16)(I_8 x H_16)).  Each thread then owns 8 tokens x 8 channels of the rotated
// tile Y (64 registers, channel pairs packed as float2): every statistics update of the Sinkhorn
// iteration is p = Y a (FMUL2), sum += p (FADD2), sum of squares += p p (FFMA2) over two elements;
// token sums reduce over 16 lanes by shuffles, channel sums over the two half-warps by a shuffle
// and over the 8 warps through shared memory.
#include <climits>
#include <type_traits>

#include "kvarn_common.cuh"
#include "kvarn_internal.h"

namespace kvarn {

// Set by the encoder when a TMA copy never completes (bounded wait); read by kvarn_device_error.
__device__ unsigned int g_encode_error = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;

constexpr int kPadded = kTile + kTile / 16;
__host__ __device__ constexpr int pad(int i) { return i + (i >> 4); }

struct EncodeSmem {
    __nv_bfloat16 xs[kTile * kTile];       // TMA destination (32 KB)
    union {
        float ys[kTile * kYStride];        // FWHT staging (72 KB), dead after the second pass
        struct {
            float2 red[kWarps][4][32];     // cross-warp partial sums (8 KB)
            float cmean[kTile];            // channel means: the shift of a second channel pass
            alignas(16) uint32_t codes[kTile * 16];  // packed rows (up to 8 KB)
        } late;
    } u;
    float cinv[kTile];                     // inverse channel factor 1 / c
    // per-group and per-other-axis arrays, indexed through pad(): a half-warp reads the 8 tokens
    // tg + 16 k of its lanes' slots, which pad() spreads over 8 banks
    float logf_[kPadded];                  // log of the other-axis factor
    float grp_min[kPadded];
    float grp_scale[kPadded];
    float grp_z[kPadded];                  // zero-point (value of the FP16 code)
    float grp_inv_s1[kPadded];             // 1 / S1 (0 where S1 = 0)
    float grp_s1[kPadded];                 // S1
    float oth_inv_s2[kPadded];             // 1 / s2 along the other axis
    float bred[kWarps];                    // per-warp partial sums of the log factors
    float2 bmax[kWarps];                   // per-warp partial maxima of (S, |m|) over the groups
    alignas(16) uint8_t params[KVARN_PARAM_BYTES];
    alignas(8) uint64_t bar;
};

// Element (token slot k, channel h + 16 i) of a thread's rotated tile held as channel pairs.
__device__ __forceinline__ float& yel(float2 (&y)[8][4], int k, int i) {
    return (i & 1) ? y[k][i >> 1].y : y[k][i >> 1].x;
}

// Power-of-two tile factor: largest S/g in (128, 256] unless |m|/g would pass 32768.
__device__ __forceinline__ float tile_factor(float s_max, float m_max) {
    int e = INT_MIN;
    if (s_max > 0.f) e = ceil_log2(s_max) - 8;
    if (m_max > 0.f) e = max(e, ceil_log2(m_max) - 15);
    return e == INT_MIN ? 1.f : ldexpf(1.f, e);
}

// Thread coordinates within the tile: the thread owns channels h + 16 i of tokens tg + 16 (k ^ kown).
struct TileLanes {
    int tid, lane, warp, h, tsub, tg, kown;
    __device__ __forceinline__ TileLanes() {
        tid = threadIdx.x;
        lane = tid & 31;
        warp = tid >> 5;
        h = lane & 15;
        tsub = lane >> 4;
        tg = 2 * warp + tsub;
        kown = ((h >> 3) & 1) * 4 + ((h >> 2) & 1) * 2 + ((h >> 1) & 1);
    }
};

// Stage 1 of a tile, the same for K and V: the tile in sm.xs (already arrived) is rotated into y
// and normalised; on return the thread holds Y in y, the inverse token factor of its token kown in
// b_own, and the inverse channel factors are in sm.cinv.  next: the tile this CTA encodes after it
// (its copy starts once sm.xs is consumed), or null.
__device__ __forceinline__ void rotate_normalise(EncodeSmem& sm, const TileLanes& L, const __nv_bfloat16* next,
                                                 float2 (&y)[8][4], float& b_out, int iters, int rotate,
                                                 int normalize) {
    constexpr uint32_t kTileBytes = kTile * kTile * 2;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int h = lane & 15;                 // channel lane: channels h + 16 i
    const int tsub = lane >> 4;
    const int tg = 2 * warp + tsub;          // token group: tokens tg + 16 k
    const __nv_bfloat16* xs = sm.xs;

    // ---- rotation pass 1: H_16 over channel bits 0..3, 16 contiguous channels per item ----
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + kThreads * it;
        const int t = idx >> 3, c = idx & 7;
        float2 f[8];  // channels 16 c + 2 m, 16 c + 2 m + 1 in f[m]
        {
            // the two 16-byte halves are read in a lane-dependent order (bank-conflict free)
            const int sw = (c >> 2) & 1;
            const uint4 ra = *reinterpret_cast<const uint4*>(xs + t * kTile + 16 * c + 8 * sw);
            const uint4 rb = *reinterpret_cast<const uint4*>(xs + t * kTile + 16 * c + 8 * (sw ^ 1));
            const uint4 r0 = sw ? rb : ra, r1 = sw ? ra : rb;
            const __nv_bfloat162* p0 = reinterpret_cast<const __nv_bfloat162*>(&r0);
            const __nv_bfloat162* p1 = reinterpret_cast<const __nv_bfloat162*>(&r1);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                f[m] = __bfloat1622float2(p0[m]);
                f[4 + m] = __bfloat1622float2(p1[m]);
            }
        }
        if (rotate) fwht_pairs<8>(f);
        float* dst = sm.u.ys + t * kYStride + 16 * c;
        {
            // 16-byte chunk q (channels 16 c + 4 q .. + 3) goes to position q ^ ((c >> 1) & 3) of the
            // row's 16-channel group: the XOR spreads one store instruction's lanes over all banks
            const int swz = (c >> 1) & 3;
            *reinterpret_cast<float4*>(dst + 4 * (0 ^ swz)) = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
            *reinterpret_cast<float4*>(dst + 4 * (1 ^ swz)) = make_float4(f[2].x, f[2].y, f[3].x, f[3].y);
            *reinterpret_cast<float4*>(dst + 4 * (2 ^ swz)) = make_float4(f[4].x, f[4].y, f[5].x, f[5].y);
            *reinterpret_cast<float4*>(dst + 4 * (3 ^ swz)) = make_float4(f[6].x, f[6].y, f[7].x, f[7].y);
        }
    }
    __syncthreads();
    // the bf16 slot is free again: prefetch this CTA's next tile into it
    if (tid == 0 && next != nullptr) {
        fence_proxy_async();
        mbar_expect_tx(&sm.bar, kTileBytes);
        bulk_g2s(sm.xs, next, kTileBytes, &sm.bar);
    }

    // ---- rotation pass 2: H_8 over channel bits 4..6; thread keeps Y ----
    // Register slot k of a thread holds token tg + 16 (k ^ kown), kown = channel-lane bits 3..1
    // as a 3-bit number: the partner lanes of the token reductions (h ^ 8, h ^ 4, h ^ 2) then
    // hold each other's tokens in complementary slots, so every lane keeps and sends the same
    // slots and no per-lane selection is needed; after the reduction lane h owns token kown.
    const int kown = L.kown;
    // y[k][m]: token slot k, channels h + 16 (2 m) (.x) and h + 16 (2 m + 1) (.y).  Channel 16 i + h
    // sits at 16 i + 4 (((h >> 2) & 3) ^ ((i >> 1) & 3)) + (h & 3) of its row (the swizzle of pass 1):
    // for i = 2 q and 2 q + 1 the offset within the 16-channel group is off[q]
    int off[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) off[q] = 4 * (((h >> 2) & 3) ^ q) + (h & 3);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int t = tg + 16 * (k ^ kown);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            y[k][q] = make_float2(sm.u.ys[t * kYStride + 32 * q + off[q]], sm.u.ys[t * kYStride + 32 * q + 16 + off[q]]);
        if (rotate) {
            fwht_pairs<4>(y[k]);
#pragma unroll
            for (int q = 0; q < 4; ++q) y[k][q] = fmul2(y[k][q], make_float2(kInvSqrt128, kInvSqrt128));
        }
    }
    // the staging area is reused for the reductions and the packed rows below
    __syncthreads();

    // ---- dual-axis variance normalisation ----
    // token step:   r_t = std_j(Y_tj / c_j)   (lane owns token kown of its 8 for the update)
    // channel step: c_j = std_t(Y_tj / r_t)
    // The factors are kept as their inverses b = 1/r, a = 1/c (one rsqrt each).
    // Each step sums p and p^2 (p = Y a, resp. Y b) and takes var = E[p^2] - E[p]^2.  In fp32 that
    // loses ~log2(ms / var) bits to cancellation when a row or column is dominated by its mean (K
    // with a large per-channel bias, V with a per-token offset after the rotation moves it into one
    // channel); so a step in which some row (column) has var < ms / 8 is summed again over
    // d = p - mean, with the mean just found as the shift: E[d^2] - E[d]^2 has no cancellation.
    // Ordinary tiles never take that second pass (the first pass alone is exact to ~1e-7 there).
    constexpr float kRedo = 0.125f;
    float b_own = 1.f;
    float2 a2[4];  // (a, a) of channels h + 16 (2 m), h + 16 (2 m + 1)
#pragma unroll
    for (int m = 0; m < 4; ++m) a2[m] = make_float2(1.f, 1.f);
    if (tid < kTile) sm.cinv[tid] = 1.f;
    // lane holding the statistics of this thread's token slot k (k ^ kown is that lane's kown)
    auto slot_src = [&](int k) {
        const int kt = k ^ kown;
        return (lane & 16) | (((kt >> 2) & 1) << 3) | (((kt >> 1) & 1) << 2) | ((kt & 1) << 1);
    };
    // token step sums (sum d, sum d^2), d = Y a + sh, over the 128 channels of this lane's token
    // kown: thread partials, then a transposing reduction over the 16 channel lanes
    auto token_sums = [&](auto shifted, const float2 (&sh)[8]) -> float2 {
        float2 acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float2 p = decltype(shifted)::value ? ffma2(y[k][0], a2[0], sh[k]) : fmul2(y[k][0], a2[0]);
            float2 s1 = p, s2 = fmul2(p, p);
#pragma unroll
            for (int m = 1; m < 4; ++m) {
                p = decltype(shifted)::value ? ffma2(y[k][m], a2[m], sh[k]) : fmul2(y[k][m], a2[m]);
                s1 = fadd2(s1, p);
                s2 = ffma2(p, p, s2);
            }
            acc[k] = make_float2(s1.x + s1.y, s2.x + s2.y);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 send = acc[q + 4];
            acc[q] = fadd2(acc[q], make_float2(__shfl_xor_sync(0xffffffffu, send.x, 8),
                                               __shfl_xor_sync(0xffffffffu, send.y, 8)));
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float2 send = acc[q + 2];
            acc[q] = fadd2(acc[q], make_float2(__shfl_xor_sync(0xffffffffu, send.x, 4),
                                               __shfl_xor_sync(0xffffffffu, send.y, 4)));
        }
        float2 keep = fadd2(acc[0], make_float2(__shfl_xor_sync(0xffffffffu, acc[1].x, 2),
                                                __shfl_xor_sync(0xffffffffu, acc[1].y, 2)));
        return fadd2(keep, make_float2(__shfl_xor_sync(0xffffffffu, keep.x, 1),
                                       __shfl_xor_sync(0xffffffffu, keep.y, 1)));
    };
    // channel step partial sums (sum d, sum d^2), d = Y b + csh, of this thread's 8 tokens for its
    // 8 channels, combined over the half-warp pair into the cross-warp scratch
    float2 bb[8];
    auto channel_sums = [&](auto shifted, const float2 (&csh)[4]) {
        float2 acc[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float2 p = decltype(shifted)::value ? ffma2(y[0][m], bb[0], csh[m]) : fmul2(y[0][m], bb[0]);
            float2 s1 = p, s2 = fmul2(p, p);
#pragma unroll
            for (int k = 1; k < 8; ++k) {
                p = decltype(shifted)::value ? ffma2(y[k][m], bb[k], csh[m]) : fmul2(y[k][m], bb[k]);
                s1 = fadd2(s1, p);
                s2 = ffma2(p, p, s2);
            }
            acc[2 * m] = make_float2(s1.x, s2.x);
            acc[2 * m + 1] = make_float2(s1.y, s2.y);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float2 send = tsub ? acc[q] : acc[q + 4];
            float2 keep = tsub ? acc[q + 4] : acc[q];
            keep = fadd2(keep, make_float2(__shfl_xor_sync(0xffffffffu, send.x, 16),
                                           __shfl_xor_sync(0xffffffffu, send.y, 16)));
            sm.u.late.red[warp][q][lane] = keep;  // channel h + 16 (q + 4 tsub)
        }
    };
    // channel tid's total over the 8 warps (threads 0..127)
    auto channel_total = [&]() -> float2 {
        const int hj = tid & 15, ij = tid >> 4;
        const int src_lane = ((ij >> 2) << 4) | hj, q = ij & 3;
        float2 s = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s = fadd2(s, sm.u.late.red[w][q][src_lane]);
        return s;
    };
    const float2 no_shift8[8] = {};
    const float2 no_shift4[4] = {};
    const int n_it = normalize ? iters : 0;
    for (int itn = 0; itn < n_it; ++itn) {
        {
            const float2 t1 = token_sums(std::false_type(), no_shift8);
            const float mean = t1.x * (1.f / kTile);
            const float ms = t1.y * (1.f / kTile);
            const float var = ms - mean * mean;
            // the factors of the first pass go out at once; the warp vote on a mean-dominated row
            // comes after them, off the path from the sums to the channel step
            float b_new = var > kDegenerateRel * ms ? rsqrtf(var) : b_own;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float b = __shfl_sync(0xffffffffu, b_new, slot_src(k));
                bb[k] = make_float2(b, b);
            }
            if (__any_sync(0xffffffffu, var < kRedo * ms)) {  // warp-uniform, rare
                float2 sh[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float mk = __shfl_sync(0xffffffffu, mean, slot_src(k));
                    sh[k] = make_float2(-mk, -mk);
                }
                const float2 t2 = token_sums(std::true_type(), sh);
                const float dm = t2.x * (1.f / kTile);
                const float var2 = t2.y * (1.f / kTile) - dm * dm;
                b_new = var2 > kDegenerateRel * ms ? rsqrtf(var2) : b_own;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float b = __shfl_sync(0xffffffffu, b_new, slot_src(k));
                    bb[k] = make_float2(b, b);
                }
            }
            b_own = b_new;
        }

        channel_sums(std::false_type(), no_shift4);
        __syncthreads();
        float cms = 0.f, cmean = 0.f;
        bool redo = false;
        if (tid < kTile) {
            const float2 t = channel_total();
            cmean = t.x * (1.f / kTile);
            cms = t.y * (1.f / kTile);
            const float var = cms - cmean * cmean;
            redo = var < kRedo * cms;
            if (!redo && var > kDegenerateRel * cms) sm.cinv[tid] = rsqrtf(var);
        }
        if (__syncthreads_or(redo)) {  // block-uniform, rare: some column is dominated by its mean
            if (tid < kTile) sm.u.late.cmean[tid] = cmean;  // the shift of the second pass
            __syncthreads();
            float2 csh[4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
                csh[m] = make_float2(-sm.u.late.cmean[h + 32 * m], -sm.u.late.cmean[h + 32 * m + 16]);
            channel_sums(std::true_type(), csh);
            __syncthreads();
            if (tid < kTile) {
                const float2 t = channel_total();
                const float dm = t.x * (1.f / kTile);
                const float var = t.y * (1.f / kTile) - dm * dm;
                if (var > kDegenerateRel * cms) sm.cinv[tid] = rsqrtf(var);
            }
            __syncthreads();
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) a2[m] = make_float2(sm.cinv[h + 32 * m], sm.cinv[h + 32 * m + 16]);
    }
    b_out = b_own;
}

// Stage 2 of a tile, by kind: the scale split (s2, g, S1, Z), round-to-nearest codes, packing and the
// stores to output slot otile.  y, b_own and sm.cinv as rotate_normalise leaves them.
template <int BITS, int KIND>
__device__ __forceinline__ void split_quantise_store(EncodeSmem& sm, const TileLanes& L, float2 (&y)[8][4],
                                                     float b_own, uint8_t* __restrict__ codes_out,
                                                     uint8_t* __restrict__ params_out,
                                                     float* __restrict__ scale_out, int64_t otile, int rotate) {
    constexpr int kLevels = (1 << BITS) - 1;
    const int tid = L.tid, lane = L.lane, warp = L.warp, h = L.h, tsub = L.tsub, tg = L.tg, kown = L.kown;

    // ---- scale split: s2 along the other axis (geometric mean 1, E4M3, clamped) ----
    // K: other axis = token (factor r, one lane of each lane pair h, h ^ 1 holds token
    // tg + 16 kown); V: other axis = channel (factor c, channel tid for threads 0..127).  The log
    // factors are summed per warp on the way into shared memory, so one barrier serves both.
    float lf = 0.f;
    if (KIND == KVARN_KIND_K) {
        if ((h & 1) == 0) {
            lf = -logf(b_own);
            sm.logf_[pad(tg + 16 * kown)] = lf;
        }
    } else {
        if (tid < kTile) {
            lf = -logf(sm.cinv[tid]);
            sm.logf_[pad(tid)] = lf;
        }
    }
    {
        const float ws = warp_sum(lf);
        if (lane == 0) sm.bred[warp] = ws;
    }
    __syncthreads();
    float log_sum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) log_sum += sm.bred[w];
    const float mean_log = log_sum * (1.f / kTile);
    if (tid < kTile) {
        float s2 = e4m3_value(e4m3_rn(expf(sm.logf_[pad(tid)] - mean_log)));
        s2 = fminf(fmaxf(s2, 0.001953125f), 448.f);  // [2^-9, 448]
        sm.params[128 + tid] = e4m3_rn(s2);
        sm.oth_inv_s2[pad(tid)] = 1.f / s2;
    }
    __syncthreads();

    // W = Y / s2, then per-group min / max
    float gmin_own = 0.f, gmax_own = 0.f;  // V: this lane's token kown
    if (KIND == KVARN_KIND_K) {
        float2 mm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float inv = sm.oth_inv_s2[pad(tg + 16 * (k ^ kown))];
#pragma unroll
            for (int m = 0; m < 4; ++m) y[k][m] = fmul2(y[k][m], make_float2(inv, inv));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float lo = yel(y, 0, i), hi = lo;
#pragma unroll
            for (int k = 1; k < 8; ++k) {
                lo = fminf(lo, yel(y, k, i));
                hi = fmaxf(hi, yel(y, k, i));
            }
            mm[i] = make_float2(lo, hi);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float2 send = tsub ? mm[q] : mm[q + 4];
            float2 keep = tsub ? mm[q + 4] : mm[q];
            keep.x = fminf(keep.x, __shfl_xor_sync(0xffffffffu, send.x, 16));
            keep.y = fmaxf(keep.y, __shfl_xor_sync(0xffffffffu, send.y, 16));
            sm.u.late.red[warp][q][lane] = keep;
        }
        __syncthreads();
        if (tid < kTile) {
            const int j = tid, hj = j & 15, ij = j >> 4;
            const int src_lane = ((ij >> 2) << 4) | hj, q = ij & 3;
            float lo = sm.u.late.red[0][q][src_lane].x, hi = sm.u.late.red[0][q][src_lane].y;
#pragma unroll
            for (int w = 1; w < kWarps; ++w) {
                lo = fminf(lo, sm.u.late.red[w][q][src_lane].x);
                hi = fmaxf(hi, sm.u.late.red[w][q][src_lane].y);
            }
            sm.grp_min[pad(j)] = lo;
            sm.grp_scale[pad(j)] = (hi - lo) / (float)kLevels;
            gmin_own = lo;
            gmax_own = hi;
        }
    } else {
        float inv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) inv[i] = sm.oth_inv_s2[pad(h + 16 * i)];
        float2 mm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float lo = 0.f, hi = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) y[k][m] = fmul2(y[k][m], make_float2(inv[2 * m], inv[2 * m + 1]));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float w = yel(y, k, i);
                lo = i ? fminf(lo, w) : w;
                hi = i ? fmaxf(hi, w) : w;
            }
            mm[k] = make_float2(lo, hi);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 send = mm[q + 4];
            float2 keep = mm[q];
            keep.x = fminf(keep.x, __shfl_xor_sync(0xffffffffu, send.x, 8));
            keep.y = fmaxf(keep.y, __shfl_xor_sync(0xffffffffu, send.y, 8));
            mm[q] = keep;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float2 send = mm[q + 2];
            float2 keep = mm[q];
            keep.x = fminf(keep.x, __shfl_xor_sync(0xffffffffu, send.x, 4));
            keep.y = fmaxf(keep.y, __shfl_xor_sync(0xffffffffu, send.y, 4));
            mm[q] = keep;
        }
        {
            const float2 send = mm[1];
            float2 keep = mm[0];
            keep.x = fminf(keep.x, __shfl_xor_sync(0xffffffffu, send.x, 2));
            keep.y = fmaxf(keep.y, __shfl_xor_sync(0xffffffffu, send.y, 2));
            keep.x = fminf(keep.x, __shfl_xor_sync(0xffffffffu, keep.x, 1));
            keep.y = fmaxf(keep.y, __shfl_xor_sync(0xffffffffu, keep.y, 1));
            gmin_own = keep.x;
            gmax_own = keep.y;
        }
        if ((h & 1) == 0) {
            const int t = tg + 16 * kown;
            sm.grp_min[pad(t)] = gmin_own;
            sm.grp_scale[pad(t)] = (gmax_own - gmin_own) / (float)kLevels;
        }
    }
    // per-warp maxima of S and |m| over the groups this warp's threads wrote (K: threads 0..127,
    // V: the even lanes; every other thread contributes 0), read after the barrier below
    {
        const bool writer = (KIND == KVARN_KIND_K) ? tid < kTile : (h & 1) == 0;
        float ms = writer ? (gmax_own - gmin_own) / (float)kLevels : 0.f;
        float mm = writer ? fabsf(gmin_own) : 0.f;
        ms = warp_max(ms);
        mm = warp_max(mm);
        if (lane == 0) sm.bmax[warp] = make_float2(ms, mm);
    }
    __syncthreads();

    // ---- tile factor g, group scale S1 (E4M3, rounded up) and zero-point Z (FP16) ----
    float s_max = 0.f, m_max = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const float2 bm = sm.bmax[w];
        s_max = fmaxf(s_max, bm.x);
        m_max = fmaxf(m_max, bm.y);
    }
    const float g = tile_factor(s_max, m_max);
    const float inv_g = 1.f / g;  // exact: g is a power of two
    if (tid < kTile) {
        const uint8_t s1b = e4m3_up(sm.grp_scale[pad(tid)] * inv_g);
        const float s1 = e4m3_value(s1b);
        const __half zh = __float2half_rn(sm.grp_min[pad(tid)] * inv_g);
        sm.params[tid] = s1b;
        reinterpret_cast<__half*>(sm.params + 256)[tid] = zh;
        sm.grp_z[pad(tid)] = __half2float(zh);
        sm.grp_inv_s1[pad(tid)] = s1 > 0.f ? 1.f / s1 : 0.f;
        sm.grp_s1[pad(tid)] = s1;
    }
    __syncthreads();

    // ---- codes and packing ----
    // K rows are tokens: lane h of row t holds channels h + 16 i at bits BITS*i.
    // V rows are channels: lane tg of row j holds tokens tg + 16 k at bits BITS*k.
    uint32_t packed[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) packed[q] = 0;
    {
        // group constants: K groups are this thread's 8 channels, V groups its 8 tokens
        float nz[8], is1[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int grp = (KIND == KVARN_KIND_K) ? (h + 16 * m) : (tg + 16 * (m ^ kown));
            nz[m] = -sm.grp_z[pad(grp)];
            is1[m] = sm.grp_inv_s1[pad(grp)];
        }
        // Adding 1.5 * 2^23 rounds a value in [0, 2^22) to an integer (half to even) held in the
        // low mantissa bits.  Exact half-way points occur in practice only without the rotation
        // (bf16 inputs on a coarse grid); there a product with the rounded reciprocal can land
        // on the wrong side, so near a half-way point the code is redone with a correctly
        // rounded division.  With the rotation the check is left out.
        constexpr float kRound = 12582912.f;
        // With the rotation: v = sat(d / (S1 (2^b - 1))) in [0, 1] (one saturating multiply does
        // both clamps) and r = v (2^b - 1) + kRound in one FFMA2, whose single rounding puts the
        // nearest integer (half to even) of v (2^b - 1) in r's low bits.  The two roundings of
        // 1 / (S1 (2^b - 1)) and of the product move u = (W / g - Z) / S1 by a few ulp, which
        // changes a code only within a few ulp of a half-way point.
        float is1l[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) is1l[m] = is1[m] * (1.f / (float)kLevels);
        auto quantise = [&](auto tie_check) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const int g0 = (KIND == KVARN_KIND_K) ? i : k, g1 = (KIND == KVARN_KIND_K) ? i + 1 : k;
                    const float2 d = ffma2(y[k][i >> 1], make_float2(inv_g, inv_g),
                                           make_float2(nz[g0], nz[g1]));
                    float2 rr;
                    if (!decltype(tie_check)::value) {
                        const float2 v = make_float2(mul_sat(d.x, is1l[g0]), mul_sat(d.y, is1l[g1]));
                        rr = ffma2(v, make_float2((float)kLevels, (float)kLevels), make_float2(kRound, kRound));
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int ii = i + e, ge = e ? g1 : g0;
                        float r = e ? rr.y : rr.x;
                        if (decltype(tie_check)::value) {
                            float v = fminf(fmaxf((e ? d.y : d.x) * is1[ge], 0.f), (float)kLevels);
                            r = v + kRound;
                            if (fabsf(v - (r - kRound)) > 0.4999f && is1[ge] > 0.f) {
                                const int grp = (KIND == KVARN_KIND_K) ? (h + 16 * ii) : (tg + 16 * (k ^ kown));
                                v = fminf(fmaxf(__fdiv_rn(e ? d.y : d.x, sm.grp_s1[pad(grp)]), 0.f), (float)kLevels);
                                r = v + kRound;
                            }
                        }
                        // r's bits are kRoundBits + code: add them shifted into place and take
                        // the eight shifted kRoundBits off each word once, below
                        const uint32_t rb = __float_as_uint(r);
                        if (KIND == KVARN_KIND_K)
                            packed[k] += rb << (BITS * ii);
                        else
                            packed[ii] += rb << (BITS * (k ^ kown));
                    }
                }
            }
        };
        if (rotate)
            quantise(std::integral_constant<bool, false>());
        else
            quantise(std::integral_constant<bool, true>());
        // every word received kRoundBits at the eight shifts BITS * n (the sums wrap modulo 2^32)
        constexpr uint32_t kRoundBits = 0x4B400000u;  // bits of kRound
        uint32_t offset = 0;
#pragma unroll
        for (int n = 0; n < 8; ++n) offset += kRoundBits << (BITS * n);
#pragma unroll
        for (int q = 0; q < 8; ++q) packed[q] -= offset;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int row = (KIND == KVARN_KIND_K) ? (tg + 16 * (q ^ kown)) : (h + 16 * q);
        const int lane16 = (KIND == KVARN_KIND_K) ? h : tg;
        if (BITS == 2)
            reinterpret_cast<uint16_t*>(sm.u.late.codes)[row * 16 + lane16] = (uint16_t)packed[q];
        else
            sm.u.late.codes[row * 16 + lane16] = packed[q];
    }
    __syncthreads();

    // ---- write out: codes (16-byte stores), params, tile factor ----
    {
        constexpr int kCodeBytes = kTile * 16 * BITS;
        uint4* dst = reinterpret_cast<uint4*>(codes_out + otile * kCodeBytes);
        const uint4* src = reinterpret_cast<const uint4*>(sm.u.late.codes);
#pragma unroll
        for (int v = tid; v < kCodeBytes / 16; v += kThreads) dst[v] = src[v];
        if (tid < KVARN_PARAM_BYTES / 16)
            reinterpret_cast<uint4*>(params_out + otile * KVARN_PARAM_BYTES)[tid] =
                reinterpret_cast<const uint4*>(sm.params)[tid];
        if (tid == 0) scale_out[otile] = g;
    }
    // no barrier here: the next tile starts with the copy wait's barrier, before anything
    // overwrites the packed rows or the parameters
}

// Initialises the copy barrier and starts the copy of the CTA's first tile (if any).
__device__ __forceinline__ void encode_prologue(EncodeSmem& sm, const __nv_bfloat16* first) {
    if (threadIdx.x == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && first != nullptr) {
        mbar_expect_tx(&sm.bar, kTile * kTile * 2);
        bulk_g2s(sm.xs, first, kTile * kTile * 2, &sm.bar);
    }
}

// Waits for the CTA's local-th tile.  False (uniform over the CTA) when its copy never arrived:
// the error word is then set and the copy has been waited for (bounded).
__device__ __forceinline__ bool encode_wait(EncodeSmem& sm, int local) {
    const bool ok = mbar_wait(&sm.bar, local & 1, &g_encode_error);
    if (__syncthreads_and(ok)) return true;
    if (threadIdx.x == 0) mbar_drain(&sm.bar, local & 1);
    return false;
}

// Tiles of one kind.
template <int BITS, int KIND>
__global__ void __launch_bounds__(kThreads, 2)
encode_kernel(const __nv_bfloat16* __restrict__ x, int64_t n_tiles, uint8_t* __restrict__ codes_out,
              uint8_t* __restrict__ params_out, float* __restrict__ scale_out, int iters,
              int rotate, int normalize) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    EncodeSmem& sm = *reinterpret_cast<EncodeSmem*>(smem_raw);
    encode_prologue(sm, blockIdx.x < n_tiles ? x + (int64_t)blockIdx.x * kTile * kTile : nullptr);
    const TileLanes L;
    int local = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
        if (!encode_wait(sm, local)) break;
        const int64_t nt = tile + gridDim.x;
        float2 y[8][4];
        float b_own;
        rotate_normalise(sm, L, nt < n_tiles ? x + nt * kTile * kTile : nullptr, y, b_own, iters, rotate, normalize);
        split_quantise_store<BITS, KIND>(sm, L, y, b_own, codes_out, params_out, scale_out, tile, rotate);
    }
}

// The K and V tiles of one call in one grid: virtual tile i < n_k is K tile i, else V tile i - n_k.
// With dest, input tile u (of either kind) goes to output slot dest[u] and is skipped when dest[u]
// is negative (the append path stages one slot per (sequence, kv head), most of them unused).
struct EncodeKV {
    const __nv_bfloat16* kx;
    const __nv_bfloat16* vx;
    int64_t n_k, n_v;
    uint8_t* k_codes;
    uint8_t* k_params;
    float* k_scale;
    uint8_t* v_codes;
    uint8_t* v_params;
    float* v_scale;
    const int32_t* dest;  // [n_k] output slots shared by K and V (n_k == n_v), or null
    int iters, rotate, normalize;
};

__device__ __forceinline__ const __nv_bfloat16* kv_src(const EncodeKV& a, int64_t i) {
    return i < a.n_k ? a.kx + i * kTile * kTile : a.vx + (i - a.n_k) * kTile * kTile;
}

// The first virtual tile at or after i, stepping by the grid, that is to be encoded (n if none).
__device__ __forceinline__ int64_t kv_next(const EncodeKV& a, int64_t i, int64_t n) {
    if (a.dest == nullptr) return i < n ? i : n;
    for (; i < n; i += gridDim.x)
        if (a.dest[i < a.n_k ? i : i - a.n_k] >= 0) return i;
    return n;
}

template <int KB, int VB>
__global__ void __launch_bounds__(kThreads, 2) encode_kv_kernel(EncodeKV a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    EncodeSmem& sm = *reinterpret_cast<EncodeSmem*>(smem_raw);
    const int64_t n = a.n_k + a.n_v;
    int64_t tile = kv_next(a, blockIdx.x, n);
    encode_prologue(sm, tile < n ? kv_src(a, tile) : nullptr);
    const TileLanes L;
    for (int local = 0; tile < n; ++local) {
        if (!encode_wait(sm, local)) break;
        const int64_t nt = kv_next(a, tile + gridDim.x, n);
        const __nv_bfloat16* next = nt < n ? kv_src(a, nt) : nullptr;
        const int64_t u = tile < a.n_k ? tile : tile - a.n_k;
        const int64_t slot = a.dest != nullptr ? (int64_t)a.dest[u] : u;
        // the rotation and the normalisation are the same for both kinds: their code appears once
        float2 y[8][4];
        float b_own;
        rotate_normalise(sm, L, next, y, b_own, a.iters, a.rotate, a.normalize);
        if (tile < a.n_k)
            split_quantise_store<KB, KVARN_KIND_K>(sm, L, y, b_own, a.k_codes, a.k_params, a.k_scale, slot, a.rotate);
        else
            split_quantise_store<VB, KVARN_KIND_V>(sm, L, y, b_own, a.v_codes, a.v_params, a.v_scale, slot, a.rotate);
        tile = nt;
    }
}

}  // namespace

size_t encode_smem_bytes() { return sizeof(EncodeSmem); }

cudaError_t read_and_clear_device_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_encode_error, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_encode_error, &zero, sizeof(zero));
    *out = v;
    return e;
}

cudaError_t launch_encode(int bits, int kind, const void* x, int64_t n_tiles, void* codes,
                          void* params, float* tile_scale, int iters, int rotate, int normalize,
                          cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t err = current_device(&dev, &sms);
    if (err != cudaSuccess) return err;
    const int grid = (int)(n_tiles < 2 * sms ? n_tiles : 2 * sms);  // two CTAs per SM
    const size_t smem = sizeof(EncodeSmem);
    auto run = [&](auto kern) -> cudaError_t {
        cudaError_t e = set_smem_limit_once(kern, (int)smem, true, dev);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, stream>>>(static_cast<const __nv_bfloat16*>(x), n_tiles,
                                               static_cast<uint8_t*>(codes),
                                               static_cast<uint8_t*>(params), tile_scale, iters,
                                               rotate, normalize);
        return cudaGetLastError();
    };
    if (bits == 2 && kind == KVARN_KIND_K) return run(encode_kernel<2, KVARN_KIND_K>);
    if (bits == 2 && kind == KVARN_KIND_V) return run(encode_kernel<2, KVARN_KIND_V>);
    if (bits == 4 && kind == KVARN_KIND_K) return run(encode_kernel<4, KVARN_KIND_K>);
    return run(encode_kernel<4, KVARN_KIND_V>);
}

// K then V blocks of one call in one grid of two CTAs per SM: the K and V tiles share the waves,
// so the last wave of the K tiles no longer leaves SMs idle before the V tiles start.
cudaError_t launch_encode_kv(int k_bits, int v_bits, const void* k_x, int64_t n_k, void* k_codes,
                             void* k_params, float* k_scale, const void* v_x, int64_t n_v, void* v_codes,
                             void* v_params, float* v_scale, int iters, int rotate, int normalize,
                             cudaStream_t stream, const int32_t* dest) {
    if (n_k + n_v == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t err = current_device(&dev, &sms);
    if (err != cudaSuccess) return err;
    const int64_t n = n_k + n_v;
    const int grid = (int)(n < 2 * sms ? n : 2 * sms);
    const size_t smem = sizeof(EncodeSmem);
    EncodeKV a;
    a.kx = static_cast<const __nv_bfloat16*>(k_x);
    a.vx = static_cast<const __nv_bfloat16*>(v_x);
    a.n_k = n_k;
    a.n_v = n_v;
    a.k_codes = static_cast<uint8_t*>(k_codes);
    a.k_params = static_cast<uint8_t*>(k_params);
    a.k_scale = k_scale;
    a.v_codes = static_cast<uint8_t*>(v_codes);
    a.v_params = static_cast<uint8_t*>(v_params);
    a.v_scale = v_scale;
    a.dest = dest;
    a.iters = iters;
    a.rotate = rotate;
    a.normalize = normalize;
    auto run = [&](auto kern) -> cudaError_t {
        cudaError_t e = set_smem_limit_once(kern, (int)smem, true, dev);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, stream>>>(a);
        return cudaGetLastError();
    };
    if (k_bits == 2 && v_bits == 2) return run(encode_kv_kernel<2, 2>);
    if (k_bits == 4 && v_bits == 2) return run(encode_kv_kernel<4, 2>);
    if (k_bits == 2 && v_bits == 4) return run(encode_kv_kernel<2, 4>);
    return run(encode_kv_kernel<4, 4>);
}

}  // namespace kvarn
