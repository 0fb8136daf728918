// Decode attention over the packed KVarN cache: one query per sequence, grouped-query heads.
//
// Method: the quantised cache is restored at attention read time (dimensionstp.github.io review,
// "4-2 Training strategy"); the query is rotated by the same head-wise Hadamard after RoPE, so keys
// stay in the rotated basis (paperlayer.ai summary, "A Hadamard Transform Arrangement"); the
// second scale s2 is fused into the dequantisation (paperlayer.ai, "3 Methods" and "I KVarN
// Dequantization Overhead").  Here both scales are folded out of the inner products:
//   K (groups = channels): s_t = s2_t g (sum_j q'_j S1_j code_tj + sum_j q'_j Z_j)
//   V (groups = tokens):   o_j += g s2_j (sum_t p_t S1_t code_tj + sum_t p_t Z_t)
//
// Split kernel (5th-generation tensor cores).  The full tiles of all (sequence, kv head) units form
// one stream that every CTA cuts, from the sequence lengths, into equal contiguous pieces of >= P
// tiles (P = 16, smaller for small calls); a CTA holds two warpgroup "workers", each processing its piece persistently.  Per tile,
// lane 0 of each of the worker's four warps brings one of the tile's four blocks (K codes, V codes,
// K parameters, V parameters) into a shared-memory ring with a 1-D TMA bulk copy (mbarrier-tracked);
// then thread r of the worker:
//   * masks K row r (token r) into fp16 subnormals (code * 2^shift * 2^-24, exact; no conversion)
//     and stores them in TMEM as the MMA's A operand;
//   * writes q'' = q' S1 2^-shift for channel r as fp16 hi/lo pieces into the B operand (shared
//     memory, N-contiguous) -- up to 8 heads x 2 pieces = N 16 -- and its share of sum_j q'_j Z_j;
//   * after 8 tcgen05.mma, owns token r's scores, runs the online softmax (log2 domain), writes
//     p S1 for token r as the next B and its share of sum_t p_t Z_t, masks V row r (channel r)
//     into A, and after 8 more MMAs owns channel r of sum_t p_t v_t.
// The number of MMA instructions per issuing warp, not their FLOPs, sets the tensor-core cost
// here: one warp's MMAs complete one after another (~130 cycles each for M=128, K=16, whatever N
// and whether or not they share an accumulator), while MMAs issued by different warps overlap.
// So each of the worker's 4 warps issues 2 of the 8 K-steps into its own 16-column partial
// accumulator and the partials are summed on readout; the zero-point sums stay on the CUDA cores.
// Merge kernel: one 128-thread CTA per (sequence, query head) merges the partial slots by
// log-sum-exp, applies the inverse rotation, attends to the unquantised sink and tail tokens and
// normalises.  Two launches per call, both with programmatic dependent launch.
#include <math.h>

#include "kvarn_common.cuh"
#include "kvarn_internal.h"
#include "tcgen05.cuh"

namespace kvarn {

// Set when a bounded wait (TMA data or tensor-core completion) gives up; read by kvarn_device_error.
__device__ unsigned int g_decode_error = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kWorkers = 2;                 // warpgroups per CTA
// Piece granularity P (DecodeArgs::piece): every worker's piece of the tile stream has >= P tiles and
// a unit has one partial slot per P-tile block (+1, below).  P = 16 when the stream can fill the
// GPU's workers with 16-tile pieces; smaller calls halve it (down to 2) so that more workers share
// the tiles and the call's latency is not one worker walking 16 tiles.
constexpr int kMaxPiece = 16, kMinPieceTiles = 2;
constexpr long long kFillWorkers = 512;  // device-independent stand-in for the worker count
constexpr int kIdRing = 32;                // tile-id ring of a worker
constexpr int kIdBatch = 16;               // tile ids are fetched 16 at a time, one batch ahead
constexpr int kWsStride = 132;  // floats per (sequence, query head, split): m, l, pad, pad, o[128]
constexpr uint32_t kTmemCols = 256;         // worker w: A (64) and D (4 partials x 16) at 128 w
constexpr uint32_t kBBytes = 128 * 16 * 2;  // one B operand: K = 128 x N = 16 fp16, N-contiguous
constexpr uint32_t kBKStride = 256, kBNStride = 128;  // core-matrix strides of B along K and N
// Lazy maximum: keep the running max while no score exceeds it by more than kLazy (log2 units), so
// p <= 2^kLazy; with S1 <= 256, p S1 kWScale <= 2^15 fits fp16 while small terms stay normal.
constexpr float kLazy = 4.f;
constexpr float kWScale = 8.f;
constexpr float kTwo24 = 16777216.f;
// The lo piece of a B value is stored times 2^11 (it is at most half an fp16 ulp of the hi piece,
// so it stays below |x| and never overflows): unscaled it would be an fp16 subnormal for most
// values and carry only a few bits; its column's sum is multiplied back by 2^-11 on readout.
constexpr float kLoScale = 2048.f;

// A worker's piece of the tile stream.  The stream lists, sequence by sequence and unit by unit
// (unit = kv head x head block), the full tiles of each unit; a piece is a contiguous run of it.
struct Piece {
    int b, u, j;     // first tile: sequence, unit, tile within the unit
    long long len;   // number of tiles
};

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
    const __nv_bfloat16* k_sink;  // [B][Hkv][128][128] bf16, the first sink_len tokens (or null)
    const __nv_bfloat16* v_sink;
    int sink_len;                 // 0..128 FP16 sink tokens before the packed body
    const __nv_bfloat16* k_tail;
    const __nv_bfloat16* v_tail;
    float qscale;  // softmax scale * log2(e): scores are kept in the log2 domain
    int rotate;
    int full_tail;  // the tail holds the last 1..128 tokens (else L mod 128)
    int splits;     // partial slots per (sequence, query head) = splits + 1
    int piece;      // P: minimum piece length and tiles per partial slot block
    int B;
    int units;      // units per sequence: kv heads x head blocks
    int hblocks;    // head blocks per kv head
    float* ws;
    float* out;
};


__device__ __forceinline__ int clamp_len(int len, int max_tiles, int full_tail) {
    const int cap = max_tiles * kTile + (full_tail ? kTile : kTile - 1);
    return len < 0 ? 0 : (len > cap ? cap : len);
}

// Full tiles read from the pools for a (clamped) length: all complete blocks, or all but the
// most recent one when the tail keeps a full window.
__device__ __forceinline__ int n_full_tiles(int len, int full_tail) {
    return full_tail ? (len > 0 ? (len - 1) >> 7 : 0) : len >> 7;
}

// 2^x by the hardware approximation (ex2.approx.ftz: relative error within 2 ulp; results below
// 2^-126 flush to 0, i.e. weights 2^-126 under the running maximum).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory ring stage: K codes | V codes | K params | V params, one bulk copy each.
template <int KB, int VB>
struct Stage {
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = KB * 2048;
    static constexpr uint32_t kKP = kV + VB * 2048;
    static constexpr uint32_t kVP = kKP + 512;
    static constexpr uint32_t kBytes = kVP + 512;
    // ring depth: four stages at K2V2, three at mixed widths, two at K4V4 (2 CTAs per SM must fit)
    static constexpr int kCount = (KB + VB == 4) ? 4 : (KB + VB == 6 ? 3 : 2);
};

// Byte offset of the 8 consecutive B elements (rows n0..n0+7) at K index kk.
__device__ __forceinline__ uint32_t b_off(int n0, int kk) {
    return (uint32_t)((kk >> 3) * kBKStride + (n0 >> 3) * kBNStride + (kk & 7) * 16);
}

// Position of column c (0..127) of a packed row in the MMA K order, and the power of two
// (2^-shift) the B element carries to cancel the code's 2^shift.
template <int BITS>
__device__ __forceinline__ void k_slot(int c, int& kk, float& inv_pre) {
    const int h = c & 15, i = c >> 4;
    if (BITS == 2) {
        // code i of lane h -> TMEM column 8 i + (h >> 1), half h & 1: the K order is the column order
        kk = c;
        inv_pre = ldexpf(1.f, -2 * (i <= 4 ? i : i - 5));
    } else {
        // codes (ii, ii + 4) of lane h -> TMEM column 16 ii + h, halves 0 / 1
        const int ii = i & 3;
        kk = 2 * (16 * ii + h) + (i >> 2);
        inv_pre = ldexpf(1.f, -4 * (ii <= 1 ? ii : ii - 2));
    }
}

// Mask one packed row (BITS*4 words) into 64 fp16x2 TMEM columns, in the order k_slot describes.
// A code field left in place is the fp16 subnormal code * 2^shift * 2^-24 (exact).
template <int BITS>
__device__ __forceinline__ void unpack_row_to_tmem(const uint32_t (&x)[4 * BITS], uint32_t taddr) {
    constexpr int kWords = 4 * BITS;
    constexpr int kSh = BITS == 2 ? 10 : 8;
    uint32_t xs[kWords];
#pragma unroll
    for (int w = 0; w < kWords; ++w) xs[w] = x[w] >> kSh;
#pragma unroll
    for (int chunk = 0; chunk < 4; ++chunk) {
        uint32_t r[16];
        if (BITS == 2) {
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * chunk + ii;
                const uint32_t mask = i <= 4 ? (0x00030003u << (2 * i)) : (0x00030003u << (2 * (i - 5)));
#pragma unroll
                for (int w = 0; w < 8; ++w) r[8 * ii + w] = (i <= 4 ? x[w] : xs[w]) & mask;
            }
        } else {
            const int ii = chunk;
            const uint32_t mask = ii <= 1 ? (0x000F000Fu << (4 * ii)) : (0x000F000Fu << (4 * (ii - 2)));
#pragma unroll
            for (int w = 0; w < 16; ++w) r[w] = (ii <= 1 ? x[w] : xs[w]) & mask;
        }
        tc::st16(taddr + 16 * chunk, r);
    }
}

// Read this thread's packed row (BITS*16 bytes) from shared memory.  Rows are 32 (2-bit) or 64
// (4-bit) bytes apart, so a quarter-warp's 16-byte reads meet 2- or 4-way bank conflicts; taking
// them is cheaper than reading in a lane-dependent order and putting the words back in place.
template <int BITS>
__device__ __forceinline__ void load_row(const uint8_t* base, int r, uint32_t (&x)[4 * BITS]) {
    const uint4* p = reinterpret_cast<const uint4*>(base + r * 16 * BITS);
#pragma unroll
    for (int q = 0; q < BITS; ++q) {
        const uint4 u = p[q];
        x[4 * q] = u.x;
        x[4 * q + 1] = u.y;
        x[4 * q + 2] = u.z;
        x[4 * q + 3] = u.w;
    }
}

// hi/lo fp16 pieces of GH values (lo scaled by kLoScale), packed as B rows 2h (hi) and 2h+1 (lo);
// rows >= 2*GH stay zero.
template <int GH>
__device__ __forceinline__ void store_b(uint8_t* b, int kk, const float (&x)[GH]) {
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) w[q] = 0u;
    if constexpr (GH == 1) {
        const __half hi = __float2half_rn(x[0]);
        const __half lo = __float2half_rn((x[0] - __half2float(hi)) * kLoScale);
        const __half2 v = __halves2half2(hi, lo);
        w[0] = *reinterpret_cast<const uint32_t*>(&v);
    } else {
        // two values at a time: packed conversions and residuals, then (hi, lo) per value
#pragma unroll
        for (int h = 0; h < GH; h += 2) {
            const float2 xv = make_float2(x[h], x[h + 1]);
            const __half2 hi = __floats2half2_rn(xv.x, xv.y);
            const float2 r = fmul2(ffma2(__half22float2(hi), make_float2(-1.f, -1.f), xv),
                                   make_float2(kLoScale, kLoScale));
            const __half2 lo = __floats2half2_rn(r.x, r.y);
            const uint32_t hb = *reinterpret_cast<const uint32_t*>(&hi), lb = *reinterpret_cast<const uint32_t*>(&lo);
            w[h] = __byte_perm(hb, lb, 0x5410);
            w[h + 1] = __byte_perm(hb, lb, 0x7632);
        }
    }
    *reinterpret_cast<uint4*>(b + b_off(0, kk)) = make_uint4(w[0], w[1], w[2], w[3]);
    if (GH > 4) *reinterpret_cast<uint4*>(b + b_off(8, kk)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Max over the 32 lanes of each of GH values by a transposing butterfly: afterwards every lane of
// group l >> (5 - log2 GH) holds the maximum of value (l >> (5 - log2 GH)).
template <int GH>
__device__ __forceinline__ float warp_max_multi(float (&v)[GH], int lane) {
    constexpr int kL = GH == 1 ? 0 : (GH == 2 ? 1 : (GH == 4 ? 2 : 3));
    if (kL >= 1) {
        constexpr int n = GH / 2;
        const bool up = lane & 16;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            const float send = up ? v[q] : v[q + n];
            const float keep = up ? v[q + n] : v[q];
            v[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
        }
    }
    if (kL >= 2) {
        constexpr int n = GH / 4;
        const bool up = lane & 8;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            const float send = up ? v[q] : v[q + n];
            const float keep = up ? v[q + n] : v[q];
            v[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
        }
    }
    if (kL >= 3) {
        const bool up = lane & 4;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    float m = v[0];
#pragma unroll
    for (int s = 16 >> kL; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    return m;
}

// Sum over the 32 lanes of each of GH values (transposing butterfly, as warp_max_multi): every lane
// of group l >> (5 - log2 GH) ends with the sum of value (l >> (5 - log2 GH)).
template <int GH>
__device__ __forceinline__ float warp_sum_multi(float (&v)[GH], int lane) {
    constexpr int kL = GH == 1 ? 0 : (GH == 2 ? 1 : (GH == 4 ? 2 : 3));
    if (kL >= 1) {
        constexpr int n = GH / 2;
        const bool up = lane & 16;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            const float send = up ? v[q] : v[q + n];
            const float keep = up ? v[q + n] : v[q];
            v[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    if (kL >= 2) {
        constexpr int n = GH / 4;
        const bool up = lane & 8;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            const float send = up ? v[q] : v[q + n];
            const float keep = up ? v[q + n] : v[q];
            v[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    if (kL >= 3) {
        const bool up = lane & 4;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float m = v[0];
#pragma unroll
    for (int s = 16 >> kL; s > 0; s >>= 1) m += __shfl_xor_sync(0xffffffffu, m, s);
    return m;
}

// Sum over the 4 warps of per-warp partials laid out [4 warps][8]: out[h] for h < GH.
template <int GH>
__device__ __forceinline__ void sum_warp_parts(const float* part, float (&out)[GH]) {
    if constexpr (GH >= 4) {
#pragma unroll
        for (int c = 0; c < GH / 4; ++c) {
            const float4 a = *reinterpret_cast<const float4*>(part + 4 * c);
            const float4 b = *reinterpret_cast<const float4*>(part + 8 + 4 * c);
            const float4 d = *reinterpret_cast<const float4*>(part + 16 + 4 * c);
            const float4 e = *reinterpret_cast<const float4*>(part + 24 + 4 * c);
            out[4 * c + 0] = (a.x + b.x) + (d.x + e.x);
            out[4 * c + 1] = (a.y + b.y) + (d.y + e.y);
            out[4 * c + 2] = (a.z + b.z) + (d.z + e.z);
            out[4 * c + 3] = (a.w + b.w) + (d.w + e.w);
        }
    } else {
#pragma unroll
        for (int h = 0; h < GH; ++h) out[h] = (part[h] + part[8 + h]) + (part[16 + h] + part[24 + h]);
    }
}

// tcgen05.ld of NC consecutive 32-bit columns (32x32b shape; NC = 2, 4, 8 or 16).
template <int NC>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t (&r)[NC]) {
    if constexpr (NC == 2) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr) : "memory");
    } else if constexpr (NC == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr) : "memory");
    } else if constexpr (NC == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr) : "memory");
    } else {
        tc::ld16(taddr, r);
    }
}

// Sum of the 4 partial accumulators (16 columns apart) for the 2*GH used columns: acc[2h] is head
// h's hi piece, acc[2h+1] its lo piece.
template <int GH>
__device__ __forceinline__ void read_partials(uint32_t d_taddr, float (&acc)[2 * GH]) {
    constexpr int NC = 2 * GH;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t r0[NC], r1[NC];
        ld_cols<NC>(d_taddr + 32 * half, r0);
        ld_cols<NC>(d_taddr + 32 * half + 16, r1);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float v = __uint_as_float(r0[c]) + __uint_as_float(r1[c]);
            acc[c] = half ? acc[c] + v : v;
        }
    }
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier over n threads that also returns the OR of every thread's flag.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool flag) {
    uint32_t out;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n bar.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(out)
        : "r"(id), "r"(n), "r"((uint32_t)flag)
        : "memory");
    return out != 0;
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

// Length of the body (packed tiles + tail) of sequence b: the tokens after the sink.
__device__ __forceinline__ int body_len(const DecodeArgs& a, int b) {
    const int len = a.seq_lens[b] - a.sink_len;
    return clamp_len(len, a.max_tiles, a.full_tail);
}

__device__ __forceinline__ int full_tiles(const DecodeArgs& a, int b) {
    return n_full_tiles(body_len(a, b), a.full_tail);
}

// Partial slot of (sequence b, query head hq, slot k): m, l, pad, pad, o[128].
__device__ __forceinline__ float* slot_ptr(const DecodeArgs& a, int b, int hq, int k) {
    return a.ws + (((size_t)b * a.Hq + hq) * (a.splits + 1) + k) * kWsStride;
}

// Sum of v over the CTA's kThreads threads (every thread gets it); scratch holds kThreads / 32 values.
__device__ __forceinline__ long long cta_sum(long long v, long long* scratch) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    long long t = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t += scratch[w];
    return t;
}

// The pieces of this CTA's workers.  The stream of full tiles -- sequence by sequence, unit by unit
// (unit = kv head x head block) -- is cut into w_used equal contiguous runs of >= P tiles,
// worker w taking run w (none when w >= w_used); this balances the grid to a tile whatever the
// length mix.  Every CTA computes it from the lengths (two passes over the sequences).
__device__ Piece find_piece(const DecodeArgs& a, int wk, long long* scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long long own = 0;
    for (int b = tid; b < a.B; b += kThreads) own += full_tiles(a, b);
    const long long units = a.units;
    const long long total = units * cta_sum(own, scratch);
    const long long n_workers = (long long)gridDim.x * kWorkers;
    long long w_used = total / a.piece;
    if (w_used < 1) w_used = total > 0 ? 1 : 0;
    if (w_used > n_workers) w_used = n_workers;
    long long g0[kWorkers];  // first stream tile of each of the CTA's workers (-1: no piece)
#pragma unroll
    for (int k = 0; k < kWorkers; ++k) {
        const long long w = (long long)blockIdx.x * kWorkers + k;
        g0[k] = w < w_used ? total * w / w_used : -1;
    }
    Piece e;
    e.b = e.u = e.j = 0;
    e.len = 0;
    const long long w = (long long)blockIdx.x * kWorkers + wk;
    if (w < w_used) e.len = total * (w + 1) / w_used - total * w / w_used;
    // the sequence holding tile g0 of the stream: exclusive prefix sums of the tiles per sequence
    long long carry = 0;
    __shared__ int s_b[kWorkers];
    __shared__ long long s_rem[kWorkers];
    if (tid < kWorkers) {
        s_b[tid] = 0;
        s_rem[tid] = 0;
    }
    for (int base = 0; base < a.B; base += kThreads) {
        const int b = base + tid;
        const long long v = b < a.B ? (long long)full_tiles(a, b) : 0;
        long long inc = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += y;
        }
        __syncthreads();
        if (lane == 31) scratch[warp] = inc;
        __syncthreads();
        long long before = 0, chunk = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            before += w < warp ? scratch[w] : 0;
            chunk += scratch[w];
        }
        const long long pre = carry + before + inc - v;
        if (v > 0) {
#pragma unroll
            for (int k = 0; k < kWorkers; ++k)
                if (g0[k] >= units * pre && g0[k] < units * (pre + v)) {
                    s_b[k] = b;
                    s_rem[k] = g0[k] - units * pre;
                }
        }
        carry += chunk;
    }
    __syncthreads();
    if (e.len > 0) {
        const long long nt = full_tiles(a, s_b[wk]);
        e.b = s_b[wk];
        e.u = (int)(s_rem[wk] / nt);
        e.j = (int)(s_rem[wk] % nt);
    }
    return e;
}

template <int KB, int VB, int GH>
__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(DecodeArgs a) {
    using St = Stage<KB, VB>;
    constexpr int NS = St::kCount;
    extern __shared__ __align__(1024) uint8_t dsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wk = warp >> 2, wq = warp & 3, r = tid & 127;

    // per-worker shared memory
    constexpr uint32_t kWorkerBytes = NS * St::kBytes + 2 * kBBytes + GH * kTile * 4 + 8 * 4 + 32 * 4 * 4 +
                                      kIdRing * 4 + 16;
    constexpr uint32_t kWorkerStride = (kWorkerBytes + 1023) & ~1023u;
    uint8_t* wbase = dsm + wk * kWorkerStride;
    uint8_t* bk = wbase;                                   // B operands first: 1024-byte aligned
    uint8_t* bv = bk + kBBytes;
    uint8_t* stages = bv + kBBytes;
    float* qrs = reinterpret_cast<float*>(stages + NS * St::kBytes);  // [GH][128]
    float* einv = qrs + GH * kTile;                        // [8]
    float* mpart = einv + 8;                               // [4 warps][8]
    float* lpart = mpart + 32;                             // [4 warps][8]
    float* zkpart = lpart + 32;                            // sum_j q'_j Z_j: [head] or [4 warps][8]
    float* zvpart = zkpart + 32;                           // [4 warps][8] partial sum_t p Zv_t
    int* idring = reinterpret_cast<int*>(zvpart + 32);     // [kIdRing] tile ids (producer)
    uint8_t* cta = dsm + kWorkers * kWorkerStride;
    uint64_t* full = reinterpret_cast<uint64_t*>(cta);     // [worker][NS]
    uint64_t* mmab = full + kWorkers * NS;                 // [worker]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mmab + kWorkers);

    const int hblocks = a.hblocks;
    // programmatic dependent launch: the merge grid may be scheduled early (it waits for this
    // grid before reading the workspace); this grid's prologue overlaps the previous kernel's tail
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    for (int i = tid; i < (int)(kWorkers * 2 * kBBytes / 16); i += kThreads) {
        const int wkr = i / (2 * kBBytes / 16), off = i % (2 * kBBytes / 16);
        reinterpret_cast<uint4*>(dsm + wkr * kWorkerStride)[off] = make_uint4(0, 0, 0, 0);
    }
    if (tid < kWorkers * NS) mbar_init(&full[tid], 4);  // one arrival per copy (one per warp)
    if (tid < kWorkers) mbar_init(&mmab[tid], 4);  // one tcgen05.commit per warp of the worker
    if (warp == 0) tc::alloc(tmem_slot, kTmemCols);
    fence_mbar_init();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernels' writes are visible
    __shared__ long long s_scratch[kThreads / 32];
    const Piece piece = find_piece(a, wk, s_scratch);
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const uint32_t a_col = tmem + 128 * wk, d_col = a_col + 64;  // D: 4 partials x 16 columns
    const uint32_t bk_addr = smem_addr(bk), bv_addr = smem_addr(bv);
    const int bar_id = 1 + wk;
    constexpr uint32_t kIdesc = tc::idesc_f16_f32_bmn(128, 16);
    int kk_k, kk_v;
    float pre_k, pre_v;
    k_slot<KB>(r, kk_k, pre_k);  // r as channel of a K row
    k_slot<VB>(r, kk_v, pre_v);  // r as token of a V row
    const bool producer = (r == 0);
    const uint64_t bk_desc = tc::smem_desc(bk_addr, kBKStride, kBNStride);
    const uint64_t bv_desc = tc::smem_desc(bv_addr, kBKStride, kBNStride);

    // ---- tile ids and copies ----
    // Warp 0 keeps the block-table entries of the coming 16..32 tiles of the piece in a 32-entry
    // ring in shared memory: the first 32 are loaded at the start; at every 16th tile the batch
    // loaded 16 tiles earlier (plain loads into registers) is stored and the next one is loaded.  The four
    // bulk copies of a tile (K codes, V codes, K params, V params) are issued by lane 0 of the
    // four warps, each arriving on the stage barrier with its own byte count: an issue blocks its
    // thread for ~100 cycles, so the copies are spread instead of serialised in one thread.
    int f_b = piece.b, f_u = piece.u, f_j = piece.j, f_nt = 0;  // first tile of the next batch
    long long f_left = piece.len;                                // tiles not yet fetched
    int f_pos = 0;                                               // stream position of that tile
    int pend_id = 0, pend_n = 0, pend_pos = 0;                   // a loaded, not yet stored batch
    // advance (b, u, j) of this piece's stream by n tiles (n >= 0)
    auto advance = [&](int& b, int& u, int& j, int& nt, int n) {
        j += n;
        while (j >= nt) {
            j -= nt;
            if (++u == a.units) {
                u = 0;
                do {
                    ++b;
                    nt = full_tiles(a, b);
                } while (nt == 0);
            }
        }
    };
    auto fetch_batch = [&](int width) {  // warp 0: load the ids of the next `width` tiles
        const int n = (int)min((long long)width, f_left);
        pend_n = n;
        pend_pos = f_pos;
        if (lane < n) {
            int b = f_b, u = f_u, j = f_j, nt = f_nt;
            advance(b, u, j, nt, lane);
            pend_id = a.block_table[((size_t)b * a.Hkv + u / hblocks) * a.max_tiles + j];
        }
        f_left -= n;
        f_pos += n;
        if (f_left > 0) advance(f_b, f_u, f_j, f_nt, n);
    };
    auto store_batch = [&]() {  // warp 0: the loaded ids into the ring
        if (lane < pend_n) idring[(pend_pos + lane) % kIdRing] = pend_id;
        pend_n = 0;
    };
    // copies of stream position i into its stage; every warp's lane 0 calls this for the same i
    auto issue_copies = [&](int i) {
        if (lane != 0) return;
        const int st = i % NS;
        uint8_t* sb = stages + st * St::kBytes;
        uint64_t* bar = &full[wk * NS + st];
        const int64_t tile = idring[i % kIdRing];
        fence_proxy_async();  // the consumers' reads of this stage come before the TMA writes
        if (wq == 0) {
            mbar_expect_tx(bar, KB * 2048);
            bulk_g2s(sb + St::kK, a.k_codes + tile * (KB * 2048), KB * 2048, bar);
        } else if (wq == 1) {
            mbar_expect_tx(bar, VB * 2048);
            bulk_g2s(sb + St::kV, a.v_codes + tile * (VB * 2048), VB * 2048, bar);
        } else if (wq == 2) {
            mbar_expect_tx(bar, 512);
            bulk_g2s(sb + St::kKP, a.k_params + tile * 512, 512, bar);
        } else {
            mbar_expect_tx(bar, 512);
            bulk_g2s(sb + St::kVP, a.v_params + tile * 512, 512, bar);
        }
    };
    int issued = 0;  // stream positions whose copies are issued (uniform over the worker)
    if (piece.len > 0) {
        if (wq == 0) {
            f_nt = full_tiles(a, f_b);
            fetch_batch(kIdRing);
            store_batch();
            if (f_left > 0) fetch_batch(kIdBatch);
        }
        named_sync(bar_id, 128);  // the first batch of ids is in the ring
        issued = (int)min((long long)NS, piece.len);
        for (int i = 0; i < issued; ++i) issue_copies(i);
    }

    uint32_t mma_phase = 0;
    int pos = 0;       // consumer stream position
    int c_st = 0;      // its ring stage (pos % NS) and phase parity ((pos / NS) & 1)
    uint32_t c_ph = 0;
    bool ok = true;    // this thread's waits all succeeded
    bool alive = true;  // uniform over the worker: changes only at AND-barriers
    // consumer cursor over the piece: unit (cb, cu) from tile cj, c_left tiles to go
    int cb = piece.b, cu = piece.u, cj = piece.j;
    long long c_left = piece.len;
    int c_nt = c_left > 0 ? full_tiles(a, cb) : 0;
    bool cont = false;  // the current unit was entered from the previous one (not at the piece start)
    while (c_left > 0 && alive) {
        // one segment: the tiles of unit (cb, cu) from cj on that belong to this piece
        const int kvh = cu / hblocks, hb = cu % hblocks;
        const int hq0 = kvh * a.group + hb * GH;
        const int seg_j0 = cj;
        const int n_t = (int)min((long long)(c_nt - cj), c_left);
        // rotated queries of the unit's heads, scaled so |q'| 2^E <= 2^7 (q' S1 <= 2^15 in fp16)
        for (int h = wq; h < GH; h += 4) {
            const __nv_bfloat16* qp = a.q + ((size_t)cb * a.Hq + hq0 + h) * kTile + 4 * lane;
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
            const int e = mx > 0.f ? 7 - ceil_log2(mx) : 0;
            const float s = ldexpf(1.f, e);
#pragma unroll
            for (int m = 0; m < 4; ++m) qrs[h * kTile + 4 * lane + m] = v[m] * s;
            if (lane == 0) einv[h] = ldexpf(1.f, -e) * kTwo24;  // undo the scale and the 2^-24
        }
        named_sync(bar_id, 128);

        float m_run[GH], l_part[GH], o[GH];
        // the unit's rotated query for channel r and its scale, kept in registers for small groups
        constexpr bool kQReg = GH <= 4;
        // sum_j q'_j Z_j of the score phase: with 2-bit K and four heads one warp per head (lane l:
        // channels 4l..4l+3, one warp sum); otherwise per-warp partials of every head, combined
        // after the barrier.  Measured: the first is ~1% faster there, and 1-3% slower at 4-bit K
        // or with one or two heads (where only that many warps would carry the sums).
        constexpr bool kZkPerHead = GH == 4 && KB == 2;
        float qreg[kQReg ? GH : 1], ereg[kQReg ? GH : 1];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            m_run[h] = -INFINITY;
            l_part[h] = 0.f;
            o[h] = 0.f;
            if constexpr (kQReg) {
                qreg[h] = qrs[h * kTile + r];
                ereg[h] = einv[h];
            }
        }
        for (int j = 0; j < n_t && alive; ++j, ++pos) {
            const uint8_t* sb = stages + c_st * St::kBytes;
            // tile factors by plain loads: they arrive long before the softmax needs them
            const int64_t tile_id = idring[pos % kIdRing];
            const float gk = __ldg(a.k_scale + tile_id);
            const float gv = __ldg(a.v_scale + tile_id);
            if (wq == 0 && (pos % kIdBatch) == 0 && pos > 0) {
                // the batch loaded 16 tiles ago (positions pos + 16 .. pos + 31) goes into the
                // slots of positions pos - 16 .. pos - 1, all read before this tile's barriers;
                // its first reader is the refill at pos + 14, after this tile's barrier
                store_batch();
                if (f_left > 0) fetch_batch(kIdBatch);
            }
            ok = mbar_wait(&full[wk * NS + c_st], c_ph, &g_decode_error) && ok;
            if (++c_st == NS) {
                c_st = 0;
                c_ph ^= 1u;
            }
            const float* qv = qrs;

            // ---- scores: A = K codes of token r, B = q' S1 2^-shift of channel r ----
            {
                uint32_t x[4 * KB];
                load_row<KB>(sb + St::kK, r, x);
                unpack_row_to_tmem<KB>(x, a_col + lane_off);
            }
            if constexpr (kZkPerHead) {
                float xs[GH];
                const float s1 = e4m3_value(sb[St::kKP + r]) * pre_k;
#pragma unroll
                for (int h = 0; h < GH; ++h) xs[h] = qreg[h] * s1;
                store_b<GH>(bk, kk_k, xs);
                // sum_j q'_j Z_j of head wq (one head per warp; lane l takes channels 4l..4l+3),
                // read after the barrier below
                if (wq < GH) {
                    const float4 qv4 = *reinterpret_cast<const float4*>(qv + wq * kTile + 4 * lane);
                    const uint2 zr = *reinterpret_cast<const uint2*>(sb + St::kKP + 256 + 8 * lane);
                    const float2 z01 = __half22float2(*reinterpret_cast<const __half2*>(&zr.x));
                    const float2 z23 = __half22float2(*reinterpret_cast<const __half2*>(&zr.y));
                    float t = qv4.x * z01.x;
                    t = fmaf(qv4.y, z01.y, t);
                    t = fmaf(qv4.z, z23.x, t);
                    t = fmaf(qv4.w, z23.y, t);
                    t = warp_sum(t);
                    if (lane == 0) zkpart[wq] = t;
                }
            } else {
                float xs[GH], xz[GH];
                const float s1 = e4m3_value(sb[St::kKP + r]) * pre_k;
                const float z = fp16_value(reinterpret_cast<const uint16_t*>(sb + St::kKP + 256)[r]);
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    float q;
                    if constexpr (kQReg) q = qreg[h];
                    else q = qv[h * kTile + r];
                    xs[h] = q * s1;
                    xz[h] = q * z;
                }
                store_b<GH>(bk, kk_k, xs);
                // sum_j q'_j Z_j: per-warp partials, combined after the barrier below
                const float zsum = warp_sum_multi<GH>(xz, lane);
                constexpr int kGroup = 32 / GH;
                if ((lane & (kGroup - 1)) == 0) zkpart[wq * 8 + lane / kGroup] = zsum;
            }
            fence_proxy_async();
            tc::wait_st();
            tc::fence_before();
            // this barrier also orders every reuse of the previous tile's stage, B, scratch and TMEM,
            // and makes the give-up decision uniform
            alive = named_sync_and(bar_id, 128, ok && alive);
            if (!alive) break;
            if (lane == 0) {
                // warp wq issues K-steps 2 wq and 2 wq + 1 into its own partial accumulator
                tc::fence_after();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int s = 2 * wq + u;
                    tc::mma_f16_ts(d_col + 16 * wq, a_col + 8 * s, bk_desc + (uint64_t)(s * 2 * kBKStride >> 4),
                                   kIdesc, u);
                }
                tc::commit(&mmab[wk]);
            }
            ok = mbar_wait(&mmab[wk], mma_phase, &g_decode_error) && ok;
            mma_phase ^= 1;
            tc::fence_after();
            float dsum[2 * GH];
            read_partials<GH>(d_col + lane_off, dsum);

            // ---- online softmax over the tile's 128 tokens (thread r = token r), log2 domain ----
            // Lazy maximum: p = 2^(s - m) with the running maximum m while no score of the tile
            // exceeds it by more than kLazy (p <= 2^kLazy keeps p S1 kWScale inside fp16); otherwise
            // (always on a segment's first tile) the tile maximum is taken exactly and the partial
            // sums are rescaled.
            float sc[GH], p[GH], zks[GH];
            const float tok = gk * e4m3_value(sb[St::kKP + 128 + r]);
            bool over = false;
            if constexpr (kZkPerHead) {
#pragma unroll
                for (int h = 0; h < GH; ++h) zks[h] = zkpart[h];
            } else {
                sum_warp_parts<GH>(zkpart, zks);
            }
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float zk = zks[h];
                const float dot = fmaf(dsum[2 * h + 1], 1.f / kLoScale, dsum[2 * h]);
                float ei;
                if constexpr (kQReg) ei = ereg[h];
                else ei = einv[h];
                sc[h] = fmaf(dot, ei, zk * (ei * (1.f / kTwo24))) * tok;
                over = over || !(sc[h] <= m_run[h] + kLazy);
                p[h] = fast_exp2(sc[h] - m_run[h]);
            }
            const float w = e4m3_value(sb[St::kVP + r]) * (kWScale * pre_v);
            const float zval = fp16_value(reinterpret_cast<const uint16_t*>(sb + St::kVP + 256)[r]);
            auto build_bv = [&]() {
                float xs[GH], xz[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    xs[h] = p[h] * w;
                    xz[h] = p[h] * zval;
                }
                store_b<GH>(bv, kk_v, xs);
                // sum_t p_t Zv_t: per-warp partials, combined after the barrier below
                const float zsum = warp_sum_multi<GH>(xz, lane);
                constexpr int kGroup = 32 / GH;
                if ((lane & (kGroup - 1)) == 0) zvpart[wq * 8 + lane / kGroup] = zsum;
            };
            // build_bv shuffles across the warp, so the choice must be warp-uniform; any warp with an
            // overflowing lane leaves it to the exact path (the OR below then is true as well)
            if (!__any_sync(0xffffffffu, over)) build_bv();

            // ---- PV: A = V codes of channel r, B = p S1 2^-shift of token r ----
            {
                uint32_t x[4 * VB];
                load_row<VB>(sb + St::kV, r, x);
                unpack_row_to_tmem<VB>(x, a_col + lane_off);
            }
            const float chan = gv * e4m3_value(sb[St::kVP + 128 + r]);  // channel r
            fence_proxy_async();
            tc::wait_st();
            tc::fence_before();
            // one barrier when no score overshot the lazy maximum: A, B and the partial sums are
            // then complete; otherwise the exact path below adds two
            if (named_sync_or(bar_id, 128, over)) {
                // exact tile maximum, rescale, rebuild B
                float mx[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) mx[h] = sc[h];
                {
                    const float m = warp_max_multi<GH>(mx, lane);
                    constexpr int kGroup = 32 / GH;
                    if ((lane & (kGroup - 1)) == 0) mpart[wq * 8 + lane / kGroup] = m;
                }
                named_sync(bar_id, 128);
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const float mt = fmaxf(fmaxf(mpart[h], mpart[8 + h]), fmaxf(mpart[16 + h], mpart[24 + h]));
                    const float m_new = fmaxf(m_run[h], mt);
                    const float alpha = fast_exp2(m_run[h] - m_new);
                    m_run[h] = m_new;
                    l_part[h] *= alpha;
                    o[h] *= alpha;
                    p[h] = fast_exp2(sc[h] - m_new);
                }
                build_bv();
                fence_proxy_async();
                tc::fence_before();
                named_sync(bar_id, 128);  // mpart is read; zvpart and B are complete
            }
#pragma unroll
            for (int h = 0; h < GH; ++h) l_part[h] += p[h];
            if (lane == 0) {
                tc::fence_after();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int s = 2 * wq + u;
                    tc::mma_f16_ts(d_col + 16 * wq, a_col + 8 * s, bv_desc + (uint64_t)(s * 2 * kBKStride >> 4),
                                   kIdesc, u);
                }
                tc::commit(&mmab[wk]);
            }
            // while the PV MMAs run: refill the stage the previous tile used (every thread of the
            // worker is past it: they all reached this tile's barriers)
            if (pos > 0 && issued < piece.len) {
                issue_copies(issued);
                ++issued;
            }
            ok = mbar_wait(&mmab[wk], mma_phase, &g_decode_error) && ok;
            mma_phase ^= 1;
            tc::fence_after();
            read_partials<GH>(d_col + lane_off, dsum);
            float zvs[GH];
            sum_warp_parts<GH>(zvpart, zvs);
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float zv = zvs[h];
                const float acc = fmaf(dsum[2 * h + 1], 1.f / kLoScale, dsum[2 * h]);
                o[h] = fmaf(fmaf(acc, kTwo24 / kWScale, zv), chan, o[h]);
            }
        }

        // ---- this segment's partial (m, l, o) for its heads ----
        // Slots of a unit: k < ceil(nt / 16) for the 16-tile block in which a piece starts, and
        // slot `splits` for the piece that enters the unit from the previous one.  As every piece
        // has >= P tiles, no two pieces start in one block; blocks that no piece starts in lie
        // wholly inside one segment, which marks their slots empty -- so every slot the merge
        // reads is written exactly once.
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const float ls = warp_sum(l_part[h]);
            if (lane == 0) lpart[wq * 8 + h] = ls;
        }
        alive = named_sync_and(bar_id, 128, ok && alive);
        {
            const int seg_j1 = seg_j0 + n_t;
            const int own = cont ? a.splits : seg_j0 / a.piece;
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                float* dst = slot_ptr(a, cb, hq0 + h, own);
                dst[4 + r] = o[h];
                if (r == 0) {
                    dst[0] = m_run[h];
                    dst[1] = lpart[h] + lpart[8 + h] + lpart[16 + h] + lpart[24 + h];
                }
            }
            const int n_blk = (c_nt + a.piece - 1) / a.piece;
            for (int k = r; k < n_blk; k += 128) {
                const int k0 = k * a.piece, k1 = min(k0 + a.piece, c_nt);
                if (k != own && k0 >= seg_j0 && k1 <= seg_j1) {
#pragma unroll
                    for (int h = 0; h < GH; ++h) {
                        float* dst = slot_ptr(a, cb, hq0 + h, k);
                        dst[0] = -INFINITY;
                        dst[1] = 0.f;
                    }
                }
            }
            if (!cont && seg_j0 == 0 && r == 0) {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    float* dst = slot_ptr(a, cb, hq0 + h, a.splits);
                    dst[0] = -INFINITY;
                    dst[1] = 0.f;
                }
            }
        }
        named_sync(bar_id, 128);  // lpart / qrs are rewritten by the next segment
        // advance the cursor to the next unit with full tiles
        c_left -= n_t;
        cj = 0;
        cont = true;
        if (++cu == a.units) {
            cu = 0;
            if (c_left > 0) {
                do {
                    ++cb;
                    c_nt = full_tiles(a, cb);
                } while (c_nt == 0);
            }
        }
    }
    if (producer) {
        // after a give-up, wait (bounded) for copies still in flight before the CTA exits
        for (int q = pos; q < issued; ++q) mbar_drain(&full[wk * NS + q % NS], (q / NS) & 1);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::dealloc(tmem, kTmemCols);
}

// Max and sum over the merge CTA's 128 threads (every thread gets the result); red holds 4 floats.
__device__ __forceinline__ float merge_max(float v, float* red) {
    v = warp_max(v);
    __syncthreads();  // red is free again
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}
__device__ __forceinline__ float merge_sum(float v, float* red) {
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return (red[0] + red[1]) + (red[2] + red[3]);
}

// Unnormalised Sylvester Walsh-Hadamard transform of 128 values, value i held by thread i: butterflies
// on index bits 0-4 by shuffles, bits 5-6 through shared memory (stage: 128 floats).
__device__ __forceinline__ float fwht128_block(float x, float* stage) {
    const int c = threadIdx.x;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, s);
        x = (c & s) ? y - x : x + y;
    }
#pragma unroll
    for (int s = 32; s < kTile; s <<= 1) {
        __syncthreads();
        stage[c] = x;
        __syncthreads();
        const float y = stage[c ^ s];
        x = (c & s) ? y - x : x + y;
    }
    return x;
}

// The 4 warps' float4 partials (channels 4 lane .. 4 lane + 3) summed for channel threadIdx.x.
__device__ __forceinline__ float merge_warp_parts(float4 acc, float (*part)[kTile]) {
    const int c = threadIdx.x;
    __syncthreads();  // part is free again
    *reinterpret_cast<float4*>(&part[c >> 5][4 * (c & 31)]) = acc;
    __syncthreads();
    return (part[0][c] + part[1][c]) + (part[2][c] + part[3][c]);
}

// One CTA of 128 threads per (sequence, query head), thread c owning output channel c:
//   1. log-sum-exp merge of the partial slots (slot weights one per thread; the weighted o sums
//      spread over the 4 warps, each lane reading 4 channels of a slot), then the inverse rotation;
//   2. the unquantised tokens -- the FP16 sink, then the bf16 tail, in the original basis -- 128 at
//      a time: thread t scores token t (its whole row at once), one online-softmax update per chunk,
//      and the p-weighted V rows again spread over the warps;
//   3. normalise by l.
// The kernel is a chain of dependent steps behind the split grid, so its loads are issued early:
// right after the wait, one round trip brings each thread's slot (m, l), each warp's o rows of the
// first 4 x kPreSlots = 20 slots (17 at the usual piece sizes) and the query; later loads are only for
// slots beyond those.  At <= 128 registers four CTAs fit on an SM, so B 16 x 32 heads is one wave.
constexpr int kPreSlots = 5;  // o rows prefetched per warp: slots warp, warp + 4, ..., warp + 16

__device__ __forceinline__ float4 fma4(float4 v, float w, float4 acc) {
    acc.x = fmaf(v.x, w, acc.x);
    acc.y = fmaf(v.y, w, acc.y);
    acc.z = fmaf(v.z, w, acc.z);
    acc.w = fmaf(v.w, w, acc.w);
    return acc;
}

__global__ void __launch_bounds__(kTile, 4) decode_merge_kernel(DecodeArgs a) {
    __shared__ __align__(16) float s_q[kTile];     // scaled query, original basis
    __shared__ __align__(16) float s_w[kTile];     // slot weights / token probabilities of a chunk
    __shared__ __align__(16) float s_part[4][kTile];
    __shared__ float s_red[4];
    const int c = threadIdx.x, lane = c & 31, warp = c >> 5;
    const int hq = blockIdx.x, b = blockIdx.y;
    // programmatic dependent launch: the split grid (and everything before it) is complete and
    // visible once this returns; nothing is read before it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int kvh = hq / a.group;
    const int len = body_len(a, b);
    const int nt = n_full_tiles(len, a.full_tail);
    const int tail = len - nt * kTile;  // 0..127, or 1..128 with the full window
    const int n_sink = max(0, min(a.sink_len, a.seq_lens[b]));
    const int n_tok = n_sink + tail;
    const size_t tb = ((size_t)b * a.Hkv + kvh) * kTile * kTile;
    const float* base = slot_ptr(a, b, hq, 0);
    // the slots this (sequence, head) has: one per P-tile block and the unit-entry slot
    const int n_slots = nt > 0 ? (nt + a.piece - 1) / a.piece + 1 : 0;
    auto slot_of = [&](int i) { return i + 1 == n_slots ? a.splits : i; };
    // row of unquantised token t (sink first, then tail)
    auto k_row = [&](int t) {
        const bool in_sink = t < n_sink;
        return reinterpret_cast<const uint4*>((in_sink ? a.k_sink : a.k_tail) + tb +
                                              (size_t)(in_sink ? t : t - n_sink) * kTile);
    };

    // ---- the first round trip ----
    float m0 = -INFINITY, l0 = 0.f;
    if (c < n_slots) {
        m0 = __ldcg(base + slot_of(c) * kWsStride);
        l0 = __ldcg(base + slot_of(c) * kWsStride + 1);
    }
    float4 pre[kPreSlots];
#pragma unroll
    for (int q = 0; q < kPreSlots; ++q) {
        const int j = warp + 4 * q;
        // rows of empty slots hold whatever the workspace held: loaded, never used
        pre[q] = j < n_slots ? __ldcg(reinterpret_cast<const float4*>(base + slot_of(j) * kWsStride + 4) + lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float qc = n_tok > 0 ? __bfloat162float(a.q[((size_t)b * a.Hq + hq) * kTile + c]) * a.qscale : 0.f;

    float mloc = m0;
    for (int i = c + kTile; i < n_slots; i += kTile) mloc = fmaxf(mloc, __ldcg(base + slot_of(i) * kWsStride));
    float mmax = merge_max(mloc, s_red);
    float l = 0.f, o = 0.f;
    if (mmax != -INFINITY) {  // uniform over the CTA
        float lloc = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < n_slots; k0 += kTile) {
            const int i = k0 + c;
            float w = 0.f;
            if (i < n_slots) {
                const float m = k0 == 0 ? m0 : __ldcg(base + slot_of(i) * kWsStride);
                if (m != -INFINITY) {  // an empty slot (its o is not written) weighs 0
                    w = fast_exp2(m - mmax);
                    lloc = fmaf(k0 == 0 ? l0 : __ldcg(base + slot_of(i) * kWsStride + 1), w, lloc);
                }
            }
            __syncthreads();  // s_w is free again
            s_w[c] = w;
            __syncthreads();
            const int n_c = min(kTile, n_slots - k0);
            int j = warp;
            if (k0 == 0) {
#pragma unroll
                for (int q = 0; q < kPreSlots; ++q, j += 4) {
                    if (j < n_c) {
                        const float wj = s_w[j];
                        if (wj != 0.f) acc = fma4(pre[q], wj, acc);
                    }
                }
            }
#pragma unroll 4
            for (; j < n_c; j += 4) {
                const float wj = s_w[j];
                if (wj == 0.f) continue;
                acc = fma4(__ldcg(reinterpret_cast<const float4*>(base + slot_of(k0 + j) * kWsStride + 4) + lane), wj,
                           acc);
            }
        }
        l = merge_sum(lloc, s_red);
        o = merge_warp_parts(acc, s_part);
        if (a.rotate) o = fwht128_block(o, s_w) * kInvSqrt128;
    }

    if (n_tok > 0) {
        s_q[c] = qc;
        __syncthreads();
        for (int t0 = 0; t0 < n_tok; t0 += kTile) {
            const int t = t0 + c;
            float sc = -INFINITY;
            if (t < n_tok) {
                const uint4* kr = k_row(t);
                uint4 raw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) raw[i] = __ldg(kr + i);
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __nv_bfloat162* kp = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
                    const float4 q0 = *reinterpret_cast<const float4*>(&s_q[8 * i]);
                    const float4 q1 = *reinterpret_cast<const float4*>(&s_q[8 * i + 4]);
                    const float2 k0 = __bfloat1622float2(kp[0]), k1 = __bfloat1622float2(kp[1]);
                    const float2 k2 = __bfloat1622float2(kp[2]), k3 = __bfloat1622float2(kp[3]);
                    d = fmaf(q0.x, k0.x, d);
                    d = fmaf(q0.y, k0.y, d);
                    d = fmaf(q0.z, k1.x, d);
                    d = fmaf(q0.w, k1.y, d);
                    d = fmaf(q1.x, k2.x, d);
                    d = fmaf(q1.y, k2.y, d);
                    d = fmaf(q1.z, k3.x, d);
                    d = fmaf(q1.w, k3.y, d);
                }
                sc = d;
            }
            const float m_new = fmaxf(mmax, merge_max(sc, s_red));
            const float al = fast_exp2(mmax - m_new);  // 0 while nothing came before
            const float p = t < n_tok ? fast_exp2(sc - m_new) : 0.f;
            l = fmaf(l, al, merge_sum(p, s_red));
            __syncthreads();  // s_w is free again
            s_w[c] = p;
            __syncthreads();
            const int n_c = min(kTile, n_tok - t0);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int j = warp; j < n_c; j += 4) {
                const int tt = t0 + j;
                const bool in_sink = tt < n_sink;
                const __nv_bfloat16* vr = (in_sink ? a.v_sink : a.v_tail) + tb +
                                          (size_t)(in_sink ? tt : tt - n_sink) * kTile + 4 * lane;
                const uint2 raw = __ldg(reinterpret_cast<const uint2*>(vr));
                const float2 v0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
                const float2 v1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
                const float pj = s_w[j];
                acc.x = fmaf(pj, v0.x, acc.x);
                acc.y = fmaf(pj, v0.y, acc.y);
                acc.z = fmaf(pj, v1.x, acc.z);
                acc.w = fmaf(pj, v1.y, acc.w);
            }
            o = fmaf(o, al, merge_warp_parts(acc, s_part));
            mmax = m_new;
        }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    a.out[((size_t)b * a.Hq + hq) * kTile + c] = o * inv;
}

template <int KB, int VB, int GH>
size_t split_smem_bytes() {
    using St = Stage<KB, VB>;
    constexpr uint32_t kWorkerBytes = St::kCount * St::kBytes + 2 * kBBytes + GH * kTile * 4 + 8 * 4 + 32 * 4 * 4 +
                                      kIdRing * 4 + 16;
    constexpr uint32_t kWorkerStride = (kWorkerBytes + 1023) & ~1023u;
    size_t bytes = (size_t)kWorkers * kWorkerStride + kWorkers * St::kCount * 8 + kWorkers * 8 + 16;
    // at least 80 KB, so no more than two CTAs (2 x 256 TMEM columns) share an SM
    return bytes < 80 * 1024 ? 80 * 1024 : bytes;
}

// Launch with programmatic stream serialisation: the grid may start before the previous kernel in
// the stream completes; it executes griddepcontrol.wait before reading that kernel's results.
template <typename Kern>
cudaError_t launch_dependent(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             const DecodeArgs& a) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, a);
}

// Persistent grid: two CTAs per SM, or fewer when at most max_stream_tiles full tiles (an upper
// bound the host knows: sequences x units x block-table width) cannot keep them all busy with pieces
// of >= piece tiles.
int split_grid(long long max_stream_tiles, int piece) {
    int dev = 0, sms = 0;
    if (current_device(&dev, &sms) != cudaSuccess) return -1;
    const long long pieces = (max_stream_tiles + piece - 1) / piece;
    const long long ctas = (pieces + kWorkers - 1) / kWorkers;
    return (int)(ctas < 1 ? 1 : (ctas < 2 * sms ? ctas : 2 * sms));
}

template <int KB, int VB, int GH>
cudaError_t run_split(const DecodeArgs& a, int grid, cudaStream_t stream) {
    auto kern = decode_split_kernel<KB, VB, GH>;
    const size_t smem = split_smem_bytes<KB, VB, GH>();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = set_smem_limit_once(kern, (int)smem, false, dev);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(grid), dim3(kThreads), smem, stream, a);
}

template <int KB, int VB>
cudaError_t run_split_g(const DecodeArgs& a, int gh, int grid, cudaStream_t stream) {
    if (gh == 1) return run_split<KB, VB, 1>(a, grid, stream);
    if (gh == 2) return run_split<KB, VB, 2>(a, grid, stream);
    if (gh == 4) return run_split<KB, VB, 4>(a, grid, stream);
    return run_split<KB, VB, 8>(a, grid, stream);
}

}  // namespace

// Workspace: the partial slots [B][Hq][splits + 1][132] f32, rounded up to 256 bytes.
DecodePlan plan_decode(int B, int Hq, int Hkv, int max_tiles) {
    DecodePlan p;
    const long long units = (long long)B * Hkv;
    const long long bound = units * (max_tiles > 0 ? max_tiles : 0);  // full tiles at most
    p.piece = kMaxPiece;
    while (p.piece > kMinPieceTiles && bound < kFillWorkers * p.piece) p.piece /= 2;
    p.splits = max_tiles <= 0 ? 1 : (max_tiles + p.piece - 1) / p.piece;
    // The workspace covers every block-table width up to max_tiles, so one sized for the widest
    // table serves narrower ones (which may take a finer granularity and more slots per tile):
    // for each finer P the widest table that selects it (bound < 1024 P) gives its slot count.
    long long ws_splits = p.splits;
    for (int piece = p.piece / 2; piece >= kMinPieceTiles && units > 0; piece /= 2) {
        long long m = (2 * kFillWorkers * piece + units - 1) / units - 1;  // widest table with P = piece
        if (m > max_tiles) m = max_tiles;
        if (m > 0) ws_splits = ws_splits > (m + piece - 1) / piece ? ws_splits : (m + piece - 1) / piece;
    }
    p.workspace_bytes = ((size_t)B * Hq * (ws_splits + 1) * kWsStride * sizeof(float) + 255) & ~(size_t)255;
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
                          const void* k_sink, const void* v_sink, int sink_len, const void* k_tail,
                          const void* v_tail, float softmax_scale, int rotate, int full_tail,
                          void* workspace, const DecodePlan& plan, float* out, cudaStream_t stream) {
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
    a.k_sink = static_cast<const __nv_bfloat16*>(k_sink);
    a.v_sink = static_cast<const __nv_bfloat16*>(v_sink);
    a.sink_len = sink_len;
    a.k_tail = static_cast<const __nv_bfloat16*>(k_tail);
    a.v_tail = static_cast<const __nv_bfloat16*>(v_tail);
    a.qscale = softmax_scale * kLog2e;
    a.rotate = rotate;
    a.full_tail = full_tail;
    a.splits = plan.splits;
    a.piece = plan.piece;
    a.B = B;
    // heads per unit: the largest of 8, 4, 2, 1 dividing the group (8 heads x (hi, lo) fill the 16
    // MMA columns); a larger or odd group is cut into group / gh head blocks, each a unit of its own
    // that reads the kv head's tiles again
    const int gh = group % 8 == 0 ? 8 : (group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1));
    a.hblocks = group / gh;
    a.units = Hkv * a.hblocks;
    a.ws = static_cast<float*>(workspace);
    a.out = out;
    const int grid = split_grid((long long)B * a.units * (max_tiles > 0 ? max_tiles : 0), plan.piece);
    if (grid <= 0) return cudaErrorInvalidDevice;
    cudaError_t e;
    if (k_bits == 2 && v_bits == 2) e = run_split_g<2, 2>(a, gh, grid, stream);
    else if (k_bits == 4 && v_bits == 2) e = run_split_g<4, 2>(a, gh, grid, stream);
    else if (k_bits == 2 && v_bits == 4) e = run_split_g<2, 4>(a, gh, grid, stream);
    else e = run_split_g<4, 4>(a, gh, grid, stream);
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_merge_kernel, dim3(Hq, B), dim3(kTile), 0, stream, a);
}

}  // namespace kvarn
