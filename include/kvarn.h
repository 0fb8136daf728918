/*
 * libkvarn -- the KVarN KV-cache codec on one GB300 GPU (sm_103a).
 *
 * The method (KVarN, arXiv:2606.03458) stores the KV cache of each attention head as
 * 128-token x 128-channel tiles. On write, a completed tile is rotated over its channels by an
 * orthonormal Hadamard matrix, normalised on both axes by alternating token/channel
 * standard-deviation normalisation in the log domain (Sinkhorn-Knopp style), and round-to-nearest
 * quantised to 2-bit codes (4-bit keys under the "kvarn_k4v2_g128" preset) with, per 128-element
 * group, two FP8 scales and one FP16 zero-point.  On read, attention consumes the packed cache.
 *
 * Sources (web pages describing the paper; cited by page and section):
 *   [paperlayer]  "KVarN: Variance-Normalized KV-Cache Quantization Mitigates Error Accumulation
 *                 in Reasoning Tasks", paperlayer.ai source-linked summary of arXiv v1.
 *   [dimensionstp] "KVarN: ... Review", dimensionstp.github.io study notes.
 *   [agihunt]     agihunt.info summary of arXiv:2606.03458.
 *   [pheeree]     pheeree.github.io blog post on KVarN (quotes the paper's sections verbatim).
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers of the current CUDA device; the caller owns them.
 *     The library never allocates or frees memory and never synchronises the stream; work is
 *     enqueued on `stream` (NULL = the legacy default stream).
 *   - Arguments are validated on the host before anything is enqueued. On any error the call
 *     returns a non-zero kvarn_status, enqueues nothing and leaves every output untouched;
 *     kvarn_last_error() then describes the problem (thread-local text).
 *   - A launch failure returns KVARN_ERR_CUDA (the CUDA error is consumed with cudaGetLastError).
 *   - Head dimension and tile length are fixed at 128.  Tensor pointers (x, codes, params, out,
 *     q, tails, workspace) must be 16-byte aligned; float/int32 arrays (tile_scale, k_scale,
 *     v_scale, block_table, seq_lens) 4-byte aligned.
 *
 * Packed tile format (one 128-token x 128-channel tile of one head; all little-endian)
 *   Tile axes: t = token (0..127), j = channel (0..127).  Y = X * H is the rotated tile, where
 *   H[i][j] = (-1)^popcount(i & j) / sqrt(128) (Sylvester order, orthonormal and symmetric)
 *   [paperlayer, "2 Preliminaries" and "A Hadamard Transform Arrangement"].
 *   Groups of 128 elements follow KIVI [paperlayer, "2 Preliminaries"]: for K a group is one
 *   channel (its 128 tokens); for V a group is one token (its 128 channels).  The "other axis"
 *   is the remaining one (K: token, V: channel).
 *   codes : 128 rows of 16*b bytes (b = bits).  K tiles: row = token, column = channel.  V tiles
 *           are stored transposed: row = channel, column = token (so decode can stream one
 *           channel's tokens as one row).  Each row is cut into 16 little-endian lanes of b bytes;
 *           the code of column c = 16*i + h (h = c mod 16, i = c div 16) sits in lane h at bits
 *           [b*i, b*i + b).  2-bit tile: 4096 bytes; 4-bit tile: 8192 bytes.
 *   params: 512 bytes per tile:
 *           [  0,128) S1[g]  FP8 E4M3 group scale, indexed by group
 *           [128,256) s2[o]  FP8 E4M3 other-axis scale, indexed by the other axis
 *           [256,512) Z[g]   FP16 zero-point, indexed by group
 *   tile_scale: one float32 per tile, g = a power of two that keeps S1 and Z inside their formats
 *           (the per-tile factor this library adds; 32 bits per 16384 elements).
 *   Dequantised (rotated basis):  Yhat[t][j] = g * s2[o] * (S1[grp] * code[t][j] + Z[grp]).
 *   Storage: b + (8 + 8 + 16)/128 + 32/16384 bits per element = 2.2520 (b=2), 4.2520 (b=4);
 *   the paper states 2.25 bits/element for 2-bit codes with two FP8 scales and one FP16
 *   zero-point per 128-element group [paperlayer, "D Experimental details"].
 */
#ifndef KVARN_H
#define KVARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVARN_HEAD_DIM 128
#define KVARN_TILE_TOKENS 128
#define KVARN_PARAM_BYTES 512

/* Compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* kvarn_stream_t;

typedef enum {
    KVARN_OK = 0,
    KVARN_ERR_INVALID_ARG = 1, /* a pointer, size, alignment or enum is out of range */
    KVARN_ERR_UNSUPPORTED = 2, /* a valid but unimplemented combination (e.g. 3-bit codes) */
    KVARN_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    KVARN_ERR_WORKSPACE = 4,   /* the workspace passed is smaller than required */
    KVARN_ERR_TIMEOUT = 5      /* a device-side wait gave up (reported by kvarn_device_error) */
} kvarn_status;

/* Which cache a tile belongs to; selects the group axis (K: channel, V: token). */
typedef enum { KVARN_KIND_K = 0, KVARN_KIND_V = 1 } kvarn_kind;

/* Flags for ablations: skip the Hadamard rotation and/or the variance normalisation.
 * With both set the codec is plain asymmetric RTN per channel (K) / per token (V), i.e. KIVI's
 * grouping [paperlayer, "5 Related Work"], with the scale stored as FP8 times the tile factor. */
#define KVARN_FLAG_NO_ROTATE 1u
#define KVARN_FLAG_NO_NORMALIZE 2u
/* Decode only: a full FP16 recent window [paperlayer, "D Experimental details": the most recent
 * tokens stay in FP16, R = 128].  Without the flag the tail holds the L mod 128 tokens after the
 * last full block (0..127); with it the tail holds the last ((L - 1) mod 128) + 1 tokens (1..128,
 * none when L = 0), so a block is read from the packed pool only once a newer token exists --
 * the block pseudo-decode's convention, where a block's tokens see each other unquantised. */
#define KVARN_FLAG_FULL_TAIL 4u

typedef struct {
    int32_t k_bits;         /* 2 or 4 */
    int32_t v_bits;         /* 2 or 4 */
    int32_t sinkhorn_iters; /* 0..64; the paper uses 8 [paperlayer, "4 Experiments", Efficiency] */
    uint32_t flags;         /* KVARN_FLAG_* */
} kvarn_config;

/* Fill *out from a preset name.
 *   "kvarn_k4v2_g128": 4-bit K, 2-bit V, group 128, 8 iterations (the shipped preset
 *       [dimensionstp, "3-1 Overview"]);
 *   "kvarn_k2v2_g128": all 2-bit (the paper's setting [paperlayer, "D Experimental details"]);
 *   "kvarn_k4v4_g128", "kvarn_k2v4_g128": the other bit widths (other granularities trade
 *       capacity against overhead [dimensionstp, "4-3 Engineering notes"]);
 *   ablations through the same kernels [paperlayer, "4 Experiments", "B Full Token-Scale
 *   Distribution Error"]: "hadamard_k2v2_g128" = rotation without normalisation,
 *   "kivi_k2v2_g128" = neither, plain per-channel (K) / per-token (V) RTN.
 * Returns KVARN_ERR_INVALID_ARG for a NULL pointer or an unknown name. */
kvarn_status kvarn_config_from_preset(const char* name, kvarn_config* out);

/* Bytes of packed codes per tile for b-bit codes (16*128*b: 4096 for b=2, 8192 for b=4);
 * 0 for an unsupported b. */
size_t kvarn_tile_code_bytes(int bits);

/* Bytes of per-tile parameters (S1, s2, Z): 512.  The float tile_scale is stored apart. */
size_t kvarn_tile_param_bytes(void);

/* Encode n_tiles completed tiles of one cache kind [paperlayer, "3 Methods"; agihunt, pipeline
 * paragraph: rotate -> dual-axis variance normalisation -> RTN].
 *   x_bf16     : [n_tiles][128 tokens][128 channels] bfloat16, token-major (post-RoPE K or V).
 *   codes      : [n_tiles][kvarn_tile_code_bytes(bits)] output.
 *   params     : [n_tiles][512] output.
 *   tile_scale : [n_tiles] float32 output.
 * bits = cfg->k_bits for KVARN_KIND_K, cfg->v_bits for KVARN_KIND_V.  n_tiles == 0 is a no-op.
 * Errors: NULL/misaligned pointer, n_tiles < 0, bits not in {2,4}, iterations outside 0..64. */
kvarn_status kvarn_encode_blocks(const kvarn_config* cfg, kvarn_kind kind, const void* x_bf16,
                                 int64_t n_tiles, void* codes, void* params, float* tile_scale,
                                 kvarn_stream_t stream);

/* Encode n_tiles K blocks and n_tiles V blocks (the same token range of both caches) in one
 * launch: the results are those of kvarn_encode_blocks(K) and kvarn_encode_blocks(V) on the same
 * arguments, bit for bit [paperlayer, "3 Methods" and "D Experimental details": keys and values
 * are normalised and quantised alike, with their own group axes]: one call for the usual case
 * of appending a block to both caches.  Arguments, layouts and errors as for
 * kvarn_encode_blocks, per kind (k_* with cfg->k_bits, v_* with cfg->v_bits). */
kvarn_status kvarn_encode_kv_blocks(const kvarn_config* cfg, const void* k_bf16, const void* v_bf16,
                                    int64_t n_tiles, void* k_codes, void* k_params, float* k_scale,
                                    void* v_codes, void* v_params, float* v_scale,
                                    kvarn_stream_t stream);

/* Dequantise n_tiles packed tiles to float32 [n_tiles][128][128] (token-major).
 * original_basis = 0 returns Yhat (rotated basis); 1 returns Yhat * H, the estimate of the
 * input tile [paperlayer, "I KVarN Dequantization Overhead": both scales are applied in one
 * pass].  With KVARN_FLAG_NO_ROTATE the two are the same.  Errors as for encode. */
kvarn_status kvarn_dequant(const kvarn_config* cfg, kvarn_kind kind, const void* codes,
                           const void* params, const float* tile_scale, int64_t n_tiles,
                           int original_basis, float* out, kvarn_stream_t stream);

/* Bytes of device workspace kvarn_decode_attention needs for this shape and for every narrower
 * block table (max_tiles' <= max_tiles, same B, Hq, Hkv), so one workspace sized for the widest
 * table serves all calls; never smaller for a larger max_tiles.  A call with table width m uses the
 * split-K partials [B][Hq][S + 1][132] float32, S = ceil(m / P) (m, l, 2 pad, o[128] per slot; S = 1
 * when m is 0), where P, the piece granularity, is 16, halved (down to 2) while B * Hkv * m < 512 * P:
 * calls with few tiles are cut into shorter pieces for more parallel workers.  The size is the
 * largest such slot array over m <= max_tiles, rounded up to a multiple of 256.  Returns 0 for an
 * invalid shape.  (The split-K decomposition and its
 * log-sum-exp merge are this library's; the pages only say that attention reads the cache.) */
size_t kvarn_decode_workspace_size(const kvarn_config* cfg, int B, int Hq, int Hkv,
                                   int max_tiles);

/* Decode attention, one query per sequence, grouped-query heads, over the packed cache
 * [dimensionstp, "4-2 Training strategy": the quantised cache is restored at attention read
 * time; paperlayer, "A Hadamard Transform Arrangement": the query is rotated by the same
 * head-wise Hadamard after RoPE so keys stay in the rotated basis].
 *   q_bf16      : [B][Hq][128] bfloat16 queries (original basis).
 *   k_codes, k_params, k_scale : K tile pool (bits = cfg->k_bits); v_*: V tile pool.  The two
 *                 pools are indexed by the same tile id.
 *   block_table : [B][Hkv][max_tiles] int32 tile ids; entry i of (b, kv head) is the tile
 *                 holding tokens [128 i, 128 i + 128) of that sequence.
 *   seq_lens    : [B] int32 device array, tokens of context per sequence (0 allowed).
 *   seq_lens_host: optional [B] host copy; when given, every length is checked against
 *                 128*max_tiles + 127 (+ 128 with KVARN_FLAG_FULL_TAIL) before launch (device
 *                 lengths are clamped to the same bound in any case).
 *   k_tail_bf16, v_tail_bf16 : [B][Hkv][128][128] bfloat16, original basis; with n = the number
 *                 of full tiles read from the pools (floor(L/128), or floor((L-1)/128) with
 *                 KVARN_FLAG_FULL_TAIL), tokens [128 n, L) of sequence b are rows 0 .. L-128n-1.
 *   softmax_scale: multiplies q.k before the softmax.
 *   workspace   : at least kvarn_decode_workspace_size(...) bytes of device memory.
 *   out         : [B][Hq][128] float32 attention output (original basis); a sequence of
 *                 length 0 gets zeros.
 * Hq must be a positive multiple of Hkv (Hq <= 65535).  The query heads of a kv head are taken in
 * blocks of the largest of 8, 4, 2 and 1 that divides Hq/Hkv; each block reads the kv head's tiles
 * once (so a group of 16 reads them twice, a group of 5 five times).  Tile ids are not range-checked
 * on the device: they must index the pools the caller passes. */
kvarn_status kvarn_decode_attention(const kvarn_config* cfg, const void* q_bf16, int B, int Hq,
                                    int Hkv, const void* k_codes, const void* k_params,
                                    const float* k_scale, const void* v_codes,
                                    const void* v_params, const float* v_scale,
                                    const int32_t* block_table, int max_tiles,
                                    const int32_t* seq_lens, const int32_t* seq_lens_host,
                                    const void* k_tail_bf16, const void* v_tail_bf16,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    float* out, kvarn_stream_t stream);

/* Decode attention with an FP16 sink: the first min(sink_len, L) tokens of each sequence are kept
 * unquantised [paperlayer, "D Experimental details": FP16 sink tokens, a grouped quantised body and
 * FP16 trailing tokens; S = 128, or 32 for one benchmark].  Arguments as for
 * kvarn_decode_attention, plus
 *   k_sink_bf16, v_sink_bf16 : [B][Hkv][128][128] bfloat16, original basis; rows 0 .. S'-1 hold
 *                 the sink tokens of sequence b, S' = min(sink_len, L) (may be NULL when
 *                 sink_len = 0);
 *   sink_len    : 0..128.
 * seq_lens counts all tokens (sink, body and tail); the block table and the tail then describe the
 * body of L - S' tokens exactly as kvarn_decode_attention describes a whole sequence (entry i of
 * the block table holds body tokens [128 i, 128 i + 128), i.e. tokens S + 128 i ...), and the
 * seq_lens_host bound grows by sink_len.  Attention does not depend on the order of the keys, so
 * the sink is attended like the tail.  kvarn_decode_attention is this call with sink_len = 0. */
kvarn_status kvarn_decode_attention_sink(const kvarn_config* cfg, const void* q_bf16, int B, int Hq,
                                         int Hkv, const void* k_codes, const void* k_params,
                                         const float* k_scale, const void* v_codes, const void* v_params,
                                         const float* v_scale, const int32_t* block_table, int max_tiles,
                                         const int32_t* seq_lens, const int32_t* seq_lens_host,
                                         const void* k_sink_bf16, const void* v_sink_bf16, int sink_len,
                                         const void* k_tail_bf16, const void* v_tail_bf16,
                                         float softmax_scale, void* workspace, size_t workspace_bytes,
                                         float* out, kvarn_stream_t stream);

/* Decode attention without a caller workspace.  Same arguments and results as
 * kvarn_decode_attention, minus workspace/workspace_bytes: the split-K partials go to a fixed array
 * of KVARN_STATIC_WS_BYTES (8 MiB) that the library keeps in device memory on every GPU that loads
 * it, for the life of the process.  The paper has no counterpart; this call exists for callers that
 * cannot allocate device memory where they run decode -- e.g. code inside a host callback (CUDA
 * forbids API calls such as cudaMalloc there), a plugin whose host framework owns the allocator and
 * offers no scratch, or a latency-critical loop that must not hit cudaMalloc's implicit
 * synchronisation.  Nothing is allocated: no cudaMalloc/cudaFree, no allocating library routine.
 *   - The first call on a device, with that device current, looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any stream capture.  The
 *     cached address belongs to the device's primary context: it does not survive
 *     cudaDeviceReset() (or any teardown of that context), after which the array may sit
 *     elsewhere -- a process that resets a device must not call this entry point on it again.
 *   - All calls on a device share the one array and it keeps the previous call's contents (every
 *     value a call reads is written earlier in that call).  Calls whose kernels can overlap on the
 *     GPU (different streams without ordering) race on it: serialise them.
 *   - Shapes needing more than KVARN_STATIC_WS_BYTES (see kvarn_decode_workspace_size) return
 *     KVARN_ERR_WORKSPACE before anything is enqueued; e.g. B=16, Hq=32, Hkv=8, 256 tiles needs 4.4 MiB. */
#define KVARN_STATIC_WS_BYTES (8u * 1024u * 1024u)
kvarn_status kvarn_decode_attention_static_ws(
    const kvarn_config* cfg, const void* q_bf16, int B, int Hq, int Hkv, const void* k_codes,
    const void* k_params, const float* k_scale, const void* v_codes, const void* v_params,
    const float* v_scale, const int32_t* block_table, int max_tiles, const int32_t* seq_lens,
    const int32_t* seq_lens_host, const void* k_tail_bf16, const void* v_tail_bf16,
    float softmax_scale, float* out, kvarn_stream_t stream);

/* Bytes of device workspace kvarn_append_tokens needs: one staging slot per (sequence, kv head)
 * for a K and a V block (2 x 32 KiB each) and the slots' pool tiles (int32, rounded up to 256
 * bytes).  0 for an invalid shape. */
size_t kvarn_append_workspace_size(int B, int Hkv);

/* Commit the first n_accept[b] of n_new offered tokens of each sequence to its cache
 * [paperlayer, "D Experimental details": a quantised body of 128-token blocks and unquantised
 * trailing tokens; agihunt, pipeline paragraph: a block is quantised once it is done].  The
 * accepted tokens go to the bf16 tail; a block they complete (128 tokens, or with
 * KVARN_FLAG_FULL_TAIL a full tail followed by a newer token) is encoded with cfg into the pool
 * slot block_table[b][h][block index] -- the same codes kvarn_encode_blocks gives for that
 * block -- and the tail keeps the remaining tokens.  seq_lens[b] grows by the accepted count.
 *   k_new_bf16, v_new_bf16 : [B][Hkv][n_new][128] bfloat16, original basis (post-RoPE K); n_new
 *                 1..128 tokens offered per sequence this step.
 *   n_accept    : [B] int32 device, tokens to commit (clamped to 0..n_new); NULL = all n_new
 *                 (speculative decoding commits only the accepted prefix).
 *   seq_lens    : [B] int32 device, updated in place.
 *   k_tail_bf16, v_tail_bf16 : [B][Hkv][128][128] bfloat16 tails, updated in place.
 *   pools, block_table, max_tiles : as for kvarn_decode_attention; written slots only.
 *   workspace   : >= kvarn_append_workspace_size(B, Hkv) bytes, 256-byte aligned.
 * A sequence whose completed block has no entry in the block table (index >= max_tiles) is left
 * unchanged and bit 3 (value 4) of kvarn_device_error is set.  Host-side errors as elsewhere;
 * nothing is enqueued on error.  Launches: one append kernel and one encode kernel (K and V). */
kvarn_status kvarn_append_tokens(const kvarn_config* cfg, int B, int Hkv, const void* k_new_bf16,
                                 const void* v_new_bf16, int n_new, const int32_t* n_accept,
                                 int32_t* seq_lens, void* k_tail_bf16, void* v_tail_bf16, void* k_codes,
                                 void* k_params, float* k_scale, void* v_codes, void* v_params,
                                 float* v_scale, const int32_t* block_table, int max_tiles, void* workspace,
                                 size_t workspace_bytes, kvarn_stream_t stream);

/* Reads and clears the device-side error words of the current device, after synchronising it.
 * Bit 1 (value 1): an encoder TMA bulk copy did not complete within its bounded wait (the affected
 * tiles are left unwritten).  Bit 2 (value 2): a decode wait gave up.  Bit 3 (value 4): an append
 * found no block-table slot for a completed block.  Bit 4 (value 8): the wait of
 * kvarn_check_bounded_wait gave up.  *code_out = 0 means no such event.
 * Kernels cannot return a status to the call that enqueued them (that call has returned long
 * before they run), so a device wait that gives up sets its bit, ends its kernel normally -- the
 * CUDA context stays usable -- and is reported here: the call returns KVARN_ERR_TIMEOUT when any
 * timeout bit (KVARN_DEVICE_TIMEOUT_BITS) was set, KVARN_OK otherwise (bit 3 alone is reported in
 * *code_out with KVARN_OK); *code_out is filled in both cases.  The bits stay set until read: until
 * then every bounded wait of the kernel family that set one gives up at once.
 * (A library diagnostic; the pages have no counterpart.) */
#define KVARN_DEVICE_TIMEOUT_BITS 0xBu
kvarn_status kvarn_device_error(uint32_t* code_out);

/* Self-check of the bounded device waits (a library diagnostic; the pages have no counterpart).
 * Enqueues one small kernel whose mbarrier wait cannot complete (it expects 16 bytes that no copy
 * delivers) and therefore gives up after limit_us microseconds (1..1000000): the kernel sets bit 4
 * of the device error word and ends normally.  A following kvarn_device_error returns
 * KVARN_ERR_TIMEOUT with bit 4 set, and the device stays usable.  No fault, trap or hang is
 * involved; this is how the failure path of every bounded wait in the library is tested.
 * Errors: KVARN_ERR_INVALID_ARG for limit_us outside 1..1000000. */
kvarn_status kvarn_check_bounded_wait(uint32_t limit_us, kvarn_stream_t stream);

/* Static text for a status code. */
const char* kvarn_status_string(kvarn_status status);

/* Thread-local description of the last error returned on this thread ("" if none). */
const char* kvarn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H */
