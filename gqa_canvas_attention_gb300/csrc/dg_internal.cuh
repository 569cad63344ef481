// dg_internal.cuh -- shared declarations between the translation units of libdgattn.so:
// kernel parameter blocks, operand layouts in the plan's scratch, and the host launchers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

namespace dg {

// Device status word bits (OR-ed in by kernels whose bounded waits ran out).
enum : uint32_t {
    kErrWaitProducer = 1u,
    kErrWaitMma = 2u,
    kErrWaitSoftmax = 4u,
    kErrWaitDrain = 8u,
    kErrSchedule = 16u,            // a stream-K run covered more than two pairs (host error)
    kErrRange = 32u,               // a cache V value outside the fp16 range (tensor-core path)
};

// Rows of the tensor-core query tile: the G = nh/nkv query heads of one kv group are packed
// into the MMA M dimension, row R = t * G + (h mod G) of group g = h / G.
constexpr int kTileM = 128;
// Rows of the fp32 path's query tile.
constexpr int kFp32TileM = 32;

// What the first-stage kernel writes.
enum NormOut : int {
    kOutFp32 = 0,   // q_hat [T, nh, hd], k_hat / v_hat [T, nkv, hd] fp32 (input layouts)
    kOutTc = 1,     // bf16 hi/lo planes of q_hat * log2(e) and k_hat, fp16 v_hat (tensor-core
                    // layouts)
};

struct NormRopeParams {
    const float *q, *k, *v;        // [T, nh*hd], [T, nkv*hd], [T, nkv*hd]
    const float *wq, *wk;          // [hd] or null
    const float *cos_sin;          // [T, 2*hd] or null (then computed per lane from inv_freq)
    const float4 *inv_freq;        // [hd/2] theta^(-2i/hd) in fp64, exactly x + y + z (w unused)
    int T, nh, nkv, ctx, S, S_pad, rows_pad;
    long long pos0;
    float eps;
    int do_norm, do_rope;          // 0/1 (the attention-only entry point passes 0, 0)
    int inputs_resident;           // 1: q, k, v, weights and cos_sin are complete before the
                                   // previous kernel in the stream started (DG_OPT_INPUTS_RESIDENT)
    int other_set;                 // 1: the operand arrays written here are not the ones the
                                   // previous forward's attention kernel reads (the plan
                                   // alternates two sets), so the stores need not wait for it
    // kOutFp32 destinations
    float *q_out, *k_out, *v_out;
    // kOutTc destinations
    __nv_bfloat16 *qh, *ql;        // [nkv, rows_pad, hd] elements; qh row-interleaved per 128-row
                                   // tile (unit u of row r at (tile * hd/8 + u) * 128 + r), ql too
                                   // when ql_interleaved, else row-major (a TMA operand)
    int ql_interleaved;
    __nv_bfloat16 *kh, *kl;        // [nkv, S, hd] (canvas rows ctx..ctx+T-1)
    __half *vh;                    // [nkv, S, hd] fp16 (canvas rows ctx..ctx+T-1)
    // kOutTc with a cache passed with the call: its fp32 rows [nkv, ctx, hd] are converted into
    // rows 0..ctx-1 of kh / kl / vh by the last cache_blocks blocks of the same launch
    const float *kc, *vc;
    int cache_blocks;
    uint32_t *status;              // kErrRange is OR-ed in for a V value beyond the fp16 range
};

// Conversion of a cache [nkv, ctx, hd] into the tensor-core operand arrays (rows 0..ctx-1).
// Element types of a cache handed to dg_attn_cache_prepare_typed (DG_DTYPE_*).
enum CacheType : int { kCacheF32 = 0, kCacheF16 = 1, kCacheBf16 = 2 };

struct CachePrepParams {
    const void *k_cache, *v_cache; // [nkv, ctx, hd] of `dtype`
    __nv_bfloat16 *kh, *kl;        // tensor-core layouts (k32 == nullptr) ...
    __half *vh;                    // [nkv, S, hd] fp16 (cache rows 0..ctx-1)
    float *k32, *v32;              // ... or an fp32 copy [nkv, ctx, hd] for the exact path
    int nkv, ctx, S, S_pad, hd;
    int dtype;                     // CacheType
    uint32_t *status;              // kErrRange is OR-ed in for a V value beyond the fp16 range
    __nv_bfloat16 *kh2, *kl2;      // null, or a second set of tensor-core arrays written with
    __half *vh2;                   // the same rows (the plan's other operand set)
};

struct AttnFp32Params {
    const float *q;                // q_hat [T, nh, hd]
    const float *k_cache, *v_cache;// [nkv, ctx, hd] or null when ctx == 0
    const float *k, *v;            // canvas k_hat / v_hat [T, nkv, hd]
    float *out;                    // [T, nh*hd] (splits == 1)
    float *part_o;                 // [splits, nkv, rows_pad, hd] (splits > 1)
    float2 *part_ml;               // [splits, nkv, rows_pad] (running max, denominator)
    int T, nh, nkv, ctx, S, G, rows, rows_pad;
    int splits, keys_per_split;
};

struct AttnTcParams {
    const __nv_bfloat16 *qh;       // q_hat hi, bf16, row-interleaved tiles; loaded into TMEM
    const __nv_bfloat16 *ql;       // q_hat lo: row-interleaved (into TMEM) or row-major (TMA)
    float *out;
    float *part_o;
    float2 *part_ml;
    uint32_t *status;
    unsigned long long wait_limit_ns;
    int T, nh, nkv, S, G, rows, rows_pad;
    int splits, tiles_per_split, n_tiles;
    int cluster_combine;           // 1: the splits CTAs of a query tile form a cluster and merge
                                   // their partial results through distributed shared memory
    int inject_stall;              // test hook: withhold the first P-ready signal of each CTA
    int static_keys;               // keys [0, static_keys) of every kv group (cache rows) were
                                   // complete before the kernel ahead of this one started: the
                                   // producers may load them before waiting for that kernel
    // stream-K schedule (sk_ctas > 0): CTA c takes key-tile units [sk_begin(c), sk_begin(c + 1))
    // of the qtiles * nkv pairs in order p = g * qtiles + qt, n_tiles units each; its pieces go
    // to part_o / part_ml at slot = its rank among the CTAs of that pair
    int sk_ctas, qtiles;
    long long sk_units;
    __nv_bfloat16 *out_hi, *out_lo;// null, or [T, nh*hd] in place of out: its bf16 hi / lo split
                                   // (hi = bf16(o), lo = bf16(o - hi)), written by the split
                                   // schedule's CTAs that write output rows (the layer path)
};

// Stream-K schedule: U key-tile units over C CTAs, CTA c taking [sk_begin(c), sk_begin(c + 1)).
__host__ __device__ inline long long sk_begin(int c, long long U, int C)
{
    return (long long)c * U / C;
}
// The CTA whose run holds unit u.
__host__ __device__ inline int sk_cta_of(long long u, long long U, int C)
{
    int c = (int)((u * C) / U);
    while (c + 1 < C && sk_begin(c + 1, U, C) <= u) ++c;
    while (c > 0 && sk_begin(c, U, C) > u) --c;
    return c;
}

struct CombineParams {
    const float *part_o;
    const float2 *part_ml;
    float *out;
    int T, nh, nkv, G, rows, rows_pad, splits, hd;
    int log2_domain;               // 1: weights are 2^(s - m) (tensor-core path), 0: e^(s - m)
    // stream-K pieces (sk_ctas > 0): pair (qt, g) has the pieces of CTAs sk_cta_of(p * n_tiles)
    // .. sk_cta_of((p + 1) * n_tiles - 1), p = g * qtiles + qt; part_o holds them row-interleaved
    // per 128-row tile (16-byte unit u of tile row r at u * 128 + r)
    int sk_ctas, qtiles, n_tiles;
    long long sk_units;
};

// ---- the projection step before the block (proj_tc.cu) ----
struct ProjPrepParams {            // input RMSNorm scale and the bf16 hi/lo split of x
    const float *x;                // [T, H] residual stream (or the attention output)
    float *rin;                    // [T] (mean x^2 + eps)^-1/2, or null (split only)
    __nv_bfloat16 *xh, *xl;        // [T_pad, H]
    int T, H;
    float eps;
};

struct ProjWeightParams {          // W' = W diag(ln_w), split bf16 hi/lo, rows q | k | v
    const float *wq, *wk, *wv;     // [nq, H], [nk, H], [n_rows - nq - nk, H]
    const float *ln_w;             // [H] or null
    __nv_bfloat16 *wh, *wl;        // [n_rows, H]
    int nq, nk, n_rows, H;
};

struct ProjParams {
    const float *rin;              // [T]
    const float *wq_norm, *wk_norm;// [hd] or null
    const float *cos_sin;          // [T, 2*hd]
    __nv_bfloat16 *qh, *ql, *kh, *kl;
    __half *vh;
    uint32_t *status;
    unsigned long long wait_limit_ns;
    int T, H, nh, nkv, G, ctx, S, rows_pad, rows_pad_tokens;
    int ql_interleaved, kv_shared;
    float eps;
};

struct ProjMaps {
    CUtensorMap xh, xl;            // bf16 [T_pad][H], box {64, 128}
    CUtensorMap wh, wl;            // bf16 [n_rows][H], box {64, 64}
};

// o_proj + post-attention RMSNorm + residual add (the step after the block)
struct OprojParams {
    float *y;                      // [T, H] the projection, fp32
    float *part_ss;                // [T, H/tile_n] partial sums of squares of y per column tile
    uint32_t *status;
    unsigned long long wait_limit_ns;
    int T, H, K;                   // K = nh * hd
    int tile_n;                    // output columns per CTA (128, 80 or 64)
};

struct PostNormParams {
    const float *y, *part_ss, *w;  // w [H] or null
    float *resid;                  // [T, H], updated in place
    int T, H, n_tiles;
    float eps, scale;
};

cudaError_t proj_prepare_attrs();
cudaError_t launch_oproj(const OprojParams &p, const ProjMaps &maps, cudaStream_t s);
int oproj_tile_n(int H, int T, int num_sms);   // 0: H has none of the supported tile widths
cudaError_t launch_post_norm(const PostNormParams &p, cudaStream_t s);
cudaError_t launch_hidden_prep(const ProjPrepParams &p, cudaStream_t s);
cudaError_t launch_proj_weights(const ProjWeightParams &p, cudaStream_t s);
cudaError_t launch_qkv_proj(const ProjParams &p, const ProjMaps &maps, int hd, int n_tiles,
                            cudaStream_t s);

// Tensor maps handed to the tensor-core kernel (by value, __grid_constant__).
struct TcMaps {
    CUtensorMap ql;                // bf16 [nkv][rows_pad][hd], box {64, 128, 1}
    CUtensorMap kh, kl;            // bf16 [nkv][S][hd], box {64, NK, 1}
    CUtensorMap vh;                // fp16 [nkv][S][hd], box {64, NK, 1}
};

// Tile geometry of the tensor-core kernel for a head dimension.
struct TcGeom {
    int nk;        // keys per score tile
    int vk;        // keys per V ring stage (divides nk)
    int ql_in_tmem;
};
TcGeom tc_geometry(int hd);

// Launch attribute of the kernels that may start while the previous kernel of the stream is still
// running (programmatic dependent launch): each of them calls pdl_wait() before it reads anything
// an earlier kernel writes, so only its launch and set-up overlap.
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// Run `set` (a function-attribute call, which applies to the current device only) once per device:
// `done` holds one bit per device ordinal below 64 (a higher ordinal runs `set` every time).
// Threads that race on a device's first call may both run `set`; the calls are idempotent.
template <class F> cudaError_t once_per_device(std::atomic<unsigned long long> &done, F &&set)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// float4 units of K (and of V) each thread of the first stage's cache blocks converts a pass
constexpr int kNormCacheUnroll = 4;

// Host launchers (return cudaGetLastError()).
// smem_bytes: dynamic shared memory each block asks for and does not use (see beside_smem in
// the plan code), 0 normally.
cudaError_t launch_norm_rope(const NormRopeParams &p, int hd, int mode, cudaStream_t s,
                             size_t smem_bytes = 0);
// cos|sin table [T, 2*hd] of the positions pos0 .. pos0 + T - 1 (layout of a caller's table).
cudaError_t launch_rope_table(float *cs, const float4 *inv_freq, int T, int hd, long long pos0,
                              cudaStream_t s);
cudaError_t launch_cache_prep(const CachePrepParams &p, cudaStream_t s);
cudaError_t launch_attn_fp32(const AttnFp32Params &p, int hd, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnTcParams &p, const TcMaps &maps, int hd, cudaStream_t s);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t s);
cudaError_t attn_tc_prepare(int hd);   // one-time function attributes (smem opt-in)
// The split-schedule variant that writes o_proj's bf16 hi/lo operands (p.out_hi/out_lo) in place
// of the fp32 rows (hd 128 and 256): its own launch with the configuration launch_attn_tc built,
// and its attributes.
cudaError_t launch_attn_tc_split(const cudaLaunchConfig_t &cfg, const TcMaps &maps,
                                 const AttnTcParams &p, int hd);
cudaError_t attn_tc_split_prepare(int hd);
// Clusters of `splits` CTAs the GPU can hold at once (0: that cluster launch cannot run).
int attn_tc_max_clusters(int hd, int splits, int qtiles, int nkv);
constexpr int kMaxClusterSplits = 8;   // portable cluster size
constexpr int kMaxStreamKPieces = 16;  // pieces of one pair the stream-K combine merges
size_t attn_tc_smem_bytes(int hd);

}  // namespace dg
