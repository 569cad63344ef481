// aux_kernels.cu -- the two streaming helpers around the attention kernels:
//  * cache_prep: converts an encoder cache [nkv, ctx, hd] (page "inferencelayer 0.2.3,
//    src/diffusion_gemma_gpu.rs", DgGpuCache / upload_cache: already normed and roped), given in
//    fp32 or as an f16 / bf16 twin, into the tensor-core operand arrays [nkv, S, hd] (K as a bf16
//    hi/lo pair, V rounded to fp16) or, for the exact path, into an fp32 copy;
//  * combine: merges the partial results of the key-range partitions (split-KV) of one query
//    row with the log-sum-exp rule  out = sum_s w_s O_s / sum_s w_s l_s,  w_s = b^(m_s - max m).
#include "cache_rows.cuh"
#include "dg_internal.cuh"
#include "sm103_ptx.cuh"

namespace dg {
namespace {

// Four consecutive cache elements as floats (every f16 and bf16 value is exact in fp32).
template <typename T> __device__ __forceinline__ float4 load4(const void *base, size_t i);
template <> __device__ __forceinline__ float4 load4<float>(const void *base, size_t i)
{
    return reinterpret_cast<const float4 *>(base)[i];
}
template <> __device__ __forceinline__ float4 load4<__half>(const void *base, size_t i)
{
    const uint2 u = reinterpret_cast<const uint2 *>(base)[i];
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const void *base, size_t i)
{
    const uint2 u = reinterpret_cast<const uint2 *>(base)[i];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__global__ void __launch_bounds__(256) cache_kv_kernel(CachePrepParams p)
{
    const size_t n4 = (size_t)p.nkv * p.ctx * p.hd / 4;
    bool out_of_range = false;     // a V value the fp16 operand cannot hold (or not finite)
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 k = load4<T>(p.k_cache, i);
        const float4 v = load4<T>(p.v_cache, i);
        if (p.k32) {
            // exact path: an fp32 copy in the caller's layout
            reinterpret_cast<float4 *>(p.k32)[i] = k;
            reinterpret_cast<float4 *>(p.v32)[i] = v;
            continue;
        }
        out_of_range |= cache_store4(k, v, i, p.hd, p.ctx, p.S, p.kh, p.kl, p.vh);
        if (p.kh2) cache_store4(k, v, i, p.hd, p.ctx, p.S, p.kh2, p.kl2, p.vh2);
    }
    if (__any_sync(0xffffffffu, out_of_range) && (threadIdx.x & 31) == 0 && p.status)
        atomicOr(p.status, kErrRange);
}

// One warp per (packed row R, kv group g): every lane loads the (m, l) pairs and its slice of
// the partial rows of a group of partitions at once (independent loads in flight), then the
// weights b^(m_s - max m) are applied.  8 rows per CTA.
constexpr int kMaxCombineSplits = 64;
constexpr int kCombineRowsPerCta = 8;
constexpr int kCombineBatch = 8;      // partitions whose loads are issued together

template <int HD>
__global__ void __launch_bounds__(32 * kCombineRowsPerCta) combine_kernel(CombineParams p)
{
    pdl_launch_dependents();
    pdl_wait();   // the partial results come from the attention kernel just before
    constexpr int V4 = HD / 128 > 0 ? HD / 128 : 1;   // float4 per lane (hd 256: 2, 128: 1)
    constexpr bool PART = HD < 128;                   // hd 64 / 32: lanes beyond hd/4 idle
    const int lane = threadIdx.x & 31;
    const int R = blockIdx.x * kCombineRowsPerCta + (threadIdx.x >> 5);
    const int g = blockIdx.y;
    if (R >= p.rows) return;
    const size_t stride = (size_t)p.nkv * p.rows_pad;   // rows between partitions
    const size_t row = (size_t)g * p.rows_pad + R;
    float mmax = -INFINITY;
    for (int s = lane; s < p.splits; s += 32) mmax = fmaxf(mmax, p.part_ml[s * stride + row].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    const bool active = !PART || lane < HD / 4;
    float4 acc[V4];
#pragma unroll
    for (int v = 0; v < V4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    const float4 *src = reinterpret_cast<const float4 *>(p.part_o);
    const size_t hd4 = HD / 4;
    for (int s0 = 0; s0 < p.splits; s0 += kCombineBatch) {
        float2 ml[kCombineBatch];
        float4 o[kCombineBatch][V4];
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            const int s = s0 + k;
            ml[k] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int v = 0; v < V4; ++v) o[k][v] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s < p.splits) {
                ml[k] = p.part_ml[s * stride + row];
#pragma unroll
                for (int v = 0; v < V4; ++v)
                    if (active) o[k][v] = src[(s * stride + row) * hd4 + lane + 32 * v];
            }
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            if (s0 + k >= p.splits) break;
            const float w = p.log2_domain ? exp2f(ml[k].x - mmax) : expf(ml[k].x - mmax);
            den = fmaf(w, ml[k].y, den);
#pragma unroll
            for (int v = 0; v < V4; ++v) {
                acc[v].x = fmaf(w, o[k][v].x, acc[v].x); acc[v].y = fmaf(w, o[k][v].y, acc[v].y);
                acc[v].z = fmaf(w, o[k][v].z, acc[v].z); acc[v].w = fmaf(w, o[k][v].w, acc[v].w);
            }
        }
    }
    if (!active) return;
    const float inv = 1.0f / den;
    const int t = R / p.G, h = g * p.G + R % p.G;
    float4 *dst = reinterpret_cast<float4 *>(p.out + ((size_t)t * p.nh + h) * HD);
#pragma unroll
    for (int v = 0; v < V4; ++v)
        dst[lane + 32 * v] = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv,
                                         acc[v].w * inv);
}

// Stream-K pieces: one CTA per (128-row query tile, kv group, 8 columns), one thread per row.
// The pair's pieces are those of CTAs sk_cta_of(p * n_tiles) .. sk_cta_of((p + 1) * n_tiles - 1)
// of the attention kernel, merged in that order (deterministic):
//   out = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k,  M = max_k m_k.
// Every load of a thread (the (m, l) and the 2 float4 of its columns of up to 8 pieces) is in
// flight at once: one round trip to memory and a store.  A piece's O rows are row-interleaved,
// so each load instruction of a warp reads 512 contiguous bytes; the merged rows go out through a
// shared-memory transpose, 32 contiguous bytes of 16 rows per store instruction.  (Tried on the
// GB300, 48-step workload: 32 columns per thread in 4-piece batches, 16 columns per thread, and a
// one-CTA-per-SM loop over the units; this layout was the fastest, ~8 us of a forward.)
constexpr int kSkBatch = 8;

template <int HD>
__global__ void __launch_bounds__(kTileM) combine_sk_kernel(CombineParams p)
{
    pdl_launch_dependents();
    pdl_wait();   // the pieces come from the attention kernel just before
    __shared__ float stage[kTileM / 32][32 * 12];
    const int qt = blockIdx.x, g = blockIdx.y, c8 = blockIdx.z;    // columns 8*c8 ..
    const int r = threadIdx.x, lane = r & 31, warp = r >> 5;
    const int pr = g * p.qtiles + qt;
    const long long U = p.sk_units;
    const int c0 = sk_cta_of((long long)pr * p.n_tiles, U, p.sk_ctas);
    const int np = sk_cta_of((long long)(pr + 1) * p.n_tiles - 1, U, p.sk_ctas) - c0 + 1;
    const int R = qt * kTileM + r;
    const size_t stride = (size_t)p.nkv * p.rows_pad;           // rows between slots
    const size_t row = (size_t)g * p.rows_pad + R;
    // float4 units of this tile in slot k: (slot tile base + u) * 128 + r
    const float4 *src = reinterpret_cast<const float4 *>(p.part_o) +
                        ((size_t)g * p.rows_pad + (size_t)qt * kTileM) * (HD / 4) + r;
    const size_t slot_stride = stride * (HD / 4);
    float M = -INFINITY, den = 0.f;
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int k0 = 0; k0 < np; k0 += kSkBatch) {
        float2 ml[kSkBatch];
        float4 o[kSkBatch][2];
#pragma unroll
        for (int k = 0; k < kSkBatch; ++k) {
            ml[k] = make_float2(-INFINITY, 0.f);
            o[k][0] = o[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k0 + k < np) {
                ml[k] = p.part_ml[(k0 + k) * stride + row];
#pragma unroll
                for (int v = 0; v < 2; ++v)
                    o[k][v] = src[(k0 + k) * slot_stride + (size_t)(2 * c8 + v) * kTileM];
            }
        }
        // fold the batch in with a running reference (the first batch sets it)
        float Mb = M;
#pragma unroll
        for (int k = 0; k < kSkBatch; ++k) Mb = fmaxf(Mb, ml[k].x);
        const float rescale = M == -INFINITY ? 0.f : exp2f(M - Mb);
        den *= rescale;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            acc[v].x *= rescale; acc[v].y *= rescale; acc[v].z *= rescale; acc[v].w *= rescale;
        }
#pragma unroll
        for (int k = 0; k < kSkBatch; ++k) {
            const float w = k0 + k < np ? exp2f(ml[k].x - Mb) : 0.f;
            den = fmaf(w, ml[k].y, den);
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                acc[v].x = fmaf(w, o[k][v].x, acc[v].x);
                acc[v].y = fmaf(w, o[k][v].y, acc[v].y);
                acc[v].z = fmaf(w, o[k][v].z, acc[v].z);
                acc[v].w = fmaf(w, o[k][v].w, acc[v].w);
            }
        }
        M = Mb;
    }
    const float inv = 1.0f / den;
    float *mydst = R < p.rows ? p.out + ((size_t)(R / p.G) * p.nh + g * p.G + R % p.G) * HD
                              : nullptr;
    float *stg = stage[warp];
#pragma unroll
    for (int v = 0; v < 2; ++v)
        *reinterpret_cast<float4 *>(stg + lane * 12 + 4 * v) =
            make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
    __syncwarp();
    const int sub = lane & 1, rsub = lane >> 1;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int j = 16 * k + rsub;
        float *d = reinterpret_cast<float *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mydst), j));
        if (d)
            *reinterpret_cast<float4 *>(d + 8 * c8 + 4 * sub) =
                *reinterpret_cast<const float4 *>(stg + j * 12 + 4 * sub);
    }
}

}  // namespace

cudaError_t launch_cache_prep(const CachePrepParams &p, cudaStream_t s)
{
    const size_t n4 = (size_t)p.nkv * p.ctx * p.hd / 4;
    if (n4 == 0) return cudaSuccess;
    int blocks = (int)((n4 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    switch (p.dtype) {
    case kCacheF32: cache_kv_kernel<float><<<blocks, 256, 0, s>>>(p); break;
    case kCacheF16: cache_kv_kernel<__half><<<blocks, 256, 0, s>>>(p); break;
    case kCacheBf16: cache_kv_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s)
{
    if (p.sk_ctas > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.qtiles, p.nkv, p.hd / 8);
        cfg.blockDim = dim3(kTileM);
        cfg.stream = s;
        cudaLaunchAttribute attr[1] = {pdl_attribute()};
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        switch (p.hd) {
        case 64: return cudaLaunchKernelEx(&cfg, combine_sk_kernel<64>, p);
        case 128: return cudaLaunchKernelEx(&cfg, combine_sk_kernel<128>, p);
        case 256: return cudaLaunchKernelEx(&cfg, combine_sk_kernel<256>, p);
        default: return cudaErrorInvalidValue;
        }
    }
    if (p.splits > kMaxCombineSplits) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.rows + kCombineRowsPerCta - 1) / kCombineRowsPerCta, p.nkv);
    cfg.blockDim = dim3(32 * kCombineRowsPerCta);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (p.hd) {
    case 32: return cudaLaunchKernelEx(&cfg, combine_kernel<32>, p);
    case 64: return cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
    case 128: return cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
    case 256: return cudaLaunchKernelEx(&cfg, combine_kernel<256>, p);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
