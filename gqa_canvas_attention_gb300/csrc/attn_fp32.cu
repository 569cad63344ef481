// attn_fp32.cu -- the exact-fp32 attention path on the CUDA cores (page "inferencelayer 0.2.3,
// src/diffusion_gemma_gpu.rs", item DG_ATTN): GQA bidirectional attention, scaling 1.0, no mask,
// keys j < ctx read straight from the caller's cache [nkv, ctx, hd] and keys ctx + t from the
// normed canvas [T, nkv, hd] -- the two split sources of the page's kernel.
//
// A CTA takes 32 packed query rows (the G heads of one kv group, row R = t*G + h mod G) and one
// key range; 256 threads, 8 per row.  Each 32-key tile of K and V is staged in shared memory.
// Scores use blocked summation with a compensated outer sum (8-term fp32 FMA blocks folded into a
// Knuth TwoSum pair) and stay an unrounded (hi, lo) pair until the running maximum has been
// subtracted; the online softmax keeps an fp32 running max and denominator per row (expf), and
// the P.V accumulators live in registers (hd/8 columns per thread).
#include "dg_internal.cuh"

namespace dg {
namespace {

constexpr int kBK = 32;        // keys per tile
constexpr int kThreads = 256;  // 8 threads per query row

__device__ __forceinline__ void two_sum(float &s, float &c, float b)
{
    const float t = s + b;
    const float bb = t - s;
    c += (s - (t - bb)) + (b - bb);
    s = t;
}

template <int HD>
__global__ void __launch_bounds__(kThreads) attn_fp32_kernel(AttnFp32Params p)
{
    constexpr int KPAD = HD + 4;         // K rows padded: 8 key rows per quarter-warp hit distinct banks
    constexpr int NC4 = HD / 32;         // float4 column groups per thread
    extern __shared__ __align__(16) float smem[];
    float *Qs = smem;                    // [32][HD]
    float *Ks = Qs + kFp32TileM * HD;    // [kBK][KPAD]
    float *Vs = Ks + kBK * KPAD;         // [kBK][HD]

    const int tid = threadIdx.x;
    const int r = tid >> 3;              // row of the tile
    const int c8 = tid & 7;
    const int lane = tid & 31;
    const int rowbase_lane = lane & ~7;
    const int g = blockIdx.y;
    const int split = blockIdx.z;
    const int R0 = blockIdx.x * kFp32TileM;

    // key range of this split
    const int kb = split * p.keys_per_split;
    const int ke = min(p.S, kb + p.keys_per_split);

    // stage the query tile
    for (int i = tid; i < kFp32TileM * (HD / 4); i += kThreads) {
        const int rr = i / (HD / 4), c4 = i % (HD / 4);
        const int R = R0 + rr;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (R < p.rows) {
            const int t = R / p.G, h = g * p.G + R % p.G;
            v = reinterpret_cast<const float4 *>(p.q + ((size_t)t * p.nh + h) * HD)[c4];
        }
        reinterpret_cast<float4 *>(Qs + rr * HD)[c4] = v;
    }

    float o[NC4 * 4];
#pragma unroll
    for (int i = 0; i < NC4 * 4; ++i) o[i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    for (int k0 = kb; k0 < ke; k0 += kBK) {
        __syncthreads();   // previous tile fully consumed (and Qs staged on the first pass)
        for (int i = tid; i < kBK * (HD / 4); i += kThreads) {
            const int kk = i / (HD / 4), c4 = i % (HD / 4);
            const int j = k0 + kk;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (j < ke) {
                const float *ksrc, *vsrc;
                if (j < p.ctx) {
                    ksrc = p.k_cache + ((size_t)g * p.ctx + j) * HD;
                    vsrc = p.v_cache + ((size_t)g * p.ctx + j) * HD;
                } else {
                    ksrc = p.k + ((size_t)(j - p.ctx) * p.nkv + g) * HD;
                    vsrc = p.v + ((size_t)(j - p.ctx) * p.nkv + g) * HD;
                }
                kv = reinterpret_cast<const float4 *>(ksrc)[c4];
                vv = reinterpret_cast<const float4 *>(vsrc)[c4];
            }
            reinterpret_cast<float4 *>(Ks + kk * KPAD)[c4] = kv;
            reinterpret_cast<float4 *>(Vs + kk * HD)[c4] = vv;
        }
        __syncthreads();

        // scores of row r against keys c8, c8 + 8, c8 + 16, c8 + 24
        float shi[4] = {0.f, 0.f, 0.f, 0.f}, slo[4] = {0.f, 0.f, 0.f, 0.f};
        const float *qrow = Qs + r * HD;
#pragma unroll 2
        for (int i0 = 0; i0 < HD; i0 += 8) {
            const float4 qa = *reinterpret_cast<const float4 *>(qrow + i0);
            const float4 qb = *reinterpret_cast<const float4 *>(qrow + i0 + 4);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float *krow = Ks + (c8 + 8 * m) * KPAD + i0;
                const float4 ka = *reinterpret_cast<const float4 *>(krow);
                const float4 kc = *reinterpret_cast<const float4 *>(krow + 4);
                float b = qa.x * ka.x;
                b = fmaf(qa.y, ka.y, b); b = fmaf(qa.z, ka.z, b); b = fmaf(qa.w, ka.w, b);
                b = fmaf(qb.x, kc.x, b); b = fmaf(qb.y, kc.y, b); b = fmaf(qb.z, kc.z, b);
                b = fmaf(qb.w, kc.w, b);
                two_sum(shi[m], slo[m], b);
            }
        }
        // the maximum takes the rounded scores; the exponent below takes the unrounded pair
        // (a score of ~60 rounded to fp32 is off by up to 2e-6, which moves the output by as much
        // as 1e-5), with the maximum subtracted from the high part first (exact near the top)
        float mx = -INFINITY;
        bool live[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            live[m] = k0 + c8 + 8 * m < ke;
            if (live[m]) mx = fmaxf(mx, shi[m] + slo[m]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = expf(m_run - m_new);   // 0 on the first tile (m_run = -inf)
        float pv[4], psum = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            pv[m] = live[m] ? expf((shi[m] - m_new) + slo[m]) : 0.f;
            psum += pv[m];
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        psum += __shfl_xor_sync(0xffffffffu, psum, 4);
        l_run = l_run * alpha + psum;
        m_run = m_new;
#pragma unroll
        for (int i = 0; i < NC4 * 4; ++i) o[i] *= alpha;

#pragma unroll 4
        for (int kk = 0; kk < kBK; ++kk) {
            const float pk = __shfl_sync(0xffffffffu, pv[kk >> 3], rowbase_lane + (kk & 7));
            const float *vrow = Vs + kk * HD;
#pragma unroll
            for (int q = 0; q < NC4; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(vrow + 4 * (c8 + 8 * q));
                o[4 * q + 0] = fmaf(pk, v.x, o[4 * q + 0]);
                o[4 * q + 1] = fmaf(pk, v.y, o[4 * q + 1]);
                o[4 * q + 2] = fmaf(pk, v.z, o[4 * q + 2]);
                o[4 * q + 3] = fmaf(pk, v.w, o[4 * q + 3]);
            }
        }
    }

    const int R = R0 + r;
    if (R >= p.rows) return;
    if (p.splits == 1) {
        const int t = R / p.G, h = g * p.G + R % p.G;
        float *dst = p.out + ((size_t)t * p.nh + h) * HD;
        const float inv = 1.0f / l_run;
#pragma unroll
        for (int q = 0; q < NC4; ++q)
            reinterpret_cast<float4 *>(dst)[c8 + 8 * q] =
                make_float4(o[4 * q] * inv, o[4 * q + 1] * inv, o[4 * q + 2] * inv,
                            o[4 * q + 3] * inv);
    } else {
        const size_t row = ((size_t)split * p.nkv + g) * p.rows_pad + R;
        float *dst = p.part_o + row * HD;
#pragma unroll
        for (int q = 0; q < NC4; ++q)
            reinterpret_cast<float4 *>(dst)[c8 + 8 * q] =
                make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        if (c8 == 0) p.part_ml[row] = make_float2(m_run, l_run);
    }
}

template <int HD>
cudaError_t launch_hd(const AttnFp32Params &p, cudaStream_t s)
{
    const size_t smem = sizeof(float) * ((size_t)kFp32TileM * HD + (size_t)kBK * (HD + 4) +
                                         (size_t)kBK * HD);
    // the shared-memory opt-in is a per-device setting of the function
    static std::atomic<unsigned long long> attr_set{0};
    cudaError_t e = once_per_device(attr_set, [&] {
        return cudaFuncSetAttribute(attn_fp32_kernel<HD>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    dim3 grid((p.rows + kFp32TileM - 1) / kFp32TileM, p.nkv, p.splits);
    attn_fp32_kernel<HD><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fp32(const AttnFp32Params &p, int hd, cudaStream_t s)
{
    switch (hd) {
    case 32: return launch_hd<32>(p, s);
    case 64: return launch_hd<64>(p, s);
    case 128: return launch_hd<128>(p, s);
    case 256: return launch_hd<256>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
