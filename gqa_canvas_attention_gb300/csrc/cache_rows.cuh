// cache_rows.cuh -- the conversion of encoder-cache rows (page "inferencelayer 0.2.3,
// src/diffusion_gemma_gpu.rs", DgGpuCache: already normed and roped) into the tensor-core
// operand layouts, shared by the cache preparation kernel and the first-stage kernel (which
// converts a cache passed with the call in the same launch as the canvas rows).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dg {

constexpr float kF16Max = 65504.0f;   // largest finite fp16 value

// Four consecutive elements, float4 unit i of a cache [nkv, ctx, hd], into row j of kv head g of
// the operand arrays [nkv, S, hd] (g = row / ctx, j = row % ctx): K as a bf16 hi/lo pair
// (hi = bf16(k), lo = bf16(k - hi)), V rounded to fp16.  Returns true when a V value lies beyond
// the fp16 range or is not finite.
__device__ __forceinline__ bool cache_store4(float4 k, float4 v, size_t i, int hd, int ctx, int S,
                                             __nv_bfloat16 *kh, __nv_bfloat16 *kl, __half *vh)
{
    // row = g * ctx + j < nkv * ctx < 2^31: 32-bit divisions (a 64-bit one is a subroutine call)
    const unsigned hd4 = (unsigned)hd / 4;
    const unsigned row = (unsigned)(i / hd4);
    const unsigned c4 = (unsigned)(i - (size_t)row * hd4);
    const unsigned g = row / (unsigned)ctx, j = row - g * (unsigned)ctx;
    const size_t dst = ((size_t)g * S + j) * hd + 4 * (size_t)c4;
    // two 16-bit values per 32-bit word, element 2w in the low half
    auto bf2 = [](float a, float b) {
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
    };
    const float kx[4] = {k.x, k.y, k.z, k.w};
    float kr[4];                                   // k - bf16(k), exact in fp32
#pragma unroll
    for (int e = 0; e < 4; ++e) kr[e] = kx[e] - __bfloat162float(__float2bfloat16_rn(kx[e]));
    const uint2 uh = make_uint2(bf2(k.x, k.y), bf2(k.z, k.w));
    const uint2 ul = make_uint2(bf2(kr[0], kr[1]), bf2(kr[2], kr[3]));
    const uint2 uv = make_uint2(
        (uint32_t)__half_as_ushort(__float2half_rn(v.x)) |
            ((uint32_t)__half_as_ushort(__float2half_rn(v.y)) << 16),
        (uint32_t)__half_as_ushort(__float2half_rn(v.z)) |
            ((uint32_t)__half_as_ushort(__float2half_rn(v.w)) << 16));
    *reinterpret_cast<uint2 *>(kh + dst) = uh;
    *reinterpret_cast<uint2 *>(kl + dst) = ul;
    *reinterpret_cast<uint2 *>(vh + dst) = uv;
    return !(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))) <= kF16Max);
}

}  // namespace dg
