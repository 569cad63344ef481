// norm_rope.cu -- first stage of the canvas attention block (page "inferencelayer 0.2.3,
// src/diffusion_gemma_gpu.rs", item DG_HEADNORM_ROPE and the three head-norm dispatches of
// canvas_forward): per (token, head) RMSNorm with optional weight, NeoX rotate-half RoPE on q
// and k, the weightless un-roped norm on v.
//
// One warp per (canvas token, chunk of up to 512/hd of its nh + 2*nkv heads): the warp requests
// every row of its chunk, its norm weights and its cos/sin row before any arithmetic, then
// normalises, rotates and stores the rows, 256/hd rows per instruction.  The cos/sin rows come from a table (the
// caller's, or the plan's, built once per set of positions by rope_table_kernel); without one each
// lane computes those of its own elements.  Either way the angle (pos0 + t) * theta^(-2i/hd) is
// reduced modulo 2*pi without rounding anything that matters: the fp64 frequency arrives exactly
// as three floats, the position is an integer below 2^24 (exact in fp32), the large products are
// split exactly with FMAs, 2*pi is a three-float split (Cody & Waite, "Software Manual for the
// Elementary Functions", 1980, with Dekker's exact products), and the pieces are summed with
// Knuth's TwoSum into r_hi + r_lo, |r_lo| <= half an ulp of r_hi.  CUDA's sincosf of r_hi, moved
// to first order in r_lo, then gives cos and sin of the fp64 angle to fp32 accuracy at every
// position.  (fp32 angles would be off by up to ~1e-3 rad at positions near 8192.)
//
// A row is held by hd/8 lanes, 8 elements each (elements 4l..4l+3 and hd/2+4l..hd/2+4l+3 of
// sub-lane l), so a warp instruction covers 256/hd rows; the RMS is a shuffle reduction over the
// row's lanes and the rotate-half partner of element i (i +- hd/2) is in the same lane.
//
// For the tensor-core layouts q-hat (times log2 e) and k-hat are written as bf16 hi/lo pairs and
// v-hat as fp16, next to the cache rows of the same kv head.
#include "cache_rows.cuh"
#include "dg_internal.cuh"
#include "sm103_ptx.cuh"

namespace dg {
namespace {

// A row of hd values is held by hd/8 consecutive lanes ("sub-lanes"), 8 values each: sub-lane l
// holds elements 4l..4l+3 (slots 0-3) and hd/2+4l..hd/2+4l+3 (slots 4-7), so the rotate-half
// partner of slot e is slot e^4 of the same lane, and a warp instruction covers 32/(hd/8) rows.
template <int HD>
struct Rows {
    static constexpr int LPR = HD / 8;         // lanes per row
    static constexpr int RPI = 32 / LPR;       // rows per warp instruction
    static constexpr int HALF = HD / 2;
    __device__ static __forceinline__ int idx(int l, int e)
    {
        return e < 4 ? 4 * l + e : HALF + 4 * l + (e - 4);
    }
    __device__ static __forceinline__ void load(const float *row, int l, float (&x)[8])
    {
        const float4 a = reinterpret_cast<const float4 *>(row)[l];
        const float4 b = reinterpret_cast<const float4 *>(row + HALF)[l];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    // A row read exactly once (the canvas inputs): no L1 allocation, and an L2 policy that
    // evicts these lines first, so the stream does not push the attention kernel's cache tiles
    // out of L2.
    __device__ static __forceinline__ void load_once(const float *row, int l, uint64_t pol,
                                                     float (&x)[8])
    {
        const float4 *a = reinterpret_cast<const float4 *>(row) + l;
        const float4 *b = reinterpret_cast<const float4 *>(row + HALF) + l;
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3])
                     : "l"(a), "l"(pol));
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7])
                     : "l"(b), "l"(pol));
    }
    __device__ static __forceinline__ void store(float *row, int l, const float (&x)[8])
    {
        reinterpret_cast<float4 *>(row)[l] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4 *>(row + HALF)[l] = make_float4(x[4], x[5], x[6], x[7]);
    }
    // 16-bit values: 8 bytes per half row
    template <typename H, typename H2>
    __device__ static __forceinline__ void store_16(H *row, int l, const H (&x)[8])
    {
        uint2 u, w;
        H2 a, b;
        a.x = x[0]; a.y = x[1]; b.x = x[2]; b.y = x[3];
        u.x = *reinterpret_cast<uint32_t *>(&a); u.y = *reinterpret_cast<uint32_t *>(&b);
        a.x = x[4]; a.y = x[5]; b.x = x[6]; b.y = x[7];
        w.x = *reinterpret_cast<uint32_t *>(&a); w.y = *reinterpret_cast<uint32_t *>(&b);
        reinterpret_cast<uint2 *>(row)[l] = u;
        reinterpret_cast<uint2 *>(row + HALF)[l] = w;
    }
};

// Q operand rows for the tensor-core kernel, "row-interleaved": 16-byte unit u (8 values) of row r
// of 128-row tile T sits at unit index (T * (HD/8) + u) * 128 + r, so that 32 threads each
// loading their own row read 512 contiguous bytes per instruction.  `tile` points at unit 0 of
// the tile; sub-lane `l` holds the elements Rows<HD>::idx(l, e): two runs of 4, each half a unit.
template <int HD>
__device__ __forceinline__ void store_q_interleaved(__nv_bfloat16 *tile, int r, int l,
                                                    const __nv_bfloat16 (&x)[8])
{
    char *base = reinterpret_cast<char *>(tile);
#pragma unroll
    for (int g4 = 0; g4 < 2; ++g4) {
        const int i = Rows<HD>::idx(l, 4 * g4);
        __nv_bfloat162 a, b;
        a.x = x[4 * g4]; a.y = x[4 * g4 + 1]; b.x = x[4 * g4 + 2]; b.y = x[4 * g4 + 3];
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(base + ((size_t)(i / 8) * 128 + r) * 16 + (i % 8) * 2) = u;
    }
}

// a + b = s + e exactly (Knuth's TwoSum; no multiplication, so nothing for the compiler to fuse)
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// cos and sin of p * f for an integer position p < 2^24 and the fp64 frequency f held exactly as
// f.x + f.y + f.z (see the file comment for the method).
__device__ __forceinline__ void rope_angle_cos_sin(float pf, float4 f, float &c, float &s)
{
    // 2*pi = kC1 + kC2 + kC3 to 72 bits (the rest is below 5e-23)
    const float kC1 = 0x1.921fb6p+2f, kC2 = -0x1.777a5cp-23f, kC3 = -0x1.ee59dap-48f;
    const float kInvTwoPi = 0.15915494309189535f;
    // the angle: p*f.x = A1 + e1 and p*f.y = A2 + e2 exactly, p*f.z below 2^-23 * p*f.x
    const float A1 = __fmul_rn(pf, f.x), e1 = fmaf(pf, f.x, -A1);
    const float A2 = __fmul_rn(pf, f.y), e2 = fmaf(pf, f.y, -A2);
    const float A3 = __fmul_rn(pf, f.z);
    // kq turns of 2*pi: kq*kC1 = P1 + E1 and kq*kC2 = P2 + E2 exactly
    const float kq = rintf(A1 * kInvTwoPi);
    const float P1 = __fmul_rn(kq, kC1), E1 = fmaf(kq, kC1, -P1);
    const float P2 = __fmul_rn(kq, kC2), E2 = fmaf(kq, kC2, -P2);
    const float P3 = __fmul_rn(kq, kC3);
    // the reduced angle (A1 - P1) + e1 - E1 + A2 - P2 + (e2 - E2 + A3 - P3): A1 - P1 is exact
    // (Sterbenz), the next four terms are summed without loss, the last ones are tiny
    float r = __fsub_rn(A1, P1), lo = 0.f, t;
    two_sum(r, e1, r, t);
    lo = __fadd_rn(lo, t);
    two_sum(r, -E1, r, t);
    lo = __fadd_rn(lo, t);
    two_sum(r, A2, r, t);
    lo = __fadd_rn(lo, t);
    two_sum(r, -P2, r, t);
    lo = __fadd_rn(lo, t);
    lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(e2, E2), __fsub_rn(A3, P3)));
    // r_hi + r_lo with |r_lo| <= half an ulp of r_hi; cos(r_hi + r_lo) to first order in r_lo
    const float r_hi = __fadd_rn(r, lo);
    const float r_lo = __fsub_rn(lo, __fsub_rn(r_hi, r));
    float sd, cd;
    sincosf(r_hi, &sd, &cd);
    c = fmaf(-sd, r_lo, cd);
    s = fmaf(cd, r_lo, sd);
}

// Rows (heads) of one token that one warp takes: 16 values per lane in registers, two rows per
// lane (more warps, each with a shorter chain of dependent instructions, measured faster than 32
// or 64 values per lane).
template <int HD> constexpr int kChunkRows = 2 * Rows<HD>::RPI;

// A cache passed with the call, converted by the last blocks of the first-stage launch: each
// thread takes kNormCacheUnroll float4 units of K and of V a pass, every load of the pass issued
// before the first store.  The waits are the canvas rows' (a cache is an input like q).
constexpr int kCacheUnroll = kNormCacheUnroll;

template <int HD>
__device__ __forceinline__ void convert_cache(const float4 *kc, const float4 *vc, int nkv, int ctx,
                                              int S, int blocks, unsigned blk, bool wait_stores,
                                              __nv_bfloat16 *kh, __nv_bfloat16 *kl, __half *vh,
                                              uint32_t *status)
{
    const size_t n4 = (size_t)nkv * ctx * HD / 4;
    const size_t stride = (size_t)blocks * 128;
    bool out_of_range = false;     // a V value the fp16 operand cannot hold (or not finite)
    for (size_t i0 = (size_t)blk * 128 + threadIdx.x; i0 < n4; i0 += kCacheUnroll * stride) {
        float4 k[kCacheUnroll], v[kCacheUnroll];
#pragma unroll
        for (int u = 0; u < kCacheUnroll; ++u) {
            const size_t i = i0 + u * stride;
            k[u] = i < n4 ? kc[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[u] = i < n4 ? vc[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the rows written here are read by the previous forward's attention kernel until it
        // ends, unless the plan alternates operand sets
        if (wait_stores) {
            pdl_wait();
            wait_stores = false;
        }
#pragma unroll
        for (int u = 0; u < kCacheUnroll; ++u) {
            const size_t i = i0 + u * stride;
            if (i < n4) out_of_range |= cache_store4(k[u], v[u], i, HD, ctx, S, kh, kl, vh);
        }
    }
    if (wait_stores) pdl_wait();
    if (__any_sync(0xffffffffu, out_of_range) && (threadIdx.x & 31) == 0 && status)
        atomicOr(status, kErrRange);
}

template <int HD, int MODE>
__global__ void __launch_bounds__(128) norm_rope_kernel(NormRopeParams p, int chunks)
{
    using R = Rows<HD>;
    constexpr int LPR = R::LPR, RPI = R::RPI;
    constexpr int RG = 2;                         // rows per lane
    // The inputs may come from the kernel before this one in the stream: wait for it first,
    // unless the caller has declared them resident.  Then, if the arrays written here are the
    // ones the previous forward's attention kernel reads, only the stores below wait (the loads
    // and arithmetic overlap the end of that kernel); if they are the other operand set, nothing
    // waits but one thread at the very end, which keeps this grid from completing before the
    // kernel ahead of it.
    pdl_launch_dependents();
    if (!p.inputs_resident) pdl_wait();
    if constexpr (MODE == kOutTc) {
        if ((int)blockIdx.x >= (int)gridDim.x - p.cache_blocks) {
            convert_cache<HD>(reinterpret_cast<const float4 *>(p.kc),
                              reinterpret_cast<const float4 *>(p.vc), p.nkv, p.ctx, p.S,
                              p.cache_blocks, blockIdx.x - (gridDim.x - p.cache_blocks),
                              p.inputs_resident && !p.other_set, p.kh, p.kl, p.vh, p.status);
            return;
        }
    }
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int t = gw / chunks;
    if (t >= p.T) return;
    const int jobs = p.nh + 2 * p.nkv;
    const int j0 = (gw % chunks) * kChunkRows<HD>;
    const int nj = min(kChunkRows<HD>, jobs - j0);
    const int G = p.nh / p.nkv;
    auto src_row = [&](int job) -> const float * {
        if (job < p.nh) return p.q + ((size_t)t * p.nh + job) * HD;
        if (job < p.nh + p.nkv) return p.k + ((size_t)t * p.nkv + (job - p.nh)) * HD;
        return p.v + ((size_t)t * p.nkv + (job - p.nh - p.nkv)) * HD;
    };

    // every row of the chunk is requested before any arithmetic; lanes past the chunk's last row
    // hold zeros (they join the shuffles, store nothing)
    float x[RG][8];
    uint64_t stream_pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream_pol));
#pragma unroll
    for (int g = 0; g < RG; ++g) {
        const int r = g * RPI + rsub;
        if (r < nj) {
            R::load_once(src_row(j0 + r), sub, stream_pol, x[g]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[g][e] = 0.f;
        }
    }

    // the norm weights of the kinds present in the chunk (vector loads, once per warp)
    float wq[8], wk[8];
    const bool has_q = j0 < p.nh, has_k = j0 < p.nh + p.nkv && j0 + nj > p.nh;
    if (p.do_norm && p.wq && has_q) R::load(p.wq, sub, wq);
    if (p.do_norm && p.wk && has_k) R::load(p.wk, sub, wk);

    // cos and sin of this lane's elements at position pos0 + t; the sine carries the sign of the
    // rotate-half partner (-x[i + hd/2] in the first half), so the rotation is two FMAs
    float cs[8], sn[8];
    if (p.do_rope && (has_q || has_k)) {
        if (p.cos_sin) {
            const float *row = p.cos_sin + (size_t)t * 2 * HD;
            R::load(row, sub, cs);
            R::load(row + HD, sub, sn);
        } else {
            // slots e and e + 4 share the frequency of element 4 * sub + e
            const float pf = (float)(p.pos0 + t);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                rope_angle_cos_sin(pf, p.inv_freq[4 * sub + e], cs[e], sn[e]);
                cs[e + 4] = cs[e];
                sn[e + 4] = sn[e];
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sn[e] = -sn[e];
    }

#pragma unroll
    for (int g = 0; g < RG; ++g) {
        const int job = j0 + g * RPI + rsub;
        const int kind = job < p.nh ? 0 : job < p.nh + p.nkv ? 1 : 2;
        float *xr = x[g];
        if (p.do_norm) {
            float rn;
            if constexpr (MODE == kOutFp32) {
                // the exact path: the sum of squares and the scale in fp64 (one scale per row),
                // so a canvas key's scale -- which moves every score of that key, by up to
                // |s| * 2^-22 from a 2-ulp rsqrtf at |s| ~ 60 -- carries only its final rounding
                double ss = 0.0;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fma((double)xr[e], (double)xr[e], ss);
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                rn = (float)(1.0 / sqrt(ss / (double)HD + (double)p.eps));
            } else {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(xr[e], xr[e], ss);
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                rn = rsqrtf(ss * (1.0f / (float)HD) + p.eps);
            }
            const bool use_q = kind == 0 && p.wq, use_k = kind == 1 && p.wk;
            if (use_q || use_k) {
#pragma unroll
                for (int e = 0; e < 8; ++e) xr[e] = (xr[e] * rn) * (use_q ? wq[e] : wk[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xr[e] *= rn;
            }
        }
        if (p.do_rope && kind != 2) {
            float part[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) part[e] = xr[e ^ 4];
#pragma unroll
            for (int e = 0; e < 8; ++e) xr[e] = fmaf(xr[e], cs[e], part[e] * sn[e]);
        }
    }

    // the operand arrays are read by the previous forward's attention kernel until it ends
    if (p.inputs_resident && !p.other_set) pdl_wait();

#pragma unroll
    for (int g = 0; g < RG; ++g) {
        const int r = g * RPI + rsub;
        if (r >= nj) continue;
        const int job = j0 + r;
        const int kind = job < p.nh ? 0 : job < p.nh + p.nkv ? 1 : 2;
        const int head = kind == 0 ? job : kind == 1 ? job - p.nh : job - p.nh - p.nkv;
        const float *xr = x[g];
        if constexpr (MODE == kOutFp32) {
            float *dst = kind == 0 ? p.q_out + ((size_t)t * p.nh + head) * HD
                       : kind == 1 ? p.k_out + ((size_t)t * p.nkv + head) * HD
                                   : p.v_out + ((size_t)t * p.nkv + head) * HD;
            R::store(dst, sub, x[g]);
        } else {
            if (kind == 2) {
                __half v[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const __half2 h = __floats2half2_rn(xr[e], xr[e + 1]);
                    v[e] = h.x;
                    v[e + 1] = h.y;
                }
                R::template store_16<__half, __half2>(p.vh + ((size_t)head * p.S + p.ctx + t) * HD,
                                                      sub, v);
            } else {
                // q-hat is scaled by log2(e) (one fp32 rounding) so that the tensor-core kernel
                // gets its scores in the log2 units of its exponentials
                const float sc = kind == 0 ? 1.4426950408889634f : 1.0f;
                // hi = bf16(y), lo = bf16(y - hi), two elements per conversion
                __nv_bfloat16 hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float y0 = xr[e] * sc, y1 = xr[e + 1] * sc;
                    const __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
                    const float2 hf = __bfloat1622float2(h);
                    const __nv_bfloat162 l = __floats2bfloat162_rn(y0 - hf.x, y1 - hf.y);
                    hi[e] = h.x; hi[e + 1] = h.y;
                    lo[e] = l.x; lo[e + 1] = l.y;
                }
                if (kind == 0) {
                    // Q hi row-interleaved (the attention kernel's threads load it into TMEM);
                    // Q lo likewise when it goes to TMEM, else row-major for TMA
                    const int gk = head / G, Rw = t * G + head % G;
                    const size_t tile = ((size_t)gk * (p.rows_pad / 128) + Rw / 128) * HD * 128;
                    store_q_interleaved<HD>(p.qh + tile, Rw % 128, sub, hi);
                    if (p.ql_interleaved)
                        store_q_interleaved<HD>(p.ql + tile, Rw % 128, sub, lo);
                    else
                        R::template store_16<__nv_bfloat16, __nv_bfloat162>(
                            p.ql + ((size_t)gk * p.rows_pad + Rw) * HD, sub, lo);
                } else {
                    const size_t off = ((size_t)head * p.S + p.ctx + t) * HD;
                    R::template store_16<__nv_bfloat16, __nv_bfloat162>(p.kh + off, sub, hi);
                    R::template store_16<__nv_bfloat16, __nv_bfloat162>(p.kl + off, sub, lo);
                }
            }
        }
    }
    // With the other operand set nothing above waited.  One thread waits here, so that this grid
    // completes only after the kernel ahead of it: the attention kernel that follows relies on
    // that before it writes the output and partial buffers the one ahead also writes.
    if (p.other_set && p.inputs_resident && blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
}

// The cos|sin table of the canvas positions pos0 .. pos0 + T - 1: row t = cos(hd) | sin(hd), both
// halves of each equal, one thread per (t, frequency).
__global__ void rope_table_kernel(float *cs, const float4 *inv_freq, int T, int hd, long long pos0)
{
    const int half = hd / 2;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * half) return;
    const int t = (int)(i / half), k = (int)(i % half);
    float c, s;
    rope_angle_cos_sin((float)(pos0 + t), inv_freq[k], c, s);
    float *row = cs + (size_t)t * 2 * hd;
    row[k] = c;
    row[k + half] = c;
    row[hd + k] = s;
    row[hd + k + half] = s;
}

template <int HD>
cudaError_t launch_hd(const NormRopeParams &p, int mode, cudaStream_t s, size_t smem_bytes)
{
    const int jobs = p.nh + 2 * p.nkv;
    const int chunks = (jobs + kChunkRows<HD> - 1) / kChunkRows<HD>;
    const long long warps = (long long)p.T * chunks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + 3) / 4 + p.cache_blocks));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (mode == kOutFp32) return cudaLaunchKernelEx(&cfg, norm_rope_kernel<HD, kOutFp32>, p, chunks);
    if constexpr (HD >= 64) {
        return cudaLaunchKernelEx(&cfg, norm_rope_kernel<HD, kOutTc>, p, chunks);
    } else {
        return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_rope_table(float *cs, const float4 *inv_freq, int T, int hd, long long pos0,
                              cudaStream_t s)
{
    const long long n = (long long)T * (hd / 2);
    rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cs, inv_freq, T, hd, pos0);
    return cudaGetLastError();
}

cudaError_t launch_norm_rope(const NormRopeParams &p, int hd, int mode, cudaStream_t s,
                             size_t smem_bytes)
{
    switch (hd) {
    case 32: return launch_hd<32>(p, mode, s, smem_bytes);
    case 64: return launch_hd<64>(p, mode, s, smem_bytes);
    case 128: return launch_hd<128>(p, mode, s, smem_bytes);
    case 256: return launch_hd<256>(p, mode, s, smem_bytes);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
