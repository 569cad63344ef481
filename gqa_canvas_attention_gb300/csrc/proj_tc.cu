// proj_tc.cu -- the step before the attention block on the tensor cores (page "inferencelayer
// 0.2.3, src/diffusion_gemma_gpu.rs", canvas_forward, attention branch): the input RMSNorm of the
// residual stream (`rms!(&cur, &l.ln_in, 1, &nb)`, item DG_RMSNORM), the q / k / v projections
// (`gemm!` on GLin weights: y = x W^T, W stored [n, k]; with no value projection, v is the raw k
// projection), and then -- fused into the GEMM's epilogue -- the block's own first stage (the
// per-head qk-norm + NeoX RoPE and the weightless v-norm of DG_HEADNORM_ROPE), written straight
// into the attention kernel's operand arrays.
//
// Precision: fp32 inputs and weights.  The input norm's per-token scale r_t = (mean x^2 + eps)^-1/2
// is applied in the epilogue; the norm weight is folded into W once (W' = W diag(ln_w), one fp32
// rounding).  x and W' are split into bf16 hi/lo pairs and the product is taken as
// x_hi W'_hi + x_hi W'_lo + x_lo W'_hi (three kind::f16 MMAs, fp32 accumulation in TMEM), about
// 16 significant bits per operand, as in the attention kernel's scores.
//
// Work unit: one CTA per (128 tokens, 128 output columns).  Columns are taken in groups of 64
// (one 128-byte swizzled panel of W rows).  A CTA holds two groups whose columns are RoPE partners
// (i and i + hd/2): hd = 128 -> one head; hd = 256 -> half a head (groups c and c + 2), the two
// halves of a head being a cluster of 2 CTAs that exchange one partial sum of squares per token.
// Roles: warp 0 TMA producer (6-stage ring), warp 1 MMA issuer and TMEM owner, warps 2-9
// epilogue (two threads per token row = TMEM lane, each taking half of the columns).  Every
// mbarrier wait is bounded.
//
// Every kernel here is launched with programmatic dependent launch: after its own set-up it waits
// for the kernel before it (pdl_wait) and only then lets the next kernel of the stream be
// scheduled, so launches and set-ups overlap the tail of the kernel ahead.  Because no kernel
// signals before its wait, everything enqueued ahead of a kernel's predecessor has completed
// by the time the kernel starts: the GEMM producers rely on that when they request the prepared
// weights before their own wait.  A kernel is launched only once every CTA of the one before it
// has started, so CTAs scheduled early never keep that one from running.
#include "dg_internal.cuh"
#include "sm103_ptx.cuh"

namespace dg {
namespace {

// Steps of 32 along the contraction (64-byte swizzled rows), six stages deep: with the
// producer refilling a slot only once the MMAs that read it have completed, the ring must hold
// enough steps ahead to cover the load latency (three 64-wide steps measured 2 kcycles a step).
constexpr int kProjStages = 6;
constexpr int kProjThreads = 192;                         // o_proj: producer, MMA, 4 epilogue warps
constexpr int kQkvThreads = 320;                          // projection: producer, MMA, 8 epilogue warps
constexpr int kStepK = 32;
constexpr int kPanelBytes = kTileM * kStepK * 2;            // 128 rows x 32 bf16
constexpr int kStageBytes = 4 * kPanelBytes;                // A hi, A lo, B hi, B lo
constexpr int kProjBarOff = kProjStages * kStageBytes;
constexpr int kProjSmem = kProjBarOff + 256 + 1536 + 1024;  // barriers, sum exchange, alignment

__global__ void __launch_bounds__(256) hidden_prep_kernel(ProjPrepParams p)
{
    // one CTA per token row: r_t and the bf16 hi/lo split of the row (each thread's loads of the
    // row are issued together)
    __shared__ float red[8];
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x;
    const float4 *x = reinterpret_cast<const float4 *>(p.x + (size_t)t * p.H);
    uint2 *xh = reinterpret_cast<uint2 *>(p.xh + (size_t)t * p.H);
    uint2 *xl = reinterpret_cast<uint2 *>(p.xl + (size_t)t * p.H);
    float ss = 0.f;
#pragma unroll 4
    for (int i = threadIdx.x; i < p.H / 4; i += 256) {
        const float4 v = x[i];
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
        uint2 uh, ul;
        uh.x = *reinterpret_cast<const uint32_t *>(&h01);
        uh.y = *reinterpret_cast<const uint32_t *>(&h23);
        ul.x = *reinterpret_cast<const uint32_t *>(&l01);
        ul.y = *reinterpret_cast<const uint32_t *>(&l23);
        xh[i] = uh;
        xl[i] = ul;
    }
    if (!p.rin) return;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int w = 0; w < 8; ++w) tot += red[w];
        p.rin[t] = rsqrtf(tot / (float)p.H + p.eps);
    }
}

__global__ void __launch_bounds__(256) proj_weights_kernel(ProjWeightParams p)
{
    // W' = W diag(ln_w) split into bf16 hi/lo, rows in the order q | k | v
    const size_t n4 = (size_t)p.n_rows * p.H / 4;
    const int h4 = p.H / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / h4;
        const int c4 = (int)(i % h4);
        const float *src = row < (size_t)p.nq ? p.wq + row * p.H
                         : row < (size_t)(p.nq + p.nk) ? p.wk + (row - p.nq) * p.H
                                                       : p.wv + (row - p.nq - p.nk) * p.H;
        float4 v = reinterpret_cast<const float4 *>(src)[c4];
        if (p.ln_w) {
            const float4 w = reinterpret_cast<const float4 *>(p.ln_w)[c4];
            v.x *= w.x; v.y *= w.y; v.z *= w.z; v.w *= w.w;
        }
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
        uint2 uh, ul;
        uh.x = *reinterpret_cast<const uint32_t *>(&h01);
        uh.y = *reinterpret_cast<const uint32_t *>(&h23);
        ul.x = *reinterpret_cast<const uint32_t *>(&l01);
        ul.y = *reinterpret_cast<const uint32_t *>(&l23);
        reinterpret_cast<uint2 *>(p.wh)[i] = uh;
        reinterpret_cast<uint2 *>(p.wl)[i] = ul;
    }
}

// N values of a token row as bf16 into 2N contiguous bytes.
template <int N>
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16 *dst, const float *v)
{
#pragma unroll
    for (int u = 0; u < N / 8; ++u) {
        uint4 w;
        uint32_t *pw = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * u + 2 * e], v[8 * u + 2 * e + 1]);
            pw[e] = *reinterpret_cast<const uint32_t *>(&h);
        }
        reinterpret_cast<uint4 *>(dst)[u] = w;
    }
}

// The bf16 hi/lo split of N values: hi = bf16(v) (exact in fp32), lo = v - hi (rounded to bf16
// when stored).
template <int N>
__device__ __forceinline__ void split_n(const float *v, float *hi, float *lo)
{
#pragma unroll
    for (int e = 0; e < N; e += 2) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[e], v[e + 1]);
        const float2 f = __bfloat1622float2(h);
        hi[e] = f.x;
        hi[e + 1] = f.y;
        lo[e] = v[e] - f.x;
        lo[e + 1] = v[e + 1] - f.y;
    }
}

// The q operand's row-interleaved layout (see the first-stage kernel): 16-byte unit u of tile
// row r at (tile * hd/8 + u) * 128 + r.  Writes the N/8 units of N columns starting at c0.
template <int N>
__device__ __forceinline__ void store_q_rows(__nv_bfloat16 *tile_base, int r, int c0, const float *v)
{
    uint4 *base = reinterpret_cast<uint4 *>(tile_base);
#pragma unroll
    for (int u = 0; u < N / 8; ++u) {
        uint4 w;
        uint32_t *pw = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * u + 2 * e], v[8 * u + 2 * e + 1]);
            pw[e] = *reinterpret_cast<const uint32_t *>(&h);
        }
        base[(size_t)(c0 / 8 + u) * kTileM + r] = w;
    }
}

// ---- the bf16x3 split GEMM main loop shared by the two projection kernels ----
// D[128 x 128] (TMEM, fp32) = sum over H of A_hi B_hi + A_hi B_lo + A_lo B_hi, A rows m0..m0+127
// of maps.xh / maps.xl, B rows brow0..brow0+63 and brow1..brow1+63 of maps.wh / maps.wl, in
// kStepK-wide steps of the contraction through a kProjStages ring.

// TMA producer (one thread): returns false when a wait ran out.  The weights were prepared
// before the kernel ahead of this one started, so the first stages' W panels are requested
// before this thread waits for that kernel (pdl_wait), and the activation panels after it.
__device__ __forceinline__ bool gemm_load_loop(uint8_t *smem, uint64_t *full, uint64_t *empty,
                                               const ProjMaps &maps, int m0, int brow0, int brow1,
                                               int nk, uint64_t limit, int b_rows = 128)
{
    // brow1 >= 0: two boxes of 64 W rows; brow1 < 0: one box of b_rows rows from brow0
    const uint32_t tx = 2 * kPanelBytes + 2 * (uint32_t)b_rows * kStepK * 2;
    auto load_w = [&](int it) {
        const int s = it % kProjStages, k0 = it * kStepK;
        uint8_t *st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], tx);
        tma_load_3d(st + 2 * kPanelBytes, &maps.wh, &full[s], k0, brow0, 0);
        tma_load_3d(st + 3 * kPanelBytes, &maps.wl, &full[s], k0, brow0, 0);
        if (brow1 >= 0) {
            tma_load_3d(st + 2 * kPanelBytes + kPanelBytes / 2, &maps.wh, &full[s], k0, brow1, 0);
            tma_load_3d(st + 3 * kPanelBytes + kPanelBytes / 2, &maps.wl, &full[s], k0, brow1, 0);
        }
    };
    const int pre = nk < kProjStages ? nk : kProjStages;
    for (int it = 0; it < pre; ++it) load_w(it);
    pdl_wait();
    bool ok = true;
    int issued[kProjStages] = {};
    for (int it = 0; it < nk; ++it) {
        const int s = it % kProjStages;
        if (it >= pre) {
            if (!mbar_wait_bounded(&empty[s], ((it / kProjStages) - 1) & 1, limit)) {
                ok = false;
                break;
            }
            load_w(it);
        }
        uint8_t *st = smem + s * kStageBytes;
        const int k0 = it * kStepK;
        tma_load_3d(st, &maps.xh, &full[s], k0, m0, 0);
        tma_load_3d(st + kPanelBytes, &maps.xl, &full[s], k0, m0, 0);
        ++issued[s];
    }
    // let every load issued here land before the CTA can exit
    for (int s = 0; s < kProjStages; ++s)
        if (issued[s] > 0) mbar_wait_bounded(&full[s], (issued[s] - 1) & 1, limit);
    return ok;
}

// MMA issuer (a whole warp: warp-uniform loop and descriptors, one elected lane issues the
// tcgen05 instructions): accumulates into tacc, signals acc_full; drains before returning.
// Returns a DG status bit, or 0 (the same in every lane).
template <int N = 128>
__device__ __forceinline__ uint32_t gemm_mma_loop(uint8_t *smem, uint64_t *full, uint64_t *empty,
                                                  uint64_t *acc_full, uint64_t *drain,
                                                  uint32_t tacc, int nk, uint64_t limit)
{
    constexpr uint32_t idesc = make_idesc(1, 0, 0, kTileM, N);
    const uint32_t leader = elect_one_sync();
    const uint64_t d0 = smem_desc_sw64(smem_u32(smem));
    uint32_t err = 0;
    bool ok = true;
    for (int it = 0; ok && it < nk; ++it) {
        const int s = it % kProjStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (it / kProjStages) & 1, limit));
        if (!ok) break;
        tc_fence_after();
        const uint64_t base = d0 + (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
        for (int sub = 0; sub < kStepK / 16; ++sub) {
            const uint64_t ah = base + (uint64_t)((sub * 32) >> 4);
            const uint64_t al = base + (uint64_t)((kPanelBytes + sub * 32) >> 4);
            const uint64_t bh = base + (uint64_t)((2 * kPanelBytes + sub * 32) >> 4);
            const uint64_t bl = base + (uint64_t)((3 * kPanelBytes + sub * 32) >> 4);
            mma_bf16_ss_by(leader, tacc, ah, bh, idesc, (it > 0 || sub > 0) ? 1u : 0u);
            mma_bf16_ss_by(leader, tacc, ah, bl, idesc, 1u);
            mma_bf16_ss_by(leader, tacc, al, bh, idesc, 1u);
        }
        mma_commit_by(leader, &empty[s]);
    }
    if (ok) mma_commit_by(leader, acc_full);
    else err |= kErrWaitMma;
    mma_commit_by(leader, drain);   // no tcgen05 operation of this warp may still run when TMEM goes
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(drain, 0, limit))) err |= kErrWaitDrain;
    return err;
}

template <int HD>
__global__ void __launch_bounds__(kQkvThreads, 1)
qkv_proj_kernel(const __grid_constant__ ProjMaps maps, const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kProjBarOff);
    uint64_t *full = bars;
    uint64_t *empty = full + kProjStages;
    uint64_t *acc_full = empty + kProjStages;
    uint64_t *drain = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    float *ss_ex = reinterpret_cast<float *>(smem + kProjBarOff + 256);   // [128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const int m0 = blockIdx.y * kTileM;
    const int j = blockIdx.x;
    // the two column groups of this CTA (RoPE partners) and the head they belong to
    const int head = HD == 256 ? j / 2 : j;
    const int g0 = HD == 256 ? 4 * head + (j & 1) : 2 * head;
    const int g1 = g0 + HD / 128;
    const int c0 = (g0 % (HD / 64)) * 64;                    // first column of g0 in its head
    const int nk = p.H / kStepK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kProjStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
        prefetch_tmap(&maps.xh);
        prefetch_tmap(&maps.xl);
        prefetch_tmap(&maps.wh);
        prefetch_tmap(&maps.wl);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tacc = *tmem_slot;
    // (the producer thread waits inside gemm_load_loop, after its weight requests)
    if (warp != 0) {
        pdl_wait();
        pdl_launch_dependents();
    }

    // Epilogue: eight warps, two per TMEM lane quarter.  Thread (row r, half h) takes columns
    // 32h..32h+31 of each of the two groups (RoPE partners stay in one thread).
    constexpr int CW = 32;
    float a[CW], b[CW];           // the token row's values of groups g0 and g1 (this half)
    float ss_local = 0.f;
    bool epi_ok = false;
    const int half = warp >= 2 ? (warp - 2) >> 2 : 0;
    float *ss_part = ss_ex + kTileM;                         // [2][128] per-half partial sums

    if (warp == 0) {
        if (lane == 0 && !gemm_load_loop(smem, full, empty, maps, m0, g0 * 64, g1 * 64, nk, limit))
            atomicOr(p.status, kErrWaitProducer);
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t e = gemm_mma_loop(smem, full, empty, acc_full, drain, tacc, nk, limit);
        if (e && lane == 0) atomicOr(p.status, e);
        __syncwarp();
    } else {
        // part 1: accumulator columns into registers, input-norm scale, partial sum of squares
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(acc_full, 0, limit));
        if (ok && head < p.nh + p.nkv) {
            // Every MMA has completed, so the operand ring is free: the eight warps copy the cos
            // and sin of columns c0..c0+63 of the tile's 128 rows into it with row-contiguous
            // loads (two 256-byte rows per warp instruction); the rotation below reads them back
            // (row pitch 68 floats, conflict-free for float4), ordered by the barrier that follows.
            // 4096 float4 over 256 threads: each thread's 16 loads are all issued before its
            // first store (one memory round trip, not sixteen)
            float *cs_s = reinterpret_cast<float *>(smem);
            constexpr int kItems = kTileM * 2 * 16 / 256;
            float4 v[kItems];
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const int it = (int)threadIdx.x - 64 + 256 * k;
                const int row = it >> 5, w = (it >> 4) & 1, q4 = it & 15;
                const int tt = m0 + row;
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tt < p.T)
                    v[k] = *reinterpret_cast<const float4 *>(p.cos_sin + (size_t)tt * 2 * HD +
                                                             w * HD + c0 + 4 * q4);
            }
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const int it = (int)threadIdx.x - 64 + 256 * k;
                const int row = it >> 5, w = (it >> 4) & 1, q4 = it & 15;
                *reinterpret_cast<float4 *>(cs_s + (row * 2 + w) * 68 + 4 * q4) = v[k];
            }
        }
        if (ok) {
            tc_fence_after();
            uint32_t u[32];
            tmem_ld32(tacc + lane_off + CW * half, u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < CW; ++i) a[i] = __uint_as_float(u[i]);
            tmem_ld32(tacc + lane_off + 64 + CW * half, u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < CW; ++i) b[i] = __uint_as_float(u[i]);
            const int t = m0 + r;
            const float rs = t < p.T ? p.rin[t] : 0.f;
#pragma unroll
            for (int i = 0; i < CW; ++i) {
                a[i] *= rs;
                b[i] *= rs;
                ss_local = fmaf(a[i], a[i], fmaf(b[i], b[i], ss_local));
            }
            epi_ok = true;
        } else if (lane == 0) {
            atomicOr(p.status, kErrWaitSoftmax);
        }
        ss_part[half * kTileM + r] = ss_local;
        named_barrier_sync(1, 256);                          // the eight epilogue warps
        if (half == 0) ss_ex[r] = ss_part[r] + ss_part[kTileM + r];
    }

    // hd = 256: the two halves of a head exchange their partial sums of squares
    if constexpr (HD == 256) {
        __syncwarp();
        cluster_sync_all();
    } else {
        __syncthreads();
    }

    if (warp >= 2 && epi_ok) {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int t = m0 + r;
        float ss = ss_ex[r];
        if constexpr (HD == 256)
            ss += dsmem_ld_f32(dsmem_map(smem_u32(&ss_ex[r]), cluster_ctarank() ^ 1u));
        const float rn = rsqrtf(ss / (float)HD + p.eps);
        const int nq = p.nh, nkh = p.nkv;
        const int kind = head < nq ? 0 : head < nq + nkh ? 1 : 2;   // q, k, v
        const int hh = kind == 0 ? head : kind == 1 ? head - nq : head - nq - nkh;
        const int ca = c0 + CW * half, cb = ca + HD / 2;         // first columns (in the head)
        if (t < p.T) {
            // v-hat: the weightless, un-roped norm (of the k projection when v is not projected)
            if (kind == 2 || (kind == 1 && p.kv_shared)) {
                __half *vrow = p.vh + ((size_t)hh * p.S + p.ctx + t) * HD;
#pragma unroll
                for (int u = 0; u < CW / 8; ++u) {
                    uint4 wa, wb;
                    uint32_t *pa = reinterpret_cast<uint32_t *>(&wa);
                    uint32_t *pb = reinterpret_cast<uint32_t *>(&wb);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 8 * u + 2 * e;
                        const __half2 ha = __floats2half2_rn(a[i] * rn, a[i + 1] * rn);
                        const __half2 hb = __floats2half2_rn(b[i] * rn, b[i + 1] * rn);
                        pa[e] = *reinterpret_cast<const uint32_t *>(&ha);
                        pb[e] = *reinterpret_cast<const uint32_t *>(&hb);
                    }
                    reinterpret_cast<uint4 *>(vrow + ca)[u] = wa;
                    reinterpret_cast<uint4 *>(vrow + cb)[u] = wb;
                }
            }
            if (kind < 2) {
                // q-hat / k-hat: norm, weight, NeoX rotation of the pairs (ca + i, cb + i)
                const float *w = kind == 0 ? p.wq_norm : p.wk_norm;
                // this row's cos / sin of columns ca.., staged in shared memory above
                const float *cs = reinterpret_cast<const float *>(smem) + r * 2 * 68 + CW * half;
                const float sc = kind == 0 ? 1.4426950408889634f : 1.0f;   // q in log2 units
#pragma unroll
                for (int i = 0; i < CW; i += 4) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(cs + i);
                    const float4 s4 = *reinterpret_cast<const float4 *>(cs + 68 + i);
                    float4 wa = make_float4(1.f, 1.f, 1.f, 1.f), wb = wa;
                    if (w) {
                        wa = *reinterpret_cast<const float4 *>(w + ca + i);
                        wb = *reinterpret_cast<const float4 *>(w + cb + i);
                    }
                    const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
                    const float ww[4] = {wa.x, wa.y, wa.z, wa.w}, vv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float ya = a[i + e] * rn * ww[e], yb = b[i + e] * rn * vv[e];
                        a[i + e] = fmaf(ya, cc[e], -yb * sn[e]) * sc;
                        b[i + e] = fmaf(yb, cc[e], ya * sn[e]) * sc;
                    }
                }
                float hi[CW], lo[CW];
                if (kind == 0) {
                    const int g = hh / p.G, R = t * p.G + hh % p.G;
                    const size_t tile = ((size_t)g * (p.rows_pad / kTileM) + R / kTileM) * HD * kTileM;
                    const size_t qrow = ((size_t)g * p.rows_pad + R) * HD;
                    split_n<CW>(a, hi, lo);
                    store_q_rows<CW>(p.qh + tile, R % kTileM, ca, hi);
                    if (p.ql_interleaved) store_q_rows<CW>(p.ql + tile, R % kTileM, ca, lo);
                    else store_bf16_row<CW>(p.ql + qrow + ca, lo);
                    split_n<CW>(b, hi, lo);
                    store_q_rows<CW>(p.qh + tile, R % kTileM, cb, hi);
                    if (p.ql_interleaved) store_q_rows<CW>(p.ql + tile, R % kTileM, cb, lo);
                    else store_bf16_row<CW>(p.ql + qrow + cb, lo);
                } else {
                    const size_t row = ((size_t)hh * p.S + p.ctx + t) * HD;
                    split_n<CW>(a, hi, lo);
                    store_bf16_row<CW>(p.kh + row + ca, hi);
                    store_bf16_row<CW>(p.kl + row + ca, lo);
                    split_n<CW>(b, hi, lo);
                    store_bf16_row<CW>(p.kh + row + cb, hi);
                    store_bf16_row<CW>(p.kl + row + cb, lo);
                }
            }
        }
    }

    // no CTA leaves while its peer may still read its partial sums; TMEM is released last
    if constexpr (HD == 256) {
        __syncwarp();
        cluster_sync_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tacc, 128);
    }
}

// The step after the block: y = attn W_o^T (the same split GEMM: A = the attention output, B = W_o,
// one CTA per 128 tokens x N output columns, N chosen per H so that the CTAs fill the GPU), y and
// its partial sums of squares to memory; the
// post-attention RMSNorm needs the whole row of H columns, so it and the residual add run in
// post_norm_kernel.
template <int N>
__global__ void __launch_bounds__(kProjThreads, 1)
oproj_kernel(const __grid_constant__ ProjMaps maps, const OprojParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kProjBarOff);
    uint64_t *full = bars;
    uint64_t *empty = full + kProjStages;
    uint64_t *acc_full = empty + kProjStages;
    uint64_t *drain = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const int m0 = blockIdx.y * kTileM, n0 = blockIdx.x * N;
    const int nk = p.K / kStepK;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kProjStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
        prefetch_tmap(&maps.xh);
        prefetch_tmap(&maps.xl);
        prefetch_tmap(&maps.wh);
        prefetch_tmap(&maps.wl);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tacc = *tmem_slot;
    // (the producer thread waits inside gemm_load_loop, after its weight requests)
    if (warp != 0) {
        pdl_wait();
        pdl_launch_dependents();
    }

    if (warp == 0) {
        if (lane == 0 && !gemm_load_loop(smem, full, empty, maps, m0, n0, -1, nk, limit, N))
            atomicOr(p.status, kErrWaitProducer);
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t e = gemm_mma_loop<N>(smem, full, empty, acc_full, drain, tacc, nk, limit);
        if (e && lane == 0) atomicOr(p.status, e);
        __syncwarp();
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int t = m0 + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(acc_full, 0, limit));
        if (ok) {
            tc_fence_after();
            float ss = 0.f;
            // Every MMA has completed, so the operand ring is free: each warp stages 16 columns
            // of its 32 rows at a time (row pitch 20 floats, conflict-free for float4) and writes
            // them back row-contiguous, 8 rows x 64 bytes per store instruction.
            float *stage = reinterpret_cast<float *>(smem) + quarter * (32 * 20);
            const int j0 = lane >> 2, q4 = lane & 3;
#pragma unroll 1
            for (int c = 0; c < N / 16; ++c) {
                uint32_t u[16];
                tmem_ld16(tacc + lane_off + 16 * c, u);
                tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 f = make_float4(__uint_as_float(u[4 * v]), __uint_as_float(u[4 * v + 1]),
                                                 __uint_as_float(u[4 * v + 2]), __uint_as_float(u[4 * v + 3]));
                    ss = fmaf(f.x, f.x, fmaf(f.y, f.y, fmaf(f.z, f.z, fmaf(f.w, f.w, ss))));
                    *reinterpret_cast<float4 *>(stage + lane * 20 + 4 * v) = f;
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int jr = 8 * k + j0;                     // row of the warp's 32
                    const int tr = m0 + quarter * 32 + jr;
                    if (tr < p.T)
                        *reinterpret_cast<float4 *>(p.y + (size_t)tr * p.H + n0 + 16 * c + 4 * q4) =
                            *reinterpret_cast<const float4 *>(stage + jr * 20 + 4 * q4);
                }
                __syncwarp();
            }
            if (t < p.T) p.part_ss[(size_t)t * gridDim.x + blockIdx.x] = ss;
        } else if (lane == 0) {
            atomicOr(p.status, kErrWaitSoftmax);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tacc, 128);
    }
}

// resid = (resid + y (mean y^2 + eps)^-1/2 w) * scale, one CTA per token row.
__global__ void __launch_bounds__(256) post_norm_kernel(PostNormParams p)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    float ss = 0.f;     // every warp sums the row's partial sums itself
    for (int i = lane; i < p.n_tiles; i += 32) ss += p.part_ss[(size_t)t * p.n_tiles + i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rn = rsqrtf(ss / (float)p.H + p.eps);
    const float4 *y = reinterpret_cast<const float4 *>(p.y + (size_t)t * p.H);
    float4 *x = reinterpret_cast<float4 *>(p.resid + (size_t)t * p.H);
    const float4 *w = reinterpret_cast<const float4 *>(p.w);
#pragma unroll 4
    for (int i = threadIdx.x; i < p.H / 4; i += 256) {
        const float4 a = y[i];
        float4 r = x[i];
        const float4 ww = w ? w[i] : make_float4(1.f, 1.f, 1.f, 1.f);
        r.x = (r.x + a.x * rn * ww.x) * p.scale;
        r.y = (r.y + a.y * rn * ww.y) * p.scale;
        r.z = (r.z + a.z * rn * ww.z) * p.scale;
        r.w = (r.w + a.w * rn * ww.w) * p.scale;
        x[i] = r;
    }
}

template <int HD>
cudaError_t launch_proj_hd(const ProjParams &p, const ProjMaps &maps, int n_tiles, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_tiles, p.rows_pad_tokens / kTileM);
    cfg.blockDim = dim3(kQkvThreads);
    cfg.dynamicSmemBytes = kProjSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = HD == 256 ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = HD == 256 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, qkv_proj_kernel<HD>, maps, p);
}

}  // namespace

cudaError_t proj_prepare_attrs()
{
    cudaError_t e = cudaFuncSetAttribute(qkv_proj_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(qkv_proj_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kProjSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(oproj_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kProjSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(oproj_kernel<80>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kProjSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(oproj_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kProjSmem);
    return e;
}

int oproj_tile_n(int H, int T, int num_sms)
{
    // the column tile giving the fewest waves x columns per CTA (time per CTA ~ its columns)
    const int opts[3] = {128, 80, 64};
    int best = 0;
    long long best_cost = -1;
    for (int n : opts) {
        if (H % n) continue;
        const long long ctas = (long long)(H / n) * ((T + kTileM - 1) / kTileM);
        const long long cost = ((ctas + num_sms - 1) / num_sms) * n;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = n;
        }
    }
    return best;
}

// A launch configuration with programmatic dependent launch on stream s.
static cudaLaunchConfig_t pdl_config(dim3 grid, int threads, size_t smem, cudaStream_t s,
                                     cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t launch_oproj(const OprojParams &p, const ProjMaps &maps, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        pdl_config(dim3(p.H / p.tile_n, (p.T + kTileM - 1) / kTileM), kProjThreads, kProjSmem, s, attr);
    switch (p.tile_n) {
    case 128: return cudaLaunchKernelEx(&cfg, oproj_kernel<128>, maps, p);
    case 80: return cudaLaunchKernelEx(&cfg, oproj_kernel<80>, maps, p);
    case 64: return cudaLaunchKernelEx(&cfg, oproj_kernel<64>, maps, p);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_post_norm(const PostNormParams &p, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(dim3(p.T), 256, 0, s, attr);
    return cudaLaunchKernelEx(&cfg, post_norm_kernel, p);
}

cudaError_t launch_hidden_prep(const ProjPrepParams &p, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(dim3(p.T), 256, 0, s, attr);
    return cudaLaunchKernelEx(&cfg, hidden_prep_kernel, p);
}

cudaError_t launch_proj_weights(const ProjWeightParams &p, cudaStream_t s)
{
    const size_t n4 = (size_t)p.n_rows * p.H / 4;
    int blocks = (int)((n4 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    proj_weights_kernel<<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_qkv_proj(const ProjParams &p, const ProjMaps &maps, int hd, int n_tiles,
                            cudaStream_t s)
{
    switch (hd) {
    case 128: return launch_proj_hd<128>(p, maps, n_tiles, s);
    case 256: return launch_proj_hd<256>(p, maps, n_tiles, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
