// attn_tc_kernel.cuh -- tensor-core attention for the canvas block (page "inferencelayer 0.2.3,
// src/diffusion_gemma_gpu.rs", item DG_ATTN: GQA bidirectional attention, scaling 1.0, no mask,
// keys = [cache | canvas] of kv head g = h / (nh/nkv)), written for sm_103a.
//
// Work unit: one CTA per (128-row query tile, kv group, key-range partition) with the split
// schedule (2..8 partitions of a query tile form a thread-block cluster and merge in the kernel);
// with the stream-K schedule one CTA per SM, each an equal run of key tiles over the (query tile,
// kv group) pairs in order, so a CTA may hold the end of one pair and the start of the next (two
// "pieces", merged afterwards by the combine kernel).  The G query heads of a kv group are packed
// into the MMA M dimension (row R = t*G + h mod G), so each K/V tile is staged once for all of
// them.
//
// Precision (scores reach |s| ~ 90 because of scaling 1.0, so one TF32 rounding of q or k moves
// outputs by ~1e-2): Q.K^T is computed as  qh.kh + qh.kl + ql.kh  with bf16 hi/lo splits of both
// operands (three kind::f16 MMAs, ~16 significant bits per operand).  P.V runs with P and V
// rounded to fp16: the same 10 explicit mantissa bits as TF32 with round to nearest, P <= 2^15 and
// the normed V well inside the fp16 range, at twice the TF32 rate and half the bytes of V.
// K and V tiles are read by every query tile of their kv group, and the cache part by every
// forward of a denoising loop: their loads carry an L2 evict-last policy.
//
// Roles (32 * (7 + NQI) threads):
//   warp 0   K producer: TMA of the K hi/lo tile into a KST-deep ring (and the Q lo tile when it
//            lives in shared memory);
//   warp 1   P.V issuer and TMEM owner;
//   warp 2   V producer: TMA of the fp16 V tile ([keys, hd], an MN-major operand) into a
//            VST-deep ring of VK-key stages;
//   warp 3, 8.. Q.K^T issuers.  Key tiles are dealt round-robin to NQI issuers; issuer q owns
//            the score buffers and K ring slots of the tiles j = q (mod NQI), so every mbarrier
//            keeps a single in-order consumer.
//            An issuing warp runs its loop as a whole (warp-uniform indices and descriptors) and
//            one elected lane issues the tcgen05 instructions: from a lone lane in a divergent
//            branch the same 48 MMAs of a tile took ~40% longer to hand over, and at NK = 64
//            that hand-over, not the tensor pipe, set the pace of the loop;
//   warps 4-7 softmax: thread = one query row = one TMEM lane.  They put Q into TMEM, turn each
//            score tile S (TMEM) into P = 2^(s*log2e - m) rounded to fp16, packed two per column
//            over the start of S, keep the fp32 running max m and the denominator l (the sum of
//            those fp16 values), rescale O in TMEM when the max has grown by more than 15 (log2
//            units; so P <= 2^15 in between), and write the output.
// TMEM: O [128 x hd] fp32, Q hi (bf16 pairs), Q lo (hd <= 128), NSP score/probability buffers.
// hd = 256 uses 64-key score tiles in two buffers (TMEM holds 128 columns for them): the product
// ql.kh takes its Q lo operand from shared memory (4 KiB per k-step), so wider tiles read it
// fewer times per key; 16- and 32-key tiles in 8 and 4 buffers were slower.
// Every mbarrier wait is bounded; a wait that runs out sets a status bit and the CTA unwinds.
#pragma once
#include "dg_internal.cuh"
#include "sm103_ptx.cuh"

namespace dg {
namespace {

// A score chunk of W columns (32 or 16) from TMEM, and its fp16 probabilities (W/2 columns) back.
template <int W> __device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[W])
{
    if constexpr (W == 32) tmem_ld32(taddr, r);
    else tmem_ld16(taddr, r);
}
template <int W> __device__ __forceinline__ void tmem_st_half_chunk(uint32_t taddr, const uint32_t *r)
{
    if constexpr (W == 32) tmem_st16(taddr, r);
    else tmem_st8(taddr, r);
}

template <int HD> struct Cfg;
template <> struct Cfg<256> {
    static constexpr int NK = 64, VK = 32, NSP = 2, KST = 2, VST = 2, NQI = 1;
    static constexpr bool QL_TMEM = false;
    static constexpr int O_COL = 0, QH_COL = 256, QL_COL = 0, SP_COL = 384;
};
template <> struct Cfg<128> {
    static constexpr int NK = 64, VK = 64, NSP = 4, KST = 4, VST = 4, NQI = 2;
    static constexpr bool QL_TMEM = true;
    static constexpr int O_COL = 0, QH_COL = 128, QL_COL = 192, SP_COL = 256;
};
template <> struct Cfg<64> {
    static constexpr int NK = 128, VK = 128, NSP = 3, KST = 3, VST = 3, NQI = 1;
    static constexpr bool QL_TMEM = true;
    static constexpr int O_COL = 0, QH_COL = 64, QL_COL = 96, SP_COL = 128;
};

template <int HD> struct Layout {
    using C = Cfg<HD>;
    static constexpr int KPANELS = HD / 64;                 // 128-byte bf16 panels of a K row
    static constexpr int VPANELS = HD / 64;                 // 128-byte fp16 panels of a V row
    static constexpr int QL_BYTES = C::QL_TMEM ? 0 : kTileM * HD * 2;
    static constexpr int KPANEL_BYTES = C::NK * 128;
    static constexpr int KSTAGE_BYTES = 2 * KPANELS * KPANEL_BYTES;   // hi + lo
    static constexpr int VPANEL_BYTES = C::VK * 128;       // VK key rows of 64 hd values
    static constexpr int VSTAGE_BYTES = VPANELS * VPANEL_BYTES;
    static constexpr int K_OFF = QL_BYTES;
    static constexpr int V_OFF = K_OFF + C::KST * KSTAGE_BYTES;
    static constexpr int BAR_OFF = V_OFF + C::VST * VSTAGE_BYTES;
    static constexpr int NBARS = 2 * C::KST + 2 * C::VST + 3 * C::NSP + 5 + (C::NQI + 1);
    static constexpr int THREADS = 32 * (7 + C::NQI);
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + TMEM slot + alignment
    // In-cluster combine, once every MMA has completed (operand rings free): O of the tile
    // (row pitch HD + 4 floats: a float4 store per lane is conflict-free), the (m, l) of each
    // row, the merge weights and output row pointers of the rows this CTA writes.
    static constexpr int STG_PITCH = HD + 4;
    static constexpr int ML_OFF = kTileM * STG_PITCH * 4;
    static constexpr int WGT_OFF = ML_OFF + kTileM * 8;
    static constexpr int DST_OFF = WGT_OFF + kTileM * kMaxClusterSplits * 4;
    static constexpr int CMB_END = DST_OFF + kTileM * 8;
    static_assert(CMB_END <= BAR_OFF, "combine staging fits below the barriers");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(C::SP_COL + C::NSP * C::NK <= 512, "TMEM budget");
    static_assert(C::NSP % C::NQI == 0 && C::KST % C::NQI == 0, "issuer-owned buffers and slots");
    static_assert(C::NK % C::VK == 0 && C::VK % 16 == 0, "V stages tile a score tile");
};

// log2 units.  Each row's reference m is the row maximum seen at the last rescale (or over the
// first score tile), so it never exceeds the row's running maximum: the largest P of a row is
// >= 1, and every key within 14 of the row maximum gets a normal fp16 P with its full 11-bit
// precision.  Keys further below fall into the fp16 subnormal range, each off by at most 2^-25
// against a denominator >= 1, so even S = 8704 such keys move the weights by at most 2.6e-4
// relative.  O is rescaled when a row's maximum exceeds m + 15, so P <= 2^15 (inside the fp16
// range, 65504) in between.
constexpr float kRescaleThreshold = 15.0f;
constexpr float kHeadroom = 0.0f;

// Four output values as the bf16 hi / lo pair the o_proj GEMM takes (hi = bf16(o),
// lo = bf16(o - hi)), at element i of the two [T, nh*hd] arrays.
__device__ __forceinline__ void store_split4(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t i,
                                             float4 v)
{
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
    *reinterpret_cast<uint2 *>(hi + i) = make_uint2(*reinterpret_cast<const uint32_t *>(&h01),
                                                    *reinterpret_cast<const uint32_t *>(&h23));
    *reinterpret_cast<uint2 *>(lo + i) = make_uint2(*reinterpret_cast<const uint32_t *>(&l01),
                                                    *reinterpret_cast<const uint32_t *>(&l23));
}

// Rows [r0, r0 + nr) of the in-cluster merge of P partitions: out = sum_p w_p O_p with the
// per-row weights w (already divided by the merged denominator).  The peers' staged O rows are
// read through distributed shared memory, whose latency is long: each thread takes U float4
// columns (of different rows) at once, so U * P loads are in flight per thread.  The CTA's own
// rows (partition `self`) are read through the local shared-memory path.
template <int P, int HD, int THREADS, int PITCH, bool SPLIT>
__device__ __forceinline__ void cluster_merge_rows(uint32_t smem_base, int self, int r0, int nr,
                                                   const float *wgt, float *const *dst,
                                                   const float *out, __nv_bfloat16 *out_hi,
                                                   __nv_bfloat16 *out_lo)
{
    constexpr int V4 = HD / 4;
    constexpr int U = P <= 2 ? 4 : (P <= 4 ? 2 : 1);
    uint32_t peer[P];
#pragma unroll
    for (int q = 0; q < P; ++q) peer[q] = dsmem_map(smem_base, q);
    const int n = nr * V4;
    for (int base = threadIdx.x; base < n; base += U * THREADS) {
        float4 v[U][P];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int item = base + u * THREADS;
            if (item < n) {
                const uint32_t off = (uint32_t)(((r0 + item / V4) * PITCH + 4 * (item % V4)) * 4);
#pragma unroll
                for (int q = 0; q < P; ++q)
                    v[u][q] = q == self ? lds_f4(smem_base + off) : dsmem_ld_f4(peer[q] + off);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int item = base + u * THREADS;
            if (item >= n) continue;
            const int i = item / V4;
            float *d = dst[i];
            if (!d) continue;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const float w = wgt[i * kMaxClusterSplits + q];
                acc.x = fmaf(w, v[u][q].x, acc.x);
                acc.y = fmaf(w, v[u][q].y, acc.y);
                acc.z = fmaf(w, v[u][q].z, acc.z);
                acc.w = fmaf(w, v[u][q].w, acc.w);
            }
            if constexpr (SPLIT)
                store_split4(out_hi, out_lo, (size_t)(d - out) + 4 * (item % V4), acc);
            else
                *reinterpret_cast<float4 *>(d + 4 * (item % V4)) = acc;
        }
    }
}

// SK: the stream-K schedule (a CTA may hold two pieces); its bookkeeping is compiled only into
// that instantiation (it costs the split schedule ~2% at hd = 256 otherwise).  SPLIT (split
// schedule only): the CTAs that write output rows write their bf16 hi / lo split into
// p.out_hi / p.out_lo instead of the fp32 rows (the o_proj GEMM reads only the split; an SM
// sends ~13.5 bytes per cycle, so every byte written counts); an instantiation of its own, since
// even an untaken branch there cost the kernel 1-2.5%.
template <int HD, bool SK, bool SPLIT = false>
__global__ void __launch_bounds__(Layout<HD>::THREADS, 1)
attn_tc_kernel(const __grid_constant__ TcMaps maps, const AttnTcParams p)
{
    using C = Cfg<HD>;
    using Lay = Layout<HD>;
    constexpr int NK = C::NK, NSP = C::NSP, KST = C::KST, VST = C::VST, NQI = C::NQI;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::BAR_OFF);
    uint64_t *k_full = bars;
    uint64_t *k_empty = k_full + KST;
    uint64_t *v_full = k_empty + KST;
    uint64_t *v_empty = v_full + VST;
    uint64_t *s_full = v_empty + VST;
    uint64_t *p_full = s_full + NSP;
    uint64_t *sp_free = p_full + NSP;
    uint64_t *o_final = sp_free + NSP;
    uint64_t *q_full = o_final + 1;
    uint64_t *q_ready = q_full + 1;
    uint64_t *qk_done = q_ready + 1;        // every Q.K^T of the first piece has completed
    uint64_t *o_free = qk_done + 1;         // O of the first piece has been read out of TMEM
    uint64_t *drain = o_free + 1;           // [NQI + 1]: one per MMA-issuing thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + NQI + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;

    // The pieces of work of this CTA, each (query tile qt, kv group g, key tiles [t0, t0 + n)):
    // one with the split schedule; one or two with the stream-K schedule (the end of a pair's
    // key tiles and the start of the next pair's).  All roles walk the same sequence of
    // n_all = n[0] + n[1] tiles; ring slots and barrier phases run on across the two pieces.
    int pq[2] = {0, 0}, pg[2] = {0, 0}, pt0[2] = {0, 0}, pn[2] = {0, 0}, pslot[2] = {0, 0};
    int nseg = 1;
    if constexpr (!SK) {
        pq[0] = blockIdx.x;
        pg[0] = blockIdx.y;
        pslot[0] = blockIdx.z;
        pt0[0] = blockIdx.z * p.tiles_per_split;
        pn[0] = min(p.n_tiles, pt0[0] + p.tiles_per_split) - pt0[0];
    } else {
        const long long U = p.sk_units;
        long long u = sk_begin(blockIdx.x, U, p.sk_ctas);
        const long long u1 = sk_begin(blockIdx.x + 1, U, p.sk_ctas);
        nseg = 0;
        while (u < u1 && nseg < 2) {
            const int pr = (int)(u / p.n_tiles);
            const int t0 = (int)(u - (long long)pr * p.n_tiles);
            const int n = (int)min((long long)(p.n_tiles - t0), u1 - u);
            pq[nseg] = pr % p.qtiles;
            pg[nseg] = pr / p.qtiles;
            pt0[nseg] = t0;
            pn[nseg] = n;
            pslot[nseg] = (int)blockIdx.x - sk_cta_of((long long)pr * p.n_tiles, U, p.sk_ctas);
            ++nseg;
            u += n;
        }
        if (u < u1 && threadIdx.x == 0) atomicOr(p.status, kErrSchedule);
    }
    const int n_all = SK ? pn[0] + pn[1] : pn[0];
    // piece of tile `it` of the sequence, and the tile's index within its pair's key range
    auto piece_of = [&](int it) -> int {
        if constexpr (SK) return it < pn[0] ? 0 : 1;
        else return 0;
    };
    auto key_tile = [&](int it) -> int {
        if constexpr (SK) return it < pn[0] ? pt0[0] + it : pt0[1] + (it - pn[0]);
        else return pt0[0] + it;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < KST; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
        for (int i = 0; i < VST; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
        for (int i = 0; i < NSP; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&sp_free[i], 1);
        }
        mbar_init(o_final, 1);
        mbar_init(q_full, 1);
        mbar_init(q_ready, 128);
        mbar_init(qk_done, NQI);
        mbar_init(o_free, 128);
        for (int i = 0; i <= NQI; ++i) mbar_init(&drain[i], 1);
        fence_mbar_init();
        prefetch_tmap(&maps.kh);
        prefetch_tmap(&maps.kl);
        prefetch_tmap(&maps.vh);
        if (!C::QL_TMEM) prefetch_tmap(&maps.ql);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // The operands are written by the kernel before this one in the stream: every thread waits
    // for it before its role touches them, except that the producers first load the ring stages
    // of cache rows that were complete before that kernel started (keys < p.static_keys).
    // Only after its wait may a thread let the next kernel of the stream be scheduled.  With
    // resident inputs the plan alternates two operand sets, and the next forward's first stage
    // writes the set this kernel does not read without waiting for anything; its start after
    // this point is what guarantees that the attention kernel before this one, the last reader
    // of that set, has finished.
    auto wait_previous = [&]() {
        pdl_wait();
        pdl_launch_dependents();
    };
    // ring stages of this CTA's first tiles whose keys are all such cache rows
    auto static_prefix = [&](int stages, int keys_per_stage) -> int {
        int n = 0;
        const int per_tile = NK / keys_per_stage;
        while (n < stages && n < n_all * per_tile &&
               key_tile(n / per_tile) * NK + (n % per_tile + 1) * keys_per_stage <= p.static_keys)
            ++n;
        return n;
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- K producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            bool ok = true;
            int issued[KST] = {};
            int cur = -1, q_loads = 0;
            auto load_k = [&](int it) {
                const int s = it % KST;
                uint8_t *kst = smem + Lay::K_OFF + s * Lay::KSTAGE_BYTES;
                const int key0 = key_tile(it) * NK, g = pg[piece_of(it)];
                mbar_arrive_expect_tx(&k_full[s], Lay::KSTAGE_BYTES);
                for (int pn = 0; pn < Lay::KPANELS; ++pn) {
                    tma_load_3d_hint(kst + pn * Lay::KPANEL_BYTES, &maps.kh, &k_full[s], pn * 64,
                                     key0, g, pol);
                    tma_load_3d_hint(kst + (Lay::KPANELS + pn) * Lay::KPANEL_BYTES, &maps.kl,
                                     &k_full[s], pn * 64, key0, g, pol);
                }
                ++issued[s];
            };
            const int pre = static_prefix(KST, NK);
            for (int it = 0; it < pre; ++it) load_k(it);
            wait_previous();
            for (int it = 0; it < n_all; ++it) {
                const int sg = piece_of(it), g = pg[sg];
                if (sg != cur) {
                    cur = sg;
                    if (!C::QL_TMEM) {
                        // the Q lo tile of the piece's pair; the second replaces the first once
                        // every Q.K^T of the first piece has completed
                        if (sg > 0 && !mbar_wait_bounded(qk_done, 0, limit)) { ok = false; break; }
                        uint8_t *qls = smem;
                        mbar_arrive_expect_tx(q_full, Lay::QL_BYTES);
                        for (int pn = 0; pn < Lay::KPANELS; ++pn)
                            tma_load_3d(qls + pn * (kTileM * 128), &maps.ql, q_full, pn * 64,
                                        pq[sg] * kTileM, g);
                        ++q_loads;
                    }
                }
                if (it < pre) continue;             // loaded before the wait
                const int s = it % KST;
                if (it >= KST && !mbar_wait_bounded(&k_empty[s], ((it / KST) - 1) & 1, limit)) {
                    ok = false;
                    break;
                }
                load_k(it);
            }
            if (!ok) atomicOr(p.status, kErrWaitProducer);
            // let every load issued by this thread land before the CTA can exit
            for (int s = 0; s < KST; ++s)
                if (issued[s] > 0) mbar_wait_bounded(&k_full[s], (issued[s] - 1) & 1, limit);
            if (q_loads > 0) mbar_wait_bounded(q_full, (q_loads - 1) & 1, limit);
        } else {
            wait_previous();
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------------------- V producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            bool ok = true;
            int issued[VST] = {};
            // VK-key stages, NK/VK of them per score tile
            constexpr int VPT = NK / C::VK;
            auto load_v = [&](int it) {
                const int s = it % VST;
                uint8_t *vst = smem + Lay::V_OFF + s * Lay::VSTAGE_BYTES;
                const int tile = it / VPT;
                const int key0 = key_tile(tile) * NK + (it % VPT) * C::VK;
                const int g = pg[piece_of(tile)];
                mbar_arrive_expect_tx(&v_full[s], Lay::VSTAGE_BYTES);
                for (int pn = 0; pn < Lay::VPANELS; ++pn)
                    tma_load_3d_hint(vst + pn * Lay::VPANEL_BYTES, &maps.vh, &v_full[s], pn * 64,
                                     key0, g, pol);
                ++issued[s];
            };
            const int pre = static_prefix(VST, C::VK);
            for (int it = 0; it < pre; ++it) load_v(it);
            wait_previous();
            for (int it = pre; it < n_all * VPT; ++it) {
                const int s = it % VST;
                if (it >= VST && !mbar_wait_bounded(&v_empty[s], ((it / VST) - 1) & 1, limit)) {
                    ok = false;
                    break;
                }
                load_v(it);
            }
            if (!ok) atomicOr(p.status, kErrWaitProducer);
            for (int s = 0; s < VST; ++s)
                if (issued[s] > 0) mbar_wait_bounded(&v_full[s], (issued[s] - 1) & 1, limit);
        } else {
            wait_previous();
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3 || warp >= 8) {
        // ---------------------------------------------------------------- MMA issuers
        // The whole warp runs the issue loop, so tile indices and descriptors are warp-uniform
        // values; the lane chosen by elect.sync issues every tcgen05 instruction (the same lane
        // each time, so its commits track all of its MMAs).
        wait_previous();
        const uint32_t leader = elect_one_sync();
        constexpr uint32_t idesc_qk = make_idesc(1, 0, 0, kTileM, NK);
        constexpr uint32_t idesc_pv = make_idesc(0, 0, 1, kTileM, HD);   // fp16, B MN-major
        const uint32_t t_o = tbase + C::O_COL;
        const uint32_t t_qh = tbase + C::QH_COL;
        const uint32_t t_ql = tbase + C::QL_COL;
        const uint32_t t_sp = tbase + C::SP_COL;
        // Descriptors are built once; per stage / k-step only the start address moves
        // (the 14-bit address field cannot carry: shared addresses are < 256 KiB).
        const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + Lay::K_OFF), 16, 1024);
        // V is MN-major: 64-wide hd panels VK rows apart (leading offset), 8-key groups 1 KiB
        // apart (stride offset)
        const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + Lay::V_OFF), Lay::VPANEL_BYTES, 1024);
        const uint64_t qdesc0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
        const int me = warp == 1 ? 0 : 1 + (warp == 3 ? 0 : warp - 7);   // drain slot
        bool ok = true;
        if (warp == 1) {
            // P.V, in tile order: O += P_i V_i
            constexpr int VPT = NK / C::VK;                 // V stages per score tile
            for (int i = 0; ok && i < n_all; ++i) {
                const int b = i % NSP;
                const int sg = piece_of(i), first = sg == 0 ? 0 : pn[0];
                if (sg > 0 && i == first) {
                    // the second piece accumulates into O afresh once the first piece's O has
                    // been read out
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_free, 0, limit));
                    if (!ok) break;
                    tc_fence_after();
                }
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&p_full[b], (i / NSP) & 1, limit));
                for (int h = 0; ok && h < VPT; ++h) {
                    const int c = i * VPT + h, vs = c % VST;
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&v_full[vs], (c / VST) & 1, limit));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vd = vdesc0 + (uint64_t)((vs * Lay::VSTAGE_BYTES) >> 4);
#pragma unroll
                    for (int ks = 0; ks < C::VK / 16; ++ks) {
                        // keys 16ks..16ks+15 of the stage: two 8-row groups, 2 KiB into every
                        // hd panel; the P columns of key 16k start at 8k
                        const uint64_t bdesc = vd + (uint64_t)((ks * 16 * 128) >> 4);
                        const int kk = h * (C::VK / 16) + ks;
                        mma_bf16_ts_by(leader, t_o, t_sp + b * NK + kk * 8, bdesc, idesc_pv,
                                       (i > first || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_by(leader, &v_empty[vs]);
                }
                if (!ok) break;
                mma_commit_by(leader, &sp_free[b]);
                // O of a piece is complete after its last tile (o_final completes once per piece)
                if (i == first + pn[sg] - 1) mma_commit_by(leader, o_final);
            }
        } else {
            // Q.K^T of the tiles j = q (mod NQI): S_j = qh.kh + qh.kl + ql.kh
            const int q = warp == 3 ? 0 : warp - 7;
            int next_q = 0;                     // next phase of q_ready / q_full to wait for
            bool done0 = false;                 // qk_done committed
            for (int j = q; ok && j < n_all; j += NQI) {
                const int sg = piece_of(j);
                // Q of the piece's pair (hi, and lo when it lives in TMEM, in TMEM; lo in shared
                // memory otherwise).  Phases are waited for in order: a parity wait for phase 1
                // would pass while phase 0 is still open.  Before the second piece, every
                // Q.K^T of the first issued here is committed to qk_done (Q may be replaced once
                // they complete).
                for (; ok && next_q <= sg; ++next_q) {
                    if (next_q > 0 && !done0) {
                        mma_commit_by(leader, qk_done);
                        done0 = true;
                    }
                    ok = mbar_wait_bounded(q_ready, next_q & 1, limit);
                    if (ok && !C::QL_TMEM) ok = mbar_wait_bounded(q_full, next_q & 1, limit);
                    ok = __all_sync(0xffffffffu, ok);
                    tc_fence_after();
                }
                if (!ok) break;
                const int b = j % NSP, s = j % KST;
                if (j >= NSP) ok = mbar_wait_bounded(&sp_free[b], ((j / NSP) - 1) & 1, limit);
                if (ok) ok = mbar_wait_bounded(&k_full[s], (j / KST) & 1, limit);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint64_t kd = kdesc0 + (uint64_t)((s * Lay::KSTAGE_BYTES) >> 4);
                const uint32_t d = t_sp + b * NK;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const int pn = kk >> 2, sub = kk & 3;
                    const uint64_t bh = kd + (uint64_t)((pn * Lay::KPANEL_BYTES + sub * 32) >> 4);
                    const uint64_t bl = kd + (uint64_t)(((Lay::KPANELS + pn) * Lay::KPANEL_BYTES + sub * 32) >> 4);
                    mma_bf16_ts_by(leader, d, t_qh + kk * 8, bh, idesc_qk, kk > 0 ? 1u : 0u);
                    mma_bf16_ts_by(leader, d, t_qh + kk * 8, bl, idesc_qk, 1u);
                    if constexpr (C::QL_TMEM) {
                        mma_bf16_ts_by(leader, d, t_ql + kk * 8, bh, idesc_qk, 1u);
                    } else {
                        const uint64_t ad = qdesc0 + (uint64_t)((pn * (kTileM * 128) + sub * 32) >> 4);
                        mma_bf16_ss_by(leader, d, ad, bh, idesc_qk, 1u);
                    }
                }
                mma_commit_by(leader, &k_empty[s]);
                mma_commit_by(leader, &s_full[b]);
            }
            if (ok && nseg > 1 && !done0) mma_commit_by(leader, qk_done);
        }
        if (!ok && leader) atomicOr(p.status, kErrWaitMma);
        // no tcgen05 operation of this warp may still run when TMEM is released
        mma_commit_by(leader, &drain[me]);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&drain[me], 0, limit)) && leader)
            atomicOr(p.status, kErrWaitDrain);
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ---------------------------------------------------------------- softmax / epilogue
        wait_previous();
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                  // tile row == TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        bool ok = true;
        // Scores arrive in log2 units: the first stage scaled q-hat by log2(e) before its
        // hi/lo split, so P = 2^(s - m) needs no multiply here.
        float m_used = -INFINITY;
        float2 l2 = make_float2(0.f, 0.f);   // running denominator, two partial sums

        // A stream-K piece's result (O unnormalised, once o_final of the piece has completed):
        // its (m, l) per row, and its O rows row-interleaved per 128-row tile (16-byte unit u of
        // row r at u * 128 + r), so every store instruction of a warp writes 512 contiguous
        // bytes straight from the TMEM registers (no shared memory: the rings may be busy with
        // the next piece).
        auto write_piece = [&](int sg, float m, float l) {
            const size_t prow = ((size_t)pslot[sg] * p.nkv + pg[sg]) * p.rows_pad;
            p.part_ml[prow + (size_t)pq[sg] * kTileM + r] = make_float2(m, l);
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + (prow + (size_t)pq[sg] * kTileM) * HD) + r;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(tbase + lane_off + C::O_COL + 32 * c, orr);
                tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    dst[(size_t)(8 * c + v) * kTileM] =
                        make_float4(__uint_as_float(orr[4 * v]), __uint_as_float(orr[4 * v + 1]),
                                    __uint_as_float(orr[4 * v + 2]), __uint_as_float(orr[4 * v + 3]));
            }
        };

        for (int sg = 0; ok && sg < nseg; ++sg) {
            const int qt = pq[sg], g = pg[sg];
            const int base = sg == 0 ? 0 : pn[0];               // first tile of the piece in the CTA
            const int nloc = pn[sg], tile0 = pt0[sg];
            if (sg > 0) {
                // Q of the second pair replaces the first once every Q.K^T of the first piece is done
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(qk_done, 0, limit));
                if (!ok) break;
                tc_fence_after();
            }

            // Q hi (and Q lo) rows into TMEM: HD bf16 = HD/2 32-bit columns each.  Every load of the
            // row is issued before the first TMEM store (one memory round trip, not one per chunk).
            {
                // the operand is row-interleaved: 16-byte unit u of tile row r at (tile*HD/8 + u)*128
                // + r, so each load instruction of a warp reads 512 contiguous bytes
                constexpr int NCH = (HD / 64) * (C::QL_TMEM ? 2 : 1);   // 32-column chunks
                const size_t tile = ((size_t)g * (p.rows_pad / kTileM) + qt) * (HD / 8) * kTileM;
                const uint4 *src_h = reinterpret_cast<const uint4 *>(p.qh) + tile + r;
                const uint4 *src_l = reinterpret_cast<const uint4 *>(p.ql) + tile + r;
                uint4 w[NCH][8];
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        w[c][v] = c < HD / 64 ? src_h[(c * 8 + v) * kTileM]
                                              : src_l[((c - HD / 64) * 8 + v) * kTileM];
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    uint32_t u[32];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        u[4 * v] = w[c][v].x; u[4 * v + 1] = w[c][v].y;
                        u[4 * v + 2] = w[c][v].z; u[4 * v + 3] = w[c][v].w;
                    }
                    const int col = c < HD / 64 ? C::QH_COL + 32 * c : C::QL_COL + 32 * (c - HD / 64);
                    tmem_st32(tbase + lane_off + col, u);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(q_ready);
            }
            if (sg > 0) {
                // the first piece's O goes out while the tensor pipe starts on the second piece's
                // scores; then the second piece's P.V may overwrite O
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_final, 0, limit));
                if (!ok) break;
                tc_fence_after();
                write_piece(0, m_used, l2.x + l2.y);
                tc_fence_before();
                mbar_arrive(o_free);
            }
            m_used = -INFINITY;
            l2 = make_float2(0.f, 0.f);
            // The reference starts at -inf: the first score tile of the piece takes the rescale
            // branch below with alpha = 0 and sets it from that tile's maximum (a separate pass
            // over the first tile for its maximum cost an extra read of the tile).
            for (int it = base; ok && it < base + nloc; ++it) {
                const int b = it % NSP;
                ok = mbar_wait_bounded(&s_full[b], (it / NSP) & 1, limit);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }   // TMEM access is warp-wide
                tc_fence_after();
                const uint32_t tsp = tbase + lane_off + C::SP_COL + b * NK;
                // The whole score row stays in registers (one pass over TMEM) when the register
                // budget allows: always at NK <= 64, and at NK = 128 with 256 threads (~194
                // registers; at hd = 64 this single pass took the kernel from 137.7 to 109.3 us
                // on the 4-canvas workload).  Otherwise the maximum is taken in a first pass and
                // the scores are read again.
                constexpr bool ROW_REGS = NK <= 64 || Lay::THREADS <= 256;
                constexpr int CW = NK % 32 == 0 ? 32 : 16;            // columns per score chunk
                constexpr int RC = ROW_REGS ? NK / CW : 1;
                uint32_t sr[RC][CW];
                // keys of this tile below S; only the last tile of the key range is partial, so the
                // masking branch is warp-uniform and almost never taken
                const int valid = p.S - (tile0 + (it - base)) * NK;
                float mx;
                if constexpr (ROW_REGS) {
#pragma unroll
                    for (int c = 0; c < RC; ++c) tmem_ld_chunk<CW>(tsp + CW * c, sr[c]);
                    tmem_wait_ld();
                    if (valid < NK) {
#pragma unroll
                        for (int c = 0; c < RC; ++c)
#pragma unroll
                            for (int i = 0; i < CW; ++i)
                                if (CW * c + i >= valid) sr[c][i] = __float_as_uint(-INFINITY);
                    }
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < RC; ++c)
#pragma unroll
                        for (int i = 0; i < CW; i += 2)
                            m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], __uint_as_float(sr[c][i]),
                                                     __uint_as_float(sr[c][i + 1]));
                    mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
                } else {
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
                    for (int c = 0; c < NK / 32; ++c) {
                        tmem_ld32(tsp + 32 * c, sr[0]);
                        tmem_wait_ld();
                        if (32 * c + 32 > valid) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (32 * c + i >= valid) sr[0][i] = __float_as_uint(-INFINITY);
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], __uint_as_float(sr[0][i]),
                                                     __uint_as_float(sr[0][i + 1]));
                    }
                    mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
                }
                const bool need = mx > m_used + kRescaleThreshold;
                // A rescale moves the reference first and P of this tile is computed against the
                // new one; O (in TMEM) is scaled only afterwards, once the previous P.V product
                // has landed -- by then it usually has, so the softmax does not stall on it.
                float alpha = 1.0f;
                bool rescale_o = false;
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = fmaxf(m_used, mx + kHeadroom);
                    alpha = exp2f(m_used - m_new);          // 0 while nothing is accumulated
                    l2 = mul_f32x2(l2, make_float2(alpha, alpha));
                    m_used = m_new;
                    rescale_o = it > base;                  // warp-uniform
                }
                // P in fp16, two keys per 32-bit column, written over the start of the score buffer
                // (chunk c of 32 scores lands in columns 16c..16c+15, already read).  The denominator
                // sums the same fp16 values that P.V multiplies (widened exactly), so numerator and
                // denominator carry one set of roundings: a single dominant key returns its V.
                const float2 mm = make_float2(m_used, m_used);
                if constexpr (ROW_REGS) {
#pragma unroll
                    for (int c = 0; c < RC; ++c) {
                        uint32_t pw[CW / 2];
#pragma unroll
                        for (int i = 0; i < CW / 2; ++i) {
                            const float2 d = sub_f32x2(make_float2(__uint_as_float(sr[c][2 * i]),
                                                                   __uint_as_float(sr[c][2 * i + 1])), mm);
                            const __half2 h = __floats2half2_rn(ex2_approx(d.x), ex2_approx(d.y));
                            pw[i] = *reinterpret_cast<const uint32_t *>(&h);
                            add_f16x2_to_f32x2(l2, pw[i]);
                        }
                        tmem_st_half_chunk<CW>(tsp + (CW / 2) * c, pw);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < NK / 32; ++c) {
                        tmem_ld32(tsp + 32 * c, sr[0]);
                        tmem_wait_ld();
                        if (32 * c + 32 > valid) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (32 * c + i >= valid) sr[0][i] = __float_as_uint(-INFINITY);
                        }
                        uint32_t pw[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 d = sub_f32x2(make_float2(__uint_as_float(sr[0][2 * i]),
                                                                   __uint_as_float(sr[0][2 * i + 1])), mm);
                            const __half2 h = __floats2half2_rn(ex2_approx(d.x), ex2_approx(d.y));
                            pw[i] = *reinterpret_cast<const uint32_t *>(&h);
                            add_f16x2_to_f32x2(l2, pw[i]);
                        }
                        tmem_st16(tsp + 16 * c, pw);
                    }
                }
                tmem_wait_st();
                if (rescale_o) {
                    // O is only touched once the previous P.V product (buffer (it-1) mod NSP) has
                    // landed; two 32-column chunks per round trip to TMEM
                    const int pb = (it - 1) % NSP;
                    if (!mbar_wait_bounded(&sp_free[pb], ((it - 1) / NSP) & 1, limit)) ok = false;
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                    for (int c = 0; c < HD / 32; c += 2) {
                        uint32_t o0[32], o1[32];
                        tmem_ld32(tbase + lane_off + C::O_COL + 32 * c, o0);
                        tmem_ld32(tbase + lane_off + C::O_COL + 32 * c + 32, o1);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 x0 = mul_f32x2(
                                make_float2(__uint_as_float(o0[i]), __uint_as_float(o0[i + 1])), a2);
                            const float2 x1 = mul_f32x2(
                                make_float2(__uint_as_float(o1[i]), __uint_as_float(o1[i + 1])), a2);
                            o0[i] = __float_as_uint(x0.x);
                            o0[i + 1] = __float_as_uint(x0.y);
                            o1[i] = __float_as_uint(x1.x);
                            o1[i + 1] = __float_as_uint(x1.y);
                        }
                        tmem_st32(tbase + lane_off + C::O_COL + 32 * c, o0);
                        tmem_st32(tbase + lane_off + C::O_COL + 32 * c + 32, o1);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                if (!(p.inject_stall && it == 0)) mbar_arrive(&p_full[b]);
            }
        }   // pieces
        const float l_run = l2.x + l2.y;
        if (ok && !mbar_wait_bounded(o_final, (nseg - 1) & 1, limit)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) atomicOr(p.status, kErrWaitSoftmax);
        } else if (SK) {
            tc_fence_after();
            write_piece(nseg - 1, m_used, l_run);
        } else {
            tc_fence_after();
            const int qt = pq[0], g = pg[0], split = pslot[0];
            const int Rg = qt * kTileM + r;                 // packed row in the group
            // Every MMA has completed, so the K ring is free: each warp stages its 32 rows x 32
            // columns of O in a shared-memory tile (row pitch 36 floats, conflict-free for float4)
            // and writes it back row-contiguous: a store instruction covers 128 bytes of each of
            // 4 output rows.  Each lane computes its own row's destination once.
            if (p.cluster_combine) {
                // unnormalised O row and its (m, l), for the merge across the cluster
                float *stg = reinterpret_cast<float *>(smem) + r * Lay::STG_PITCH;
                reinterpret_cast<float2 *>(smem + Lay::ML_OFF)[r] = make_float2(m_used, l_run);
#pragma unroll 1
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(tbase + lane_off + C::O_COL + 32 * c, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        *reinterpret_cast<float4 *>(stg + 32 * c + 4 * v) =
                            make_float4(__uint_as_float(orr[4 * v]), __uint_as_float(orr[4 * v + 1]),
                                        __uint_as_float(orr[4 * v + 2]), __uint_as_float(orr[4 * v + 3]));
                }
            } else {
            float *stage = reinterpret_cast<float *>(smem + Lay::K_OFF) + quarter * (32 * 36);
            float scale;
            float *mydst = nullptr;
            if (p.splits == 1) {
                scale = 1.0f / l_run;
                if (Rg < p.rows) {
                    const int t = Rg / p.G, h = g * p.G + Rg % p.G;
                    mydst = p.out + ((size_t)t * p.nh + h) * HD;
                }
            } else {
                scale = 1.0f;
                const size_t row = ((size_t)split * p.nkv + g) * p.rows_pad + Rg;
                if (Rg < p.rows) {
                    p.part_ml[row] = make_float2(m_used, l_run);
                    mydst = p.part_o + row * HD;
                }
            }
            const int sub = lane & 7, rsub = lane >> 3;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(tbase + lane_off + C::O_COL + 32 * c, orr);
                tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    *reinterpret_cast<float4 *>(stage + lane * 36 + 4 * v) =
                        make_float4(__uint_as_float(orr[4 * v]) * scale,
                                    __uint_as_float(orr[4 * v + 1]) * scale,
                                    __uint_as_float(orr[4 * v + 2]) * scale,
                                    __uint_as_float(orr[4 * v + 3]) * scale);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 4 * k + rsub;
                    float *d = reinterpret_cast<float *>(
                        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mydst), j));
                    if (d) {
                        const float4 o4 = *reinterpret_cast<const float4 *>(stage + j * 36 + 4 * sub);
                        if constexpr (SPLIT)
                            store_split4(p.out_hi, p.out_lo,
                                         (size_t)(d - p.out) + 32 * c + 4 * sub, o4);
                        else
                            *reinterpret_cast<float4 *>(d + 32 * c + 4 * sub) = o4;
                    }
                }
                __syncwarp();
            }
            }
        }
    }

    if (p.cluster_combine) {
        // The splits CTAs of this query tile are one cluster.  After the barrier every CTA's
        // staged O and (m, l) are visible cluster-wide; CTA k merges rows [k*128/P, (k+1)*128/P):
        //   out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p,
        // reading the P partial rows through distributed shared memory, in partition order.
        __syncwarp();
        cluster_sync_all();
        const int P = p.splits;
        const int rank = (int)cluster_ctarank();
        const int r0 = rank * kTileM / P, r1 = (rank + 1) * kTileM / P, nr = r1 - r0;
        float *wgt = reinterpret_cast<float *>(smem + Lay::WGT_OFF);
        float **dst = reinterpret_cast<float **>(smem + Lay::DST_OFF);
        const uint32_t ml_base = smem_u32(smem + Lay::ML_OFF);
        if ((int)threadIdx.x < nr) {
            const int i = threadIdx.x, r = r0 + i;
            float m[kMaxClusterSplits], l[kMaxClusterSplits];
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplits; ++q) {
                if (q < P) {
                    const float2 v = dsmem_ld_f2(dsmem_map(ml_base + r * 8, q));
                    m[q] = v.x;
                    l[q] = v.y;
                    M = fmaxf(M, v.x);
                }
            }
            float L = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplits; ++q) {
                if (q < P) {
                    m[q] = exp2f(m[q] - M);
                    L += l[q] * m[q];
                }
            }
            const float inv = 1.0f / L;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplits; ++q)
                if (q < P) wgt[i * kMaxClusterSplits + q] = m[q] * inv;
            const int Rg = pq[0] * kTileM + r;
            dst[i] = Rg < p.rows ? p.out + ((size_t)(Rg / p.G) * p.nh + pg[0] * p.G + Rg % p.G) * HD
                                 : nullptr;
        }
        __syncthreads();
        const uint32_t sb = smem_u32(smem);
        constexpr int TH = Lay::THREADS, PI = Lay::STG_PITCH;
        float *const o = p.out;
        __nv_bfloat16 *const oh = p.out_hi, *const ol = p.out_lo;
        constexpr bool SP = SPLIT;
        switch (P) {
        case 2: cluster_merge_rows<2, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        case 3: cluster_merge_rows<3, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        case 4: cluster_merge_rows<4, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        case 5: cluster_merge_rows<5, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        case 6: cluster_merge_rows<6, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        case 7: cluster_merge_rows<7, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        default: cluster_merge_rows<8, HD, TH, PI, SP>(sb, rank, r0, nr, wgt, dst, o, oh, ol); break;
        }
        // no CTA leaves (or frees its shared memory) while a peer may still read it
        cluster_sync_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace
}  // namespace dg
