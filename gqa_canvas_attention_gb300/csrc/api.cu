// api.cu -- the C ABI of libdgattn.so (declared in include/dg_attn.h): plan creation and scratch
// layout, argument checks, TMA descriptor set-up, the choice of key-range partitions, and the
// enqueueing of the kernels of one forward on the caller's stream.
//
// The plan's scratch, all device-resident and allocated once at creation:
//   inv_freq  [hd/2] float4        theta^(-2i/hd) in fp64, held exactly as the sum of three floats
//   fp32 path: q_hat [T, nh, hd], k_hat / v_hat [T, nkv, hd]
//   tensor-core path: Q hi/lo bf16 [nkv, rows_pad, hd] (row R = t*G + h mod G, padded to 128),
//             K hi/lo bf16 [nkv, S, hd] (S = ctx + T) with the cache in rows 0..ctx-1 and the
//             canvas in rows ctx..ctx+T-1; V in fp16, same layout; with DG_OPT_INPUTS_RESIDENT
//             a second set of these five arrays, the forwards alternating between the two
//   partials  O [splits, nkv, rows_pad, hd] and (m, l) [splits, nkv, rows_pad]
//   status    one uint32 that kernels OR their wait failures into
#include "../../include/dg_attn.h"
#include "dg_internal.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <new>
#include <utility>
#include <vector>

namespace {

thread_local char g_last_error[512] = "";
// devices on which the projection kernels' shared-memory opt-in has been made
std::atomic<unsigned long long> g_proj_attrs{0};

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

int cuda_fail(cudaError_t e, const char *what)
{
    set_error("%s: %s", what, cudaGetErrorString(e));
    return DG_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A buffer as the byte range [p, p + bytes) (p may be NULL: no range).
struct Range {
    const void *p;
    size_t bytes;
};

bool overlap(Range a, Range b)
{
    if (!a.p || !b.p || !a.bytes || !b.bytes) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
    return x < y + b.bytes && y < x + a.bytes;
}

// DG_ERR_ARG when an output range overlaps an input range or another output.
int check_no_overlap(std::initializer_list<Range> outs, std::initializer_list<Range> ins)
{
    for (auto o = outs.begin(); o != outs.end(); ++o) {
        for (const Range &i : ins)
            if (overlap(*o, i)) {
                set_error("an output buffer overlaps an input buffer");
                return DG_ERR_ARG;
            }
        for (auto o2 = o + 1; o2 != outs.end(); ++o2)
            if (overlap(*o, *o2)) {
                set_error("two output buffers overlap");
                return DG_ERR_ARG;
            }
    }
    return DG_OK;
}

// The driver's tensor-map encoder, looked up once (a function-local static: its initialisation
// is thread-safe, so plans may be created from several host threads at once).
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
    }();
    return fn;
}

// 3-D tiled map over [d2][d1][d0] (rows of `row` elements, row >= d0) with a 128-byte
// swizzle; box {b0, b1, 1}; reads outside the dims return zeros.
bool encode_3d(CUtensorMap *m, CUtensorMapDataType dt, int esize, void *base, uint64_t d0,
               uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint64_t row,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B)
{
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {row * esize, row * d1 * esize};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The operand arrays the first stage writes and the tensor-core attention kernel reads, with the
// kernel's tensor maps over them.
struct OperandSet {
    __nv_bfloat16 *qh, *ql;      // [nkv, rows_pad, hd] q-hat bf16 hi / lo (kernel layouts)
    __nv_bfloat16 *kh, *kl;      // [nkv, S, hd] k-hat bf16 hi / lo: cache rows, then canvas rows
    __half *vh;                  // [nkv, S, hd] v-hat fp16
    dg::TcMaps maps;
};

}  // namespace

struct dg_attn_plan {
    int nh, nkv, hd, ctx, T, G, S, S_pad, rows, rows_pad;
    float eps, theta;
    long long pos0;
    int path;
    int splits_opt;
    int schedule_opt;            // DG_SCHEDULE_AUTO / _SPLIT / _STREAM_K
    long long wait_limit_ms;
    int profile;
    int inject_stall;
    int inputs_resident;
    int device, num_sms;
    int smem_per_sm, smem_reserved;     // shared memory of an SM, reserved per block
    int attn_ctas;                      // CTAs of the last tensor-core attention launch
    bool tc_ok;
    // clusters of s CTAs (s = 2..8) the tensor-core kernel can hold at once (0: not launchable)
    int max_clusters[dg::kMaxClusterSplits + 1];
    // scratch
    float4 *inv_freq;
    float *rope_cs;              // [T, 2*hd] cos|sin of the positions pos0 .. pos0 + T - 1
    bool rope_dirty;             // rope_cs does not hold the current pos0 yet
    uint32_t *status;
    float *q32, *k32, *v32;
    // Tensor-core operands: `op` is the set the next attention kernel reads.  With resident
    // inputs a second set `alt` is allocated and each forward swaps the two, so that a forward's
    // first stage writes the set the previous forward's attention kernel is not reading.
    OperandSet op, alt;
    bool alt_cache;              // alt holds the prepared cache rows too
    // A cache conversion was enqueued after the last attention kernel.  The attention kernel
    // loads cache rows before its dependency wait only when they were written before the kernel
    // ahead of it started, which the first-stage kernel (it signals before it waits) does not
    // guarantee for a conversion right before it: the next attention kernel waits first.
    bool cache_fresh;
    unsigned long long attn_launched;   // tensor-core attention kernels enqueued
    float *part_o;
    float2 *part_ml;
    int part_capacity;           // partitions the partial buffers hold
    size_t scratch_bytes;
    // prepared cache
    bool cache_ready;
    const float *prep_k, *prep_v;   // fp32 path: the caller's buffers, or c32k / c32v
    float *c32k, *c32v;             // fp32 path: copy of a 16-bit cache (made on first need)
    dg::TcMaps maps;
    // profiling: per stage, pairs of events (start, stop) recorded around launches
    std::vector<cudaEvent_t> ev[6];
    size_t ev_used[6];
    // projection step (dg_attn_proj_prepare / dg_attn_forward_hidden)
    int H;                          // hidden size the projection weights were prepared for
    int proj_rows;                  // rows of W: (nh + nkv [+ nkv]) * hd
    bool kv_shared;                 // no value projection: v is the raw k projection
    bool proj_ready;
    __nv_bfloat16 *wh, *wl;         // [proj_rows, H] W diag(ln_in_w), bf16 hi / lo
    __nv_bfloat16 *xh, *xl;         // [T_pad, H] the residual stream, bf16 hi / lo
    float *rin;                     // [T] input-norm scale
    dg::ProjMaps pmaps;
    // o_proj step (dg_attn_oproj_prepare / dg_attn_oproj_residual / dg_attn_forward_layer)
    int oH;                         // hidden size W_o was prepared for
    int otile;                      // o_proj output columns per CTA
    bool oproj_ready, has_ln_post;
    bool split_attn;                // the attention variant writing aoh / aol is set up (hd 128, 256)
    __nv_bfloat16 *woh, *wol;       // [oH, nh*hd] W_o, bf16 hi / lo
    __nv_bfloat16 *aoh, *aol;       // [T_pad, nh*hd] the attention output, bf16 hi / lo
    float *ybuf, *part_ss;          // [T, oH] the projection, [T, oH/128] its partial sums
    float *ln_post;                 // [oH] post-attention norm weight
    float *attn_buf;                // [T, nh*hd] the block's output inside dg_attn_forward_layer
    dg::ProjMaps omaps;
};

namespace {

void *dalloc(dg_attn_plan *p, size_t bytes, cudaError_t &err)
{
    if (err != cudaSuccess || bytes == 0) return nullptr;
    void *ptr = nullptr;
    err = cudaMalloc(&ptr, bytes);
    if (err == cudaSuccess) {
        p->scratch_bytes += bytes;
        err = cudaMemset(ptr, 0, bytes);
    }
    return ptr;
}

void free_scratch(dg_attn_plan *p)
{
    void *ptrs[] = {p->woh, p->wol, p->aoh, p->aol, p->ybuf, p->part_ss, p->ln_post, p->attn_buf,
                    p->wh, p->wl, p->xh, p->xl, p->rin, p->c32k, p->c32v, p->inv_freq, p->rope_cs,
                    p->status, p->q32, p->k32, p->v32, p->op.qh, p->op.ql, p->op.kh, p->op.kl,
                    p->op.vh, p->alt.qh, p->alt.ql, p->alt.kh, p->alt.kl, p->alt.vh, p->part_o,
                    p->part_ml};
    for (void *x : ptrs)
        if (x) cudaFree(x);
    for (auto &v : p->ev) {
        for (cudaEvent_t e : v) cudaEventDestroy(e);
        v.clear();
    }
}

int n_tiles_for(const dg_attn_plan *p)
{
    if (p->path == DG_PATH_TC) {
        const int nk = dg::tc_geometry(p->hd).nk;
        return (p->S + nk - 1) / nk;
    }
    return (p->S + 31) / 32;
}

int qtiles_for(const dg_attn_plan *p)
{
    const int tm = p->path == DG_PATH_TC ? dg::kTileM : dg::kFp32TileM;
    return ((p->rows + tm - 1) / tm) * p->nkv;
}

// Key-range partitions: minimise (waves of CTAs) x (tiles per CTA + the fixed start-up and drain
// cost of a CTA) + the combine kernel's cost, all in units of one key tile's time.  The
// tensor-core constants (0.9 us per tile, 8 us of start-up plus epilogue per CTA) were fitted on
// the GB300; sweeps of the partition count on the hd = 256, 128 and 64 workloads found the same
// counts as this model.  The combine reads the partitions' rows once.
// The tensor-core path merges 2..8 partitions inside the kernel (one cluster per query tile)
// when such clusters fit on the GPU; other partition counts go through the combine kernel.
bool cluster_combine(const dg_attn_plan *p, int splits)
{
    return p->path == DG_PATH_TC && splits >= 2 && splits <= dg::kMaxClusterSplits &&
           p->max_clusters[splits] > 0;
}

// Cost of s partitions, or 1e300 when s is not a partition count that leaves none empty.
double split_cost(const dg_attn_plan *p, int s)
{
    const int nt = n_tiles_for(p);
    const int qt = qtiles_for(p);
    const bool tc = p->path == DG_PATH_TC;
    const int per_sm = tc ? 1 : 2;
    const int slots = p->num_sms * per_sm;
    const double tile_us = tc ? 0.9 : 2.0;
    const double startup = tc ? 8.0 / tile_us : 1.0;
    const double rows = (double)qt * (tc ? dg::kTileM : dg::kFp32TileM);
    if (s < 1 || s > nt) return 1e300;
    const int tps = (nt + s - 1) / s;
    const int s_eff = (nt + tps - 1) / tps;
    if (s_eff != s) return 1e300;
    const bool cl = cluster_combine(p, s);
    // co-resident CTAs: whole clusters only (they are placed within one GPC each)
    const int slots_s = cl ? std::min(slots, p->max_clusters[s] * s) : slots;
    if (slots_s < 1) return 1e300;
    const int waves = (qt * s + slots_s - 1) / slots_s;
    double cost = waves * (tps + startup);
    if (s > 1 && cl) {
        cost += 1.5 / tile_us;                     // in-kernel merge through shared memory
    } else if (s > 1) {
        const double bytes = rows * p->hd * 4.0 * (s + 1);
        cost += (3.0 + bytes / 3.0e6) / tile_us;   // launch + traffic at ~3 TB/s (bytes/us)
    }
    return cost;
}

int auto_splits(const dg_attn_plan *p)
{
    const int nt = n_tiles_for(p);
    int best = 1;
    double best_cost = 1e300;
    for (int s = 1; s <= nt && s <= 64; ++s) {
        const double cost = split_cost(p, s);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Stream-K layout of the tensor-core kernel: one CTA per SM (fewer when there are fewer key
// tiles), at least one per (query tile, kv group) pair so that a CTA's run of key tiles covers at
// most two pairs; kmax = the most pieces any pair is cut into (the partial slots needed).
struct SkLayout {
    int ctas = 0, kmax = 0;
    long long units = 0;
};

bool sk_layout(const dg_attn_plan *p, SkLayout &L)
{
    if (p->path != DG_PATH_TC) return false;
    const int nt = n_tiles_for(p);
    const int pairs = qtiles_for(p);
    const long long U = (long long)pairs * nt;
    long long C = p->num_sms;
    if (C > U) C = U;
    // no pair in more pieces than the combine merges: fewer CTAs when the pairs are few
    const long long c_cap = (long long)pairs * (dg::kMaxStreamKPieces - 1);
    if (C > c_cap) C = c_cap;
    if (C < pairs) return false;
    int kmax = 0;
    for (;;) {
        kmax = 0;
        for (int pr = 0; pr < pairs; ++pr) {
            const int k = dg::sk_cta_of((long long)(pr + 1) * nt - 1, U, (int)C) -
                          dg::sk_cta_of((long long)pr * nt, U, (int)C) + 1;
            if (k > kmax) kmax = k;
        }
        if (kmax <= dg::kMaxStreamKPieces || C <= pairs) break;
        --C;
    }
    if (kmax > dg::kMaxStreamKPieces) return false;
    L.ctas = (int)C;
    L.units = U;
    L.kmax = kmax;
    return true;
}

// Cost of the stream-K schedule in the units of auto_splits (one key tile's time): the longest
// run, the CTA's start-up, the switch between two pieces (Q reload, O written out) and the
// combine kernel, which reads every piece once from L2.  Measured on the GB300 (hd = 256, 48-step
// workload): the kernel 57.4 us against 62.5 us for four clustered partitions, but the combine
// ~8 us of a forward, so the clustered split stays ahead on the workloads measured.
double sk_cost(const dg_attn_plan *p, const SkLayout &L)
{
    const double tile_us = 0.9, startup = 8.0 / tile_us;
    const double run = (double)((L.units + L.ctas - 1) / L.ctas);
    const double pieces = (double)L.ctas + qtiles_for(p);
    const double bytes = pieces * dg::kTileM * p->hd * 4.0 + (double)p->rows * p->nkv * p->hd * 4.0;
    return run + startup + 2.0 + (8.0 + bytes / 8.0e6) / tile_us;   // L2 at ~8 TB/s (bytes/us)
}

// The schedule the next forward uses.
bool use_stream_k(const dg_attn_plan *p, SkLayout &L)
{
    if (p->path != DG_PATH_TC || p->schedule_opt == DG_SCHEDULE_SPLIT) return false;
    if (!sk_layout(p, L)) return false;
    if (p->schedule_opt == DG_SCHEDULE_STREAM_K) return true;
    if (p->splits_opt > 0) return false;           // an explicit partition count asks for splits
    return sk_cost(p, L) < split_cost(p, auto_splits(p));
}

// Partitions actually used: the option (clamped so that none is empty) or the automatic choice.
void split_layout(const dg_attn_plan *p, int &splits, int &tiles_per_split, int &n_tiles)
{
    n_tiles = n_tiles_for(p);
    int s = p->splits_opt > 0 ? p->splits_opt : auto_splits(p);
    if (s > n_tiles) s = n_tiles;
    if (s > p->part_capacity) s = p->part_capacity > 0 ? p->part_capacity : 1;
    if (s < 1) s = 1;
    tiles_per_split = (n_tiles + s - 1) / s;
    splits = (n_tiles + tiles_per_split - 1) / tiles_per_split;
}

// Partial-result slots per (query tile, kv group): the split schedule needs one per partition
// when it has two or more (a single partition writes the output itself); the stream-K schedule
// needs kmax of them, even 1 (every piece goes through the combine).
int split_slots(int splits) { return splits > 1 ? splits : 0; }

int ensure_partials(dg_attn_plan *p, int slots)
{
    const int splits = slots;
    if (splits <= 0 || splits <= p->part_capacity) return DG_OK;
    if (p->part_o) cudaFree(p->part_o);
    if (p->part_ml) cudaFree(p->part_ml);
    p->part_o = nullptr;
    p->part_ml = nullptr;
    p->part_capacity = 0;
    cudaError_t err = cudaSuccess;
    const size_t rows = (size_t)splits * p->nkv * p->rows_pad;
    p->part_o = (float *)dalloc(p, rows * p->hd * sizeof(float), err);
    p->part_ml = (float2 *)dalloc(p, rows * sizeof(float2), err);
    if (err != cudaSuccess) return cuda_fail(err, "allocating split-KV partials");
    p->part_capacity = splits;
    return DG_OK;
}

int record_event(dg_attn_plan *p, int stage, cudaStream_t s)
{
    if (!p->profile) return DG_OK;
    auto &v = p->ev[stage];
    size_t &used = p->ev_used[stage];
    if (used >= v.size()) {
        const size_t grow = v.size() ? v.size() : 1024;
        for (size_t i = 0; i < grow; ++i) {
            cudaEvent_t e;
            cudaError_t err = cudaEventCreate(&e);
            if (err != cudaSuccess) return cuda_fail(err, "cudaEventCreate");
            v.push_back(e);
        }
    }
    // Inside a stream capture a plain record only orders the graph's nodes; the external flag
    // makes each replay of the graph record the event, so the timings stay readable.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(s, &cap);
    if (err != cudaSuccess) return cuda_fail(err, "cudaStreamIsCapturing");
    err = cap == cudaStreamCaptureStatusActive
              ? cudaEventRecordWithFlags(v[used++], s, cudaEventRecordExternal)
              : cudaEventRecord(v[used++], s);
    return err == cudaSuccess ? DG_OK : cuda_fail(err, "cudaEventRecord");
}

// Allocate one operand set and encode its tensor maps.
int alloc_set(dg_attn_plan *p, OperandSet &o)
{
    const size_t nqt = (size_t)p->nkv * p->rows_pad * p->hd, nkt = (size_t)p->nkv * p->S * p->hd;
    cudaError_t err = cudaSuccess;
    o.qh = (__nv_bfloat16 *)dalloc(p, nqt * 2, err);
    o.ql = (__nv_bfloat16 *)dalloc(p, nqt * 2, err);
    o.kh = (__nv_bfloat16 *)dalloc(p, nkt * 2, err);
    o.kl = (__nv_bfloat16 *)dalloc(p, nkt * 2, err);
    o.vh = (__half *)dalloc(p, nkt * 2, err);
    if (err != cudaSuccess) {
        const size_t sizes[5] = {nqt * 2, nqt * 2, nkt * 2, nkt * 2, nkt * 2};
        void *ptrs[5] = {o.qh, o.ql, o.kh, o.kl, o.vh};
        for (int i = 0; i < 5; ++i)
            if (ptrs[i]) {
                cudaFree(ptrs[i]);
                p->scratch_bytes -= sizes[i];
            }
        o = OperandSet{};
        return cuda_fail(err, "allocating the tensor-core operand arrays");
    }
    const dg::TcGeom geo = dg::tc_geometry(p->hd);
    const int nk = geo.nk;
    bool ok = true;
    ok &= encode_3d(&o.maps.ql, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.ql, p->hd, p->rows_pad,
                    p->nkv, 64, dg::kTileM, p->hd);
    ok &= encode_3d(&o.maps.kh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.kh, p->hd, p->S, p->nkv,
                    64, nk, p->hd);
    ok &= encode_3d(&o.maps.kl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.kl, p->hd, p->S, p->nkv,
                    64, nk, p->hd);
    ok &= encode_3d(&o.maps.vh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, o.vh, p->hd, p->S, p->nkv,
                    64, geo.vk, p->hd);
    if (!ok) {
        set_error("cuTensorMapEncodeTiled failed (or the driver entry point is missing)");
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

dg::NormRopeParams norm_params(const dg_attn_plan *p)
{
    dg::NormRopeParams n{};
    n.inv_freq = p->inv_freq;
    n.T = p->T; n.nh = p->nh; n.nkv = p->nkv; n.ctx = p->ctx; n.S = p->S; n.S_pad = p->S_pad;
    n.rows_pad = p->rows_pad;
    n.pos0 = p->pos0;
    n.eps = p->eps;
    n.do_norm = 1; n.do_rope = 1;
    n.inputs_resident = p->inputs_resident;
    n.q_out = p->q32; n.k_out = p->k32; n.v_out = p->v32;
    n.qh = p->op.qh; n.ql = p->op.ql; n.kh = p->op.kh; n.kl = p->op.kl; n.vh = p->op.vh;
    n.ql_interleaved = p->tc_ok ? dg::tc_geometry(p->hd).ql_in_tmem : 0;
    n.status = p->status;
    return n;
}

// Hand a per-call cache to the first-stage launch (its last blocks convert it).
void fuse_cache(const dg_attn_plan *p, dg::NormRopeParams &n, const float *k_cache,
                const float *v_cache)
{
    const long long n4 = (long long)p->nkv * p->ctx * p->hd / 4;
    const long long per_block = 128ll * dg::kNormCacheUnroll;
    n.kc = k_cache;
    n.vc = v_cache;
    n.cache_blocks = (int)std::min<long long>((n4 + per_block - 1) / per_block,
                                              (long long)p->num_sms * 16);
}

// With resident inputs on the tensor-core path, make the other operand set the current one and
// return 1: the first stage then writes a set the previous forward's attention kernel does not
// read, and need not wait for that kernel (the ordering argument is in the first-stage and
// attention kernels).  A prepared cache is copied into a set that lacks it, once, on the stream.
int swap_sets(dg_attn_plan *p, cudaStream_t s, int &other)
{
    other = 0;
    if (p->path != DG_PATH_TC || !p->inputs_resident || !p->alt.qh) return DG_OK;
    if (p->ctx > 0 && p->cache_ready && !p->alt_cache) {
        const size_t pitch = (size_t)p->S * p->hd * 2, width = (size_t)p->ctx * p->hd * 2;
        cudaError_t err = cudaSuccess;
        const void *src[3] = {p->op.kh, p->op.kl, p->op.vh};
        void *dst[3] = {p->alt.kh, p->alt.kl, p->alt.vh};
        for (int i = 0; i < 3 && err == cudaSuccess; ++i)
            err = cudaMemcpy2DAsync(dst[i], pitch, src[i], pitch, width, p->nkv,
                                    cudaMemcpyDeviceToDevice, s);
        if (err != cudaSuccess) return cuda_fail(err, "copying the prepared cache rows");
        p->alt_cache = true;
    }
    std::swap(p->op, p->alt);
    other = 1;
    return DG_OK;
}

// A call that swapped the sets and then failed before its attention kernel was enqueued swaps
// them back: the current set must stay the one the last enqueued attention kernel reads.
int unswap_unless_launched(dg_attn_plan *p, int rc, int other, unsigned long long launched)
{
    if (rc != DG_OK && other && p->attn_launched == launched) std::swap(p->op, p->alt);
    return rc;
}

// Attention + (when partitioned) combine, reading the operands the first stage left in scratch.
// `fresh_cache`: the cache rows were converted by this call's first-stage launch, so the
// tensor-core kernel may not load them before its wait for that launch.  `split` (the layer
// path): where the attention kernel writes the output itself, have it also write the bf16 hi /
// lo split the o_proj GEMM reads (p->aoh / p->aol), and set *split to say so.
int enqueue_attention(dg_attn_plan *p, const float *k_cache, const float *v_cache, float *out,
                      cudaStream_t s, bool fresh_cache = false, bool *split = nullptr)
{
    if (split) *split = false;
    int splits, tps, nt;
    split_layout(p, splits, tps, nt);
    SkLayout sk;
    const bool stream_k = use_stream_k(p, sk);
    if (stream_k) {
        splits = sk.kmax;           // partial slots per pair
        tps = nt;
        if (int rc = ensure_partials(p, sk.kmax)) return rc;
        if (!p->part_o || !p->part_ml || p->part_capacity < sk.kmax) {
            set_error("stream-K schedule without room for its partial results");
            return DG_ERR_STATE;
        }
    }
    int rc = record_event(p, DG_STAGE_ATTENTION, s);
    if (rc) return rc;
    cudaError_t err;
    if (p->path == DG_PATH_TC) {
        dg::AttnTcParams a{};
        a.qh = p->op.qh; a.ql = p->op.ql; a.out = out; a.part_o = p->part_o; a.part_ml = p->part_ml;
        a.status = p->status;
        a.wait_limit_ns = (unsigned long long)p->wait_limit_ms * 1000000ull;
        a.T = p->T; a.nh = p->nh; a.nkv = p->nkv; a.S = p->S; a.G = p->G;
        a.rows = p->rows; a.rows_pad = p->rows_pad;
        a.splits = splits; a.tiles_per_split = tps; a.n_tiles = nt;
        a.cluster_combine = !stream_k && cluster_combine(p, splits) ? 1 : 0;
        a.inject_stall = p->inject_stall;
        a.static_keys = fresh_cache || p->cache_fresh ? 0 : p->ctx;
        if (split && p->split_attn && p->aoh && !stream_k && (splits == 1 || a.cluster_combine)) {
            a.out_hi = p->aoh;
            a.out_lo = p->aol;
        }
        if (stream_k) {
            a.sk_ctas = sk.ctas;
            a.sk_units = sk.units;
            a.qtiles = p->rows_pad / dg::kTileM;
        }
        err = dg::launch_attn_tc(a, p->op.maps, p->hd, s);
        if (err != cudaSuccess) return cuda_fail(err, "tensor-core attention launch");
        ++p->attn_launched;
        p->cache_fresh = false;
        p->attn_ctas = a.sk_ctas ? a.sk_ctas
                                 : ((a.rows + dg::kTileM - 1) / dg::kTileM) * a.nkv * a.splits;
        if (split) *split = a.out_hi != nullptr;
    } else {
        dg::AttnFp32Params a{};
        a.q = p->q32; a.k = p->k32; a.v = p->v32;
        a.k_cache = k_cache; a.v_cache = v_cache;
        a.out = out; a.part_o = p->part_o; a.part_ml = p->part_ml;
        a.T = p->T; a.nh = p->nh; a.nkv = p->nkv; a.ctx = p->ctx; a.S = p->S; a.G = p->G;
        a.rows = p->rows; a.rows_pad = p->rows_pad;
        a.splits = splits; a.keys_per_split = tps * 32;
        err = dg::launch_attn_fp32(a, p->hd, s);
        if (err != cudaSuccess) return cuda_fail(err, "fp32 attention launch");
    }
    rc = record_event(p, DG_STAGE_ATTENTION, s);
    if (rc) return rc;
    if (stream_k || (splits > 1 && !cluster_combine(p, splits))) {
        dg::CombineParams c{};
        c.part_o = p->part_o; c.part_ml = p->part_ml; c.out = out;
        c.T = p->T; c.nh = p->nh; c.nkv = p->nkv; c.G = p->G; c.rows = p->rows;
        c.rows_pad = p->rows_pad; c.splits = splits; c.hd = p->hd;
        c.log2_domain = p->path == DG_PATH_TC ? 1 : 0;
        if (stream_k) {
            c.sk_ctas = sk.ctas;
            c.sk_units = sk.units;
            c.qtiles = p->rows_pad / dg::kTileM;
            c.n_tiles = nt;
        }
        if ((rc = record_event(p, DG_STAGE_COMBINE, s))) return rc;
        err = dg::launch_combine(c, s);
        if (err != cudaSuccess) return cuda_fail(err, "combine launch");
        if ((rc = record_event(p, DG_STAGE_COMBINE, s))) return rc;
    }
    return DG_OK;
}

// Resolve which cache the attention reads.  A per-call cache on the tensor-core path is
// converted into the current operand set: by the first-stage launch when `fused` is given (set
// to true here; the caller hands the cache to that launch), else by a launch of its own.
int resolve_cache(dg_attn_plan *p, const float *&k_cache, const float *&v_cache, cudaStream_t s,
                  bool *fused = nullptr)
{
    if (fused) *fused = false;
    if (p->ctx == 0) {
        if (k_cache || v_cache) {
            set_error("ctx == 0: k_cache and v_cache must be NULL");
            return DG_ERR_ARG;
        }
        return DG_OK;
    }
    if (!k_cache && !v_cache) {
        if (!p->cache_ready) {
            set_error("no cache given and none prepared (dg_attn_cache_prepare)");
            return DG_ERR_STATE;
        }
        if (p->path == DG_PATH_FP32) {
            k_cache = p->prep_k;
            v_cache = p->prep_v;
        }
        return DG_OK;
    }
    if (!k_cache || !v_cache) {
        set_error("k_cache and v_cache must both be given or both be NULL");
        return DG_ERR_ARG;
    }
    if (!aligned16(k_cache) || !aligned16(v_cache)) {
        set_error("cache pointers must be 16-byte aligned");
        return DG_ERR_ALIGN;
    }
    if (p->path == DG_PATH_TC) {
        // the per-call conversion overwrites the plan's cache copy
        p->cache_ready = p->alt_cache = false;
        if (fused) {
            *fused = true;
            return DG_OK;
        }
        dg::CachePrepParams c{k_cache, v_cache, p->op.kh, p->op.kl, p->op.vh, nullptr, nullptr,
                              p->nkv, p->ctx, p->S, p->S_pad, p->hd, dg::kCacheF32, p->status,
                              nullptr, nullptr, nullptr};
        int rc = record_event(p, DG_STAGE_CACHE, s);
        if (rc) return rc;
        cudaError_t err = dg::launch_cache_prep(c, s);
        if (err != cudaSuccess) return cuda_fail(err, "cache conversion launch");
        p->cache_fresh = true;
        if ((rc = record_event(p, DG_STAGE_CACHE, s))) return rc;
    }
    return DG_OK;
}

// A first stage that runs beside the previous forward's attention kernel (resident inputs, the
// other operand set) asks for shared memory it does not use: just enough that none of its blocks
// fits on an SM holding an attention CTA, when that kernel's grid leaves SMs idle and a few KB
// suffice.  Its blocks then run on the idle SMs and leave the attention kernel's SMs alone (on
// the 48-step hd = 256 workload 0.8 us per forward; where the attention grid covers every SM the
// stage keeps all of them).
size_t beside_smem(const dg_attn_plan *p, const dg::NormRopeParams &n)
{
    if (p->path != DG_PATH_TC || !n.inputs_resident || !n.other_set || p->attn_ctas <= 0 ||
        p->attn_ctas >= p->num_sms)
        return 0;
    const long long free_bytes = (long long)p->smem_per_sm - (long long)dg::attn_tc_smem_bytes(p->hd) -
                                 p->smem_reserved;
    if (free_bytes < p->smem_reserved) return 0;     // no block fits beside an attention CTA
    const long long need = free_bytes - p->smem_reserved + 128;
    return need <= 8192 ? (size_t)need : 0;
}

// Without a caller's table the first stage reads the plan's cos|sin table, rebuilt on the stream
// (ahead of the work that reads it) after a change of position.  *built: the table was enqueued
// just now, so a first stage launched next must wait for it before reading anything (with
// resident inputs it would otherwise read the table before its dependency wait).
int rope_table(dg_attn_plan *p, const float *&cos_sin, cudaStream_t s, bool *built = nullptr)
{
    if (built) *built = false;
    if (cos_sin) return DG_OK;
    if (p->rope_dirty) {
        cudaError_t err = dg::launch_rope_table(p->rope_cs, p->inv_freq, p->T, p->hd, p->pos0, s);
        if (err != cudaSuccess) return cuda_fail(err, "cos/sin table launch");
        p->rope_dirty = false;
        if (built) *built = true;
    }
    cos_sin = p->rope_cs;
    return DG_OK;
}

int check_plan(const dg_attn_plan *p)
{
    if (!p) {
        set_error("NULL plan");
        return DG_ERR_ARG;
    }
    return DG_OK;
}

}  // namespace

extern "C" {

dg_attn_plan *dg_attn_plan_create(int nh, int nkv, int hd, int ctx, int T, float eps,
                                  float rope_theta)
{
    if (nh < 1 || nkv < 1 || T < 1 || ctx < 0 || nh % nkv != 0) {
        set_error("bad sizes: nh=%d nkv=%d T=%d ctx=%d (need nh %% nkv == 0, nh, nkv, T >= 1, "
                  "ctx >= 0)", nh, nkv, T, ctx);
        return nullptr;
    }
    if (hd != 32 && hd != 64 && hd != 128 && hd != 256) {
        set_error("hd=%d not supported (32, 64, 128 or 256)", hd);
        return nullptr;
    }
    if (!(eps >= 0.f) || !(rope_theta > 0.f)) {
        set_error("eps must be >= 0 and rope_theta > 0");
        return nullptr;
    }
    if ((long long)ctx + T >= (1ll << 24)) {
        set_error("positions must stay below 2^24");
        return nullptr;
    }
    if ((long long)nkv * ctx >= (1ll << 32)) {
        // the cache conversion numbers its rows (kv head, cache row) in 32 bits
        set_error("nkv * ctx must stay below 2^32");
        return nullptr;
    }
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    cudaDeviceProp prop;
    if (err == cudaSuccess) err = cudaGetDeviceProperties(&prop, dev);
    if (err != cudaSuccess) {
        cuda_fail(err, "querying the current device");
        return nullptr;
    }
    if (!(prop.major == 10 && prop.minor == 3)) {
        set_error("device %s is sm_%d%d; this library is built for sm_103a only", prop.name,
                  prop.major, prop.minor);
        return nullptr;
    }
    dg_attn_plan *p = new (std::nothrow) dg_attn_plan();
    if (!p) {
        set_error("out of host memory");
        return nullptr;
    }
    p->nh = nh; p->nkv = nkv; p->hd = hd; p->ctx = ctx; p->T = T;
    p->G = nh / nkv; p->S = ctx + T; p->rows = T * p->G;
    p->S_pad = ((p->S + 31) / 32) * 32;
    p->rows_pad = ((p->rows + dg::kTileM - 1) / dg::kTileM) * dg::kTileM;
    p->eps = eps; p->theta = rope_theta; p->pos0 = ctx;
    p->tc_ok = (hd == 64 || hd == 128 || hd == 256);
    p->path = p->tc_ok ? DG_PATH_TC : DG_PATH_FP32;
    p->splits_opt = 0;
    p->schedule_opt = DG_SCHEDULE_AUTO;
    p->wait_limit_ms = 2000;
    p->device = dev;
    p->num_sms = prop.multiProcessorCount;
    p->smem_per_sm = (int)prop.sharedMemPerMultiprocessor;
    p->smem_reserved = (int)prop.reservedSharedMemPerBlock;

    const size_t nq = (size_t)T * nh * hd, nk = (size_t)T * nkv * hd;
    p->inv_freq = (float4 *)dalloc(p, sizeof(float4) * (hd / 2), err);
    p->rope_cs = (float *)dalloc(p, sizeof(float) * 2 * (size_t)T * hd, err);
    p->rope_dirty = true;
    p->status = (uint32_t *)dalloc(p, sizeof(uint32_t) * 4, err);
    p->q32 = (float *)dalloc(p, nq * sizeof(float), err);
    p->k32 = (float *)dalloc(p, nk * sizeof(float), err);
    p->v32 = (float *)dalloc(p, nk * sizeof(float), err);
    if (err != cudaSuccess) {
        cuda_fail(err, "allocating plan scratch");
        free_scratch(p);
        delete p;
        return nullptr;
    }
    // each fp64 frequency as three floats whose sum is exactly it (24 + 24 + the last 5 bits)
    std::vector<float4> f(hd / 2);
    for (int i = 0; i < hd / 2; ++i) {
        const double v = std::pow((double)rope_theta, -2.0 * i / (double)hd);
        const float a = (float)v;
        const float b = (float)(v - (double)a);
        const float c = (float)(v - (double)a - (double)b);
        f[i] = make_float4(a, b, c, 0.f);
    }
    err = cudaMemcpy(p->inv_freq, f.data(), sizeof(float4) * f.size(), cudaMemcpyHostToDevice);
    if (err == cudaSuccess && p->tc_ok) err = dg::attn_tc_prepare(hd);
    for (int sp = 0; sp <= dg::kMaxClusterSplits; ++sp)
        p->max_clusters[sp] = (err == cudaSuccess && p->tc_ok)
                                  ? dg::attn_tc_max_clusters(hd, sp, p->rows_pad / dg::kTileM, nkv)
                                  : 0;
    int rc = (err == cudaSuccess) ? DG_OK : cuda_fail(err, "plan set-up");
    if (rc == DG_OK && p->tc_ok) rc = alloc_set(p, p->op);
    if (rc == DG_OK) {
        // room for the partitions both paths would pick
        const int saved = p->path;
        int need = 0;
        for (int path : {DG_PATH_TC, DG_PATH_FP32}) {
            if (path == DG_PATH_TC && !p->tc_ok) continue;
            p->path = path;
            const int s = split_slots(auto_splits(p));
            if (s > need) need = s;
            SkLayout L;
            if (use_stream_k(p, L) && L.kmax > need) need = L.kmax;
        }
        p->path = saved;
        rc = ensure_partials(p, need);
    }
    if (rc != DG_OK) {
        free_scratch(p);
        delete p;
        return nullptr;
    }
    return p;
}

int dg_attn_schedule_info(int nh, int nkv, int hd, int ctx, int T, int num_sms,
                          const int *max_clusters, int schedule, long long *out)
{
    if (!out || nh < 1 || nkv < 1 || T < 1 || ctx < 0 || nh % nkv != 0 || num_sms < 1 ||
        (hd != 64 && hd != 128 && hd != 256) ||
        (schedule != DG_SCHEDULE_AUTO && schedule != DG_SCHEDULE_SPLIT &&
         schedule != DG_SCHEDULE_STREAM_K)) {
        set_error("dg_attn_schedule_info: bad arguments");
        return DG_ERR_ARG;
    }
    // the plan fields the schedule choice reads, as dg_attn_plan_create sets them
    dg_attn_plan p{};
    p.nh = nh; p.nkv = nkv; p.hd = hd; p.ctx = ctx; p.T = T;
    p.G = nh / nkv; p.S = ctx + T; p.rows = T * p.G;
    p.rows_pad = ((p.rows + dg::kTileM - 1) / dg::kTileM) * dg::kTileM;
    p.tc_ok = true;
    p.path = DG_PATH_TC;
    p.splits_opt = 0;
    p.schedule_opt = schedule;
    p.num_sms = num_sms;
    p.part_capacity = 1 << 30;   // no clamp by buffers
    for (int s = 0; s <= dg::kMaxClusterSplits; ++s)
        p.max_clusters[s] = s < 2 ? 0 : (max_clusters ? max_clusters[s] : num_sms / s);
    SkLayout L;
    if (use_stream_k(&p, L)) {
        out[0] = DG_SCHEDULE_STREAM_K;
        out[1] = L.kmax;
        out[2] = L.ctas;
        out[3] = (L.units + L.ctas - 1) / L.ctas;
    } else {
        int s, tps, nt;
        split_layout(&p, s, tps, nt);
        out[0] = DG_SCHEDULE_SPLIT;
        out[1] = s;
        out[2] = (long long)qtiles_for(&p) * s;
        out[3] = tps;
    }
    return DG_OK;
}

void dg_attn_plan_destroy(dg_attn_plan *p)
{
    if (!p) return;
    free_scratch(p);
    delete p;
}

int dg_attn_set_option(dg_attn_plan *p, int key, long long value)
{
    if (int rc = check_plan(p)) return rc;
    switch (key) {
    case DG_OPT_PATH:
        if (value == DG_PATH_TC && !p->tc_ok) {
            set_error("the tensor-core path needs hd in {64, 128, 256}");
            return DG_ERR_UNSUPPORTED;
        }
        if (value != DG_PATH_TC && value != DG_PATH_FP32) {
            set_error("unknown path %lld", value);
            return DG_ERR_ARG;
        }
        if (p->path != (int)value) p->cache_ready = p->alt_cache = false;
        p->path = (int)value;
        return DG_OK;
    case DG_OPT_POS0:
        if (value < 0 || value + p->T >= (1ll << 24)) {
            set_error("pos0 out of range");
            return DG_ERR_ARG;
        }
        if (p->pos0 != value) p->rope_dirty = true;
        p->pos0 = value;
        return DG_OK;
    case DG_OPT_SPLITS: {
        if (value < 0 || value > 64) {
            set_error("splits must be in [0, 64]");
            return DG_ERR_ARG;
        }
        p->splits_opt = (int)value;
        int s, tps, nt;
        const int cap = p->part_capacity;
        p->part_capacity = 1 << 30;   // size the request before clamping to the buffers
        split_layout(p, s, tps, nt);
        p->part_capacity = cap;
        return ensure_partials(p, split_slots(s));
    }
    case DG_OPT_SCHEDULE: {
        if (value != DG_SCHEDULE_AUTO && value != DG_SCHEDULE_SPLIT && value != DG_SCHEDULE_STREAM_K) {
            set_error("schedule must be DG_SCHEDULE_AUTO, _SPLIT or _STREAM_K");
            return DG_ERR_ARG;
        }
        p->schedule_opt = (int)value;
        SkLayout L;
        return use_stream_k(p, L) ? ensure_partials(p, L.kmax) : DG_OK;
    }
    case DG_OPT_WAIT_LIMIT_MS:
        if (value < 1 || value > 600000) {
            set_error("wait limit must be in [1, 600000] ms");
            return DG_ERR_ARG;
        }
        p->wait_limit_ms = value;
        return DG_OK;
    case DG_OPT_INJECT_STALL:
        p->inject_stall = value ? 1 : 0;
        return DG_OK;
    case DG_OPT_INPUTS_RESIDENT:
        if (value && p->tc_ok && !p->alt.qh) {
            if (int rc = alloc_set(p, p->alt)) return rc;
            p->alt_cache = false;
        }
        p->inputs_resident = value ? 1 : 0;
        return DG_OK;
    case DG_OPT_PROFILE:
        p->profile = value ? 1 : 0;
        for (size_t &u : p->ev_used) u = 0;
        return DG_OK;
    default:
        set_error("unknown option %d", key);
        return DG_ERR_ARG;
    }
}

int dg_attn_get_option(const dg_attn_plan *p, int key, long long *value)
{
    if (int rc = check_plan(p)) return rc;
    if (!value) {
        set_error("NULL value pointer");
        return DG_ERR_ARG;
    }
    int s, tps, nt;
    switch (key) {
    case DG_OPT_PATH: *value = p->path; return DG_OK;
    case DG_OPT_POS0: *value = p->pos0; return DG_OK;
    case DG_OPT_SPLITS: *value = p->splits_opt; return DG_OK;
    case DG_OPT_WAIT_LIMIT_MS: *value = p->wait_limit_ms; return DG_OK;
    case DG_OPT_PROFILE: *value = p->profile; return DG_OK;
    case DG_OPT_INJECT_STALL: *value = p->inject_stall; return DG_OK;
    case DG_OPT_INPUTS_RESIDENT: *value = p->inputs_resident; return DG_OK;
    case DG_OPT_SCHEDULE: *value = p->schedule_opt; return DG_OK;
    case DG_INFO_SPLITS_USED: {
        SkLayout L;
        if (use_stream_k(p, L)) {
            *value = L.kmax;        // the most pieces of one pair
            return DG_OK;
        }
        split_layout(p, s, tps, nt);
        *value = s;
        return DG_OK;
    }
    case DG_INFO_SCHEDULE_USED: {
        SkLayout L;
        *value = use_stream_k(p, L) ? DG_SCHEDULE_STREAM_K : DG_SCHEDULE_SPLIT;
        return DG_OK;
    }
    case DG_INFO_SCRATCH_BYTES: *value = (long long)p->scratch_bytes; return DG_OK;
    case DG_INFO_CACHE_READY: *value = p->cache_ready ? 1 : 0; return DG_OK;
    case DG_INFO_LAUNCHES: {
        split_layout(p, s, tps, nt);
        SkLayout L;
        const bool combine = use_stream_k(p, L) || (s > 1 && !cluster_combine(p, s));
        *value = 2 + (combine ? 1 : 0) + (p->rope_dirty ? 1 : 0);
        return DG_OK;
    }
    default:
        set_error("unknown option %d", key);
        return DG_ERR_ARG;
    }
}

int dg_attn_cache_prepare(dg_attn_plan *p, const float *k_cache, const float *v_cache,
                          cudaStream_t s)
{
    return dg_attn_cache_prepare_typed(p, k_cache, v_cache, DG_DTYPE_F32, s);
}

int dg_attn_cache_prepare_typed(dg_attn_plan *p, const void *k_cache, const void *v_cache,
                                int dtype, cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    if (dtype != DG_DTYPE_F32 && dtype != DG_DTYPE_F16 && dtype != DG_DTYPE_BF16) {
        set_error("unknown cache element type %d", dtype);
        return DG_ERR_ARG;
    }
    if (p->ctx == 0) {
        set_error("ctx == 0: there is no cache to prepare");
        return DG_ERR_ARG;
    }
    if (!k_cache || !v_cache) {
        set_error("k_cache and v_cache are required");
        return DG_ERR_ARG;
    }
    if (!aligned16(k_cache) || !aligned16(v_cache)) {
        set_error("cache pointers must be 16-byte aligned");
        return DG_ERR_ALIGN;
    }
    const int type = dtype == DG_DTYPE_F16 ? dg::kCacheF16
                   : dtype == DG_DTYPE_BF16 ? dg::kCacheBf16 : dg::kCacheF32;
    dg::CachePrepParams c{k_cache, v_cache, p->op.kh, p->op.kl, p->op.vh, nullptr, nullptr,
                          p->nkv, p->ctx, p->S, p->S_pad, p->hd, type, p->status,
                          nullptr, nullptr, nullptr};
    if (p->path == DG_PATH_FP32) {
        if (dtype == DG_DTYPE_F32) {
            p->prep_k = static_cast<const float *>(k_cache);
            p->prep_v = static_cast<const float *>(v_cache);
            p->cache_ready = true;
            return DG_OK;
        }
        // a 16-bit cache is widened once into the plan's own fp32 copy
        if (!p->c32k) {
            cudaError_t err = cudaSuccess;
            const size_t bytes = (size_t)p->nkv * p->ctx * p->hd * sizeof(float);
            p->c32k = (float *)dalloc(p, bytes, err);
            p->c32v = (float *)dalloc(p, bytes, err);
            if (err != cudaSuccess) return cuda_fail(err, "allocating the fp32 cache copy");
        }
        c.k32 = p->c32k;
        c.v32 = p->c32v;
    }
    int rc = record_event(p, DG_STAGE_CACHE, s);
    if (rc) return rc;
    if (p->path == DG_PATH_TC && p->alt.qh) {
        // the second operand set gets the same rows in the same pass
        c.kh2 = p->alt.kh; c.kl2 = p->alt.kl; c.vh2 = p->alt.vh;
    }
    cudaError_t err = dg::launch_cache_prep(c, s);
    if (err != cudaSuccess) return cuda_fail(err, "cache conversion launch");
    p->cache_fresh = true;
    if ((rc = record_event(p, DG_STAGE_CACHE, s))) return rc;
    p->alt_cache = p->path == DG_PATH_TC && p->alt.qh;
    if (p->path == DG_PATH_FP32) {
        p->prep_k = p->c32k;
        p->prep_v = p->c32v;
    }
    p->cache_ready = true;
    return DG_OK;
}

static int check_canvas_args(const dg_attn_plan *p, const float *a, const float *b, const float *c,
                             const float *wq, const float *wk, const float *cs, const float *o1,
                             const float *o2, const float *o3)
{
    if (!a || !b || !c || !o1 || (o2 == nullptr) != (o3 == nullptr)) {
        set_error("a required pointer is NULL");
        return DG_ERR_ARG;
    }
    const void *all[] = {a, b, c, wq, wk, cs, o1, o2, o3};
    for (const void *x : all)
        if (x && !aligned16(x)) {
            set_error("pointers must be 16-byte aligned");
            return DG_ERR_ALIGN;
        }
    (void)p;
    return DG_OK;
}

int dg_attn_forward(dg_attn_plan *p, const float *q, const float *k_canvas, const float *v_canvas,
                    const float *k_cache, const float *v_cache, const float *q_norm_w,
                    const float *k_norm_w, const float *cos_sin, float *out, cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    if (int rc = check_canvas_args(p, q, k_canvas, v_canvas, q_norm_w, k_norm_w, cos_sin, out,
                                   nullptr, nullptr))
        return rc;
    const size_t qb = (size_t)p->T * p->nh * p->hd * 4, kb = (size_t)p->T * p->nkv * p->hd * 4;
    const size_t cb = (size_t)p->nkv * p->ctx * p->hd * 4, wb = (size_t)p->hd * 4;
    if (int rc = check_no_overlap({{out, qb}}, {{q, qb}, {k_canvas, kb}, {v_canvas, kb},
                                                {k_cache, cb}, {v_cache, cb}, {q_norm_w, wb},
                                                {k_norm_w, wb}, {cos_sin, 2 * (size_t)p->T * wb}}))
        return rc;
    int other;
    if (int rc = swap_sets(p, s, other)) return rc;
    const unsigned long long launched = p->attn_launched;
    auto run = [&]() -> int {
        bool fused;
        if (int rc = resolve_cache(p, k_cache, v_cache, s, &fused)) return rc;
        bool built;
        if (int rc = rope_table(p, cos_sin, s, &built)) return rc;
        dg::NormRopeParams n = norm_params(p);
        n.q = q; n.k = k_canvas; n.v = v_canvas; n.wq = q_norm_w; n.wk = k_norm_w;
        n.cos_sin = cos_sin;
        n.other_set = other;
        if (built) n.inputs_resident = 0;
        if (fused) fuse_cache(p, n, k_cache, v_cache);
        const int mode = p->path == DG_PATH_TC ? dg::kOutTc : dg::kOutFp32;
        int rc = record_event(p, DG_STAGE_NORM_ROPE, s);
        if (rc) return rc;
        cudaError_t err = dg::launch_norm_rope(n, p->hd, mode, s, beside_smem(p, n));
        if (err != cudaSuccess) return cuda_fail(err, "norm/rope launch");
        if ((rc = record_event(p, DG_STAGE_NORM_ROPE, s))) return rc;
        return enqueue_attention(p, k_cache, v_cache, out, s, fused);
    };
    return unswap_unless_launched(p, run(), other, launched);
}

int dg_attn_norm_rope(dg_attn_plan *p, const float *q, const float *k_canvas,
                      const float *v_canvas, const float *q_norm_w, const float *k_norm_w,
                      const float *cos_sin, float *q_hat, float *k_hat, float *v_hat,
                      cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    if (int rc = check_canvas_args(p, q, k_canvas, v_canvas, q_norm_w, k_norm_w, cos_sin, q_hat,
                                   k_hat, v_hat))
        return rc;
    if (!k_hat) {
        set_error("k_hat and v_hat are required");
        return DG_ERR_ARG;
    }
    const size_t qb = (size_t)p->T * p->nh * p->hd * 4, kb = (size_t)p->T * p->nkv * p->hd * 4;
    const size_t wb = (size_t)p->hd * 4;
    if (int rc = check_no_overlap({{q_hat, qb}, {k_hat, kb}, {v_hat, kb}},
                                  {{q, qb}, {k_canvas, kb}, {v_canvas, kb}, {q_norm_w, wb},
                                   {k_norm_w, wb}, {cos_sin, 2 * (size_t)p->T * wb}}))
        return rc;
    bool built;
    if (int rc = rope_table(p, cos_sin, s, &built)) return rc;
    dg::NormRopeParams n = norm_params(p);
    n.q = q; n.k = k_canvas; n.v = v_canvas; n.wq = q_norm_w; n.wk = k_norm_w; n.cos_sin = cos_sin;
    n.q_out = q_hat; n.k_out = k_hat; n.v_out = v_hat;
    if (built) n.inputs_resident = 0;
    cudaError_t err = dg::launch_norm_rope(n, p->hd, dg::kOutFp32, s);
    if (err != cudaSuccess) return cuda_fail(err, "norm/rope launch");
    return DG_OK;
}

int dg_attn_attend(dg_attn_plan *p, const float *q_hat, const float *k_hat, const float *v_hat,
                   const float *k_cache, const float *v_cache, float *out, cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    if (int rc = check_canvas_args(p, q_hat, k_hat, v_hat, nullptr, nullptr, nullptr, out,
                                   nullptr, nullptr))
        return rc;
    {
        const size_t qb = (size_t)p->T * p->nh * p->hd * 4;
        const size_t kb = (size_t)p->T * p->nkv * p->hd * 4;
        const size_t cb = (size_t)p->nkv * p->ctx * p->hd * 4;
        if (int rc = check_no_overlap({{out, qb}}, {{q_hat, qb}, {k_hat, kb}, {v_hat, kb},
                                                    {k_cache, cb}, {v_cache, cb}}))
            return rc;
    }
    int other;
    if (int rc = swap_sets(p, s, other)) return rc;
    const unsigned long long launched = p->attn_launched;
    auto run = [&]() -> int {
        bool fused;
        if (int rc = resolve_cache(p, k_cache, v_cache, s, &fused)) return rc;
        // the first-stage kernel with norm and rope switched off only re-lays the operands out
        dg::NormRopeParams n = norm_params(p);
        n.q = q_hat; n.k = k_hat; n.v = v_hat;
        n.other_set = other;
        if (fused) fuse_cache(p, n, k_cache, v_cache);
        n.do_norm = 0; n.do_rope = 0;
        const int mode = p->path == DG_PATH_TC ? dg::kOutTc : dg::kOutFp32;
        cudaError_t err = dg::launch_norm_rope(n, p->hd, mode, s, beside_smem(p, n));
        if (err != cudaSuccess) return cuda_fail(err, "operand layout launch");
        return enqueue_attention(p, k_cache, v_cache, out, s, fused);
    };
    return unswap_unless_launched(p, run(), other, launched);
}

int dg_attn_proj_prepare(dg_attn_plan *p, int H, const float *ln_in_w, const float *wq,
                         const float *wk, const float *wv, cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    if (!p->tc_ok || (p->hd != 128 && p->hd != 256)) {
        set_error("the projection step needs the tensor-core path with hd 128 or 256");
        return DG_ERR_UNSUPPORTED;
    }
    if (H < 64 || H % 64 != 0) {
        set_error("H=%d: the hidden size must be a positive multiple of 64", H);
        return DG_ERR_ARG;
    }
    if (!wq || !wk) {
        set_error("wq and wk are required");
        return DG_ERR_ARG;
    }
    const void *all[] = {ln_in_w, wq, wk, wv};
    for (const void *x : all)
        if (x && !aligned16(x)) {
            set_error("pointers must be 16-byte aligned");
            return DG_ERR_ALIGN;
        }
    cudaError_t err = dg::once_per_device(g_proj_attrs, dg::proj_prepare_attrs);
    if (err != cudaSuccess) return cuda_fail(err, "projection kernel attributes");
    const bool shared = wv == nullptr;
    const int rows = (p->nh + p->nkv + (shared ? 0 : p->nkv)) * p->hd;
    const int t_pad = ((p->T + dg::kTileM - 1) / dg::kTileM) * dg::kTileM;
    if (H != p->H || rows != p->proj_rows) {
        void *old[] = {p->wh, p->wl, p->xh, p->xl, p->rin};
        for (void *x : old)
            if (x) cudaFree(x);
        p->wh = p->wl = p->xh = p->xl = nullptr;
        p->rin = nullptr;
        p->proj_ready = false;
        p->H = 0;
        p->wh = (__nv_bfloat16 *)dalloc(p, (size_t)rows * H * 2, err);
        p->wl = (__nv_bfloat16 *)dalloc(p, (size_t)rows * H * 2, err);
        p->xh = (__nv_bfloat16 *)dalloc(p, (size_t)t_pad * H * 2, err);
        p->xl = (__nv_bfloat16 *)dalloc(p, (size_t)t_pad * H * 2, err);
        p->rin = (float *)dalloc(p, (size_t)p->T * sizeof(float), err);
        if (err != cudaSuccess) return cuda_fail(err, "allocating the projection operands");
        bool ok = true;
        const auto sw64 = CU_TENSOR_MAP_SWIZZLE_64B;   // 32-wide steps of the contraction
        ok &= encode_3d(&p->pmaps.xh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->xh, H, t_pad, 1, 32,
                        dg::kTileM, H, sw64);
        ok &= encode_3d(&p->pmaps.xl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->xl, H, t_pad, 1, 32,
                        dg::kTileM, H, sw64);
        ok &= encode_3d(&p->pmaps.wh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->wh, H, rows, 1, 32,
                        64, H, sw64);
        ok &= encode_3d(&p->pmaps.wl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->wl, H, rows, 1, 32,
                        64, H, sw64);
        if (!ok) {
            set_error("cuTensorMapEncodeTiled failed for the projection operands");
            return DG_ERR_CUDA;
        }
        p->H = H;
        p->proj_rows = rows;
    }
    dg::ProjWeightParams w{wq, wk, wv, ln_in_w, p->wh, p->wl, p->nh * p->hd, p->nkv * p->hd, rows,
                           H};
    err = dg::launch_proj_weights(w, s);
    if (err != cudaSuccess) return cuda_fail(err, "projection weight preparation launch");
    p->kv_shared = shared;
    p->proj_ready = true;
    return DG_OK;
}

}  // extern "C"

namespace {

// dg_attn_forward_hidden, and (with `split`) the first half of dg_attn_forward_layer.
int forward_hidden_impl(dg_attn_plan *p, const float *x, const float *k_cache,
                        const float *v_cache, const float *q_norm_w, const float *k_norm_w,
                        const float *cos_sin, float *out, cudaStream_t s, bool *split)
{
    if (int rc = check_plan(p)) return rc;
    if (!p->proj_ready) {
        set_error("no projection weights prepared (dg_attn_proj_prepare)");
        return DG_ERR_STATE;
    }
    if (p->path != DG_PATH_TC) {
        set_error("the projection step runs on the tensor-core path only");
        return DG_ERR_UNSUPPORTED;
    }
    if (!x || !out) {
        set_error("x and out are required");
        return DG_ERR_ARG;
    }
    const void *all[] = {x, q_norm_w, k_norm_w, cos_sin, out};
    for (const void *a : all)
        if (a && !aligned16(a)) {
            set_error("pointers must be 16-byte aligned");
            return DG_ERR_ALIGN;
        }
    {
        const size_t ob = (size_t)p->T * p->nh * p->hd * 4, xb = (size_t)p->T * p->H * 4;
        const size_t cb = (size_t)p->nkv * p->ctx * p->hd * 4, wb = (size_t)p->hd * 4;
        if (int rc = check_no_overlap({{out, ob}}, {{x, xb}, {k_cache, cb}, {v_cache, cb},
                                                    {q_norm_w, wb}, {k_norm_w, wb},
                                                    {cos_sin, 2 * (size_t)p->T * wb}}))
            return rc;
    }
    if (int rc = resolve_cache(p, k_cache, v_cache, s)) return rc;
    if (int rc = rope_table(p, cos_sin, s)) return rc;
    int rc = record_event(p, DG_STAGE_PROJECTION, s);
    if (rc) return rc;
    dg::ProjPrepParams pp{x, p->rin, p->xh, p->xl, p->T, p->H, p->eps};
    cudaError_t err = dg::launch_hidden_prep(pp, s);
    if (err != cudaSuccess) return cuda_fail(err, "input norm launch");
    dg::ProjParams q{};
    q.rin = p->rin;
    q.wq_norm = q_norm_w;
    q.wk_norm = k_norm_w;
    q.cos_sin = cos_sin;
    q.qh = p->op.qh; q.ql = p->op.ql; q.kh = p->op.kh; q.kl = p->op.kl; q.vh = p->op.vh;
    q.status = p->status;
    q.wait_limit_ns = (unsigned long long)p->wait_limit_ms * 1000000ull;
    q.T = p->T; q.H = p->H; q.nh = p->nh; q.nkv = p->nkv; q.G = p->G; q.ctx = p->ctx; q.S = p->S;
    q.rows_pad = p->rows_pad;
    q.rows_pad_tokens = ((p->T + dg::kTileM - 1) / dg::kTileM) * dg::kTileM;
    q.ql_interleaved = dg::tc_geometry(p->hd).ql_in_tmem;
    q.kv_shared = p->kv_shared ? 1 : 0;
    q.eps = p->eps;
    err = dg::launch_qkv_proj(q, p->pmaps, p->hd, p->proj_rows / 128, s);
    if (err != cudaSuccess) return cuda_fail(err, "projection launch");
    if ((rc = record_event(p, DG_STAGE_PROJECTION, s))) return rc;
    return enqueue_attention(p, k_cache, v_cache, out, s, false, split);
}

}  // namespace

extern "C" {

int dg_attn_forward_hidden(dg_attn_plan *p, const float *x, const float *k_cache,
                           const float *v_cache, const float *q_norm_w, const float *k_norm_w,
                           const float *cos_sin, float *out, cudaStream_t s)
{
    return forward_hidden_impl(p, x, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, out, s,
                               nullptr);
}

int dg_attn_oproj_prepare(dg_attn_plan *p, int H, const float *wo, const float *ln_post_w,
                          cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    const int tile = dg::oproj_tile_n(H, p->T, p->num_sms);
    if (H < 64 || tile == 0) {
        set_error("H=%d: the hidden size must be a positive multiple of 64", H);
        return DG_ERR_ARG;
    }
    if (!wo) {
        set_error("wo is required");
        return DG_ERR_ARG;
    }
    if (!aligned16(wo) || (ln_post_w && !aligned16(ln_post_w))) {
        set_error("pointers must be 16-byte aligned");
        return DG_ERR_ALIGN;
    }
    cudaError_t err = dg::once_per_device(g_proj_attrs, dg::proj_prepare_attrs);
    if (err != cudaSuccess) return cuda_fail(err, "projection kernel attributes");
    // The layer path's attention variant is set up (and so loaded) here, not with the plan: a
    // plan that never runs the layer keeps only the default attention kernels on the device.
    if (p->tc_ok && (p->hd == 128 || p->hd == 256)) {
        err = dg::attn_tc_split_prepare(p->hd);
        if (err != cudaSuccess) return cuda_fail(err, "attention kernel attributes");
        p->split_attn = true;
    }
    const int K = p->nh * p->hd;
    const int t_pad = ((p->T + dg::kTileM - 1) / dg::kTileM) * dg::kTileM;
    if (H != p->oH) {
        p->otile = tile;
        void *old[] = {p->woh, p->wol, p->aoh, p->aol, p->ybuf, p->part_ss, p->ln_post, p->attn_buf};
        for (void *x : old)
            if (x) cudaFree(x);
        p->woh = p->wol = p->aoh = p->aol = nullptr;
        p->ybuf = p->part_ss = p->ln_post = p->attn_buf = nullptr;
        p->oproj_ready = false;
        p->oH = 0;
        p->woh = (__nv_bfloat16 *)dalloc(p, (size_t)H * K * 2, err);
        p->wol = (__nv_bfloat16 *)dalloc(p, (size_t)H * K * 2, err);
        p->aoh = (__nv_bfloat16 *)dalloc(p, (size_t)t_pad * K * 2, err);
        p->aol = (__nv_bfloat16 *)dalloc(p, (size_t)t_pad * K * 2, err);
        p->ybuf = (float *)dalloc(p, (size_t)p->T * H * 4, err);
        p->part_ss = (float *)dalloc(p, (size_t)p->T * (H / tile) * 4, err);
        p->ln_post = (float *)dalloc(p, (size_t)H * 4, err);
        p->attn_buf = (float *)dalloc(p, (size_t)p->T * K * 4, err);
        if (err != cudaSuccess) return cuda_fail(err, "allocating the o_proj operands");
        bool ok = true;
        const auto sw64 = CU_TENSOR_MAP_SWIZZLE_64B;
        ok &= encode_3d(&p->omaps.xh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->aoh, K, t_pad, 1, 32,
                        dg::kTileM, K, sw64);
        ok &= encode_3d(&p->omaps.xl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->aol, K, t_pad, 1, 32,
                        dg::kTileM, K, sw64);
        ok &= encode_3d(&p->omaps.wh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->woh, K, H, 1, 32, tile,
                        K, sw64);
        ok &= encode_3d(&p->omaps.wl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->wol, K, H, 1, 32, tile,
                        K, sw64);
        if (!ok) {
            set_error("cuTensorMapEncodeTiled failed for the o_proj operands");
            return DG_ERR_CUDA;
        }
        p->oH = H;
    }
    dg::ProjWeightParams w{wo, nullptr, nullptr, nullptr, p->woh, p->wol, H, 0, H, K};
    err = dg::launch_proj_weights(w, s);
    if (err == cudaSuccess && ln_post_w)
        err = cudaMemcpyAsync(p->ln_post, ln_post_w, (size_t)H * 4, cudaMemcpyDeviceToDevice, s);
    if (err != cudaSuccess) return cuda_fail(err, "o_proj weight preparation");
    p->has_ln_post = ln_post_w != nullptr;
    p->oproj_ready = true;
    return DG_OK;
}

}  // extern "C"

namespace {

// dg_attn_oproj_residual; `split_ready`: the attention kernel has already written the bf16 hi /
// lo split of attn_out into p->aoh / p->aol, so the operand split kernel is skipped.
int oproj_residual_impl(dg_attn_plan *p, const float *attn_out, float *resid, cudaStream_t s,
                        bool split_ready)
{
    if (int rc = check_plan(p)) return rc;
    if (!p->oproj_ready) {
        set_error("no o_proj weights prepared (dg_attn_oproj_prepare)");
        return DG_ERR_STATE;
    }
    if (!attn_out || !resid) {
        set_error("attn_out and resid are required");
        return DG_ERR_ARG;
    }
    if (!aligned16(attn_out) || !aligned16(resid)) {
        set_error("pointers must be 16-byte aligned");
        return DG_ERR_ALIGN;
    }
    const int K = p->nh * p->hd;
    int rc = record_event(p, DG_STAGE_OPROJ, s);
    if (rc) return rc;
    cudaError_t err = cudaSuccess;
    if (!split_ready) {
        dg::ProjPrepParams pp{attn_out, nullptr, p->aoh, p->aol, p->T, K, p->eps};
        err = dg::launch_hidden_prep(pp, s);
        if (err != cudaSuccess) return cuda_fail(err, "o_proj operand launch");
    }
    dg::OprojParams o{p->ybuf, p->part_ss, p->status,
                      (unsigned long long)p->wait_limit_ms * 1000000ull, p->T, p->oH, K, p->otile};
    err = dg::launch_oproj(o, p->omaps, s);
    if (err != cudaSuccess) return cuda_fail(err, "o_proj launch");
    dg::PostNormParams n{p->ybuf, p->part_ss, p->has_ln_post ? p->ln_post : nullptr, resid, p->T,
                         p->oH, p->oH / p->otile, p->eps, 1.0f};
    err = dg::launch_post_norm(n, s);
    if (err != cudaSuccess) return cuda_fail(err, "post-attention norm launch");
    return record_event(p, DG_STAGE_OPROJ, s);
}

}  // namespace

extern "C" {

int dg_attn_oproj_residual(dg_attn_plan *p, const float *attn_out, float *resid, cudaStream_t s)
{
    return oproj_residual_impl(p, attn_out, resid, s, false);
}

int dg_attn_forward_layer(dg_attn_plan *p, float *resid, const float *k_cache,
                          const float *v_cache, const float *q_norm_w, const float *k_norm_w,
                          const float *cos_sin, cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    if (!p->proj_ready || !p->oproj_ready || p->H != p->oH) {
        set_error("the layer needs dg_attn_proj_prepare and dg_attn_oproj_prepare with one H");
        return DG_ERR_STATE;
    }
    // the attention kernel writes o_proj's bf16 operand split itself where it writes the output
    // (then attn_buf is left unwritten: nothing after it reads the fp32 rows)
    bool split = false;
    if (int rc = forward_hidden_impl(p, resid, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin,
                                     p->attn_buf, s, &split))
        return rc;
    return oproj_residual_impl(p, p->attn_buf, resid, s, split);
}

int dg_attn_sync_status(dg_attn_plan *p, cudaStream_t s)
{
    if (int rc = check_plan(p)) return rc;
    cudaError_t err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return cuda_fail(err, "cudaStreamSynchronize");
    uint32_t st = 0;
    err = cudaMemcpy(&st, p->status, sizeof(st), cudaMemcpyDeviceToHost);
    if (err == cudaSuccess) err = cudaMemset(p->status, 0, sizeof(uint32_t));
    if (err != cudaSuccess) return cuda_fail(err, "reading the status word");
    if (st & (dg::kErrWaitProducer | dg::kErrWaitMma | dg::kErrWaitSoftmax | dg::kErrWaitDrain)) {
        set_error("a device wait ran out (status bits 0x%x: 1 producer, 2 mma, 4 softmax, 8 drain)",
                  st);
        return DG_ERR_TIMEOUT;
    }
    if (st & dg::kErrSchedule) {
        set_error("a stream-K run covered more than two (query tile, kv group) pairs (status 0x%x)",
                  st);
        return DG_ERR_STATE;
    }
    if (st & dg::kErrRange) {
        set_error("a cache V value lies outside the fp16 range (|v| > 65504 or not finite): the "
                  "tensor-core path cannot hold it (status 0x%x); the exact path can", st);
        return DG_ERR_RANGE;
    }
    return DG_OK;
}

int dg_attn_profile_read(dg_attn_plan *p, int stage, double *total_ms, long long *launches)
{
    if (int rc = check_plan(p)) return rc;
    if (!total_ms || !launches || stage < 0 || stage > 5) {
        set_error("bad stage or NULL output pointer");
        return DG_ERR_ARG;
    }
    double tot = 0.0;
    long long n = 0;
    auto &v = p->ev[stage];
    for (size_t i = 0; i + 1 < p->ev_used[stage]; i += 2) {
        cudaError_t err = cudaEventSynchronize(v[i + 1]);
        float ms = 0.f;
        if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, v[i], v[i + 1]);
        if (err != cudaSuccess) return cuda_fail(err, "reading profiling events");
        tot += ms;
        ++n;
    }
    p->ev_used[stage] = 0;
    *total_ms = tot;
    *launches = n;
    return DG_OK;
}

const char *dg_attn_status_string(int status)
{
    switch (status) {
    case DG_OK: return "ok";
    case DG_ERR_ARG: return "invalid argument";
    case DG_ERR_ALIGN: return "misaligned pointer";
    case DG_ERR_CUDA: return "CUDA error";
    case DG_ERR_TIMEOUT: return "device wait timed out";
    case DG_ERR_UNSUPPORTED: return "unsupported";
    case DG_ERR_STATE: return "missing plan state";
    case DG_ERR_RANGE: return "value outside the range of the tensor-core operands";
    default: return "unknown status";
    }
}

const char *dg_attn_last_error(void) { return g_last_error; }

#ifndef DG_BUILD_ID
#define DG_BUILD_ID "sha1:unknown"
#endif
const char *dg_attn_build_id(void) { return DG_BUILD_ID; }

}  // extern "C"
