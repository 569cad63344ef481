// noalloc.cu -- dg_attn_forward_noalloc: the exact-fp32 forward without a plan and without any
// device allocation.
//
// Some callers cannot call cudaMalloc at the point where they run attention: code that runs
// inside a memory pool or arena it does not own, an allocator hook, or a process whose device
// memory is fully reserved up front.  This entry point serves them: its working memory (the
// normed q/k/v and the RoPE frequencies) lives in one file-scope __device__ array of fixed size,
// so it needs only the caller's inputs and output.
//
// The array is kDgNoallocScratchBytes (16 MiB) on every GPU that loads the library and stays
// there until the process exits.  All calls share it and it keeps the last call's contents;
// every call writes all of the scratch it reads before reading it, so nothing has to be cleared
// in between.  Calls that overlap on the GPU (two streams, or two host threads) race on it and
// must be serialised by the caller.  In host code the array's name is only a host-side handle,
// so its device address is looked up once per device with cudaGetSymbolAddress; the first call
// on each device does that set-up, so make that first call before any stream capture.
#include "../../include/dg_attn.h"
#include "dg_internal.cuh"

#include <cmath>
#include <cstdio>
#include <mutex>

namespace {

constexpr size_t kDgNoallocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kDgNoallocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};
thread_local char g_err[256] = "";

// theta^(-2i/hd) in fp64, held exactly as the sum of three floats, one thread per frequency.
__global__ void noalloc_inv_freq_kernel(float4 *out, int half, int hd, double theta)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= half) return;
    const double v = pow(theta, -2.0 * i / (double)hd);
    const float a = (float)v;
    const float b = (float)(v - (double)a);
    out[i] = make_float4(a, b, (float)(v - (double)a - (double)b), 0.f);
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" const char *dg_attn_noalloc_last_error(void) { return g_err; }

extern "C" int dg_attn_forward_noalloc(int nh, int nkv, int hd, int ctx, int T, float eps,
                                       float rope_theta, long long pos0, const float *q,
                                       const float *k_canvas, const float *v_canvas,
                                       const float *k_cache, const float *v_cache,
                                       const float *q_norm_w, const float *k_norm_w,
                                       const float *cos_sin, float *out, cudaStream_t stream)
{
    if (nh < 1 || nkv < 1 || T < 1 || ctx < 0 || nh % nkv != 0 ||
        (hd != 32 && hd != 64 && hd != 128 && hd != 256) || !(eps >= 0.f) ||
        !(rope_theta > 0.f)) {
        snprintf(g_err, sizeof(g_err), "bad sizes: nh=%d nkv=%d hd=%d ctx=%d T=%d", nh, nkv, hd,
                 ctx, T);
        return DG_ERR_ARG;
    }
    if (pos0 < 0) pos0 = ctx;
    if (pos0 + T >= (1ll << 24)) {
        snprintf(g_err, sizeof(g_err), "positions must stay below 2^24");
        return DG_ERR_ARG;
    }
    if (!q || !k_canvas || !v_canvas || !out || (ctx > 0 && (!k_cache || !v_cache)) ||
        (ctx == 0 && (k_cache || v_cache))) {
        snprintf(g_err, sizeof(g_err), "a required pointer is NULL (or a cache given with ctx=0)");
        return DG_ERR_ARG;
    }
    // the kernels move every row with 16-byte vector loads and stores
    const void *all[] = {q, k_canvas, v_canvas, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, out};
    for (const void *x : all)
        if (x && !aligned16(x)) {
            snprintf(g_err, sizeof(g_err), "pointers must be 16-byte aligned");
            return DG_ERR_ALIGN;
        }
    // the scratch regions, each rounded up to 256 bytes: the RoPE frequencies (hd/2 float4),
    // q-hat [T, nh, hd], k-hat and v-hat [T, nkv, hd] (fp32)
    const size_t freq_b = align256(sizeof(float4) * (size_t)(hd / 2));
    const size_t q_b = align256(sizeof(float) * (size_t)T * nh * hd);
    const size_t kv_b = align256(sizeof(float) * (size_t)T * nkv * hd);
    const size_t need = freq_b + q_b + 2 * kv_b;
    if (need > kDgNoallocScratchBytes) {
        snprintf(g_err, sizeof(g_err),
                 "needs %zu bytes of scratch for T=%d nh=%d nkv=%d hd=%d; the fixed array holds "
                 "%zu (the sum of hd*8, T*nh*hd*4 and twice T*nkv*hd*4, each rounded up to 256)",
                 need, T, nh, nkv, hd, kDgNoallocScratchBytes);
        return DG_ERR_ARG;
    }
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        snprintf(g_err, sizeof(g_err), "cudaGetDevice: %s", cudaGetErrorString(err));
        return DG_ERR_CUDA;
    }
    unsigned char *base;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_addr[dev]) {
            void *ptr = nullptr;
            err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (err != cudaSuccess || !ptr) {
                snprintf(g_err, sizeof(g_err), "cudaGetSymbolAddress: %s", cudaGetErrorString(err));
                return DG_ERR_CUDA;
            }
            g_scratch_addr[dev] = ptr;
        }
        base = static_cast<unsigned char *>(g_scratch_addr[dev]);
    }
    float4 *inv_freq = reinterpret_cast<float4 *>(base);
    float *qh = reinterpret_cast<float *>(base + freq_b);
    float *kh = reinterpret_cast<float *>(base + freq_b + q_b);
    float *vh = reinterpret_cast<float *>(base + freq_b + q_b + kv_b);

    noalloc_inv_freq_kernel<<<1, 128, 0, stream>>>(inv_freq, hd / 2, hd, (double)rope_theta);
    err = cudaGetLastError();
    if (err != cudaSuccess) {
        snprintf(g_err, sizeof(g_err), "frequency kernel: %s", cudaGetErrorString(err));
        return DG_ERR_CUDA;
    }
    dg::NormRopeParams n{};
    n.q = q; n.k = k_canvas; n.v = v_canvas; n.wq = q_norm_w; n.wk = k_norm_w;
    n.cos_sin = cos_sin; n.inv_freq = inv_freq;
    n.T = T; n.nh = nh; n.nkv = nkv; n.ctx = ctx; n.S = ctx + T; n.S_pad = ctx + T;
    n.rows_pad = T * (nh / nkv);
    n.pos0 = pos0; n.eps = eps; n.do_norm = 1; n.do_rope = 1;
    n.q_out = qh; n.k_out = kh; n.v_out = vh;
    err = dg::launch_norm_rope(n, hd, dg::kOutFp32, stream);
    if (err != cudaSuccess) {
        snprintf(g_err, sizeof(g_err), "norm/rope launch: %s", cudaGetErrorString(err));
        return DG_ERR_CUDA;
    }
    dg::AttnFp32Params a{};
    a.q = qh; a.k = kh; a.v = vh; a.k_cache = k_cache; a.v_cache = v_cache; a.out = out;
    a.T = T; a.nh = nh; a.nkv = nkv; a.ctx = ctx; a.S = ctx + T; a.G = nh / nkv;
    a.rows = T * (nh / nkv); a.rows_pad = a.rows;
    a.splits = 1; a.keys_per_split = ctx + T;
    err = dg::launch_attn_fp32(a, hd, stream);
    if (err != cudaSuccess) {
        snprintf(g_err, sizeof(g_err), "fp32 attention launch: %s", cudaGetErrorString(err));
        return DG_ERR_CUDA;
    }
    return DG_OK;
}
