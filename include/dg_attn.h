/*
 * dg_attn.h -- C ABI of libdgattn.so: DiffusionGemma's canvas-forward attention block on one
 * GB300 (sm_103a).
 *
 * The operation (page "inferencelayer 0.2.3, src/diffusion_gemma_gpu.rs"):
 *   - items DG_HEADNORM_ROPE and the three head-norm dispatches of canvas_forward:
 *       q-hat = RoPE(RMSNorm(q) * w_q), k-hat = RoPE(RMSNorm(k_canvas) * w_k),
 *       v-hat = RMSNorm(v_canvas) (no weight, no RoPE),
 *       RMSNorm(x) = x * (mean(x^2) + eps)^-1/2 per (token, head); RoPE is NeoX rotate-half at
 *       position pos0 + t with frequencies rope_theta^(-2i/hd) (both halves equal);
 *   - item DG_ATTN and its dispatch: GQA bidirectional softmax attention with scaling 1.0 and no
 *     mask over the split key/value set [cache (ctx rows) | canvas (T rows)], kv head of q head
 *     h = h / (nh / nkv).
 *
 * Layouts (all fp32, dense, row-major, on the current CUDA device):
 *   q         [T, nh*hd]           k_canvas, v_canvas [T, nkv*hd] (raw, before the norms)
 *   k_cache   [nkv, ctx, hd]       v_cache [nkv, ctx, hd] (used as given: already normed/roped)
 *   q_norm_w  [hd] or NULL         k_norm_w [hd] or NULL (NULL = unweighted)
 *   cos_sin   [T, 2*hd] or NULL    row t = cos(hd) | sin(hd); NULL = the plan's own table of the
 *                                  positions pos0 + t, built on the device by the first call after
 *                                  plan creation or a change of DG_OPT_POS0 (one extra kernel)
 *   out       [T, nh*hd]
 *
 * Ownership: the caller owns every buffer passed in; inputs are only read.  A plan owns its
 * device scratch (normed operands, split-KV partials), allocated by dg_attn_plan_create on the
 * current device and released by dg_attn_plan_destroy.
 *
 * Execution: every call that takes a stream only enqueues work on it (no host synchronisation,
 * no allocation), so it can be recorded into a CUDA graph.  One plan must not be used by two
 * streams at the same time: its scratch is shared between calls.
 *
 * Errors: calls return a DG_* status; the text of the last host-side error of the calling thread
 * is in dg_attn_last_error().  Device-side waits are bounded: a wait that runs out sets a status
 * word in the plan instead of hanging; dg_attn_sync_status() reads (and clears) it.
 */
#ifndef DG_ATTN_H
#define DG_ATTN_H

#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dg_attn_plan dg_attn_plan;

/* Status codes. */
#define DG_OK              0
#define DG_ERR_ARG         1  /* bad size or NULL pointer */
#define DG_ERR_ALIGN       2  /* a pointer is not 16-byte aligned */
#define DG_ERR_CUDA        3  /* a CUDA call or launch failed; see dg_attn_last_error() */
#define DG_ERR_TIMEOUT     4  /* a bounded device wait ran out (the kernel gave up cleanly) */
#define DG_ERR_UNSUPPORTED 5  /* the request needs something this build or device lacks */
#define DG_ERR_STATE       6  /* the call needs state the plan does not hold */
#define DG_ERR_RANGE       7  /* (dg_attn_sync_status) a cache V value lies outside the fp16 range
                                 that the tensor-core P.V operand holds (|v| > 65504 or not
                                 finite); the outputs of that forward are not valid */

/* Arithmetic paths (option DG_OPT_PATH). */
#define DG_PATH_TC   0  /* tensor cores: Q.K^T as three bf16 MMAs (hi/lo split), P.V in fp16 (10-bit
                           mantissa, the TF32 rounding); cache V must lie within fp16 range */
#define DG_PATH_FP32 1  /* exact fp32 on the CUDA cores */

/* Option keys for dg_attn_set_option / dg_attn_get_option. */
#define DG_OPT_PATH          1  /* DG_PATH_TC (default when hd is 64, 128 or 256) or DG_PATH_FP32;
                                   the exact path keeps the page's all-f32 contract (module doc) */
#define DG_OPT_POS0          2  /* position of canvas row 0 (default ctx, the cache length): the page's
                                   canvas_forward ropes canvas row t at rope_cos_sin(cache.seq_len
                                   + t, ...), and a sliding layer's cache may be shorter than seq_len */
#define DG_OPT_SPLITS        3  /* key-range partitions per query tile (0..64); 0 = chosen per plan.
                                   Scheduling only (the page's DG_ATTN runs one workgroup per row
                                   and head over all keys); results agree within rounding */
#define DG_OPT_WAIT_LIMIT_MS 4  /* device wait limit in ms (default 2000); no counterpart on the page */
#define DG_OPT_PROFILE       5  /* 1 = record CUDA events around each kernel launch, per stage (inside a
                                   stream capture as external records, taken on every replay);
                                   measurement only, no counterpart on the page */
#define DG_OPT_INJECT_STALL  6  /* test hook: 1 = the tensor-core kernel's softmax withholds its
                                   first "P ready" signal, so the bounded waits behind it run out
                                   and the forward ends with DG_ERR_TIMEOUT (no fault, no hang);
                                   no counterpart on the page */
#define DG_OPT_INPUTS_RESIDENT 7 /* 1 = the caller guarantees that the inputs of every call (q,
                                   k_canvas, v_canvas, weights, cos_sin, and a cache passed with
                                   the call) are complete before the
                                   work enqueued ahead of that call on the stream started, e.g.
                                   canvases already resident in device memory: the first stage then
                                   reads them while the previous call's attention kernel is still
                                   running.  Default 0: the first stage waits for the preceding
                                   kernel before reading anything.  On the tensor-core path,
                                   switching it on allocates a second set of operand arrays (the
                                   size of the first, DG_INFO_SCRATCH_BYTES grows); forwards then
                                   alternate between the two sets, so a forward's first stage
                                   writes the set the previous attention kernel is not reading and
                                   waits for nothing.  Consecutive calls must then share one
                                   stream, or the caller orders them.  Scheduling only (the page
                                   records all dispatches of a forward into one pass) */
#define DG_OPT_SCHEDULE      8  /* how the tensor-core kernel deals key tiles to CTAs: one of
                                   DG_SCHEDULE_AUTO (default), DG_SCHEDULE_SPLIT,
                                   DG_SCHEDULE_STREAM_K.  Scheduling only, as DG_OPT_SPLITS */
#define DG_SCHEDULE_AUTO     0  /* the cheaper of the two for the plan's geometry (a cost model) */
#define DG_SCHEDULE_SPLIT    1  /* one CTA per (query tile, kv group, key partition), partitions
                                   set by DG_OPT_SPLITS; 2..8 partitions merge inside the kernel,
                                   more through the combine kernel */
#define DG_SCHEDULE_STREAM_K 2  /* one CTA per SM: the (query tile, kv group) pairs, in order, are
                                   cut into key tiles and every CTA takes an equal run of them
                                   (a run may cover the end of one pair and the start of the
                                   next); the combine kernel merges each pair's pieces.  Ignores
                                   DG_OPT_SPLITS */
/* Read-only (dg_attn_get_option): */
#define DG_INFO_SPLITS_USED  16 /* partitions the next forward will use */
#define DG_INFO_SCRATCH_BYTES 17 /* device bytes the plan holds */
#define DG_INFO_CACHE_READY  18 /* 1 when dg_attn_cache_prepare has filled the plan's cache copy */
#define DG_INFO_LAUNCHES     19 /* kernels the next dg_attn_forward enqueues with the current options
                                   (without a caller's cos_sin table) */
#define DG_INFO_SCHEDULE_USED 20 /* DG_SCHEDULE_SPLIT or DG_SCHEDULE_STREAM_K: what the next forward
                                   uses (DG_SCHEDULE_SPLIT on the fp32 path) */

/* Create a plan for one geometry on the current device (page: the per-layer geometry that
 * DgGpu::new checks -- n_kv, head_dim, nh % n_kv -- and the scratch buffers canvas_forward sizes
 * for the normed q/k/v; the page's head_dim <= 128 limit is lifted).  Requires nh % nkv == 0,
 * nh, nkv, T >= 1, ctx >= 0, hd in {32, 64, 128, 256} (the tensor-core path needs hd in
 * {64, 128, 256}), eps >= 0, rope_theta > 0, ctx + T < 2^24, nkv * ctx < 2^32.  Returns NULL
 * on error (see
 * dg_attn_last_error()).  Allocates the plan's device scratch with cudaMalloc; the plan is tied
 * to the device that was current at creation. */
dg_attn_plan *dg_attn_plan_create(int nh, int nkv, int hd, int ctx, int T, float eps,
                                  float rope_theta);

/* The schedule of the tensor-core attention kernel that a plan of this geometry would use, on a
 * device with `num_sms` SMs on which max_clusters[s] thread-block clusters of s CTAs (s = 2..8;
 * entries 0 and 1 unused) fit at once, or num_sms / s of each when max_clusters is NULL; with
 * DG_OPT_SPLITS left at 0.  schedule: DG_SCHEDULE_AUTO, _SPLIT or _STREAM_K, as for
 * DG_OPT_SCHEDULE (a stream-K request the geometry cannot take falls back to the split schedule,
 * as a forward would).  Host arithmetic only: touches no device and needs no GPU.
 * out[4]: [0] DG_SCHEDULE_SPLIT or DG_SCHEDULE_STREAM_K; [1] key partitions per query tile
 * (split) or the most pieces any (query tile, kv group) pair is cut into (stream-K); [2] CTAs of
 * the attention kernel; [3] key tiles in the longest CTA's run.  hd must be 64, 128 or 256.
 * Returns DG_ERR_ARG (with dg_attn_last_error()) for a bad geometry or a NULL out. */
int dg_attn_schedule_info(int nh, int nkv, int hd, int ctx, int T, int num_sms,
                          const int *max_clusters, int schedule, long long *out);

/* The whole block (page: canvas_forward's attention branch from the three DG_HEADNORM_ROPE
 * dispatches -- q weighted + RoPE, k weighted + RoPE, v weightless without RoPE -- through the
 * DG_ATTN dispatch): norms + RoPE, attention, output.  k_cache and v_cache are [nkv, ctx, hd];
 * with ctx == 0 they must be NULL (the page's 1-float stub cache).  With ctx > 0 and both NULL
 * the plan uses the cache copy made by the last dg_attn_cache_prepare (DG_ERR_STATE if there is
 * none).  v_canvas may alias k_canvas (the page's k_eq_v layers, whose V is the raw K
 * projection).  out must not overlap any input (DG_ERR_ARG; checked on the byte ranges the plan's
 * sizes give).  Every pointer must be 16-byte aligned (DG_ERR_ALIGN).  Enqueued on `stream`; on
 * the tensor-core path a cache V outside the fp16 range is reported by dg_attn_sync_status
 * (DG_ERR_RANGE), and a cache passed with the call is converted by the first-stage launch
 * itself (it replaces the prepared cache copy: DG_INFO_CACHE_READY becomes 0). */
int dg_attn_forward(dg_attn_plan *plan, const float *q, const float *k_canvas,
                    const float *v_canvas, const float *k_cache, const float *v_cache,
                    const float *q_norm_w, const float *k_norm_w, const float *cos_sin, float *out,
                    cudaStream_t stream);

/* Copy a cache [nkv, ctx, hd] (K and V) into the plan in the tensor-core operand format, once
 * per cache (page: DgGpuCache / upload_cache, the encoder cache rebuilt once per canvas block).  A denoising loop that keeps its cache fixed for many steps calls this once, then
 * dg_attn_forward with k_cache = v_cache = NULL.  The copy is taken on `stream`; the caller may
 * reuse its own buffers once that stream has passed this point.  On the fp32 path the plan
 * keeps the two pointers instead (the caller must keep the buffers alive and unchanged). */
int dg_attn_cache_prepare(dg_attn_plan *plan, const float *k_cache, const float *v_cache,
                          cudaStream_t stream);

/* Element types of a cache for dg_attn_cache_prepare_typed. */
#define DG_DTYPE_F32  0
#define DG_DTYPE_F16  1  /* IEEE half */
#define DG_DTYPE_BF16 2  /* bfloat16 */

/* dg_attn_cache_prepare for a cache held as fp32, or as a 16-bit twin (the f16 K/V twin the page
 * names as a follow-up of its flash kernel: half the bytes to upload and read), [nkv, ctx, hd] of
 * `dtype` each, 16-byte aligned.  Every f16 and bf16 value is exact in fp32, so the result equals
 * dg_attn_cache_prepare on the widened cache.  On the tensor-core path the values go straight
 * into the operand arrays; on the exact path a 16-bit cache is widened into an fp32 copy owned
 * by the plan, allocated (cudaMalloc) by the first such call.  DG_ERR_ARG for an unknown dtype. */
int dg_attn_cache_prepare_typed(dg_attn_plan *plan, const void *k_cache, const void *v_cache,
                                int dtype, cudaStream_t stream);

/* The first stage alone (page: item DG_HEADNORM_ROPE and its three dispatches -- RMSNorm +
 * weight + RoPE on q and k, RMSNorm on v), in fp32, written in the input layouts: q_hat
 * [T, nh*hd], k_hat and v_hat [T, nkv*hd] (not overlapping any input: DG_ERR_ARG). */
int dg_attn_norm_rope(dg_attn_plan *plan, const float *q, const float *k_canvas,
                      const float *v_canvas, const float *q_norm_w, const float *k_norm_w,
                      const float *cos_sin, float *q_hat, float *k_hat, float *v_hat,
                      cudaStream_t stream);

/* The attention stage alone (page: item DG_ATTN and its dispatch), on operands that are already
 * normed and roped (q_hat [T, nh*hd], k_hat / v_hat [T, nkv*hd], cache as in dg_attn_forward),
 * with the plan's current path; out must not overlap an input (DG_ERR_ARG). */
int dg_attn_attend(dg_attn_plan *plan, const float *q_hat, const float *k_hat,
                   const float *v_hat, const float *k_cache, const float *v_cache, float *out,
                   cudaStream_t stream);

/* Set one DG_OPT_* option of a plan (see the keys above for the page item each one follows).
 * DG_ERR_ARG for an unknown key or a value out of range, DG_ERR_UNSUPPORTED for the tensor-core
 * path at hd = 32; changing DG_OPT_SPLITS or DG_OPT_SCHEDULE may grow the plan's partial-result
 * buffers (cudaMalloc). */
int dg_attn_set_option(dg_attn_plan *plan, int key, long long value);
/* Read a DG_OPT_* option or a DG_INFO_* value into *value (host only). */
int dg_attn_get_option(const dg_attn_plan *plan, int key, long long *value);

/* Synchronise `stream`, then read and clear the plan's device status word: DG_OK;
 * DG_ERR_TIMEOUT when a kernel gave up on a bounded wait since the last call; DG_ERR_STATE when a
 * stream-K CTA was handed a run it cannot hold (more than two pairs; the host layout rules this
 * out); DG_ERR_RANGE when a cache converted for the tensor-core path held a V value outside the
 * fp16 range.  No counterpart on the page (its dispatches cannot fail on the device). */
int dg_attn_sync_status(dg_attn_plan *plan, cudaStream_t stream);

/* Stages for dg_attn_profile_read. */
#define DG_STAGE_NORM_ROPE 0  /* the norm + RoPE kernel */
#define DG_STAGE_ATTENTION 1  /* the attention kernel (tensor-core or fp32) */
#define DG_STAGE_COMBINE   2  /* the split-KV combine kernel */
#define DG_STAGE_CACHE     3  /* the cache conversion kernel (dg_attn_cache_prepare, and a cache
                                 passed to dg_attn_forward_hidden; dg_attn_forward and
                                 dg_attn_attend convert one inside the norm + RoPE launch) */
#define DG_STAGE_PROJECTION 4 /* the input norm + q/k/v projection kernels (dg_attn_forward_hidden) */
#define DG_STAGE_OPROJ      5 /* the o_proj, post-attention norm and residual kernels */

/* With DG_OPT_PROFILE on: synchronise on the recorded events, then return the summed device time
 * (ms) and the count of the launches of one stage recorded since the last read of that stage
 * (or since profiling was switched on), and reset that stage's record. */
int dg_attn_profile_read(dg_attn_plan *plan, int stage, double *total_ms, long long *launches);

void dg_attn_plan_destroy(dg_attn_plan *plan);

/* The step before the block (page, canvas_forward, attention branch): the input RMSNorm of the
 * residual stream (`rms!(cur, ln_in)`, item DG_RMSNORM) and the q / k / v projections (`gemm!`:
 * y = x W^T with W [n, k] as GLin stores it), on the tensor cores, with the block's first stage
 * (qk-norm + RoPE, v-norm) fused into the projection's epilogue.
 *
 * dg_attn_proj_prepare stores W diag(ln_in_w) in the plan (bf16 hi/lo, like the block's other
 * tensor-core operands), once per set of weights:
 *   H          hidden size, a positive multiple of 64;
 *   ln_in_w    [H] or NULL (unweighted);
 *   wq [nh*hd, H], wk [nkv*hd, H], wv [nkv*hd, H] or NULL (no value projection: v is the raw k
 *   projection, the page's k_eq_v layers).
 * The weights are read on `stream`; the caller may reuse them once the stream has passed this
 * point.  The first call (and a call with another H or another wv-NULLness) allocates the plan's
 * projection scratch with cudaMalloc.  Needs the tensor-core path and hd 128 or 256
 * (DG_ERR_UNSUPPORTED otherwise); DG_ERR_ARG for a bad H or a NULL wq/wk. */
int dg_attn_proj_prepare(dg_attn_plan *plan, int H, const float *ln_in_w, const float *wq,
                         const float *wk, const float *wv, cudaStream_t stream);

/* The block from the residual stream x [T, H] (fp32): input norm, projections, first stage,
 * attention, output as dg_attn_forward.  Cache, weights, table and out as in dg_attn_forward.
 * DG_ERR_STATE without dg_attn_proj_prepare; DG_ERR_UNSUPPORTED on the exact path. */
int dg_attn_forward_hidden(dg_attn_plan *plan, const float *x, const float *k_cache,
                           const float *v_cache, const float *q_norm_w, const float *k_norm_w,
                           const float *cos_sin, float *out, cudaStream_t stream);

/* The step after the block (page, canvas_forward, attention branch): `gemm!(sb, o)` (o_proj,
 * y = attn W_o^T, W_o [H, nh*hd]), `rms!(nb, ln_post_attn)` (weighted RMSNorm of y, item
 * DG_RMSNORM) and `add_scale!(cur, sb, 1.0)` (item DG_ADD_SCALE): resid = resid + RMSNorm(y) w.
 * The product runs on the tensor cores (bf16 hi/lo split, like the projection step); the norm,
 * which needs whole rows of H, and the residual add run in a second kernel.
 *
 * dg_attn_oproj_prepare stores W_o [H, nh*hd] (and ln_post_w [H], or NULL for unweighted) in the
 * plan, once per set of weights; H a positive multiple of 64.  The first call (and a call with
 * another H) allocates the plan's o_proj scratch with cudaMalloc.
 * dg_attn_oproj_residual applies the step to attn_out [T, nh*hd] (fp32, e.g. dg_attn_forward's
 * out) and updates resid [T, H] (fp32) in place.  DG_ERR_STATE without preparation. */
int dg_attn_oproj_prepare(dg_attn_plan *plan, int H, const float *wo, const float *ln_post_w,
                          cudaStream_t stream);
int dg_attn_oproj_residual(dg_attn_plan *plan, const float *attn_out, float *resid,
                           cudaStream_t stream);

/* The whole attention branch of a decoder layer on the residual stream resid [T, H], in place:
 * input norm and projections (dg_attn_proj_prepare), the block, o_proj, post-attention norm and
 * residual add (dg_attn_oproj_prepare, same H).  The block's output stays inside the plan and
 * is not returned: as o_proj's bf16 hi/lo operands, written by the attention kernel itself, or
 * in fp32 first under the schedules that finish in a combine kernel. */
int dg_attn_forward_layer(dg_attn_plan *plan, float *resid, const float *k_cache,
                          const float *v_cache, const float *q_norm_w, const float *k_norm_w,
                          const float *cos_sin, cudaStream_t stream);

/* Allocation-free forward.  The pages have no counterpart: this entry point exists for callers
 * that cannot call cudaMalloc when they run attention (code inside a memory pool or arena it does
 * not own, or a process whose device memory is reserved up front).  It computes the same block
 * as dg_attn_forward on the exact-fp32 path with one key-range partition, without a plan: its
 * working memory is a fixed 16 MiB __device__ array inside the library (held on every GPU that
 * loads the library until the process exits), so it allocates nothing.  Sizes must satisfy
 * a(hd*8) + a(T*nh*hd*4) + 2*a(T*nkv*hd*4) <= 16 MiB, where a(x) rounds x up to a multiple of
 * 256 (checked on the host: DG_ERR_ARG otherwise); every pointer must be 16-byte aligned (checked
 * on the host: DG_ERR_ALIGN); other requirements as for dg_attn_plan_create / dg_attn_forward;
 * pos0 < 0 means pos0 = ctx.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress), so make it before any stream
 * capture.  Calls share the array: calls that overlap on the GPU race and must be serialised by
 * the caller.  Host-side errors are described by dg_attn_noalloc_last_error(). */
int dg_attn_forward_noalloc(int nh, int nkv, int hd, int ctx, int T, float eps,
                            float rope_theta, long long pos0, const float *q,
                            const float *k_canvas, const float *v_canvas, const float *k_cache,
                            const float *v_cache, const float *q_norm_w, const float *k_norm_w,
                            const float *cos_sin, float *out, cudaStream_t stream);
const char *dg_attn_noalloc_last_error(void);

/* A static description of a DG_* status code. */
const char *dg_attn_status_string(int status);
/* The text of the calling thread's last host-side error (a static thread-local buffer). */
const char *dg_attn_last_error(void);
/* The build identity of the loaded library: "sha1:<hex>" of the CUDA sources and this header it
 * was compiled from, hashed by the build script (a static string). */
const char *dg_attn_build_id(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_ATTN_H */
