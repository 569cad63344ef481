"""ctypes binding of libdgattn.so (include/dg_attn.h), names unchanged.

Argument marshalling only: torch tensors become device pointers, the current torch stream becomes
the ``cudaStream_t``.  Every step of the block runs in the library's CUDA kernels; if the library
is missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdgattn.so")

# status codes and option keys (mirrors include/dg_attn.h)
DG_OK, DG_ERR_ARG, DG_ERR_ALIGN, DG_ERR_CUDA, DG_ERR_TIMEOUT, DG_ERR_UNSUPPORTED, DG_ERR_STATE = range(7)
DG_ERR_RANGE = 7
DG_PATH_TC, DG_PATH_FP32 = 0, 1
DG_OPT_PATH, DG_OPT_POS0, DG_OPT_SPLITS, DG_OPT_WAIT_LIMIT_MS, DG_OPT_PROFILE = 1, 2, 3, 4, 5
DG_OPT_INJECT_STALL = 6
DG_OPT_INPUTS_RESIDENT = 7
DG_OPT_SCHEDULE = 8
DG_SCHEDULE_AUTO, DG_SCHEDULE_SPLIT, DG_SCHEDULE_STREAM_K = 0, 1, 2
DG_DTYPE_F32, DG_DTYPE_F16, DG_DTYPE_BF16 = 0, 1, 2
DG_INFO_SPLITS_USED, DG_INFO_SCRATCH_BYTES, DG_INFO_CACHE_READY, DG_INFO_LAUNCHES = 16, 17, 18, 19
DG_INFO_SCHEDULE_USED = 20
DG_STAGE_NORM_ROPE, DG_STAGE_ATTENTION, DG_STAGE_COMBINE, DG_STAGE_CACHE = 0, 1, 2, 3
DG_STAGE_PROJECTION = 4
DG_STAGE_OPROJ = 5

EXPORTED = [
    "dg_attn_plan_create", "dg_attn_forward", "dg_attn_cache_prepare",
    "dg_attn_cache_prepare_typed", "dg_attn_proj_prepare", "dg_attn_forward_hidden",
    "dg_attn_oproj_prepare", "dg_attn_oproj_residual", "dg_attn_forward_layer",
    "dg_attn_norm_rope",
    "dg_attn_attend", "dg_attn_set_option", "dg_attn_get_option", "dg_attn_sync_status",
    "dg_attn_profile_read", "dg_attn_plan_destroy", "dg_attn_status_string", "dg_attn_last_error",
    "dg_attn_forward_noalloc", "dg_attn_noalloc_last_error", "dg_attn_schedule_info",
    "dg_attn_build_id",
]

_lib = None


class DgAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)}): {last_error()}")


def load(path: str = LIB_PATH):
    """Load the library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with gqa_canvas_attention_gb300.build")
    lib = ctypes.CDLL(path)
    P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    lib.dg_attn_plan_create.argtypes = [I, I, I, I, I, ctypes.c_float, ctypes.c_float]
    lib.dg_attn_plan_create.restype = P
    lib.dg_attn_forward.argtypes = [P] * 11
    lib.dg_attn_forward.restype = I
    lib.dg_attn_cache_prepare.argtypes = [P, P, P, P]
    lib.dg_attn_cache_prepare.restype = I
    lib.dg_attn_cache_prepare_typed.argtypes = [P, P, P, I, P]
    lib.dg_attn_cache_prepare_typed.restype = I
    lib.dg_attn_proj_prepare.argtypes = [P, I, P, P, P, P, P]
    lib.dg_attn_proj_prepare.restype = I
    lib.dg_attn_forward_hidden.argtypes = [P] * 9
    lib.dg_attn_forward_hidden.restype = I
    lib.dg_attn_oproj_prepare.argtypes = [P, I, P, P, P]
    lib.dg_attn_oproj_prepare.restype = I
    lib.dg_attn_oproj_residual.argtypes = [P, P, P, P]
    lib.dg_attn_oproj_residual.restype = I
    lib.dg_attn_forward_layer.argtypes = [P] * 8
    lib.dg_attn_forward_layer.restype = I
    lib.dg_attn_norm_rope.argtypes = [P] * 11
    lib.dg_attn_norm_rope.restype = I
    lib.dg_attn_attend.argtypes = [P] * 8
    lib.dg_attn_attend.restype = I
    lib.dg_attn_set_option.argtypes = [P, I, LL]
    lib.dg_attn_set_option.restype = I
    lib.dg_attn_get_option.argtypes = [P, I, ctypes.POINTER(LL)]
    lib.dg_attn_get_option.restype = I
    lib.dg_attn_sync_status.argtypes = [P, P]
    lib.dg_attn_sync_status.restype = I
    lib.dg_attn_profile_read.argtypes = [P, I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(LL)]
    lib.dg_attn_profile_read.restype = I
    lib.dg_attn_plan_destroy.argtypes = [P]
    lib.dg_attn_plan_destroy.restype = None
    lib.dg_attn_status_string.argtypes = [I]
    lib.dg_attn_status_string.restype = ctypes.c_char_p
    lib.dg_attn_last_error.argtypes = []
    lib.dg_attn_last_error.restype = ctypes.c_char_p
    lib.dg_attn_forward_noalloc.argtypes = ([I] * 5 + [ctypes.c_float, ctypes.c_float, LL] +
                                            [P] * 10)
    lib.dg_attn_forward_noalloc.restype = I
    lib.dg_attn_noalloc_last_error.argtypes = []
    lib.dg_attn_noalloc_last_error.restype = ctypes.c_char_p
    lib.dg_attn_schedule_info.argtypes = [I, I, I, I, I, I, P, I, P]
    lib.dg_attn_schedule_info.restype = I
    lib.dg_attn_build_id.argtypes = []
    lib.dg_attn_build_id.restype = ctypes.c_char_p
    _lib = lib
    return lib


def dg_attn_schedule_info(nh, nkv, hd, ctx, T, num_sms, max_clusters=None,
                          schedule=DG_SCHEDULE_AUTO):
    """The tensor-core schedule a plan of this geometry would use (host arithmetic, no GPU):
    (schedule, partitions or most pieces of a pair, CTAs, key tiles of the longest run)."""
    lib = _lib or load()
    out = (ctypes.c_longlong * 4)()
    mc = None
    if max_clusters is not None:
        mc = (ctypes.c_int * len(max_clusters))(*max_clusters)
    rc = lib.dg_attn_schedule_info(nh, nkv, hd, ctx, T, num_sms,
                                   ctypes.cast(mc, ctypes.c_void_p) if mc is not None else None,
                                   schedule, out)
    if rc != DG_OK:
        raise DgAttnError(rc, "dg_attn_schedule_info")
    return tuple(int(v) for v in out)


def build_id() -> str:
    """The loaded library's build identity ("sha1:<hex>" of its sources)."""
    return load().dg_attn_build_id().decode()


def status_string(status: int) -> str:
    return load().dg_attn_status_string(int(status)).decode()


def last_error() -> str:
    return load().dg_attn_last_error().decode()


def _ptr(t):
    """Address of a tensor (or a raw integer address), or None.  A tensor must be contiguous:
    the library reads dense row-major buffers."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("the library reads dense row-major buffers: pass a contiguous tensor")
    return t.data_ptr()


def _check_tensors(device, *specs):
    """Reject, before any library call, a tensor the library would misread.  Each spec is
    (tensor or None, name, element count[, dtypes]); every tensor is first checked for its type,
    dtype (float32 unless given), contiguity and element count, then all of them for living on
    the plan's CUDA device."""
    import torch
    for spec in specs:
        t, name, numel = spec[:3]
        dtypes = spec[3] if len(spec) > 3 else (torch.float32,)
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
        if t.dtype not in dtypes:
            raise ValueError(f"{name}: dtype {t.dtype}, expected {' or '.join(map(str, dtypes))}")
        if not t.is_contiguous():
            raise ValueError(f"{name}: must be contiguous (dense row-major)")
        if t.numel() != numel:
            raise ValueError(f"{name}: {t.numel()} elements ({tuple(t.shape)}), expected {numel}")
    for spec in specs:
        t, name = spec[:2]
        if t is not None and (t.device.type != "cuda" or
                              (device is not None and t.device.index != device)):
            raise ValueError(f"{name}: must live on cuda:{device} (the plan's device), not "
                             f"{t.device}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != DG_OK:
        raise DgAttnError(rc, what)


def dg_attn_plan_create(nh, nkv, hd, ctx, T, eps, rope_theta):
    h = load().dg_attn_plan_create(nh, nkv, hd, ctx, T, float(eps), float(rope_theta))
    if not h:
        raise RuntimeError(f"dg_attn_plan_create: {last_error()}")
    return h


def dg_attn_plan_destroy(plan):
    load().dg_attn_plan_destroy(plan)


def dg_attn_forward(plan, q, k_canvas, v_canvas, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin,
                    out, stream=None):
    rc = load().dg_attn_forward(plan, _ptr(q), _ptr(k_canvas), _ptr(v_canvas), _ptr(k_cache),
                                _ptr(v_cache), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(cos_sin),
                                _ptr(out), _stream(stream))
    _check(rc, "dg_attn_forward")


def dg_attn_cache_prepare(plan, k_cache, v_cache, stream=None):
    _check(load().dg_attn_cache_prepare(plan, _ptr(k_cache), _ptr(v_cache), _stream(stream)),
           "dg_attn_cache_prepare")


def dg_attn_proj_prepare(plan, H, ln_in_w, wq, wk, wv=None, stream=None):
    _check(load().dg_attn_proj_prepare(plan, int(H), _ptr(ln_in_w), _ptr(wq), _ptr(wk), _ptr(wv),
                                       _stream(stream)), "dg_attn_proj_prepare")


def dg_attn_forward_hidden(plan, x, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, out,
                           stream=None):
    _check(load().dg_attn_forward_hidden(plan, _ptr(x), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(q_norm_w), _ptr(k_norm_w), _ptr(cos_sin), _ptr(out),
                                         _stream(stream)), "dg_attn_forward_hidden")


def dg_attn_oproj_prepare(plan, H, wo, ln_post_w=None, stream=None):
    _check(load().dg_attn_oproj_prepare(plan, int(H), _ptr(wo), _ptr(ln_post_w), _stream(stream)),
           "dg_attn_oproj_prepare")


def dg_attn_oproj_residual(plan, attn_out, resid, stream=None):
    _check(load().dg_attn_oproj_residual(plan, _ptr(attn_out), _ptr(resid), _stream(stream)),
           "dg_attn_oproj_residual")


def dg_attn_forward_layer(plan, resid, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin,
                          stream=None):
    _check(load().dg_attn_forward_layer(plan, _ptr(resid), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(q_norm_w), _ptr(k_norm_w), _ptr(cos_sin),
                                        _stream(stream)), "dg_attn_forward_layer")


def dg_attn_cache_prepare_typed(plan, k_cache, v_cache, dtype, stream=None):
    _check(load().dg_attn_cache_prepare_typed(plan, _ptr(k_cache), _ptr(v_cache), int(dtype),
                                              _stream(stream)),
           "dg_attn_cache_prepare_typed")


def dg_attn_norm_rope(plan, q, k_canvas, v_canvas, q_norm_w, k_norm_w, cos_sin, q_hat, k_hat,
                      v_hat, stream=None):
    rc = load().dg_attn_norm_rope(plan, _ptr(q), _ptr(k_canvas), _ptr(v_canvas), _ptr(q_norm_w),
                                  _ptr(k_norm_w), _ptr(cos_sin), _ptr(q_hat), _ptr(k_hat),
                                  _ptr(v_hat), _stream(stream))
    _check(rc, "dg_attn_norm_rope")


def dg_attn_attend(plan, q_hat, k_hat, v_hat, k_cache, v_cache, out, stream=None):
    rc = load().dg_attn_attend(plan, _ptr(q_hat), _ptr(k_hat), _ptr(v_hat), _ptr(k_cache),
                               _ptr(v_cache), _ptr(out), _stream(stream))
    _check(rc, "dg_attn_attend")


def dg_attn_forward_noalloc(nh, nkv, hd, ctx, T, eps, rope_theta, pos0, q, k_canvas, v_canvas,
                            k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, out, stream=None):
    """The allocation-free fp32 forward (no plan); returns the status code."""
    return load().dg_attn_forward_noalloc(nh, nkv, hd, ctx, T, float(eps), float(rope_theta),
                                          int(pos0), _ptr(q), _ptr(k_canvas), _ptr(v_canvas),
                                          _ptr(k_cache), _ptr(v_cache), _ptr(q_norm_w),
                                          _ptr(k_norm_w), _ptr(cos_sin), _ptr(out),
                                          _stream(stream))


def dg_attn_set_option(plan, key, value):
    _check(load().dg_attn_set_option(plan, int(key), int(value)), "dg_attn_set_option")


def dg_attn_get_option(plan, key) -> int:
    v = ctypes.c_longlong(0)
    _check(load().dg_attn_get_option(plan, int(key), ctypes.byref(v)), "dg_attn_get_option")
    return v.value


def dg_attn_sync_status(plan, stream=None) -> int:
    """Returns the device status (DG_OK, DG_ERR_TIMEOUT or DG_ERR_RANGE) instead of raising."""
    rc = load().dg_attn_sync_status(plan, _stream(stream))
    if rc not in (DG_OK, DG_ERR_TIMEOUT, DG_ERR_RANGE):
        raise DgAttnError(rc, "dg_attn_sync_status")
    return rc


def dg_attn_profile_read(plan, stage):
    ms = ctypes.c_double(0.0)
    n = ctypes.c_longlong(0)
    _check(load().dg_attn_profile_read(plan, int(stage), ctypes.byref(ms), ctypes.byref(n)),
           "dg_attn_profile_read")
    return ms.value, n.value


class Plan:
    """Owning handle around a dg_attn_plan (created on the current CUDA device)."""

    def __init__(self, nh, nkv, hd, ctx, T, eps=1e-6, rope_theta=10000.0):
        import torch
        self.nh, self.nkv, self.hd, self.ctx, self.T = nh, nkv, hd, ctx, T
        self.H = self.oH = None
        self.device = torch.cuda.current_device()
        self.handle = dg_attn_plan_create(nh, nkv, hd, ctx, T, eps, rope_theta)

    # element counts of the buffers of this geometry
    def _nq(self):
        return self.T * self.nh * self.hd

    def _nk(self):
        return self.T * self.nkv * self.hd

    def _nc(self):
        return self.nkv * self.ctx * self.hd

    def _check_canvas(self, q, k_canvas, v_canvas, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin,
                      out, q_name="q", k_name="k_canvas", v_name="v_canvas"):
        _check_tensors(self.device, (q, q_name, self._nq()), (k_canvas, k_name, self._nk()),
                       (v_canvas, v_name, self._nk()), (k_cache, "k_cache", self._nc()),
                       (v_cache, "v_cache", self._nc()), (q_norm_w, "q_norm_w", self.hd),
                       (k_norm_w, "k_norm_w", self.hd), (cos_sin, "cos_sin", 2 * self.T * self.hd),
                       (out, "out", self._nq()))

    def close(self):
        if self.handle:
            dg_attn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set(self, key, value):
        dg_attn_set_option(self.handle, key, value)
        return self

    def get(self, key):
        return dg_attn_get_option(self.handle, key)

    def forward(self, q, k_canvas, v_canvas, k_cache=None, v_cache=None, q_norm_w=None,
                k_norm_w=None, cos_sin=None, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((self.T, self.nh * self.hd), dtype=torch.float32, device=q.device)
        self._check_canvas(q, k_canvas, v_canvas, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin,
                           out)
        dg_attn_forward(self.handle, q, k_canvas, v_canvas, k_cache, v_cache, q_norm_w, k_norm_w,
                        cos_sin, out, stream)
        return out

    def proj_prepare(self, H, ln_in_w, wq, wk, wv=None, stream=None):
        _check_tensors(self.device, (ln_in_w, "ln_in_w", H), (wq, "wq", self.nh * self.hd * H),
                       (wk, "wk", self.nkv * self.hd * H), (wv, "wv", self.nkv * self.hd * H))
        dg_attn_proj_prepare(self.handle, H, ln_in_w, wq, wk, wv, stream)
        self.H = H

    def forward_hidden(self, x, k_cache=None, v_cache=None, q_norm_w=None, k_norm_w=None,
                       cos_sin=None, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((self.T, self.nh * self.hd), dtype=torch.float32, device=x.device)
        if self.H is not None:
            _check_tensors(self.device, (x, "x", self.T * self.H))
        self._check_canvas(out, None, None, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, None,
                           q_name="out")
        dg_attn_forward_hidden(self.handle, x, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, out,
                               stream)
        return out

    def oproj_prepare(self, H, wo, ln_post_w=None, stream=None):
        _check_tensors(self.device, (wo, "wo", H * self.nh * self.hd), (ln_post_w, "ln_post_w", H))
        dg_attn_oproj_prepare(self.handle, H, wo, ln_post_w, stream)
        self.oH = H

    def oproj_residual(self, attn_out, resid, stream=None):
        _check_tensors(self.device, (attn_out, "attn_out", self._nq()),
                       (resid, "resid", self.T * self.oH if self.oH is not None else resid.numel()))
        dg_attn_oproj_residual(self.handle, attn_out, resid, stream)

    def forward_layer(self, resid, k_cache=None, v_cache=None, q_norm_w=None, k_norm_w=None,
                      cos_sin=None, stream=None):
        if self.H is not None:
            _check_tensors(self.device, (resid, "resid", self.T * self.H))
        self._check_canvas(None, None, None, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin, None)
        dg_attn_forward_layer(self.handle, resid, k_cache, v_cache, q_norm_w, k_norm_w, cos_sin,
                              stream)
        return resid

    def cache_prepare(self, k_cache, v_cache, stream=None):
        """fp32, float16 or bfloat16 cache tensors [nkv, ctx, hd] (both of one dtype)."""
        import torch
        types = {torch.float32: DG_DTYPE_F32, torch.float16: DG_DTYPE_F16,
                 torch.bfloat16: DG_DTYPE_BF16}
        if k_cache.dtype not in types or v_cache.dtype != k_cache.dtype:
            raise ValueError("cache tensors must both be float32, float16 or bfloat16")
        _check_tensors(self.device, (k_cache, "k_cache", self._nc(), (k_cache.dtype,)),
                       (v_cache, "v_cache", self._nc(), (k_cache.dtype,)))
        dg_attn_cache_prepare_typed(self.handle, k_cache, v_cache, types[k_cache.dtype], stream)

    def norm_rope(self, q, k_canvas, v_canvas, q_norm_w=None, k_norm_w=None, cos_sin=None,
                  stream=None):
        import torch
        self._check_canvas(q, k_canvas, v_canvas, None, None, q_norm_w, k_norm_w, cos_sin, None)
        qh = torch.empty_like(q)
        kh = torch.empty_like(k_canvas)
        vh = torch.empty_like(v_canvas)
        dg_attn_norm_rope(self.handle, q, k_canvas, v_canvas, q_norm_w, k_norm_w, cos_sin, qh, kh,
                          vh, stream)
        return qh, kh, vh

    def attend(self, q_hat, k_hat, v_hat, k_cache=None, v_cache=None, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((self.T, self.nh * self.hd), dtype=torch.float32, device=q_hat.device)
        self._check_canvas(q_hat, k_hat, v_hat, k_cache, v_cache, None, None, None, out,
                           "q_hat", "k_hat", "v_hat")
        dg_attn_attend(self.handle, q_hat, k_hat, v_hat, k_cache, v_cache, out, stream)
        return out

    def sync_status(self, stream=None) -> int:
        return dg_attn_sync_status(self.handle, stream)
