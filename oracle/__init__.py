"""fp64 CPU oracle for the DiffusionGemma canvas attention block -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import this
package.  The product library never calls it and shares no code with it.

The arithmetic lives in ``dg_oracle.c`` (plain C, fp64, written from the page
"inferencelayer 0.2.3, src/diffusion_gemma_gpu.rs": items DG_HEADNORM_ROPE and DG_ATTN and the
head-norm / attention dispatches of ``canvas_forward``).  This module only compiles it with gcc
and marshals numpy arrays across ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_oracle.c")
_LIB = os.path.join(_HERE, "libdgoracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile dg_oracle.c into oracle/libdgoracle.so with gcc (-O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.dgo_norm_rope.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                      ctypes.c_double, ctypes.c_int, ctypes.c_longlong,
                                      ctypes.c_double, P, P]
        lib.dgo_norm_rope.restype = None
        lib.dgo_attention.argtypes = [P, P, P, P, P] + [ctypes.c_int] * 7 + [P]
        lib.dgo_attention.restype = None
        lib.dgo_forward.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_double,
                                    ctypes.c_longlong] + [P] * 8 + [ctypes.c_int, ctypes.c_int, P])
        lib.dgo_forward.restype = ctypes.c_int
        lib.dgo_rmsnorm_rows.argtypes = [P, ctypes.c_int, ctypes.c_int, P, ctypes.c_double, P]
        lib.dgo_rmsnorm_rows.restype = None
        lib.dgo_linear.argtypes = [P, ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P]
        lib.dgo_linear.restype = None
        lib.dgo_oproj_residual.argtypes = [P, ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P,
                                           ctypes.c_double, ctypes.c_double, P, P]
        lib.dgo_oproj_residual.restype = None
        lib.dgo_set_threads.argtypes = [ctypes.c_int]
        lib.dgo_set_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f32(a):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (n > 0) and return the count in force."""
    return _load().dgo_set_threads(int(n))


def norm_rope(x, heads: int, hd: int, w=None, eps: float = 1e-6, rope: bool = True,
              pos0: int = 0, theta: float = 10000.0, cos_sin=None) -> np.ndarray:
    """Per-(row, head) RMSNorm (optional weight) then optional NeoX RoPE; x is [rows, heads*hd].

    Returns fp64 [rows, heads, hd]."""
    x = _f32(x).reshape(-1, heads * hd)
    rows = x.shape[0]
    w = _f32(w)
    cs = _f32(cos_sin)
    if cs is not None:
        cs = cs.reshape(rows, 2 * hd)
    out = np.empty((rows, heads, hd), dtype=np.float64)
    _load().dgo_norm_rope(_ptr(x), rows, heads, hd, _ptr(w), float(eps), int(bool(rope)),
                          int(pos0), float(theta), _ptr(cs), _ptr(out))
    return out


def attention(qhat, khat, vhat, k_cache, v_cache, nh: int, nkv: int, hd: int,
              rows=None) -> np.ndarray:
    """Attention core on already-normed canvas inputs (fp64 [T, nh|nkv, hd]) and a cache
    ([nkv, ctx, hd], used as given).  Returns fp64 [T, nh, hd] (rows outside ``rows`` are 0)."""
    qhat = _f64(qhat).reshape(-1, nh, hd)
    T = qhat.shape[0]
    khat = _f64(khat).reshape(T, nkv, hd)
    vhat = _f64(vhat).reshape(T, nkv, hd)
    if k_cache is None or np.asarray(k_cache).size == 0:
        ctx = 0
        kc = vc = None
    else:
        kc = _f32(k_cache).reshape(nkv, -1, hd)
        vc = _f32(v_cache).reshape(nkv, -1, hd)
        ctx = kc.shape[1]
    r0, r1 = (0, T) if rows is None else rows
    out = np.zeros((T, nh, hd), dtype=np.float64)
    _load().dgo_attention(_ptr(qhat), _ptr(khat), _ptr(vhat), _ptr(kc), _ptr(vc), T, ctx, nh,
                          nkv, hd, int(r0), int(r1), _ptr(out))
    return out


def forward(q, k_canvas, v_canvas, k_cache, v_cache, nh: int, nkv: int, hd: int,
            q_norm_w=None, k_norm_w=None, cos_sin=None, eps: float = 1e-6,
            theta: float = 10000.0, pos0=None, rows=None) -> np.ndarray:
    """The whole attention block on fp32 inputs.  Returns fp64 out [T, nh*hd].

    q [T, nh*hd]; k_canvas, v_canvas [T, nkv*hd] (raw); k_cache, v_cache [nkv, ctx, hd] or
    None when ctx = 0; norm weights [hd] or None; cos_sin [T, 2*hd] or None; pos0 defaults to
    ctx.  ``rows=(r0, r1)`` restricts the computed query rows (others are left 0)."""
    q = _f32(q)
    T = q.size // (nh * hd)
    q = q.reshape(T, nh * hd)
    kcv = _f32(k_canvas).reshape(T, nkv * hd)
    vcv = _f32(v_canvas).reshape(T, nkv * hd)
    if k_cache is None or np.asarray(k_cache).size == 0:
        ctx, kc, vc = 0, None, None
    else:
        kc = _f32(k_cache).reshape(nkv, -1, hd)
        vc = _f32(v_cache).reshape(nkv, -1, hd)
        ctx = kc.shape[1]
    if pos0 is None:
        pos0 = ctx
    cs = _f32(cos_sin)
    if cs is not None:
        cs = cs.reshape(T, 2 * hd)
    r0, r1 = (0, T) if rows is None else rows
    wq, wk = _f32(q_norm_w), _f32(k_norm_w)
    out = np.zeros((T, nh * hd), dtype=np.float64)
    rc = _load().dgo_forward(nh, nkv, hd, ctx, T, float(eps), float(theta), int(pos0), _ptr(q),
                             _ptr(kcv), _ptr(vcv), _ptr(kc), _ptr(vc), _ptr(wq), _ptr(wk),
                             _ptr(cs), int(r0), int(r1), _ptr(out))
    if rc != 0:
        raise ValueError("oracle: bad sizes")
    return out


def rmsnorm_rows(x, w=None, eps: float = 1e-6) -> np.ndarray:
    """Row RMSNorm of x [rows, h] (fp32) with optional weight [h]; fp64 [rows, h]."""
    x = _f32(x)
    rows, h = x.shape
    out = np.empty((rows, h), dtype=np.float64)
    _load().dgo_rmsnorm_rows(_ptr(x), rows, h, _ptr(_f32(w)), float(eps), _ptr(out))
    return out


def linear(xhat, W) -> np.ndarray:
    """y = xhat W^T with xhat [rows, k] (fp64) and W [n, k] (fp32); fp64 [rows, n]."""
    xhat = _f64(xhat)
    W = _f32(W)
    rows, k = xhat.shape
    n = W.shape[0]
    assert W.shape[1] == k
    out = np.empty((rows, n), dtype=np.float64)
    _load().dgo_linear(_ptr(xhat), rows, k, _ptr(W), n, _ptr(out))
    return out


def project_qkv(x, ln_in_w, wq, wk, wv=None, eps: float = 1e-6):
    """The attention branch's input RMSNorm and q / k / v projections (fp64).  With wv None the
    value projection is the raw k projection (the page's k_eq_v layers)."""
    xhat = rmsnorm_rows(x, ln_in_w, eps)
    q = linear(xhat, wq)
    k = linear(xhat, wk)
    v = k.copy() if wv is None else linear(xhat, wv)
    return q, k, v


def forward_hidden(x, ln_in_w, wq, wk, wv, k_cache, v_cache, nh: int, nkv: int, hd: int,
                   q_norm_w=None, k_norm_w=None, cos_sin=None, eps: float = 1e-6,
                   theta: float = 10000.0, pos0=None, rows=None) -> np.ndarray:
    """Projection then the block: the projections enter the block as fp32 (the page's buffers
    hold them in f32).  Returns fp64 out [T, nh*hd]."""
    q, k, v = project_qkv(x, ln_in_w, wq, wk, wv, eps)
    f = lambda a: a.astype(np.float32)
    return forward(f(q), f(k), f(v), k_cache, v_cache, nh, nkv, hd, q_norm_w, k_norm_w,
                   cos_sin=cos_sin, eps=eps, theta=theta, pos0=pos0, rows=rows)


def oproj_residual(attn, wo, ln_post_w, resid, eps: float = 1e-6, scale: float = 1.0):
    """The residual stream after the attention branch: (resid + RMSNorm(attn Wo^T) w) * scale,
    attn [T, k], Wo [h, k], w [h] or None, resid [T, h] (all fp32).  fp64 [T, h]."""
    attn = _f32(attn)
    rows, k = attn.shape
    wo = _f32(wo)
    h = wo.shape[0]
    assert wo.shape[1] == k
    resid = _f32(resid).reshape(rows, h)
    out = np.empty((rows, h), dtype=np.float64)
    _load().dgo_oproj_residual(_ptr(attn), rows, k, _ptr(wo), h, _ptr(_f32(ln_post_w)),
                               float(eps), float(scale), _ptr(resid), _ptr(out))
    return out
