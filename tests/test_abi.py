"""CPU-side checks of the C ABI: the library builds, loads, and exports every entry point that
include/dg_attn.h declares; host-side errors come back as status codes without a GPU."""
import os
import re

import pytest

from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dg_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_attn_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert len(syms) >= 12
    for s in syms:
        assert hasattr(lib, s), f"{s} missing from libdgattn.so"
    assert sorted(B.EXPORTED) == syms


def test_status_strings(lib):
    assert B.status_string(B.DG_OK) == "ok"
    assert "timed out" in B.status_string(B.DG_ERR_TIMEOUT)
    assert B.status_string(99) == "unknown status"


def test_bad_geometry_is_rejected_before_any_device_call(lib):
    for args in [(6, 4, 64, 0, 8), (4, 2, 48, 0, 8), (4, 2, 64, -1, 8), (4, 2, 64, 0, 0)]:
        h = lib.dg_attn_plan_create(*args, 1e-6, 10000.0)
        assert not h
        assert B.last_error()
    # positions: ctx + T < 2^24
    assert not lib.dg_attn_plan_create(2, 1, 64, (1 << 24) - 8, 8, 1e-6, 10000.0)
    assert "2^24" in B.last_error()
    # cache rows (kv head, row) are numbered in 32 bits: nkv * ctx < 2^32
    assert not lib.dg_attn_plan_create(512, 512, 64, 1 << 23, 8, 1e-6, 10000.0)
    assert "2^32" in B.last_error()


def test_null_plan_is_an_argument_error(lib):
    assert lib.dg_attn_set_option(None, B.DG_OPT_SPLITS, 2) == B.DG_ERR_ARG
    assert lib.dg_attn_forward(None, *([None] * 10)) == B.DG_ERR_ARG


def test_header_option_values_match_binding():
    src = open(os.path.join(ROOT, "include", "dg_attn.h")).read()
    vals = dict(re.findall(r"#define\s+(DG_\w+)\s+(\d+)", src))
    for name, v in vals.items():
        assert getattr(B, name) == int(v), name


def test_noalloc_entry_point_checks_sizes_on_the_host(lib):
    # rejected before any CUDA call: nh % nkv != 0, and a size beyond the fixed scratch
    assert B.dg_attn_forward_noalloc(6, 4, 64, 0, 8, 1e-6, 1e4, -1, 16, 16, 16, None, None,
                                     None, None, None, 16, stream=0) == B.DG_ERR_ARG
    assert B.dg_attn_forward_noalloc(16, 16, 64, 0, 4096, 1e-6, 1e4, -1, 16, 16, 16, None,
                                     None, None, None, None, 16, stream=0) == B.DG_ERR_ARG
    assert "scratch" in lib.dg_attn_noalloc_last_error().decode()


def test_noalloc_entry_point_checks_alignment_and_its_bound_on_the_host(lib):
    """A misaligned pointer is DG_ERR_ALIGN and one canvas row beyond the fixed scratch is
    DG_ERR_ARG, both before any CUDA call (the pointers here are never dereferenced).  The bound
    is the sum of four regions rounded up to 256 bytes: for nh = nkv = 1, hd = 128, ctx = 0 that
    is 64 * 16 + 3 * T * 512 <= 16 MiB (the frequencies as four floats each), so T = 10922 fits
    exactly (run on the GPU) and T = 10923 does not."""
    args = (1, 1, 128, 0)
    ok = 1 << 20                                  # a 16-byte-aligned stand-in address
    assert B.dg_attn_forward_noalloc(*args, 8, 1e-6, 1e4, -1, ok + 4, ok, ok, None, None, None,
                                     None, None, ok, stream=0) == B.DG_ERR_ALIGN
    assert B.dg_attn_forward_noalloc(*args, 8, 1e-6, 1e4, -1, ok, ok, ok, None, None, None,
                                     None, ok + 8, ok, stream=0) == B.DG_ERR_ALIGN
    assert "aligned" in lib.dg_attn_noalloc_last_error().decode()
    assert B.dg_attn_forward_noalloc(*args, 10923, 1e-6, 1e4, -1, ok, ok, ok, None, None, None,
                                     None, None, ok, stream=0) == B.DG_ERR_ARG
    assert "scratch" in lib.dg_attn_noalloc_last_error().decode()
    assert 64 * 16 + 3 * 10922 * 512 == 16 << 20


def test_null_plan_is_an_argument_error_for_every_entry_point(lib):
    """Every entry point that takes a plan checks it on the host before any CUDA call."""
    assert lib.dg_attn_cache_prepare_typed(None, None, None, B.DG_DTYPE_F16, None) == B.DG_ERR_ARG
    assert lib.dg_attn_proj_prepare(None, 64, None, None, None, None, None) == B.DG_ERR_ARG
    assert lib.dg_attn_forward_hidden(None, *([None] * 8)) == B.DG_ERR_ARG
    assert lib.dg_attn_oproj_prepare(None, 128, None, None, None) == B.DG_ERR_ARG
    assert lib.dg_attn_oproj_residual(None, None, None, None) == B.DG_ERR_ARG
    assert lib.dg_attn_forward_layer(None, *([None] * 7)) == B.DG_ERR_ARG
    assert lib.dg_attn_norm_rope(None, *([None] * 10)) == B.DG_ERR_ARG
    assert lib.dg_attn_attend(None, *([None] * 7)) == B.DG_ERR_ARG


def _cpu_plan(nh=4, nkv=2, hd=64, ctx=16, T=8):
    """A Plan object with its geometry but no library handle (no GPU here): enough to show that
    its methods reject bad tensors before any library call."""
    p = object.__new__(B.Plan)
    p.nh, p.nkv, p.hd, p.ctx, p.T = nh, nkv, hd, ctx, T
    p.H = p.oH = None
    p.device = 0
    p.handle = None
    return p


def test_binding_rejects_bad_tensors_before_the_library():
    import torch
    p = _cpu_plan()
    T, nh, nkv, hd, ctx = p.T, p.nh, p.nkv, p.hd, p.ctx
    good = dict(q=torch.zeros(T, nh * hd), k_canvas=torch.zeros(T, nkv * hd),
                v_canvas=torch.zeros(T, nkv * hd), k_cache=torch.zeros(nkv, ctx, hd),
                v_cache=torch.zeros(nkv, ctx, hd), out=torch.zeros(T, nh * hd))
    cases = {
        "dtype": dict(good, q=torch.zeros(T, nh * hd, dtype=torch.float64)),
        "contiguous": dict(good, q=torch.zeros(nh * hd, T).t()),
        "elements": dict(good, k_canvas=torch.zeros(T - 1, nkv * hd)),
        "cache elements": dict(good, v_cache=torch.zeros(nkv, ctx + 1, hd)),
        "half cache": dict(good, k_cache=torch.zeros(nkv, ctx, hd, dtype=torch.float16)),
        "out elements": dict(good, out=torch.zeros(T, nh * hd + 4)),
    }
    msgs = {"dtype": "dtype", "contiguous": "contiguous", "elements": "elements",
            "cache elements": "elements", "half cache": "dtype", "out elements": "elements"}
    for name, kw in cases.items():
        with pytest.raises(ValueError, match=msgs[name]):
            p.forward(**kw)
    # right dtype, layout and size, but host memory: the device check
    with pytest.raises(ValueError, match="cuda"):
        p.forward(**good)
    with pytest.raises(ValueError, match="elements"):
        p.forward(**good, q_norm_w=torch.ones(hd + 1))
    with pytest.raises(ValueError, match="elements"):
        p.forward(**good, cos_sin=torch.ones(T, hd))
    with pytest.raises(ValueError, match="both be"):
        p.cache_prepare(torch.zeros(nkv, ctx, hd, dtype=torch.float16),
                        torch.zeros(nkv, ctx, hd, dtype=torch.float32))
    with pytest.raises(ValueError, match="elements"):
        p.attend(good["q"], good["k_canvas"], torch.zeros(3), out=good["out"])
    with pytest.raises(ValueError, match="elements"):
        p.proj_prepare(128, None, torch.zeros(nh * hd, 127), torch.zeros(nkv * hd, 128))
    with pytest.raises(ValueError, match="contiguous"):
        B._ptr(torch.zeros(4, 4).t())


def test_build_id_matches_the_sources(lib):
    assert B.build_id() == build_mod.source_id()
