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
