"""The allocation-free entry point, checked against the planned entry point.

dg_attn_forward_noalloc is for callers that cannot allocate device memory when they run
attention (code inside a memory pool it does not own, or a process whose device memory is
reserved up front); it keeps its working memory in a fixed array inside the library.  Here it is
called twice in a row through the C ABI, with different inputs, and each output must match
dg_attn_forward on the fp32 path within the fp32 parity tolerance.  This file is collected last.
"""
import numpy as np
import pytest
import torch

from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300 import build as build_mod
from gqa_canvas_attention_gb300.workloads import EPS, ROPE_THETA, make_inputs

pytestmark = pytest.mark.gpu
FP32_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.load()


def planned(d, nh, nkv, hd, ctx, T):
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, B.DG_PATH_FP32)
    out = plan.forward(d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"],
                       d["q_norm_w"], d["k_norm_w"])
    assert plan.sync_status() == B.DG_OK
    return out


def test_noalloc_matches_planned_forward_twice_in_a_row():
    T, ctx, nh, nkv, hd = 48, 300, 4, 2, 128
    outs = []
    for seed in (21, 22):
        d = {k: (v.cuda() if v is not None else None)
             for k, v in make_inputs(T, ctx, nh, nkv, hd, seed=seed, weighted=True).items()}
        out = torch.full((T, nh * hd), float("nan"), device="cuda")
        rc = B.dg_attn_forward_noalloc(nh, nkv, hd, ctx, T, EPS, ROPE_THETA, -1, d["q"],
                                       d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"],
                                       d["q_norm_w"], d["k_norm_w"], None, out)
        assert rc == B.DG_OK, B.load().dg_attn_noalloc_last_error().decode()
        torch.cuda.synchronize()
        ref = planned(d, nh, nkv, hd, ctx, T)
        err = (out.double() - ref.double()).abs().max().item()
        assert np.isfinite(out.cpu().numpy()).all()
        assert err <= FP32_TOL, err
        outs.append(out.clone())
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    T, nh, nkv, hd = 4096, 16, 16, 64          # needs 48 MiB of scratch
    q = torch.zeros(8, device="cuda")
    rc = B.dg_attn_forward_noalloc(nh, nkv, hd, 0, T, EPS, ROPE_THETA, -1, q, q, q, None, None,
                                   None, None, None, q)
    assert rc == B.DG_ERR_ARG
    assert "scratch" in B.load().dg_attn_noalloc_last_error().decode()
