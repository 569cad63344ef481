"""The allocation-free entry point, checked against the planned entry point and the oracle.

dg_attn_forward_noalloc is for callers that cannot allocate device memory when they run
attention (code inside a memory pool it does not own, or a process whose device memory is
reserved up front); it keeps its working memory in a fixed array inside the library.  Each case
calls it twice in a row through the C ABI, with different inputs, and each output must match
dg_attn_forward on the fp32 path and the fp64 oracle within the fp32 parity tolerance
(max <= 1e-5, mean <= 1e-6).  This file is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300 import build as build_mod
from gqa_canvas_attention_gb300.workloads import EPS, ROPE_THETA, make_inputs

pytestmark = pytest.mark.gpu
FP32_MAX, FP32_MEAN = 1e-5, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.load()


def planned(d, nh, nkv, hd, ctx, T, cos_sin, pos0):
    """dg_attn_forward on the fp32 path with one key partition: the arithmetic of the
    allocation-free entry point, so the two agree to rounding."""
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, B.DG_PATH_FP32).set(B.DG_OPT_SPLITS, 1)
    if pos0 >= 0:
        plan.set(B.DG_OPT_POS0, pos0)
    out = plan.forward(d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"],
                       d["q_norm_w"], d["k_norm_w"], cos_sin)
    assert plan.sync_status() == B.DG_OK
    plan.close()
    return out


def oracle_rows(h, nh, nkv, hd, cos_sin, pos0, rows=None):
    f = lambda x: None if x is None else x.numpy()
    return oracle.forward(f(h["q"]), f(h["k_canvas"]), f(h["v_canvas"]), f(h["k_cache"]),
                          f(h["v_cache"]), nh, nkv, hd, f(h["q_norm_w"]), f(h["k_norm_w"]),
                          cos_sin=f(cos_sin), eps=EPS, theta=ROPE_THETA,
                          pos0=None if pos0 < 0 else pos0, rows=rows)


def noalloc(d, nh, nkv, hd, ctx, T, cos_sin, pos0):
    out = torch.full((T, nh * hd), float("nan"), device="cuda")
    rc = B.dg_attn_forward_noalloc(nh, nkv, hd, ctx, T, EPS, ROPE_THETA, pos0, d["q"],
                                   d["k_canvas"], d["v_canvas"], d["k_cache"], d["v_cache"],
                                   d["q_norm_w"], d["k_norm_w"], cos_sin, out)
    assert rc == B.DG_OK, B.load().dg_attn_noalloc_last_error().decode()
    torch.cuda.synchronize()
    return out


CASES = [
    # T, ctx, nh, nkv, hd, caller's cos|sin table, pos0 (-1: ctx)
    (48, 300, 4, 2, 128, False, -1),
    (40, 300, 4, 2, 256, False, -1),     # the largest shared-memory variant of the fp32 kernel
    (50, 0, 4, 4, 64, False, -1),        # no cache: NULL cache pointers
    (30, 200, 4, 2, 128, True, -1),      # a caller's cos|sin table
    (30, 200, 4, 2, 128, False, 4321),   # canvas positions from 4321
    (30, 200, 4, 2, 64, False, (1 << 24) - 31),   # the largest positions (per-lane angles)
]


@pytest.mark.parametrize("case", CASES,
                         ids=lambda c: "T%d_ctx%d_nh%d_nkv%d_hd%d_table%d_pos%d" % c)
def test_noalloc_matches_planned_forward_and_oracle_twice_in_a_row(case):
    T, ctx, nh, nkv, hd, table, pos0 = case
    outs = []
    for seed in (21, 22):
        h = make_inputs(T, ctx, nh, nkv, hd, seed=seed, weighted=True)
        d = {k: (v.cuda() if v is not None else None) for k, v in h.items()}
        cs = None
        if table:
            g = torch.Generator().manual_seed(seed)
            ang = torch.rand(T, hd // 2, generator=g, dtype=torch.float64) * 6.0
            cs = torch.cat([ang.cos(), ang.cos(), ang.sin(), ang.sin()], 1).float()
        out = noalloc(d, nh, nkv, hd, ctx, T, None if cs is None else cs.cuda(), pos0)
        o = out.double().cpu().numpy()
        assert np.isfinite(o).all()
        ref = planned(d, nh, nkv, hd, ctx, T, None if cs is None else cs.cuda(), pos0)
        err = np.abs(o - ref.double().cpu().numpy())
        assert err.max() <= FP32_MAX, err.max()
        ora = oracle_rows(h, nh, nkv, hd, cs, pos0)
        e = np.abs(o - ora)
        print(f"{case} seed {seed}: vs planned {err.max():.2e}, vs oracle max {e.max():.2e} "
              f"mean {e.mean():.2e}")
        assert e.max() <= FP32_MAX and e.mean() <= FP32_MEAN
        outs.append(out.clone())
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_accepts_the_largest_size_its_scratch_holds():
    """T = 10922, nh = nkv = 1, hd = 128, ctx = 0 needs 64 * 16 + 3 * 10922 * 512 bytes = 16 MiB
    exactly (one more canvas row is refused, checked on the CPU)."""
    T, ctx, nh, nkv, hd = 10922, 0, 1, 1, 128
    h = make_inputs(T, ctx, nh, nkv, hd, seed=23, weighted=False)
    d = {k: (v.cuda() if v is not None else None) for k, v in h.items()}
    out = noalloc(d, nh, nkv, hd, ctx, T, None, -1)
    ref = planned(d, nh, nkv, hd, ctx, T, None, -1)
    assert (out.double() - ref.double()).abs().max().item() <= FP32_MAX
    for a, b in ((0, 8), (T - 8, T)):
        ora = oracle_rows(h, nh, nkv, hd, None, -1, rows=(a, b))[a:b]
        assert np.abs(out[a:b].double().cpu().numpy() - ora).max() <= FP32_MAX


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    T, nh, nkv, hd = 4096, 16, 16, 64          # needs 48 MiB of scratch
    q = torch.zeros(8, device="cuda")
    rc = B.dg_attn_forward_noalloc(nh, nkv, hd, 0, T, EPS, ROPE_THETA, -1, q, q, q, None, None,
                                   None, None, None, q)
    assert rc == B.DG_ERR_ARG
    assert "scratch" in B.load().dg_attn_noalloc_last_error().decode()
