"""Randomised parity: seeded draws of geometry and options, each forward compared with the fp64
oracle on every row (tolerances as in test_parity_gpu: tensor-core max 5e-3 / mean 5e-4, fp32
max 1e-5 / mean 1e-6).  The draws combine what the fixed cases test one at a time: head sizes,
GQA ratios, ragged row and key counts, forced partitions and schedules, resident inputs, a
prepared or per-call cache, positions anywhere below 2^24, a caller's cos|sin table, K and V
passed as one buffer."""
import random

import numpy as np
import pytest
import torch

import oracle
from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300.workloads import EPS, ROPE_THETA, make_inputs

pytestmark = pytest.mark.gpu
TOL = {B.DG_PATH_TC: (5e-3, 5e-4), B.DG_PATH_FP32: (1e-5, 1e-6)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def draw(rnd):
    hd = rnd.choice([64, 128, 256, 32])
    nkv = rnd.choice([1, 2, 3, 4, 8])
    nh = nkv * rnd.choice([1, 2, 3, 4, 8])
    T = rnd.choice([1, rnd.randint(2, 64), rnd.randint(65, 300)])
    ctx = rnd.choice([0, rnd.randint(1, 300), rnd.randint(301, 3000)])
    path = B.DG_PATH_FP32 if hd == 32 else rnd.choice([B.DG_PATH_TC, B.DG_PATH_TC,
                                                       B.DG_PATH_FP32])
    opts = {
        "splits": rnd.choice([0, 0, 1, 2, 3, 5, 9, 12]),
        "schedule": rnd.choice([B.DG_SCHEDULE_AUTO, B.DG_SCHEDULE_SPLIT,
                                B.DG_SCHEDULE_STREAM_K]),
        "resident": rnd.choice([0, 1]),
        "prepared": ctx > 0 and rnd.random() < 0.5,
        "pos0": rnd.choice([None, rnd.randint(0, (1 << 24) - 1 - T)]),
        "table": rnd.random() < 0.2,
        "weighted": rnd.random() < 0.7,
        "alias": rnd.random() < 0.15,
        "theta": rnd.choice([ROPE_THETA, 1.0e6]),
    }
    if (1 << 24) - 1 - ctx - T < 0:
        ctx = 0
    return T, ctx, nh, nkv, hd, path, opts


@pytest.mark.parametrize("seed", range(48))
def test_random_geometry_and_options(seed):
    rnd = random.Random(1000 + seed)
    T, ctx, nh, nkv, hd, path, o = draw(rnd)
    d = make_inputs(T, ctx, nh, nkv, hd, seed=2000 + seed, weighted=o["weighted"])
    if o["alias"]:
        d["v_canvas"] = d["k_canvas"]
    cs = None
    if o["table"]:
        g = torch.Generator().manual_seed(3000 + seed)
        ang = torch.rand(T, hd // 2, generator=g, dtype=torch.float64) * 6.0
        cs = torch.cat([ang.cos(), ang.cos(), ang.sin(), ang.sin()], 1).float()
    dd = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    if o["alias"]:
        dd["v_canvas"] = dd["k_canvas"]
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, o["theta"])
    plan.set(B.DG_OPT_PATH, path).set(B.DG_OPT_INPUTS_RESIDENT, o["resident"])
    if o["splits"]:
        plan.set(B.DG_OPT_SPLITS, o["splits"])
    if path == B.DG_PATH_TC:
        plan.set(B.DG_OPT_SCHEDULE, o["schedule"])
    if o["pos0"] is not None:
        plan.set(B.DG_OPT_POS0, o["pos0"])
    kc, vc = dd["k_cache"], dd["v_cache"]
    if o["prepared"]:
        plan.cache_prepare(kc, vc)
        kc = vc = None
    outs = []
    for _ in range(2):                      # twice: the second forward follows the first
        outs.append(plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], kc, vc,
                                 dd["q_norm_w"], dd["k_norm_w"],
                                 None if cs is None else cs.cuda()))
    assert plan.sync_status() == B.DG_OK
    f = lambda x: None if x is None else x.numpy()
    ref = oracle.forward(f(d["q"]), f(d["k_canvas"]), f(d["v_canvas"]), f(d["k_cache"]),
                         f(d["v_cache"]), nh, nkv, hd, f(d["q_norm_w"]), f(d["k_norm_w"]),
                         cos_sin=f(cs), eps=EPS, theta=o["theta"], pos0=o["pos0"])
    tmax, tmean = TOL[path]
    for out in outs:
        e = np.abs(out.cpu().double().numpy() - ref)
        print(f"seed {seed} T{T} ctx{ctx} nh{nh} nkv{nkv} hd{hd} path{path} {o}: "
              f"max {e.max():.2e} mean {e.mean():.2e}")
        assert np.isfinite(out.cpu().numpy()).all()
        assert e.max() <= tmax and e.mean() <= tmean
    assert torch.equal(outs[0], outs[1])
    plan.close()
