"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on the same seeded
inputs, element by element.

Tolerances (on outputs of RMS <= 1):
  tensor-core path: max |gpu - oracle| <= 5e-3 and mean <= 5e-4;
  fp32 path:        max <= 1e-5 and mean <= 1e-6.
Every output row is compared, at the full sizes of the named workloads too (the oracle does a
36.5-GFLOP forward of the 48-step workload in well under a second on 16 cores).
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300.workloads import (EPS, ROPE_THETA, WORKLOADS, make_inputs,
                                                  workload_inputs)

pytestmark = pytest.mark.gpu

TOL = {B.DG_PATH_TC: (5e-3, 5e-4), B.DG_PATH_FP32: (1e-5, 1e-6)}
PATHS = [B.DG_PATH_TC, B.DG_PATH_FP32]
PNAME = {B.DG_PATH_TC: "tc", B.DG_PATH_FP32: "fp32"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def to_dev(d):
    return {k: (v.cuda() if v is not None else None) for k, v in d.items()}


def oracle_out(d, nh, nkv, hd, rows=None, pos0=None, cos_sin=None, theta=ROPE_THETA):
    f = lambda x: None if x is None else x.numpy()
    return oracle.forward(f(d["q"]), f(d["k_canvas"]), f(d["v_canvas"]), f(d["k_cache"]),
                          f(d["v_cache"]), nh, nkv, hd, f(d["q_norm_w"]), f(d["k_norm_w"]),
                          cos_sin=cos_sin, eps=EPS, theta=theta, pos0=pos0, rows=rows)


def all_rows(T):
    return [(0, T)]


def check(out, ref, path, ranges, label=""):
    tmax, tmean = TOL[path]
    o = out.detach().cpu().double().numpy()
    errs = np.concatenate([np.abs(o[a:b] - ref[a:b]).ravel() for a, b in ranges])
    assert np.isfinite(o).all()
    mx, mn = errs.max(), errs.mean()
    print(f"{label} {PNAME[path]}: max {mx:.3e} mean {mn:.3e}")
    assert mx <= tmax, f"{label}: max err {mx:.3e} > {tmax}"
    assert mn <= tmean, f"{label}: mean err {mn:.3e} > {tmean}"


def run_forward(plan, dd, **kw):
    out = plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["k_cache"], dd["v_cache"],
                       dd["q_norm_w"], dd["k_norm_w"], **kw)
    assert plan.sync_status() == B.DG_OK
    return out


# ------------------------------------------------------------------ first stage alone

# positions: the default (pos0 = ctx), and the largest the plan takes (the last row at 2^24 - 2)
# with the global layers' rope base
POSITIONS = [(None, ROPE_THETA), ((1 << 24) - 38, 1.0e6)]


@pytest.mark.parametrize("hd", [32, 64, 128, 256])
@pytest.mark.parametrize("weighted", [True, False])
@pytest.mark.parametrize("pos", POSITIONS, ids=["pos_ctx", "pos_2e24"])
def test_norm_rope_stage(hd, weighted, pos):
    T, ctx, nh, nkv = 37, 8100, 4, 2
    pos0, theta = pos
    p0 = ctx if pos0 is None else pos0
    d = make_inputs(T, ctx, nh, nkv, hd, seed=5, weighted=weighted, draw_cache=False)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, theta)
    if pos0 is not None:
        plan.set(B.DG_OPT_POS0, pos0)
    qh, kh, vh = plan.norm_rope(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["q_norm_w"],
                                dd["k_norm_w"])
    torch.cuda.synchronize()
    w = lambda x: None if x is None else x.numpy()
    rq = oracle.norm_rope(d["q"].numpy(), nh, hd, w(d["q_norm_w"]), EPS, True, p0, theta)
    rk = oracle.norm_rope(d["k_canvas"].numpy(), nkv, hd, w(d["k_norm_w"]), EPS, True, p0,
                          theta)
    rv = oracle.norm_rope(d["v_canvas"].numpy(), nkv, hd, None, EPS, False)
    for got, ref, name in ((qh, rq, "q"), (kh, rk, "k"), (vh, rv, "v")):
        e = np.abs(got.cpu().double().numpy().reshape(ref.shape) - ref)
        print(f"hd={hd} {name}: max {e.max():.2e}")
        assert e.max() <= 2e-6, f"{name}: {e.max():.3e}"


def test_norm_rope_with_table():
    T, ctx, nh, nkv, hd = 9, 3, 2, 1, 64
    d = make_inputs(T, ctx, nh, nkv, hd, seed=6, weighted=True, draw_cache=False)
    g = torch.Generator().manual_seed(7)
    cs = torch.randn(T, 2 * hd, generator=g)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    qh, kh, _ = plan.norm_rope(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["q_norm_w"],
                               dd["k_norm_w"], cs.cuda())
    rq = oracle.norm_rope(d["q"].numpy(), nh, hd, d["q_norm_w"].numpy(), EPS, True, ctx,
                          ROPE_THETA, cos_sin=cs.numpy())
    assert np.abs(qh.cpu().double().numpy().reshape(rq.shape) - rq).max() <= 2e-6


# ------------------------------------------------------------------ whole block, named workloads

@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_parity(name, path):
    """Every row of every named workload; every canvas of a batch of canvases."""
    w = WORKLOADS[name]
    plan = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, w.theta)
    plan.set(B.DG_OPT_PATH, path)
    if w.pos0 is not None:
        plan.set(B.DG_OPT_POS0, w.pos0)
    for c in range(w.canvases):
        d = workload_inputs(w, canvas=c)
        out = run_forward(plan, to_dev(d))
        ref = oracle_out(d, w.nh, w.nkv, w.hd, pos0=w.pos0, theta=w.theta)
        check(out, ref, path, all_rows(w.T), f"{name}[{c}]")


def test_denoise_loop_steps_share_a_prepared_cache():
    """Steps 0, 1 and 47 of the 48-step loop, every row: cache prepared once, fresh canvas per
    step."""
    w = WORKLOADS["denoise48_ctx8k"]
    plan = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, ROPE_THETA)
    d0 = workload_inputs(w, step=0)
    kc, vc = d0["k_cache"].cuda(), d0["v_cache"].cuda()
    plan.cache_prepare(kc, vc)
    assert plan.get(B.DG_INFO_CACHE_READY) == 1
    for step in (0, 1, 47):
        d = workload_inputs(w, step=step)
        d["k_cache"], d["v_cache"] = d0["k_cache"], d0["v_cache"]
        dd = to_dev(d)
        out = plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"])
        assert plan.sync_status() == B.DG_OK
        check(out, oracle_out(d, w.nh, w.nkv, w.hd), B.DG_PATH_TC, all_rows(w.T), f"step{step}")


def test_denoise_loop_in_the_bench_launch_configuration():
    """The 48-step canvas exactly as the benchmark runs it: resident inputs, the cache prepared
    once, 48 forwards captured into one CUDA graph and replayed twice.  Every row of steps 0, 1
    and 47 and eight rows of every other step are compared with the oracle."""
    w = WORKLOADS["denoise48_ctx8k"]
    plan = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_INPUTS_RESIDENT, 1)
    d0 = workload_inputs(w, step=0)
    kc, vc = d0["k_cache"].cuda(), d0["v_cache"].cuda()
    steps = [workload_inputs(w, step=s) for s in range(w.steps)]
    dev = [to_dev(d) for d in steps]
    outs = [torch.empty(w.T, w.nh * w.hd, device="cuda") for _ in steps]

    def canvas():
        plan.cache_prepare(kc, vc)
        for dd, o in zip(dev, outs):
            plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                         dd["k_norm_w"], None, o)

    canvas()                                # builds the cos/sin table outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        canvas()
    for o in outs:
        o.fill_(float("nan"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert plan.sync_status() == B.DG_OK
    # With resident inputs each forward's first stage writes the operand set the previous
    # forward's attention kernel is not reading, ordered by programmatic dependent launch alone.
    # The same canvases run eagerly without the option, one kernel after the other, must give
    # the same bits for every step.
    ref = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, ROPE_THETA)
    ref.cache_prepare(kc, vc)
    for s, (dd, o) in enumerate(zip(dev, outs)):
        r = ref.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                        dd["k_norm_w"])
        assert torch.equal(o, r), f"step {s}: resident graph replay differs from eager"
    assert ref.sync_status() == B.DG_OK
    for s, (d, o) in enumerate(zip(steps, outs)):
        d["k_cache"], d["v_cache"] = d0["k_cache"], d0["v_cache"]
        rows = (0, w.T) if s in (0, 1, w.steps - 1) else (8 * (s % 60), 8 * (s % 60) + 8)
        check(o, oracle_out(d, w.nh, w.nkv, w.hd, rows=rows), B.DG_PATH_TC, [rows], f"step{s}")


# ------------------------------------------------------------------ shapes and edge cases

SHAPES = [
    # T, ctx, nh, nkv, hd
    (1, 0, 1, 1, 64),        # one key
    (1, 5, 2, 1, 128),       # single canvas row with a cache
    (3, 0, 4, 4, 64),        # MHA, ctx = 0
    (70, 33, 6, 2, 64),      # ragged: rows 210 (not a tile multiple), S = 103
    (129, 200, 2, 2, 128),   # 129 rows: two query tiles, the second with one live row
    (65, 300, 8, 1, 256),    # G = 8: 520 packed rows
    (50, 1000, 4, 2, 256),   # S = 1050, not a multiple of the key tile
    (17, 63, 4, 2, 32),      # fp32-only head size
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "T%d_ctx%d_nh%d_nkv%d_hd%d" % s)
@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_shapes(shape, path):
    T, ctx, nh, nkv, hd = shape
    if path == B.DG_PATH_TC and hd not in (64, 128, 256):
        pytest.skip("tensor-core path needs hd in {64, 128, 256}")
    d = make_inputs(T, ctx, nh, nkv, hd, seed=100 + T, weighted=True)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path)
    out = run_forward(plan, dd)
    check(out, oracle_out(d, nh, nkv, hd), path, [(0, T)], str(shape))


# Near the limits the plan accepts, compared on sampled rows (the oracle computes those rows
# only): positions up to the largest the plan takes (pos0 + T < 2^24, so the last canvas row at
# 2^24 - 2), a 256 Ki-key cache, and
# 65536 packed query rows per kv group (G = 16, 512 query tiles each).
LARGE_CASES = [
    # T, ctx, nh, nkv, hd, pos0 (None: ctx), sampled row ranges
    (4, 262144, 2, 1, 64, (1 << 24) - 5, [(0, 4)]),
    (4096, 0, 32, 2, 64, None, [(0, 8), (2041, 2047), (4088, 4096)]),
    (1024, 2048, 16, 1, 256, (1 << 24) - 1025, [(0, 4), (511, 515), (1020, 1024)]),
]


@pytest.mark.parametrize("case", LARGE_CASES, ids=lambda c: "T%d_ctx%d_nh%d_nkv%d_hd%d" % c[:5])
def test_sizes_near_the_limits(case):
    T, ctx, nh, nkv, hd, pos0, ranges = case
    d = make_inputs(T, ctx, nh, nkv, hd, seed=400 + hd, weighted=True)
    dd = to_dev(d)
    ref = np.zeros((T, nh * hd))
    for a, b in ranges:
        ref[a:b] = oracle_out(d, nh, nkv, hd, rows=(a, b), pos0=pos0)[a:b]
    for path in PATHS:
        plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
        plan.set(B.DG_OPT_PATH, path)
        if pos0 is not None:
            plan.set(B.DG_OPT_POS0, pos0)
        out = run_forward(plan, dd)
        check(out, ref, path, ranges, "large %s" % (case[:5],))
        plan.close()


def test_the_longest_cache_the_plan_accepts():
    """ctx + T = 2^24 - 1 keys with nkv = 2: each operand array holds 2.1e9 elements (past 2^31),
    the key range is cut into 64 partitions (more than a cluster merges, so through the combine
    kernel), and the one canvas row sits at position 2^24 - 2.  The cache is drawn on the device
    (seeded) and copied back for the oracle."""
    T, nh, nkv, hd = 1, 2, 2, 64
    ctx = (1 << 24) - 1 - T
    d = make_inputs(T, 0, nh, nkv, hd, seed=410, weighted=True)
    g = torch.Generator(device="cuda").manual_seed(411)
    kc = torch.randn((nkv, ctx, hd), generator=g, device="cuda")
    vc = torch.randn((nkv, ctx, hd), generator=g, device="cuda")
    dd = to_dev(d)
    dd["k_cache"], dd["v_cache"] = kc, vc
    d["k_cache"], d["v_cache"] = kc.cpu(), vc.cpu()
    ref = oracle_out(d, nh, nkv, hd)
    for path in PATHS:
        plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
        plan.set(B.DG_OPT_PATH, path)
        out = run_forward(plan, dd)
        check(out, ref, path, all_rows(T), "longest cache")
        plan.close()
        del plan
        torch.cuda.empty_cache()


# (requested partitions, cache length, partitions the tensor-core path uses): with hd = 128 a key
# tile is 64 keys, so ctx = 700 / 2000 / 2250 (+ T = 40) give 12 / 32 / 36 tiles.  2..8
# partitions merge inside the kernel (thread-block clusters); 9 and 12 use the combine kernel.
SPLIT_CASES = [(1, 700, 1), (2, 700, 2), (3, 2000, 3), (7, 2000, 7), (8, 2000, 8), (9, 2250, 9),
               (64, 700, 12)]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "splits%d_ctx%d" % c[:2])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_forced_partitions(case, path):
    splits, ctx, used = case
    T, nh, nkv, hd = 40, 4, 2, 128
    d = make_inputs(T, ctx, nh, nkv, hd, seed=11, weighted=False)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path).set(B.DG_OPT_SPLITS, splits)
    if path == B.DG_PATH_TC:
        assert plan.get(B.DG_INFO_SPLITS_USED) == used
        run_forward(plan, dd)           # the cos/sin table is built by the first forward
        assert plan.get(B.DG_INFO_LAUNCHES) == (3 if used > 8 else 2)
    out = run_forward(plan, dd)
    check(out, oracle_out(d, nh, nkv, hd), path, [(0, T)], f"splits={splits}")


# The stream-K schedule (one CTA per SM, each an equal run of key tiles over the (query tile,
# kv group) pairs in order; most runs cover the end of one pair and the start of the next).
STREAM_K_SHAPES = [
    # T, ctx, nh, nkv, hd
    (512, 8192, 8, 4, 256),  # the 48-step workload's geometry: 32 pairs x 136 tiles on 152 CTAs
    (50, 1000, 4, 2, 256),   # S = 1050: the last key tile of every pair is ragged
    (65, 300, 8, 1, 256),    # G = 8: 520 packed rows, the last query tile nearly empty
    (130, 1500, 8, 4, 256),  # 3 query tiles per kv group
    (256, 4096, 16, 8, 128), # two Q.K^T issuers per CTA
    (40, 2000, 4, 2, 128),
    (512, 0, 16, 16, 64),    # ctx = 0, 64 pairs
    (3, 5, 2, 1, 64),        # one pair, fewer key tiles than SMs
]


@pytest.mark.parametrize("shape", STREAM_K_SHAPES, ids=lambda s: "T%d_ctx%d_nh%d_nkv%d_hd%d" % s)
def test_stream_k_schedule(shape):
    T, ctx, nh, nkv, hd = shape
    d = make_inputs(T, ctx, nh, nkv, hd, seed=300 + T + hd, weighted=True)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_SCHEDULE, B.DG_SCHEDULE_STREAM_K)
    assert plan.get(B.DG_INFO_SCHEDULE_USED) == B.DG_SCHEDULE_STREAM_K
    out = run_forward(plan, dd)
    again = run_forward(plan, dd)
    assert torch.equal(out, again), "the stream-K merge order is fixed: results repeat bit for bit"
    ranges = all_rows(T)
    ref = oracle_out(d, nh, nkv, hd)
    check(out, ref, B.DG_PATH_TC, ranges, "stream-K %s" % (shape,))
    # the split schedule on the same inputs agrees within the same bound
    plan.set(B.DG_OPT_SCHEDULE, B.DG_SCHEDULE_SPLIT)
    assert plan.get(B.DG_INFO_SCHEDULE_USED) == B.DG_SCHEDULE_SPLIT
    split = run_forward(plan, dd)
    check(split, ref, B.DG_PATH_TC, ranges, "split %s" % (shape,))


def test_stream_k_under_a_cuda_graph_with_resident_inputs():
    """The bench's configuration: graph replay, resident inputs, several forwards back to back."""
    w = WORKLOADS["denoise48_ctx8k"]
    plan = B.Plan(w.nh, w.nkv, w.hd, w.ctx, w.T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_SCHEDULE, B.DG_SCHEDULE_STREAM_K).set(B.DG_OPT_INPUTS_RESIDENT, 1)
    d0 = workload_inputs(w, step=0)
    plan.cache_prepare(d0["k_cache"].cuda(), d0["v_cache"].cuda())
    steps = (0, 1, 2)
    ins = []
    for st in steps:
        d = workload_inputs(w, step=st)
        d["k_cache"], d["v_cache"] = d0["k_cache"], d0["v_cache"]
        ins.append((d, to_dev(d)))
    outs = [torch.empty(w.T, w.nh * w.hd, device="cuda") for _ in steps]
    fwd = lambda: [plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None,
                                dd["q_norm_w"], dd["k_norm_w"], None, o)
                   for (_, dd), o in zip(ins, outs)]
    fwd()                                   # builds the cos/sin table outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    for o in outs:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert plan.sync_status() == B.DG_OK
    for (d, _), o in zip(ins, outs):
        check(o, oracle_out(d, w.nh, w.nkv, w.hd), B.DG_PATH_TC, all_rows(w.T), "graph")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_k_and_v_canvas_may_alias(path):
    """Models whose V is the raw K projection pass the same buffer twice."""
    T, ctx, nh, nkv, hd = 24, 40, 4, 2, 64
    d = make_inputs(T, ctx, nh, nkv, hd, seed=12)
    d["v_canvas"] = d["k_canvas"]
    dd = to_dev(d)
    dd["v_canvas"] = dd["k_canvas"]
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path)
    out = run_forward(plan, dd)
    check(out, oracle_out(d, nh, nkv, hd), path, [(0, T)], "alias")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_pos0_option_and_table(path):
    T, ctx, nh, nkv, hd = 20, 16, 2, 1, 128
    d = make_inputs(T, ctx, nh, nkv, hd, seed=13)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path).set(B.DG_OPT_POS0, 5000)
    out = run_forward(plan, dd)
    check(out, oracle_out(d, nh, nkv, hd, pos0=5000), path, [(0, T)], "pos0")
    g = torch.Generator().manual_seed(3)
    ang = torch.rand(T, hd // 2, generator=g, dtype=torch.float64) * 6.0
    cs = torch.cat([ang.cos(), ang.cos(), ang.sin(), ang.sin()], 1).float()
    out = run_forward(plan, dd, cos_sin=cs.cuda())
    check(out, oracle_out(d, nh, nkv, hd, cos_sin=cs.numpy()), path, [(0, T)], "table")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_attend_on_oracle_normed_inputs(path):
    """The attention stage alone, on operands normed by the oracle (rounded to fp32)."""
    T, ctx, nh, nkv, hd = 48, 80, 4, 2, 256
    d = make_inputs(T, ctx, nh, nkv, hd, seed=14)
    qh = oracle.norm_rope(d["q"].numpy(), nh, hd, d["q_norm_w"].numpy(), EPS, True, ctx)
    kh = oracle.norm_rope(d["k_canvas"].numpy(), nkv, hd, d["k_norm_w"].numpy(), EPS, True, ctx)
    vh = oracle.norm_rope(d["v_canvas"].numpy(), nkv, hd, None, EPS, False)
    q32, k32, v32 = (torch.from_numpy(x.astype(np.float32)).reshape(T, -1) for x in (qh, kh, vh))
    ref = oracle.attention(q32.numpy(), k32.numpy(), v32.numpy(), d["k_cache"].numpy(),
                           d["v_cache"].numpy(), nh, nkv, hd).reshape(T, nh * hd)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path)
    out = plan.attend(q32.cuda(), k32.cuda(), v32.cuda(), d["k_cache"].cuda(), d["v_cache"].cuda())
    assert plan.sync_status() == B.DG_OK
    check(out, ref, path, [(0, T)], "attend")


@pytest.mark.parametrize("shape", [
    (32, 500, 4, 2, 128),
    (40, 333, 4, 2, 64),       # 10656 float4 units of K: a ragged last pass of its blocks
    (64, 4100, 16, 8, 256),    # 2.1 M float4 units: more than one pass of the capped block count
], ids=lambda s: "T%d_ctx%d_nh%d_nkv%d_hd%d" % s)
@pytest.mark.parametrize("resident", [0, 1])
def test_per_call_cache_and_prepared_cache_agree(shape, resident):
    """A cache passed with the call is converted by the first-stage launch itself; the prepared
    cache by its own kernel.  Both give the same operand bits, so the same outputs, and those
    match the oracle."""
    T, ctx, nh, nkv, hd = shape
    d = make_inputs(T, ctx, nh, nkv, hd, seed=15)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_INPUTS_RESIDENT, resident)
    a = run_forward(plan, dd).clone()
    assert plan.get(B.DG_INFO_CACHE_READY) == 0
    plan.cache_prepare(dd["k_cache"], dd["v_cache"])
    b = plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                     dd["k_norm_w"])
    c = run_forward(plan, dd).clone()          # per call again, after a prepared one
    assert plan.sync_status() == B.DG_OK
    assert torch.equal(a, b) and torch.equal(a, c)
    check(a, oracle_out(d, nh, nkv, hd), B.DG_PATH_TC, all_rows(T), "per-call cache")


def test_errors_are_reported_not_raised_on_device():
    T, ctx, nh, nkv, hd = 8, 16, 2, 1, 64
    d = to_dev(make_inputs(T, ctx, nh, nkv, hd, seed=16))
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    out = torch.empty(T, nh * hd, device="cuda")
    h = plan.handle
    # ctx > 0 without a cache and nothing prepared
    with pytest.raises(B.DgAttnError) as e:
        B.dg_attn_forward(h, d["q"], d["k_canvas"], d["v_canvas"], None, None, None, None, None, out)
    assert e.value.status == B.DG_ERR_STATE
    # misaligned pointer
    with pytest.raises(B.DgAttnError) as e:
        B.dg_attn_forward(h, d["q"].data_ptr() + 4, d["k_canvas"], d["v_canvas"], d["k_cache"],
                          d["v_cache"], None, None, None, out)
    assert e.value.status == B.DG_ERR_ALIGN
    # a cache on a ctx == 0 plan
    p0 = B.Plan(nh, nkv, hd, 0, T, EPS, ROPE_THETA)
    with pytest.raises(B.DgAttnError) as e:
        B.dg_attn_forward(p0.handle, d["q"], d["k_canvas"], d["v_canvas"], d["k_cache"],
                          d["v_cache"], None, None, None, out)
    assert e.value.status == B.DG_ERR_ARG
    # the fp32-only head size cannot take the tensor-core path
    p32 = B.Plan(nh, nkv, 32, ctx, T, EPS, ROPE_THETA)
    with pytest.raises(B.DgAttnError) as e:
        p32.set(B.DG_OPT_PATH, B.DG_PATH_TC)
    assert e.value.status == B.DG_ERR_UNSUPPORTED
    assert plan.sync_status() == B.DG_OK


@pytest.mark.parametrize("schedule", [B.DG_SCHEDULE_SPLIT, B.DG_SCHEDULE_STREAM_K],
                         ids=["split", "stream_k"])
def test_bounded_wait_runs_out_cleanly_and_the_context_stays_usable(schedule):
    """Failure detection without a fault: the softmax withholds one P-ready signal (a flag that
    nothing else sets), every wait behind it runs out after the short limit, the kernel unwinds
    (TMEM freed, loads drained) and the host reads DG_ERR_TIMEOUT; the next forward is exact.
    With the stream-K schedule most CTAs hold two pieces, so the waits between them (Q reload,
    O hand-over) run out too."""
    T, ctx, nh, nkv, hd = (40, 300, 4, 2, 256) if schedule == B.DG_SCHEDULE_SPLIT else \
                          (130, 1500, 8, 4, 256)
    d = make_inputs(T, ctx, nh, nkv, hd, seed=31)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_SCHEDULE, schedule)
    assert plan.get(B.DG_INFO_SCHEDULE_USED) == schedule
    plan.set(B.DG_OPT_WAIT_LIMIT_MS, 100).set(B.DG_OPT_INJECT_STALL, 1)
    plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["k_cache"], dd["v_cache"],
                 dd["q_norm_w"], dd["k_norm_w"])
    assert plan.sync_status() == B.DG_ERR_TIMEOUT
    assert plan.sync_status() == B.DG_OK          # read-and-clear
    plan.set(B.DG_OPT_INJECT_STALL, 0)
    out = run_forward(plan, dd)
    check(out, oracle_out(d, nh, nkv, hd), B.DG_PATH_TC, all_rows(T), "after-timeout")


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_forward_replays_from_a_cuda_graph(path):
    """Every call only enqueues work, so a captured cache conversion + forwards replays to the
    same result as the eager calls, and the profiling events recorded during capture are taken
    again on each replay."""
    T, ctx, nh, nkv, hd = 70, 700, 8, 2, 128
    d = make_inputs(T, ctx, nh, nkv, hd, seed=41)
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path).set(B.DG_OPT_SPLITS, 3)
    eager = run_forward(plan, dd).clone()
    out = torch.empty_like(eager)
    plan.set(B.DG_OPT_PROFILE, 1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # the library runs once outside capture on this stream
        plan.cache_prepare(dd["k_cache"], dd["v_cache"])
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.cache_prepare(dd["k_cache"], dd["v_cache"])
        for _ in range(2):
            plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                         dd["k_norm_w"], out=out)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert plan.sync_status() == B.DG_OK
    assert torch.equal(out, eager)
    ms, n = B.dg_attn_profile_read(plan.handle, B.DG_STAGE_ATTENTION)
    assert n == 2 and ms > 0.0
    check(out, oracle_out(d, nh, nkv, hd), path, [(0, T)], "graph")


@pytest.mark.parametrize("shape", [(130, 1500, 8, 4, 256), (200, 700, 16, 8, 128),
                                   (512, 0, 16, 16, 64)],
                         ids=lambda s: "T%d_ctx%d_nh%d_nkv%d_hd%d" % s)
def test_resident_inputs_give_the_same_bits(shape):
    """With DG_OPT_INPUTS_RESIDENT the first stage of each forward runs while the previous
    forward's attention kernel does, writing the other operand set; the results must be
    bit-identical to forwards that wait for each other."""
    T, ctx, nh, nkv, hd = shape
    plans, outs = [], []
    canvases = [to_dev(make_inputs(T, ctx, nh, nkv, hd, seed=50 + i)) for i in range(4)]
    for resident in (0, 1):
        plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
        plan.set(B.DG_OPT_INPUTS_RESIDENT, resident)
        assert plan.get(B.DG_OPT_INPUTS_RESIDENT) == resident
        if ctx:
            plan.cache_prepare(canvases[0]["k_cache"], canvases[0]["v_cache"])
        res = [torch.empty((T, nh * hd), device="cuda") for _ in canvases]
        for c, o in zip(canvases, res):
            plan.forward(c["q"], c["k_canvas"], c["v_canvas"], None, None, c["q_norm_w"],
                         c["k_norm_w"], out=o)
        assert plan.sync_status() == B.DG_OK
        plans.append(plan)
        outs.append(res)
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    d = make_inputs(T, ctx, nh, nkv, hd, seed=53)
    d0 = make_inputs(T, ctx, nh, nkv, hd, seed=50)
    d["k_cache"], d["v_cache"] = d0["k_cache"], d0["v_cache"]     # the prepared cache
    check(outs[1][3], oracle_out(d, nh, nkv, hd), B.DG_PATH_TC, all_rows(T), "resident")


def test_resident_operand_sets_across_entry_points_and_a_failed_call():
    """With DG_OPT_INPUTS_RESIDENT the plan keeps a second set of tensor-core operand arrays and
    each forward's first stage writes the set the previous forward's attention kernel is not
    reading.  A sequence that switches the option on after the cache is prepared (the prepared
    rows are then copied into the new set), mixes forward, attend and a per-call cache, and has a
    call in the middle that fails before any launch, must give the same bits as the same sequence
    without the option, and match the oracle."""
    T, ctx, nh, nkv, hd = 130, 700, 8, 2, 128
    hosts = [make_inputs(T, ctx, nh, nkv, hd, seed=70 + i) for i in range(4)]
    other_cache = make_inputs(T, ctx, nh, nkv, hd, seed=80)
    cv = [to_dev(h) for h in hosts]
    c2 = to_dev(other_cache)
    results = []
    for resident in (0, 1):
        plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
        base = plan.get(B.DG_INFO_SCRATCH_BYTES)
        plan.cache_prepare(cv[0]["k_cache"], cv[0]["v_cache"])
        # the attend call's inputs, complete before the sequence (resident inputs must be)
        qh, kh, vh = plan.norm_rope(cv[2]["q"], cv[2]["k_canvas"], cv[2]["v_canvas"],
                                    cv[2]["q_norm_w"], cv[2]["k_norm_w"])
        torch.cuda.synchronize()
        plan.set(B.DG_OPT_INPUTS_RESIDENT, resident)
        assert (plan.get(B.DG_INFO_SCRATCH_BYTES) > base) == bool(resident)

        def fw(c, kc=None, vc=None):
            return plan.forward(c["q"], c["k_canvas"], c["v_canvas"], kc, vc, c["q_norm_w"],
                                c["k_norm_w"])

        outs = [fw(cv[0]), fw(cv[1])]                    # the prepared cache
        outs.append(plan.attend(qh, kh, vh))
        outs.append(fw(cv[3], c2["k_cache"], c2["v_cache"]))   # replaces the prepared cache
        with pytest.raises(B.DgAttnError) as e:
            fw(cv[0])                                    # no cache given and none prepared
        assert e.value.status == B.DG_ERR_STATE
        outs.append(fw(cv[1], c2["k_cache"], c2["v_cache"]))
        plan.cache_prepare(cv[0]["k_cache"], cv[0]["v_cache"])
        outs += [fw(cv[2]), fw(cv[3])]
        assert plan.sync_status() == B.DG_OK
        results.append(outs)
    for i, (a, b) in enumerate(zip(*results)):
        assert torch.equal(a, b), i
    caches = [0, 0, 0, None, None, 0, 0]
    canvases = [0, 1, 2, 3, 1, 2, 3]
    for o, ci, ca in zip(results[1], canvases, caches):
        d = dict(hosts[ci])
        src = hosts[0] if ca == 0 else other_cache
        d["k_cache"], d["v_cache"] = src["k_cache"], src["v_cache"]
        check(o, oracle_out(d, nh, nkv, hd), B.DG_PATH_TC, all_rows(T), f"canvas{ci}")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
def test_sixteen_bit_cache_twin(dtype, path):
    """A cache held as an f16 / bf16 twin: every 16-bit value is exact in fp32, so the block must
    match the oracle run on the widened cache; the prepared cache then serves later forwards."""
    T, ctx, nh, nkv, hd = 100, 900, 8, 2, 128
    d = make_inputs(T, ctx, nh, nkv, hd, seed=61)
    k16, v16 = d["k_cache"].to(dtype), d["v_cache"].to(dtype)
    d["k_cache"], d["v_cache"] = k16.float(), v16.float()       # what the oracle sees
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path)
    plan.cache_prepare(k16.cuda(), v16.cuda())
    assert plan.get(B.DG_INFO_CACHE_READY) == 1
    out = plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                       dd["k_norm_w"])
    assert plan.sync_status() == B.DG_OK
    check(out, oracle_out(d, nh, nkv, hd), path, [(0, T)], f"twin-{dtype}")
    # the fp32 cache through the same entry point gives the same bits as the 16-bit twin
    ref = out.clone()
    plan.cache_prepare(dd["k_cache"], dd["v_cache"])
    out2 = plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                        dd["k_norm_w"])
    assert plan.sync_status() == B.DG_OK
    assert torch.equal(out2, ref)


def test_output_overlapping_an_input_is_refused_before_any_launch():
    T, ctx, nh, nkv, hd = 8, 16, 2, 1, 64
    d = to_dev(make_inputs(T, ctx, nh, nkv, hd, seed=17))
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    h = plan.handle
    big = torch.zeros(4 * T * nh * hd, device="cuda")
    for inp in ("q", "k_canvas", "v_cache", "q_norm_w"):
        args = dict(d)
        args[inp] = big[: args[inp].numel()]
        with pytest.raises(B.DgAttnError) as e:
            B.dg_attn_forward(h, args["q"], args["k_canvas"], args["v_canvas"], args["k_cache"],
                              args["v_cache"], args["q_norm_w"], args["k_norm_w"], None,
                              big[16:16 + T * nh * hd])
        assert e.value.status == B.DG_ERR_ARG and "overlap" in B.last_error()
    out = torch.empty(T, nh * hd, device="cuda")
    with pytest.raises(B.DgAttnError) as e:
        B.dg_attn_norm_rope(h, d["q"], d["k_canvas"], d["v_canvas"], None, None, None, out,
                            out[0:1], torch.empty_like(d["v_canvas"]))
    assert e.value.status == B.DG_ERR_ARG
    assert plan.sync_status() == B.DG_OK


@pytest.mark.parametrize("prepared", [True, False], ids=["prepared", "per_call"])
def test_cache_value_beyond_fp16_is_reported(prepared):
    """The tensor-core P.V takes V in fp16: a cache value beyond 65504 cannot be held, and the
    forward reports DG_ERR_RANGE instead of silently overflowing.  The exact path takes it."""
    T, ctx, nh, nkv, hd = 16, 100, 4, 2, 128
    d = make_inputs(T, ctx, nh, nkv, hd, seed=18)
    d["v_cache"][1, 37, 5] = 1.0e5
    dd = to_dev(d)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    if prepared:
        plan.cache_prepare(dd["k_cache"], dd["v_cache"])
        plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], None, None, dd["q_norm_w"],
                     dd["k_norm_w"])
    else:
        plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["k_cache"], dd["v_cache"],
                     dd["q_norm_w"], dd["k_norm_w"])
    assert plan.sync_status() == B.DG_ERR_RANGE
    assert "fp16" in B.last_error()
    assert plan.sync_status() == B.DG_OK                  # read and cleared
    plan.set(B.DG_OPT_PATH, B.DG_PATH_FP32)
    out = run_forward(plan, dd).double().cpu().numpy()
    ref = oracle_out(d, nh, nkv, hd)
    # outputs that weigh the large value are far from RMS 1: compare relative to their size
    rel = np.abs(out - ref) / np.maximum(1.0, np.abs(ref))
    print(f"range-fp32: max |ref| {np.abs(ref).max():.3e}, max relative err {rel.max():.3e}")
    assert rel.max() <= 1e-5


def test_plans_on_several_host_threads():
    """Four host threads each create their own plan (both paths, two head sizes) and run forwards
    on their own stream at the same time; each result equals the same forward run alone.  The
    library's host state (the last-error text, the tensor-map encoder and the per-device kernel
    attributes) is per thread or set up once under a thread-safe guard."""
    import threading
    cases = [(40, 300, 4, 2, 128, B.DG_PATH_TC), (40, 300, 4, 2, 256, B.DG_PATH_TC),
             (33, 100, 8, 2, 64, B.DG_PATH_FP32), (50, 0, 4, 4, 64, B.DG_PATH_TC)]
    inputs = [to_dev(make_inputs(T, ctx, nh, nkv, hd, seed=500 + i))
              for i, (T, ctx, nh, nkv, hd, _) in enumerate(cases)]
    torch.cuda.synchronize()                # the inputs are read on other streams

    def run(i, results):
        T, ctx, nh, nkv, hd, path = cases[i]
        dd = inputs[i]
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
            plan.set(B.DG_OPT_PATH, path)
            outs = [plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["k_cache"],
                                 dd["v_cache"], dd["q_norm_w"], dd["k_norm_w"],
                                 stream=stream.cuda_stream) for _ in range(3)]
            stream.synchronize()
            assert plan.sync_status(stream.cuda_stream) == B.DG_OK
            plan.close()
        results[i] = outs

    alone = {}
    for i in range(len(cases)):
        run(i, alone)
    together = {}
    threads = [threading.Thread(target=run, args=(i, together)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for i in range(len(cases)):
        assert i in together, f"thread {i} failed"
        for a, b in zip(alone[i], together[i]):
            assert torch.equal(a, b)
