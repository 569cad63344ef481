"""Stream ordering of dependent calls.  The library's kernels start early (programmatic dependent
launch) and wait for the kernel ahead of them only where they touch its results, so a call whose
input is the previous call's output is the case that would expose a missing wait.  Each test
runs such a chain back to back on one stream (eagerly and replayed from a CUDA graph) and
requires the bits of the same calls separated by device synchronisations."""
import pytest
import torch

from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300.workloads import EPS, ROPE_THETA, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def layer_plan(T, ctx, nh, nkv, hd, H, seed):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32)
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.proj_prepare(H, (1.0 + 0.1 * r(H)).cuda(), (r(nh * hd, H) / H ** 0.5).cuda(),
                      (r(nkv * hd, H) / H ** 0.5).cuda(), (r(nkv * hd, H) / H ** 0.5).cuda())
    plan.oproj_prepare(H, (r(H, nh * hd) / (nh * hd) ** 0.5).cuda(), (1.0 + 0.1 * r(H)).cuda())
    return plan, r(T, H)


@pytest.mark.parametrize("mode", ["eager", "graph"])
def test_layers_chained_on_one_residual_stream(mode):
    """Three attention branches of a layer on one residual stream, a torch kernel between them:
    each call's input norm reads what the previous call's post-attention norm wrote."""
    T, ctx, nh, nkv, hd, H = 130, 700, 8, 4, 256, 512
    d = make_inputs(T, ctx, nh, nkv, hd, seed=201)
    cu = lambda t: None if t is None else t.cuda()
    qw, kw = cu(d["q_norm_w"]), cu(d["k_norm_w"])

    def chain(plan, x, sync):
        for _ in range(3):
            plan.forward_layer(x, None, None, qw, kw)
            if sync:
                torch.cuda.synchronize()
            x.mul_(0.75)
            if sync:
                torch.cuda.synchronize()

    plan, x0 = layer_plan(T, ctx, nh, nkv, hd, H, 202)
    plan.cache_prepare(cu(d["k_cache"]), cu(d["v_cache"]))
    torch.cuda.synchronize()
    want = x0.cuda()
    chain(plan, want, sync=True)
    got = x0.cuda()
    torch.cuda.synchronize()
    if mode == "eager":
        chain(plan, got, sync=False)
    else:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain(plan, got, sync=False)
        got.copy_(x0.cuda())
        torch.cuda.synchronize()
        g.replay()
    assert plan.sync_status() == B.DG_OK
    assert torch.isfinite(want).all()
    assert torch.equal(got, want)
    plan.close()


@pytest.mark.parametrize("path", [B.DG_PATH_TC, B.DG_PATH_FP32], ids=["tc", "fp32"])
@pytest.mark.parametrize("mode", ["eager", "graph"])
def test_forwards_chained_through_their_outputs(path, mode):
    """Four forwards in which each call's queries are the previous call's output (a torch kernel
    rescales it in between) and a cache is converted right before the first: the first stage must
    wait for the attention kernel ahead of it, and the first attention kernel for the
    conversion."""
    T, ctx, nh, nkv, hd = 256, 1024, 8, 4, 256
    d = make_inputs(T, ctx, nh, nkv, hd, seed=211)
    cu = lambda t: None if t is None else t.cuda()
    k, v, qw, kw = cu(d["k_canvas"]), cu(d["v_canvas"]), cu(d["q_norm_w"]), cu(d["k_norm_w"])
    kc, vc = cu(d["k_cache"]), cu(d["v_cache"])

    def chain(plan, q, outs, sync):
        plan.cache_prepare(kc, vc)
        for o in outs:
            plan.forward(q, k, v, None, None, qw, kw, None, o)
            if sync:
                torch.cuda.synchronize()
            q = o.mul(2.0)
            if sync:
                torch.cuda.synchronize()
        return q

    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path)
    q0 = cu(d["q"])
    want = [torch.empty_like(q0) for _ in range(4)]
    chain(plan, q0, want, sync=True)
    got = [torch.empty_like(q0) for _ in range(4)]
    torch.cuda.synchronize()
    if mode == "eager":
        chain(plan, q0, got, sync=False)
    else:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain(plan, q0, got, sync=False)
        for t in got:
            t.zero_()
        torch.cuda.synchronize()
        g.replay()
    assert plan.sync_status() == B.DG_OK
    for a, b in zip(got, want):
        assert torch.isfinite(b).all()
        assert torch.equal(a, b)
    plan.close()
