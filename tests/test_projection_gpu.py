"""GPU parity of the projection step before the block (dg_attn_proj_prepare +
dg_attn_forward_hidden): input RMSNorm, q/k/v projections on the tensor cores with the block's
first stage fused into their epilogue, then the attention block, against the fp64 oracle
(oracle.forward_hidden) at the tensor-core tolerances (max 5e-3, mean 5e-4)."""
import numpy as np
import pytest
import torch

import oracle
from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300.workloads import EPS, ROPE_THETA, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def weights(H, nh, nkv, hd, seed, with_v=True):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32)
    ln = 1.0 + 0.1 * r(H)
    wq = r(nh * hd, H) / H ** 0.5
    wk = r(nkv * hd, H) / H ** 0.5
    wv = r(nkv * hd, H) / H ** 0.5 if with_v else None
    return ln, wq, wk, wv


# Geometries with 32, 12 and 24 column tiles of 128 (10 without a value projection at hd 128),
# and 5 (nh = 3, nkv = 1: an odd count).
@pytest.mark.parametrize("shape", [(130, 700, 8, 4, 256, 512), (70, 300, 8, 2, 128, 384),
                                   (256, 1024, 8, 4, 256, 1024), (40, 100, 3, 1, 128, 256)],
                         ids=lambda s: "T%d_ctx%d_nh%d_nkv%d_hd%d_H%d" % s)
@pytest.mark.parametrize("with_v", [True, False], ids=["wv", "k_eq_v"])
@pytest.mark.parametrize("schedule", [B.DG_SCHEDULE_AUTO, B.DG_SCHEDULE_STREAM_K],
                         ids=["auto", "stream_k"])
def test_hidden_to_output_parity(shape, with_v, schedule):
    T, ctx, nh, nkv, hd, H = shape
    d = make_inputs(T, ctx, nh, nkv, hd, seed=71)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(72), dtype=torch.float32)
    ln, wq, wk, wv = weights(H, nh, nkv, hd, 73, with_v)
    cu = lambda t: None if t is None else t.cuda()
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_SCHEDULE, schedule)
    if schedule == B.DG_SCHEDULE_STREAM_K:
        assert plan.get(B.DG_INFO_SCHEDULE_USED) == B.DG_SCHEDULE_STREAM_K
    plan.proj_prepare(H, cu(ln), cu(wq), cu(wk), cu(wv))
    out = plan.forward_hidden(cu(x), cu(d["k_cache"]), cu(d["v_cache"]), cu(d["q_norm_w"]),
                              cu(d["k_norm_w"]))
    assert plan.sync_status() == B.DG_OK
    n = lambda t: None if t is None else t.numpy()
    rows = (0, T)
    ref = oracle.forward_hidden(n(x), n(ln), n(wq), n(wk), n(wv), n(d["k_cache"]),
                                n(d["v_cache"]), nh, nkv, hd, n(d["q_norm_w"]), n(d["k_norm_w"]),
                                eps=EPS, theta=ROPE_THETA, rows=rows)
    o = out.cpu().double().numpy()[rows[0]:rows[1]]
    e = np.abs(o - ref[rows[0]:rows[1]])
    print(f"max {e.max():.3e} mean {e.mean():.3e}")
    assert np.isfinite(o).all()
    assert e.max() <= 5e-3 and e.mean() <= 5e-4


def test_projection_needs_prepared_weights_and_the_tensor_core_path():
    T, ctx, nh, nkv, hd, H = 8, 16, 2, 1, 128, 64
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    x = torch.zeros(T, H, device="cuda")
    with pytest.raises(B.DgAttnError) as e:
        plan.forward_hidden(x)
    assert e.value.status == B.DG_ERR_STATE
    with pytest.raises(B.DgAttnError) as e:
        plan.proj_prepare(100, None, torch.zeros(nh * hd, 100, device="cuda"),
                          torch.zeros(nkv * hd, 100, device="cuda"))
    assert e.value.status == B.DG_ERR_ARG
    p64 = B.Plan(nh, nkv, 64, ctx, T, EPS, ROPE_THETA)
    with pytest.raises(B.DgAttnError) as e:
        p64.proj_prepare(H, None, torch.zeros(nh * 64, H, device="cuda"),
                         torch.zeros(nkv * 64, H, device="cuda"))
    assert e.value.status == B.DG_ERR_UNSUPPORTED
    assert plan.sync_status() == B.DG_OK


# At T = 130, H = 512, 384, 192, 2560 give 8, 6, 3 and 40 o_proj column tiles of 64.
@pytest.mark.parametrize("H", [512, 384, 192, 2560])
def test_oproj_residual_parity(H):
    """o_proj + post-attention RMSNorm + residual add on the tensor cores against the oracle."""
    T, nh, nkv, hd = 130, 8, 4, 256
    K = nh * hd
    g = torch.Generator().manual_seed(81)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32)
    attn, wo, ln, resid = r(T, K), r(H, K) / K ** 0.5, 1.0 + 0.1 * r(H), r(T, H)
    plan = B.Plan(nh, nkv, hd, 64, T, EPS, ROPE_THETA)
    plan.oproj_prepare(H, wo.cuda(), ln.cuda())
    res_d = resid.cuda()
    plan.oproj_residual(attn.cuda(), res_d)
    assert plan.sync_status() == B.DG_OK
    ref = oracle.oproj_residual(attn.numpy(), wo.numpy(), ln.numpy(), resid.numpy(), eps=EPS)
    e = np.abs(res_d.cpu().double().numpy() - ref)
    print(f"max {e.max():.3e} mean {e.mean():.3e}")
    assert e.max() <= 1e-4 and e.mean() <= 1e-5


def test_attention_branch_of_a_layer_parity():
    """The whole attention branch on the residual stream (input norm, projections, block, o_proj,
    post-attention norm, residual add) against the oracle chain, at the block's tolerances."""
    T, ctx, nh, nkv, hd, H = 130, 700, 8, 4, 256, 512
    d = make_inputs(T, ctx, nh, nkv, hd, seed=91)
    g = torch.Generator().manual_seed(92)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32)
    x = r(T, H)
    ln, wq, wk, wv = weights(H, nh, nkv, hd, 93)
    wo, ln_post = r(H, nh * hd) / (nh * hd) ** 0.5, 1.0 + 0.1 * r(H)
    cu = lambda t: None if t is None else t.cuda()
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.proj_prepare(H, cu(ln), cu(wq), cu(wk), cu(wv))
    plan.oproj_prepare(H, cu(wo), cu(ln_post))
    xd = cu(x)
    plan.forward_layer(xd, cu(d["k_cache"]), cu(d["v_cache"]), cu(d["q_norm_w"]), cu(d["k_norm_w"]))
    assert plan.sync_status() == B.DG_OK
    n = lambda t: None if t is None else t.numpy()
    attn = oracle.forward_hidden(n(x), n(ln), n(wq), n(wk), n(wv), n(d["k_cache"]),
                                 n(d["v_cache"]), nh, nkv, hd, n(d["q_norm_w"]), n(d["k_norm_w"]),
                                 eps=EPS, theta=ROPE_THETA)
    ref = oracle.oproj_residual(attn.astype(np.float32), n(wo), n(ln_post), n(x), eps=EPS)
    e = np.abs(xd.cpu().double().numpy() - ref)
    print(f"max {e.max():.3e} mean {e.mean():.3e}")
    assert np.isfinite(e).all()
    assert e.max() <= 5e-3 and e.mean() <= 5e-4


@pytest.mark.parametrize("schedule", ["clustered", "one_partition", "stream_k", "nine_partitions"])
def test_layer_writes_the_o_proj_operands_in_the_attention_kernel(schedule):
    """Inside dg_attn_forward_layer the attention kernel, where it writes the output itself (one
    partition, or partitions merged inside a cluster), also writes the bf16 hi / lo split that
    o_proj reads, with the same arithmetic as the separate split kernel; the other schedules
    (stream-K, more than 8 partitions through the combine kernel) keep that kernel.  Either way
    the residual stream must come out bit for bit as when the two steps are called separately."""
    T, ctx, nh, nkv, hd, H = 130, 700, 8, 4, 256, 512
    d = make_inputs(T, ctx, nh, nkv, hd, seed=95)
    g = torch.Generator().manual_seed(96)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32)
    x = r(T, H)
    ln, wq, wk, wv = weights(H, nh, nkv, hd, 97)
    wo, ln_post = r(H, nh * hd) / (nh * hd) ** 0.5, 1.0 + 0.1 * r(H)
    cu = lambda t: None if t is None else t.cuda()
    results = []
    for fused in (True, False):
        plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
        if schedule == "one_partition":
            plan.set(B.DG_OPT_SPLITS, 1)
        elif schedule == "stream_k":
            plan.set(B.DG_OPT_SCHEDULE, B.DG_SCHEDULE_STREAM_K)
        elif schedule == "nine_partitions":
            plan.set(B.DG_OPT_SPLITS, 9)
        plan.proj_prepare(H, cu(ln), cu(wq), cu(wk), cu(wv))
        plan.oproj_prepare(H, cu(wo), cu(ln_post))
        xd = cu(x)
        kc, vc = cu(d["k_cache"]), cu(d["v_cache"])
        if fused:
            plan.forward_layer(xd, kc, vc, cu(d["q_norm_w"]), cu(d["k_norm_w"]))
        else:
            attn = plan.forward_hidden(xd, kc, vc, cu(d["q_norm_w"]), cu(d["k_norm_w"]))
            plan.oproj_residual(attn, xd)
        assert plan.sync_status() == B.DG_OK
        results.append(xd)
        plan.close()
    assert torch.equal(results[0], results[1])
