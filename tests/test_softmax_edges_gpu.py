"""GPU edge cases of the block's online softmax (page "inferencelayer 0.2.3,
src/diffusion_gemma_gpu.rs", item DG_ATTN: running maximum, correction factor, running
denominator), on both arithmetic paths and every head size of the tensor-core path.

RoPE would make a key depend on its row's position, so every case passes an identity cos|sin
table (cos = 1, sin = 0) and unweighted norms: q-hat is then RMSNorm(q) and a canvas key is
RMSNorm(k), while cache keys are used as given.  Each query head is c * e_0, so q-hat = r * e_0
with r = c / sqrt(c^2 / hd + eps) ~ sqrt(hd), and the score of a key is r times its component 0.
Canvas keys get component 0 = 0 (score 0) unless a case says otherwise.

Cases:
  - one dominant key returns its V (exactly its fp16 rounding on the tensor-core path);
  - a dominant key whose probability is not a power of two relative to the running reference
    (set by an earlier key 10.3 log2 units lower): numerator and denominator must carry the same
    fp16 rounding of it;
  - identical keys (all scores equal) return the mean of V;
  - scores that rise by 24 (log2 units) every 64 keys, so the running maximum jumps on every key
    tile and the accumulated output is rescaled each time;
  - many keys 14.5 to 17.5 log2 units below the maximum, whose probabilities are fp16 subnormals
    on the tensor-core path, carrying ~3% of the softmax weight.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_canvas_attention_gb300 import binding as B
from gqa_canvas_attention_gb300.workloads import EPS, ROPE_THETA

pytestmark = pytest.mark.gpu

TOL = {B.DG_PATH_TC: (5e-3, 5e-4), B.DG_PATH_FP32: (1e-5, 1e-6)}
PATHS = [B.DG_PATH_TC, B.DG_PATH_FP32]
PNAME = {B.DG_PATH_TC: "tc", B.DG_PATH_FP32: "fp32"}
LOG2E = 1.0 / math.log(2.0)
C = 3.0                      # component 0 of every query head


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def qhat0(hd):
    """Component 0 of every q-hat row (fp64)."""
    return C / math.sqrt(C * C / hd + EPS)


def base_inputs(T, ctx, nh, nkv, hd, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.zeros(T, nh * hd)
    q[:, ::hd] = C
    kc = torch.randn(T, nkv * hd, generator=g)
    kc[:, ::hd] = 0.0
    vc = torch.randn(T, nkv * hd, generator=g)
    k_cache = torch.randn(nkv, ctx, hd, generator=g)
    v_cache = torch.randn(nkv, ctx, hd, generator=g)
    table = torch.cat([torch.ones(T, hd), torch.zeros(T, hd)], 1)
    return {"q": q, "k_canvas": kc, "v_canvas": vc, "k_cache": k_cache, "v_cache": v_cache,
            "q_norm_w": None, "k_norm_w": None}, table


def run(d, table, nh, nkv, hd, path, splits=0):
    T = d["q"].shape[0]
    ctx = d["k_cache"].shape[1]
    dd = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    plan = B.Plan(nh, nkv, hd, ctx, T, EPS, ROPE_THETA)
    plan.set(B.DG_OPT_PATH, path)
    if splits:
        plan.set(B.DG_OPT_SPLITS, splits)
    out = plan.forward(dd["q"], dd["k_canvas"], dd["v_canvas"], dd["k_cache"], dd["v_cache"],
                       None, None, table.cuda())
    assert plan.sync_status() == B.DG_OK
    o = out.cpu().double().numpy()
    assert np.isfinite(o).all()
    return o


def ref_out(d, table, nh, nkv, hd):
    f = lambda x: None if x is None else x.numpy()
    return oracle.forward(f(d["q"]), f(d["k_canvas"]), f(d["v_canvas"]), f(d["k_cache"]),
                          f(d["v_cache"]), nh, nkv, hd, None, None, cos_sin=table.numpy(),
                          eps=EPS, theta=ROPE_THETA)


def check_oracle(o, ref, path, label):
    tmax, tmean = TOL[path]
    e = np.abs(o - ref)
    print(f"{label} {PNAME[path]}: max {e.max():.3e} mean {e.mean():.3e}")
    assert e.max() <= tmax, f"{label}: max err {e.max():.3e}"
    assert e.mean() <= tmean, f"{label}: mean err {e.mean():.3e}"


def rows_of_group(o, T, nh, nkv, hd, g):
    """[T, G, hd] block of the output rows that attend to kv group g."""
    G = nh // nkv
    return o.reshape(T, nh, hd)[:, g * G:(g + 1) * G, :]


def f16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().half().double().numpy()


HDS = [64, 128, 256]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
@pytest.mark.parametrize("hd", HDS)
def test_one_dominant_key_returns_its_value(hd, path):
    T, ctx, nh, nkv = 40, 700, 4, 2
    d, table = base_inputs(T, ctx, nh, nkv, hd, seed=hd)
    kc = d["k_cache"]
    kc[:, :, 0] = 0.1 * kc[:, :, 0]                 # other scores |s| < ~0.5 * sqrt(hd)
    dom = {0: 517, 1: 3}                            # a late key tile and the first one
    for g, j in dom.items():
        kc[g, j, 0] = 45.0 / qhat0(hd)              # score 45 (natural): the rest < e^-38
    o = run(d, table, nh, nkv, hd, path)
    check_oracle(o, ref_out(d, table, nh, nkv, hd), path, f"dominant hd={hd}")
    for g, j in dom.items():
        v = d["v_cache"][g, j].double().numpy()
        got = rows_of_group(o, T, nh, nkv, hd, g)
        if path == B.DG_PATH_TC:
            # V enters P.V rounded to fp16; the dominant key's own probability cancels exactly
            want = f16(v)
            assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max()
            assert np.abs(got - v).max() <= 2.0 ** -11 * np.abs(v).max() + 1e-6
        else:
            assert np.abs(got - v).max() <= 1e-5


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
@pytest.mark.parametrize("hd", HDS)
def test_dominant_key_off_a_power_of_two_keeps_numerator_and_denominator_consistent(hd, path):
    """An earlier key P sets the running reference; the dominant key D scores 10.3 log2 units
    above it (no rescale below 15), so its probability 2^10.3 is rounded to fp16 on the
    tensor-core path.  The output must be (w V_D + V_P) / (w + 1), w = 2^10.3, with that rounding
    cancelling between numerator and denominator (a denominator summed from the unrounded values
    would leave a relative error of up to 2^-11 on every element)."""
    T, ctx, nh, nkv = 24, 600, 4, 2
    d, table = base_inputs(T, ctx, nh, nkv, hd, seed=10 + hd)
    kc = d["k_cache"]
    kc[:, :, 0] = 0.1 * kc[:, :, 0]
    jP, jD = 5, 400                                 # P in the first key tile, D much later
    sP = 50.0                                       # natural units: the rest are < e^-44
    sD = sP + 10.3 / LOG2E
    for g in range(nkv):
        kc[g, jP, 0] = sP / qhat0(hd)
        kc[g, jD, 0] = sD / qhat0(hd)
    o = run(d, table, nh, nkv, hd, path, splits=1)
    check_oracle(o, ref_out(d, table, nh, nkv, hd), path, f"offset hd={hd}")
    w = 2.0 ** 10.3
    for g in range(nkv):
        vP = d["v_cache"][g, jP].double().numpy()
        vD = d["v_cache"][g, jD].double().numpy()
        got = rows_of_group(o, T, nh, nkv, hd, g)
        if path == B.DG_PATH_TC:
            want = (w * f16(vD) + f16(vP)) / (w + 1.0)
            err = np.abs(got - want).max()
            print(f"hd={hd} g={g}: |out - fp16-consistent expectation| = {err:.2e}")
            assert err <= 5e-5, err
        else:
            want = (w * vD + vP) / (w + 1.0)
            assert np.abs(got - want).max() <= 1e-5


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
@pytest.mark.parametrize("hd", HDS)
def test_identical_keys_return_the_mean_of_v(hd, path):
    """Every key is the same vector u (cache rows u-hat as given, canvas rows u, normed on the
    device to u-hat), so every score is equal and the output is the mean of all S values."""
    T, ctx, nh, nkv = 33, 450, 4, 2
    d, table = base_inputs(T, ctx, nh, nkv, hd, seed=20 + hd)
    g = torch.Generator().manual_seed(99)
    d["q"] = torch.randn(T, nh * hd, generator=g)   # any queries: the scores are still equal
    u = torch.randn(nkv, hd, generator=g, dtype=torch.float64)
    uhat = u / torch.sqrt((u * u).mean(1, keepdim=True) + EPS)
    d["k_canvas"] = u.float().reshape(1, nkv * hd).repeat(T, 1)
    d["k_cache"] = uhat.float()[:, None, :].repeat(1, ctx, 1)
    # canvas values of RMS exactly 1, so their norm is a division by sqrt(1 + eps)
    signs = torch.randint(0, 2, (T, nkv * hd), generator=g).float() * 2.0 - 1.0
    d["v_canvas"] = signs
    o = run(d, table, nh, nkv, hd, path)
    check_oracle(o, ref_out(d, table, nh, nkv, hd), path, f"identical hd={hd}")
    vhat = signs.double().numpy().reshape(T, nkv, hd) / math.sqrt(1.0 + EPS)
    for gg in range(nkv):
        mean = (d["v_cache"][gg].double().numpy().sum(0) + vhat[:, gg].sum(0)) / (ctx + T)
        got = rows_of_group(o, T, nh, nkv, hd, gg)
        tol = 2e-4 if path == B.DG_PATH_TC else 2e-6
        assert np.abs(got - mean).max() <= tol


@pytest.mark.parametrize("splits", [1, 0], ids=["one_partition", "auto_partitions"])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
@pytest.mark.parametrize("hd", HDS)
def test_scores_rising_on_every_key_tile_rescale_each_time(hd, path, splits):
    """Cache key j scores 24 * floor(j / 64) log2 units plus a jitter of up to 7 within its block
    of 64 keys, so the running maximum exceeds the rescale threshold on every key tile (64 or 128
    keys on the tensor-core path, 32 on the fp32 path) and the output accumulated so far is
    rescaled each time; the result is dominated by the last block."""
    T, ctx, nh, nkv = 30, 704, 4, 2
    d, table = base_inputs(T, ctx, nh, nkv, hd, seed=30 + hd)
    g = torch.Generator().manual_seed(7)
    j = torch.arange(ctx, dtype=torch.float64)
    for gg in range(nkv):
        s2 = 24.0 * torch.floor(j / 64) + 7.0 * torch.rand(ctx, generator=g, dtype=torch.float64)
        d["k_cache"][gg, :, 0] = (s2 / LOG2E / qhat0(hd)).float()
    o = run(d, table, nh, nkv, hd, path, splits=splits)
    check_oracle(o, ref_out(d, table, nh, nkv, hd), path, f"rising hd={hd}")


@pytest.mark.parametrize("splits", [1, 0], ids=["one_partition", "auto_partitions"])
@pytest.mark.parametrize("path", PATHS, ids=lambda p: PNAME[p])
@pytest.mark.parametrize("hd", HDS)
def test_keys_in_the_fp16_subnormal_band(hd, path, splits):
    """The top key sits in the first key tile, so the running reference is its score; 1800
    near-duplicate keys score 15.5 (+-0.05) log2 units below it -- probabilities ~2^-15.5, below
    the smallest normal fp16 number 2^-14 -- share one value vector v0 (the top key has -v0) and
    together carry ~4% of the weight.  They must count at their value: on a subnormal fp16 grid
    of 2^-24 each keeps ~724 steps.  (Were the reference 8 above the top, each would sit at
    1.4 steps, round to 1, and the output would move by ~3e-2.)"""
    T, ctx, nh, nkv = 20, 2000, 2, 1
    d, table = base_inputs(T, ctx, nh, nkv, hd, seed=40 + hd)
    g = torch.Generator().manual_seed(8)
    top = 40.0 * LOG2E                                           # log2 units
    s2 = top - 15.5 + 0.1 * (torch.rand(ctx, generator=g, dtype=torch.float64) - 0.5)
    s2[:200] = top - 60.0                                        # negligible keys
    s2[3] = top
    d["k_cache"][0, :, 0] = (s2 / LOG2E / qhat0(hd)).float()
    v0 = torch.randn(hd, generator=g)
    d["v_cache"][0, 200:] = v0
    d["v_cache"][0, 3] = -v0
    ref = ref_out(d, table, nh, nkv, hd)
    # the band's share of the weight, from the scores as stored (fp32 keys)
    s = d["k_cache"][0, :, 0].double().numpy() * qhat0(hd) * LOG2E
    p = 2.0 ** (s - s.max())
    band = p[(s <= s.max() - 14.0)].sum() / p.sum()
    assert 0.03 < band < 0.05
    o = run(d, table, nh, nkv, hd, path, splits=splits)
    check_oracle(o, ref, path, f"subnormal hd={hd}")
