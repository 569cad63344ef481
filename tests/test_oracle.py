"""Pins for the fp64 oracle, checked against things other than the oracle itself.

Each test ties one part of the oracle to a fact fixed by the page ("inferencelayer 0.2.3,
src/diffusion_gemma_gpu.rs": DG_HEADNORM_ROPE, DG_ATTN) or by mathematics: closed forms,
textbook special cases, invariants, and a brute-force restatement built a different way
(explicit rotation matrices and a dense score matrix).  The mistakes each one would catch are
named in its docstring.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def rnd(*shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(np.float32)


# ---------------------------------------------------------------- RMSNorm (DG_HEADNORM_ROPE)

def test_rmsnorm_closed_form_mean_square():
    """Unweighted y = x (m + eps)^-1/2 has mean(y^2) = m / (m + eps) exactly (m = mean x^2).
    Catches: eps outside the sqrt, sum instead of mean, a missing square root."""
    for hd in (2, 8, 64, 256):
        for eps in (1e-6, 0.25):
            x = rnd(3, hd)
            y = oracle.norm_rope(x, 1, hd, eps=eps, rope=False)[:, 0, :]
            m = (x.astype(np.float64) ** 2).mean(axis=1)
            np.testing.assert_allclose((y ** 2).mean(axis=1), m / (m + eps), rtol=1e-13)


def test_rmsnorm_weight_multiplies():
    """The weight multiplies element-wise (w, not 1 + w), after the normalisation.
    Catches: 1 + w, weight inside the mean."""
    hd = 16
    x, w = rnd(2, 3 * hd), (1.0 + 0.5 * rnd(hd))
    a = oracle.norm_rope(x, 3, hd, w=w, rope=False)
    b = oracle.norm_rope(x, 3, hd, w=None, rope=False)
    np.testing.assert_allclose(a, b * w.astype(np.float64), rtol=1e-14)


def test_rmsnorm_per_head_independent():
    """Each (row, head) is normalised on its own slice.  Catches: a norm over the whole row."""
    hd = 8
    x = rnd(1, 2 * hd)
    x[0, hd:] *= 100.0
    y = oracle.norm_rope(x, 2, hd, rope=False)
    for h in range(2):
        np.testing.assert_allclose((y[0, h] ** 2).mean(), 1.0, rtol=1e-5)


# ---------------------------------------------------------------- RoPE (DG_HEADNORM_ROPE)

def test_rope_position_zero_is_identity():
    """At p = 0 every angle is 0.  Catches: an offset in the position."""
    hd = 64
    x = rnd(1, 2 * hd)
    a = oracle.norm_rope(x, 2, hd, rope=True, pos0=0)
    b = oracle.norm_rope(x, 2, hd, rope=False)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-15)


def test_rope_hd2_is_plane_rotation_by_p_radians():
    """hd = 2 has one pair with frequency theta^0 = 1, so RoPE at position p is the textbook
    counter-clockwise rotation by p radians: (y0 cos p - y1 sin p, y1 cos p + y0 sin p).
    Catches: a sign flip of the rotate-half term, swapped cos/sin."""
    x = rnd(5, 2)
    y = oracle.norm_rope(x, 1, 2, rope=False)[:, 0, :]
    z = oracle.norm_rope(x, 1, 2, rope=True, pos0=7)[:, 0, :]
    for r in range(5):
        p = 7 + r
        R = np.array([[math.cos(p), -math.sin(p)], [math.sin(p), math.cos(p)]])
        np.testing.assert_allclose(z[r], R @ y[r], rtol=0, atol=1e-14)


def test_rope_hd4_pairs_and_frequencies():
    """hd = 4, theta = 10000: element pairs are (0, 2) and (1, 3) (rotate-half, not adjacent),
    rotated by p * 1 and p * 10000^(-1/2) = p / 100.  Catches: interleaved pairing, a wrong
    exponent (2i/hd vs i/hd), theta applied as theta^(+...)."""
    p = 123
    x = rnd(1, 4)
    y = oracle.norm_rope(x, 1, 4, rope=False)[0, 0]
    z = oracle.norm_rope(x, 1, 4, rope=True, pos0=p, theta=10000.0)[0, 0]
    for i, ang in ((0, p * 1.0), (1, p / 100.0)):
        c, s = math.cos(ang), math.sin(ang)
        np.testing.assert_allclose(z[i], y[i] * c - y[i + 2] * s, atol=1e-13)
        np.testing.assert_allclose(z[i + 2], y[i + 2] * c + y[i] * s, atol=1e-13)


def test_rope_preserves_norm():
    """A rotation keeps the Euclidean norm.  Catches: cos and sin not from the same angle."""
    hd = 128
    x = rnd(4, 3 * hd)
    y = oracle.norm_rope(x, 3, hd, rope=False)
    z = oracle.norm_rope(x, 3, hd, rope=True, pos0=9000)
    np.testing.assert_allclose(np.linalg.norm(z, axis=-1), np.linalg.norm(y, axis=-1), rtol=1e-13)


def test_rope_relative_position_property():
    """<R(p+c) a, R(p'+c) b> = <R(p) a, R(p') b>: dot products depend only on p - p'."""
    hd = 64
    a, b = rnd(1, hd), rnd(1, hd)
    for (p, pp, c) in ((3, 11, 500), (0, 8191, 17), (4000, 4000, 4096)):
        za = oracle.norm_rope(a, 1, hd, pos0=p + c)[0, 0]
        zb = oracle.norm_rope(b, 1, hd, pos0=pp + c)[0, 0]
        ya = oracle.norm_rope(a, 1, hd, pos0=p)[0, 0]
        yb = oracle.norm_rope(b, 1, hd, pos0=pp)[0, 0]
        assert abs(za @ zb - ya @ yb) < 1e-11


def test_rope_table_matches_formula():
    """A cos|sin table built from the same angles gives the same result (to fp32 rounding of
    the table), and the table is taken per element verbatim."""
    hd, T, pos0 = 32, 6, 40
    x = rnd(T, 2 * hd)
    half = hd // 2
    tab = np.zeros((T, 2 * hd), np.float32)
    for t in range(T):
        ang = (pos0 + t) * 10000.0 ** (-2.0 * (np.arange(hd) % half) / hd)
        tab[t, :hd], tab[t, hd:] = np.cos(ang), np.sin(ang)
    a = oracle.norm_rope(x, 2, hd, pos0=pos0, cos_sin=tab)
    b = oracle.norm_rope(x, 2, hd, pos0=pos0)
    np.testing.assert_allclose(a, b, atol=2e-7)
    ident = np.concatenate([np.ones((T, hd)), np.zeros((T, hd))], 1).astype(np.float32)
    np.testing.assert_allclose(oracle.norm_rope(x, 2, hd, pos0=pos0, cos_sin=ident),
                               oracle.norm_rope(x, 2, hd, rope=False), atol=0)


# ---------------------------------------------------------------- brute force (whole block)

def brute_force(q, kc, vc, kcache, vcache, nh, nkv, hd, wq, wk, eps, theta, pos0):
    """The block restated with different machinery: RMS via np.linalg.norm, RoPE as an explicit
    hd x hd block-rotation matrix, attention as one dense [rows, S] score matrix per q head with
    an explicit softmax."""
    T = q.shape[0]
    ctx = 0 if kcache is None else kcache.shape[1]
    half = hd // 2

    def rms(v, w):
        v = v.astype(np.float64)
        n = np.linalg.norm(v, axis=-1, keepdims=True) / math.sqrt(hd)
        out = v / np.sqrt(n ** 2 + eps)
        return out if w is None else out * w.astype(np.float64)

    def rot(p):
        R = np.zeros((hd, hd))
        for i in range(half):
            ang = p / theta ** (2.0 * i / hd)
            c, s = math.cos(ang), math.sin(ang)
            R[i, i], R[i, i + half] = c, -s
            R[i + half, i + half], R[i + half, i] = c, s
        return R

    Q = rms(q.reshape(T, nh, hd), wq)
    K = rms(kc.reshape(T, nkv, hd), wk)
    V = rms(vc.reshape(T, nkv, hd), None)
    for t in range(T):
        R = rot(pos0 + t)
        Q[t] = Q[t] @ R.T
        K[t] = K[t] @ R.T
    out = np.zeros((T, nh, hd))
    G = nh // nkv
    for h in range(nh):
        g = h // G
        keys = K[:, g, :]
        vals = V[:, g, :]
        if ctx:
            keys = np.concatenate([kcache[g].astype(np.float64), keys], 0)
            vals = np.concatenate([vcache[g].astype(np.float64), vals], 0)
        Sm = Q[:, h, :] @ keys.T
        Pm = np.exp(Sm - Sm.max(axis=1, keepdims=True))
        Pm /= Pm.sum(axis=1, keepdims=True)
        out[:, h, :] = Pm @ vals
    return out.reshape(T, nh * hd)


@pytest.mark.parametrize("T,ctx,nh,nkv,hd,weighted", [
    (5, 7, 4, 2, 8, True),
    (3, 0, 2, 2, 16, False),
    (4, 3, 6, 3, 4, True),
    (1, 1, 1, 1, 2, False),
    (6, 9, 8, 1, 32, True),
])
def test_forward_matches_brute_force(T, ctx, nh, nkv, hd, weighted):
    q, kc, vc = rnd(T, nh * hd), rnd(T, nkv * hd), rnd(T, nkv * hd)
    kca = rnd(nkv, ctx, hd) if ctx else None
    vca = rnd(nkv, ctx, hd) if ctx else None
    wq = (1 + 0.1 * rnd(hd)) if weighted else None
    wk = (1 + 0.1 * rnd(hd)) if weighted else None
    a = oracle.forward(q, kc, vc, kca, vca, nh, nkv, hd, wq, wk, eps=1e-6, theta=10000.0)
    b = brute_force(q, kc, vc, kca, vca, nh, nkv, hd, wq, wk, 1e-6, 10000.0, ctx)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


# ---------------------------------------------------------------- attention invariants (DG_ATTN)

def test_softmax_rows_sum_to_one_via_one_hot_values():
    """With value j = e_j (one-hot, S <= hd) the output is the probability row itself: it must
    be non-negative and sum to 1.  Catches: a missing or wrong denominator."""
    T, ctx, nh, nkv, hd = 5, 6, 2, 1, 16
    S = ctx + T
    qh = oracle.norm_rope(rnd(T, nh * hd), nh, hd, pos0=ctx)
    kh = oracle.norm_rope(rnd(T, nkv * hd), nkv, hd, pos0=ctx)
    vh = np.zeros((T, nkv, hd))
    for t in range(T):
        vh[t, 0, ctx + t] = 1.0
    kcache = rnd(nkv, ctx, hd)
    vcache = np.zeros((nkv, ctx, hd), np.float32)
    for j in range(ctx):
        vcache[0, j, j] = 1.0
    out = oracle.attention(qh, kh, vh, kcache, vcache, nh, nkv, hd)
    assert (out >= 0).all()
    np.testing.assert_allclose(out[:, :, :S].sum(-1), 1.0, atol=1e-14)
    assert np.abs(out[:, :, S:]).max() == 0.0


def test_identical_keys_give_mean_of_values():
    """All keys equal -> equal weights -> output = mean of all S values (cache and canvas)."""
    T, ctx, nh, nkv, hd = 4, 5, 2, 2, 8
    key = rnd(hd)
    qh = oracle.norm_rope(rnd(T, nh * hd), nh, hd, pos0=ctx)
    kh = np.broadcast_to(key.astype(np.float64), (T, nkv, hd)).copy()
    vh = oracle.norm_rope(rnd(T, nkv * hd), nkv, hd, rope=False)
    kcache = np.broadcast_to(key, (nkv, ctx, hd)).copy()
    vcache = rnd(nkv, ctx, hd)
    out = oracle.attention(qh, kh, vh, kcache, vcache, nh, nkv, hd)
    for h in range(nh):
        g = h // (nh // nkv)
        mean = (vcache[g].astype(np.float64).sum(0) + vh[:, g].sum(0)) / (ctx + T)
        np.testing.assert_allclose(out[:, h], np.broadcast_to(mean, (T, hd)), atol=1e-14)


def test_single_key_returns_normed_value_unroped():
    """T = 1, ctx = 0: one key, weight 1, so the output is the canvas V after the weightless,
    un-roped V norm, whatever q, k, the weights and the position are.  Catches: RoPE or the k
    weight applied to V."""
    hd = 16
    q, k, v = rnd(1, 3 * hd), rnd(1, hd), rnd(1, hd)
    out = oracle.forward(q, k, v, None, None, 3, 1, hd, q_norm_w=1 + rnd(hd),
                         k_norm_w=1 + rnd(hd), pos0=777)
    v64 = v.astype(np.float64)[0]
    expect = v64 / math.sqrt((v64 ** 2).mean() + 1e-6)
    for h in range(3):
        np.testing.assert_allclose(out[0, h * hd:(h + 1) * hd], expect, rtol=1e-13)


def test_dominant_cache_key_returns_its_value_as_given():
    """A cache key aligned with q-hat and 50x its scale dominates the softmax, so the output is
    that cache row's value exactly as stored (the cache is neither normed nor roped).
    Catches: roping or norming the cache, cache/canvas index mix-ups."""
    T, ctx, nh, nkv, hd = 1, 3, 2, 1, 32
    q, kc, vc = rnd(T, nh * hd), rnd(T, hd), rnd(T, hd)
    qh = oracle.norm_rope(q, nh, hd, pos0=ctx)
    kcache = rnd(nkv, ctx, hd)
    vcache = rnd(nkv, ctx, hd)
    for h in range(nh):
        kcache[0, 1] = (qh[0, h] * 50.0).astype(np.float32)
        out = oracle.forward(q, kc, vc, kcache, vcache, nh, nkv, hd)
        np.testing.assert_allclose(out[0, h * hd:(h + 1) * hd], vcache[0, 1], atol=1e-12)


def test_permuting_canvas_keys_and_values_jointly():
    """No mask: permuting the canvas K/V rows together leaves every output unchanged (RoPE
    switched off through an identity cos|sin table so rows carry no position)."""
    T, ctx, nh, nkv, hd = 7, 4, 4, 2, 16
    q, kc, vc = rnd(T, nh * hd), rnd(T, nkv * hd), rnd(T, nkv * hd)
    kca, vca = rnd(nkv, ctx, hd), rnd(nkv, ctx, hd)
    ident = np.concatenate([np.ones((T, hd)), np.zeros((T, hd))], 1).astype(np.float32)
    perm = RNG.permutation(T)
    a = oracle.forward(q, kc, vc, kca, vca, nh, nkv, hd, cos_sin=ident)
    b = oracle.forward(q, kc[perm], vc[perm], kca, vca, nh, nkv, hd, cos_sin=ident)
    np.testing.assert_allclose(a, b, atol=1e-13)
    # and permuting the cache rows jointly
    cp = RNG.permutation(ctx)
    c = oracle.forward(q, kc, vc, kca[:, cp], vca[:, cp], nh, nkv, hd, cos_sin=ident)
    np.testing.assert_allclose(a, c, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads():
    """nh/nkv = G consecutive q heads share kv head h // G: the result equals MHA (nkv = nh) with
    every kv head repeated G times.  Catches: h % nkv instead of h // G."""
    T, ctx, nh, nkv, hd = 5, 6, 6, 2, 8
    G = nh // nkv
    q, kc, vc = rnd(T, nh * hd), rnd(T, nkv * hd), rnd(T, nkv * hd)
    kca, vca = rnd(nkv, ctx, hd), rnd(nkv, ctx, hd)
    a = oracle.forward(q, kc, vc, kca, vca, nh, nkv, hd)
    rep = lambda x: np.repeat(x.reshape(T, nkv, hd), G, axis=1).reshape(T, nh * hd)
    b = oracle.forward(q, rep(kc), rep(vc), np.repeat(kca, G, 0), np.repeat(vca, G, 0), nh, nh,
                       hd)
    np.testing.assert_allclose(a, b, atol=1e-13)


def test_shifting_all_positions_changes_nothing_without_cache():
    """ctx = 0: every key and query is roped, so only position differences matter and a shift
    of pos0 leaves the output unchanged (the relative-position property end to end)."""
    T, nh, nkv, hd = 6, 2, 1, 32
    q, kc, vc = rnd(T, nh * hd), rnd(T, nkv * hd), rnd(T, nkv * hd)
    a = oracle.forward(q, kc, vc, None, None, nh, nkv, hd, pos0=0)
    b = oracle.forward(q, kc, vc, None, None, nh, nkv, hd, pos0=5000)
    np.testing.assert_allclose(a, b, atol=1e-10)


def test_ctx_zero_is_canvas_self_attention():
    """ctx = 0 is plain bidirectional self-attention over the T canvas rows (brute force)."""
    T, nh, nkv, hd = 9, 4, 4, 16
    q, kc, vc = rnd(T, nh * hd), rnd(T, nkv * hd), rnd(T, nkv * hd)
    a = oracle.forward(q, kc, vc, None, None, nh, nkv, hd)
    b = brute_force(q, kc, vc, None, None, nh, nkv, hd, None, None, 1e-6, 10000.0, 0)
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_rows_subset_equals_full():
    """Computing a subset of query rows gives the same numbers as the full run."""
    T, ctx, nh, nkv, hd = 8, 4, 2, 1, 8
    q, kc, vc = rnd(T, nh * hd), rnd(T, nkv * hd), rnd(T, nkv * hd)
    kca, vca = rnd(nkv, ctx, hd), rnd(nkv, ctx, hd)
    a = oracle.forward(q, kc, vc, kca, vca, nh, nkv, hd)
    b = oracle.forward(q, kc, vc, kca, vca, nh, nkv, hd, rows=(3, 6))
    np.testing.assert_array_equal(a[3:6], b[3:6])
    assert np.abs(b[:3]).max() == 0 and np.abs(b[6:]).max() == 0


def test_worked_example_by_hand():
    """A case small enough to do by hand: hd = 2, T = 1, ctx = 1, pos0 = 0 (no rotation),
    eps = 0.  q = (3, 4) -> q-hat = (3, 4) / sqrt(12.5); canvas k = (1, 1) -> (1, 1);
    canvas v = (0, 2) -> (0, sqrt 2); cache key (0, 0) (score 0), cache value (1, 0).
    The canvas score is 7 / sqrt(12.5), so out = (w0 * 1, w1 * sqrt 2) with
    w1 = 1 / (1 + e^-s) and w0 = 1 - w1."""
    q = np.array([[3.0, 4.0]], np.float32)
    k = np.array([[1.0, 1.0]], np.float32)
    v = np.array([[0.0, 2.0]], np.float32)
    kca = np.zeros((1, 1, 2), np.float32)
    vca = np.array([[[1.0, 0.0]]], np.float32)
    out = oracle.forward(q, k, v, kca, vca, 1, 1, 2, eps=0.0, pos0=0)
    s = 7.0 / math.sqrt(12.5)
    w1 = 1.0 / (1.0 + math.exp(-s))
    np.testing.assert_allclose(out[0], [1.0 - w1, w1 * math.sqrt(2.0)], rtol=1e-14)


# ---------------------------------------------------------------- input RMSNorm + projections
# (canvas_forward, attention branch: rms!(cur, ln_in) then gemm! y = x W^T on GLin weights)

def test_projection_hand_example():
    """x = [3, 4], no weight, eps = 0: mean x^2 = 12.5, so xhat = x / sqrt(12.5); with W = [[1, 2]]
    the projection is (3 + 8) / sqrt(12.5).  Catches: x W instead of x W^T, a missing norm."""
    x = np.array([[3.0, 4.0]], dtype=np.float32)
    q, k, v = oracle.project_qkv(x, None, np.array([[1.0, 2.0]], np.float32),
                                 np.array([[0.0, 1.0], [1.0, 0.0]], np.float32), eps=0.0)
    s = math.sqrt(12.5)
    assert q.shape == (1, 1) and abs(q[0, 0] - 11.0 / s) < 1e-14
    np.testing.assert_allclose(k[0], [4.0 / s, 3.0 / s], rtol=1e-14)
    np.testing.assert_array_equal(v, k)     # no value projection: v is the raw k projection


def test_projection_rows_of_w_select_columns():
    """A W row with a single 1 at column i returns column i of the normed input, so each output
    column j is row j of W dotted with the row of x: W is [n, k], applied transposed.
    Catches: transposed W, a row/column index swap, an output column offset."""
    h, n = 12, 5
    x = rnd(4, h)
    cols = [7, 0, 11, 3, 3]
    W = np.zeros((n, h), np.float32)
    for j, i in enumerate(cols):
        W[j, i] = 1.0
    lnw = 1.0 + 0.2 * rnd(h)
    q, _, _ = oracle.project_qkv(x, lnw, W, W, eps=1e-6)
    xd = x.astype(np.float64)
    m = (xd ** 2).mean(axis=1, keepdims=True)
    xhat = xd / np.sqrt(m + 1e-6) * lnw.astype(np.float64)
    np.testing.assert_allclose(q, xhat[:, cols], rtol=1e-14)


def test_input_norm_weight_scales_linearly_and_norm_is_scale_free():
    """RMSNorm removes any positive scale of x; the ln_in weight scales every projection
    linearly.  Catches: eps applied wrongly at scale, weight applied before the mean."""
    h, n = 16, 6
    x, W, lnw = rnd(3, h), rnd(n, h), 1.0 + 0.1 * rnd(h)
    q1, _, _ = oracle.project_qkv(x, lnw, W, W, eps=0.0)
    q2, _, _ = oracle.project_qkv((8.0 * x).astype(np.float32), lnw, W, W, eps=0.0)
    q3, _, _ = oracle.project_qkv(x, (2.0 * lnw).astype(np.float32), W, W, eps=0.0)
    np.testing.assert_allclose(q2, q1, rtol=1e-12)
    np.testing.assert_allclose(q3, 2.0 * q1, rtol=1e-12)


def test_projection_brute_force_with_fsum():
    """An independent restatement with Python loops and math.fsum on a small case."""
    h, n, rows = 10, 7, 3
    x, W, lnw = rnd(rows, h), rnd(n, h), 1.0 + 0.1 * rnd(h)
    eps = 1e-3
    q, _, _ = oracle.project_qkv(x, lnw, W, W, eps=eps)
    for r in range(rows):
        ms = math.fsum(float(v) * float(v) for v in x[r]) / h
        inv = 1.0 / math.sqrt(ms + eps)
        xr = [float(x[r, i]) * inv * float(lnw[i]) for i in range(h)]
        for j in range(n):
            ref = math.fsum(xr[i] * float(W[j, i]) for i in range(h))
            assert abs(q[r, j] - ref) <= 1e-12 * (1.0 + abs(ref))


# ---------------------------------------------------------------- o_proj + post-attention norm + residual
# (canvas_forward: gemm!(sb, o) then rms!(nb, ln_post_attn) then add_scale!(cur, sb, 1.0))

def test_oproj_residual_hand_example():
    """attn = [1, 2], Wo = [[1, 0], [0, 1], [1, 1]]: y = [1, 2, 3], mean y^2 = 14/3, so the update
    is y / sqrt(14/3) (eps = 0, no weight) added to the residual.  Catches: the norm over the
    input instead of the projection, a missing residual, transposed Wo."""
    attn = np.array([[1.0, 2.0]], np.float32)
    wo = np.array([[1, 0], [0, 1], [1, 1]], np.float32)
    resid = np.array([[10.0, 20.0, 30.0]], np.float32)
    out = oracle.oproj_residual(attn, wo, None, resid, eps=0.0)
    s = math.sqrt(14.0 / 3.0)
    np.testing.assert_allclose(out[0], [10 + 1 / s, 20 + 2 / s, 30 + 3 / s], rtol=1e-14)


def test_oproj_residual_is_scale_free_in_the_attention_output():
    """The post-attention RMSNorm removes any positive scale of the projected vector (eps = 0), and
    the weight multiplies the normalised update.  Catches: weight inside the mean, no norm."""
    k, h = 12, 20
    attn, wo, resid, w = rnd(3, k), rnd(h, k), rnd(3, h), 1.0 + 0.2 * rnd(h)
    o1 = oracle.oproj_residual(attn, wo, w, resid, eps=0.0)
    o2 = oracle.oproj_residual((8.0 * attn).astype(np.float32), wo, w, resid, eps=0.0)
    np.testing.assert_allclose(o2, o1, rtol=1e-12)
    upd = o1 - resid.astype(np.float64)
    np.testing.assert_allclose(((upd / w.astype(np.float64)) ** 2).mean(axis=1), 1.0, rtol=1e-12)


def test_oproj_residual_brute_force_with_fsum():
    k, h, rows = 9, 11, 2
    attn, wo, resid, w = rnd(rows, k), rnd(h, k), rnd(rows, h), 1.0 + 0.1 * rnd(h)
    eps = 1e-2
    out = oracle.oproj_residual(attn, wo, w, resid, eps=eps)
    for r in range(rows):
        y = [math.fsum(float(attn[r, i]) * float(wo[j, i]) for i in range(k)) for j in range(h)]
        inv = 1.0 / math.sqrt(math.fsum(v * v for v in y) / h + eps)
        for j in range(h):
            ref = float(resid[r, j]) + y[j] * inv * float(w[j])
            assert abs(out[r, j] - ref) <= 1e-12 * (1.0 + abs(ref))
