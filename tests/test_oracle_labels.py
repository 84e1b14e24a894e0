"""Pins for the oracle's Eq 7 (confidence), prefix survival and Eq 8 (soft acceptance label).

Eq 8 is pinned by closed forms printed on the pages: identical distributions give c* = 1 and a
one-hot draft against a uniform target gives 1/V ("DSpark -- paper verification", delta table D7);
a point-mass draft gives c* = p^t(x) and a draft supported inside E gives c* <= p^t(E)
("Phase-Conditioned Speculative Decoding", Propositions 1 and 3); and c* = 1 - TV equals the
acceptance probability of the standard speculative accept/reject rule (same page, section 3),
checked by Monte Carlo.  Eq 7 is pinned by w = 0 (c = 1/2, S_k = 2^-k exactly), by separating
the two halves of w (the d + r width check and the x_{k-1} index check recommended in the first
page's section 7).
"""
import numpy as np
import pytest
from scipy.special import expit, softmax


def test_tv_identical_is_one(oracle_mod):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 300)).astype(np.float32)
    cstar, l1 = oracle_mod.tv_label(x, x, T=0.8)
    assert np.all(cstar == 1.0) and np.all(l1 < 1e-15)


@pytest.mark.parametrize("V", [2, 7, 1000])
def test_tv_one_hot_vs_uniform(oracle_mod, V):
    d = np.zeros((1, V), np.float32)
    d[0, V // 3] = 2000.0      # exp(-2000) underflows: an exact one-hot distribution
    cstar, l1 = oracle_mod.tv_label(d, np.zeros((1, V), np.float32))
    tol = 4 * V * np.finfo(np.float64).eps       # a few ulps per summed term
    assert abs(cstar[0] - 1.0 / V) < tol
    assert abs(l1[0] - 2.0 * (1.0 - 1.0 / V)) < tol


def test_tv_point_mass_is_target_mass(oracle_mod):
    rng = np.random.default_rng(1)
    V = 257
    t = rng.standard_normal((6, V)).astype(np.float32) * 2
    d = np.zeros_like(t)
    xs = rng.integers(0, V, 6)
    d[np.arange(6), xs] = 3000.0
    cstar, _ = oracle_mod.tv_label(d, t)
    q = softmax(t.astype(np.float64), axis=1)
    np.testing.assert_allclose(cstar, q[np.arange(6), xs], rtol=0, atol=1e-14)


def test_tv_disjoint_supports_is_zero(oracle_mod):
    V = 64
    d = np.full((1, V), -3000.0, np.float32)
    t = np.full((1, V), -3000.0, np.float32)
    d[0, :10] = 0.0
    t[0, 10:] = 0.0
    cstar, l1 = oracle_mod.tv_label(d, t)
    assert cstar[0] == 0.0 and abs(l1[0] - 2.0) < 1e-14


def test_tv_equals_sum_of_minima_and_support_bound(oracle_mod):
    rng = np.random.default_rng(2)
    V, T = 500, 1.7
    d = rng.standard_normal((8, V)).astype(np.float32) * 3
    t = (d + rng.standard_normal((8, V)).astype(np.float32)).astype(np.float32)
    cstar, l1 = oracle_mod.tv_label(d, t, T=T)
    p = softmax(d.astype(np.float64) / T, axis=1)
    q = softmax(t.astype(np.float64) / T, axis=1)
    np.testing.assert_allclose(cstar, np.minimum(p, q).sum(1), rtol=0, atol=1e-12)
    # Proposition 3: draft supported inside E  =>  c* <= target mass on E
    E = np.arange(V) < 40
    dE = np.where(E, d, -3000.0).astype(np.float32)
    cE, _ = oracle_mod.tv_label(dE, t, T=T)
    assert np.all(cE <= q[:, E].sum(1) + 1e-14)


def test_tv_is_accept_probability_monte_carlo(oracle_mod):
    """c* = sum_v p_v min(1, q_v / p_v): simulate the speculative accept/reject rule."""
    rng = np.random.default_rng(3)
    V, n = 8, 1_000_000
    d = rng.standard_normal((1, V)).astype(np.float32) * 1.5
    t = rng.standard_normal((1, V)).astype(np.float32) * 1.5
    cstar, _ = oracle_mod.tv_label(d, t)
    p = softmax(d[0].astype(np.float64))
    q = softmax(t[0].astype(np.float64))
    x = rng.choice(V, size=n, p=p)
    accept = rng.random(n) < np.minimum(1.0, q[x] / p[x])
    sigma = np.sqrt(cstar[0] * (1 - cstar[0]) / n)
    assert abs(accept.mean() - cstar[0]) < 5 * sigma


def _draft_conf(oracle_mod, **kw):
    return oracle_mod.draft(head=0, T=1.0, seed=5, **kw)


def test_confidence_zero_weight_half(oracle_mod):
    rng = np.random.default_rng(4)
    B, G, V, r, d = 3, 6, 32, 4, 5
    res = _draft_conf(oracle_mod, B=B, gamma=G, V=V, r=r, d=d, W1=rng.standard_normal((V, r)),
                      W2=rng.standard_normal((V, r)), U=rng.standard_normal((B, G, V)),
                      x0=np.array([0, 1, 2]), h=rng.standard_normal((B, G, d)),
                      w=np.zeros(d + r))
    assert np.all(res.c == 0.5)
    assert np.all(res.S == 0.5 ** np.arange(1, G + 1))


def test_confidence_halves_and_index(oracle_mod):
    """w[0:d] multiplies h_k, w[d:d+r] multiplies W1[x_{k-1}] (width d + r; x_0 is the anchor).
    With r = 1 and W1[x] = x/V the embedding half reveals which token conditioned step k."""
    rng = np.random.default_rng(5)
    B, G, V, d = 2, 5, 16, 3
    W1 = (np.arange(V, dtype=np.float64) / V)[:, None]
    W2 = rng.standard_normal((V, 1))
    U = rng.standard_normal((B, G, V))
    h = rng.standard_normal((B, G, d))
    x0 = np.array([3, 9])
    forced = np.array([[4, 5, 6, 7, 8], [10, 11, 12, 13, 14]], dtype=np.int32)
    w_emb = np.concatenate([np.zeros(d), [2.0]])
    res = _draft_conf(oracle_mod, B=B, gamma=G, V=V, r=1, d=d, W1=W1, W2=W2, U=U, x0=x0, h=h,
                      w=w_emb, forced=forced)
    prev = np.concatenate([x0[:, None], forced[:, :-1]], axis=1)
    np.testing.assert_allclose(res.c, expit(2.0 * prev / V), rtol=0, atol=1e-15)
    w_hid = np.concatenate([np.array([0.5, -1.0, 2.0]), [0.0]])
    res = _draft_conf(oracle_mod, B=B, gamma=G, V=V, r=1, d=d, W1=W1, W2=W2, U=U, x0=x0, h=h,
                      w=w_hid, forced=forced)
    np.testing.assert_allclose(res.c, expit(h @ w_hid[:d]), rtol=0, atol=1e-15)


def test_survival_non_increasing_and_consistent(oracle_mod):
    rng = np.random.default_rng(6)
    B, G, V, r, d = 4, 7, 64, 8, 16
    kw = dict(B=B, gamma=G, V=V, r=r, d=d, W1=rng.standard_normal((V, r)),
              W2=rng.standard_normal((V, r)) * 0.3, U=rng.standard_normal((B, G, V)),
              x0=rng.integers(0, V, B), h=rng.standard_normal((B, G, d)),
              w=rng.standard_normal(d + r))
    res = _draft_conf(oracle_mod, **kw)
    assert np.all((res.c > 0) & (res.c < 1))
    assert np.all(np.diff(res.S, axis=1) <= 0) and np.all(res.S[:, 0] == res.c[:, 0])
    np.testing.assert_allclose(res.S, np.cumprod(res.c, axis=1), rtol=1e-14, atol=0)
    c2, S2, st = oracle_mod.confidence(B=B, gamma=G, V=V, r=r, d=d, W1=kw["W1"], h=kw["h"],
                                       w=kw["w"], x0=kw["x0"], tokens=res.tokens)
    assert st == 0 and np.array_equal(c2, res.c) and np.array_equal(S2, res.S)


def test_draft_labels_match_standalone_tv(oracle_mod):
    rng = np.random.default_rng(7)
    B, G, V, r = 2, 3, 100, 4
    U = rng.standard_normal((B, G, V)).astype(np.float32)
    target = (U + rng.standard_normal((B, G, V))).astype(np.float32)
    res = oracle_mod.draft(head=0, B=B, gamma=G, V=V, r=r, d=0, T=1.2, seed=1,
                           W1=rng.standard_normal((V, r)).astype(np.float32),
                           W2=rng.standard_normal((V, r)).astype(np.float32), U=U,
                           x0=np.array([1, 2]), target=target, want_z=True)
    cs, l1 = oracle_mod.tv_label(res.z.reshape(-1, V).astype(np.float32),
                                 target.reshape(-1, V), T=1.2)
    # z is rounded to fp32 for the standalone call; the label moves by far less than 1e-5
    np.testing.assert_allclose(res.cstar.ravel(), cs, rtol=0, atol=1e-5)
    np.testing.assert_allclose(res.l1.ravel(), l1, rtol=0, atol=2e-5)
