"""Pins of the oracle's training losses (Eqs 9-12 of "DSpark -- paper verification", section 1)
and their gradients.

* The position weights w_k = exp(-(k-1)/gamma) against the values the same page prints in its
  delta table (D2), stored in tests/golden/loss_constants.txt: [1, .78, .61, .47] at gamma = 4
  (exactly, to the printed two decimals) and [1, .87, .75, .65, .57, .49, .43] at gamma = 7 (to
  0.01: two of those entries, .57 and .43, do not round from the formula the page states, which
  gives .565 and .424).  They are read off dL/d(confidence logit) = a_conf w_k (c - c*) at
  c = 1/2, c* = 1.
* Every analytic gradient against central differences of the oracle's own loss.  c* is a label
  (no gradient through it), so the logit gradient is checked with a_conf = 0; the confidence
  logits do not move c*, so their gradient is checked with every weighting.
* L1 on probabilities, not logits (D6): logits shifted by a constant give L_tv = 0 and c* = 1.
* L_ce gathers log p at the label (D5): a uniform draft gives ln V per position, a one-hot draft 0.
* The alpha defaults (D4, in the same golden file): L = 0.1 L_ce + 0.9 L_tv + 1.0 L_conf.
* Disjoint supports give ||p - q||_1 = 2, so c* = 0 and L_conf = -sum w ln(1 - c).
"""
import os

import numpy as np
import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "loss_constants.txt")


def printed(name):
    """The numbers on the line `name` of the golden file of printed loss constants."""
    for line in open(GOLDEN):
        f = line.split()
        if f and f[0] == name:
            return [float(x) for x in f[1:]]
    raise KeyError(name)


def inputs(B, G, V, seed, noise=1.0):
    rng = np.random.default_rng(seed)
    zd = rng.normal(0, 1.5, (B, G, V)).astype(np.float32)
    zt = (zd + rng.normal(0, noise, (B, G, V))).astype(np.float32)
    lab = rng.integers(0, V, (B, G)).astype(np.int32)
    cf = rng.normal(0, 1, (B, G)).astype(np.float32)
    return zd, zt, lab, cf


@pytest.mark.parametrize("G,tol", [(4, 1e-12), (7, 0.0100001)])
def test_position_weights_match_the_printed_values(G, tol):
    V = 5
    zd = np.zeros((1, G, V), np.float32)
    r = oracle.draft_loss(T=1.0, draft_logits=zd, target_logits=zd, labels=np.zeros((1, G), np.int32),
                          conf_logits=np.zeros((1, G), np.float32), alpha=(0.1, 0.9, 1.0))
    w = -2.0 * r.grad_conf[0]  # a_conf = 1, c = 1/2, c* = 1
    assert np.all(np.abs(np.round(w, 2) - printed(f"weights_gamma{G}")) <= tol)
    assert abs(w[0] - 1.0) < 1e-15 and abs(w[-1] - np.exp(-(G - 1) / G)) < 1e-15


def loss_of(zd, zt, lab, cf, T, alpha):
    return oracle.draft_loss(T=T, draft_logits=zd, target_logits=zt, labels=lab, conf_logits=cf,
                             alpha=alpha).loss


@pytest.mark.parametrize("T,alpha", [(1.0, (0.1, 0.9, 1.0)), (0.7, (1.0, 0.0, 0.0)),
                                     (1.3, (0.0, 1.0, 0.0)), (1.0, (0.0, 0.0, 1.0)),
                                     (0.9, (0.3, 0.6, 0.0))])
def test_gradients_match_finite_differences(T, alpha):
    B, G, V = 2, 3, 7
    zd, zt, lab, cf = inputs(B, G, V, seed=11)
    r = oracle.draft_loss(T=T, draft_logits=zd, target_logits=zt, labels=lab, conf_logits=cf,
                          alpha=alpha)
    # finite differences in float64 copies (the oracle reads float32: use steps representable
    # in float32 around values of order 1)
    h = 2.0 ** -10
    rng = np.random.default_rng(3)
    for _ in range(25 if alpha[2] == 0 else 0):  # c* is a label: the logit gradient omits it
        b, j, v = rng.integers(B), rng.integers(G), rng.integers(V)
        up, dn = zd.copy(), zd.copy()
        up[b, j, v] += h
        dn[b, j, v] -= h
        fd = (loss_of(up, zt, lab, cf, T, alpha)[b] - loss_of(dn, zt, lab, cf, T, alpha)[b]) / (2 * h)
        assert abs(fd - r.grad_logits[b, j, v]) < 2e-4, (b, j, v, fd, r.grad_logits[b, j, v])
    for b in range(B):
        for j in range(G):
            up, dn = cf.copy(), cf.copy()
            up[b, j] += h
            dn[b, j] -= h
            fd = (loss_of(zd, zt, lab, up, T, alpha)[b] - loss_of(zd, zt, lab, dn, T, alpha)[b]) / (2 * h)
            assert abs(fd - r.grad_conf[b, j]) < 2e-5


def test_l1_is_on_probabilities_not_logits():
    B, G, V = 1, 4, 9
    zd, _, lab, cf = inputs(B, G, V, seed=5)
    zt = zd + np.float32(3.0)  # the same distributions, different logits
    r = oracle.draft_loss(T=1.0, draft_logits=zd, target_logits=zt, labels=lab, conf_logits=cf)
    assert abs(r.parts[0, 1]) < 1e-6
    # c* = 1: L_conf = -sum w ln c
    w = np.exp(-np.arange(G) / G)
    c = 1 / (1 + np.exp(-cf[0].astype(np.float64)))
    assert abs(r.parts[0, 2] - (-(w * np.log(c)).sum())) < 1e-6


def test_cross_entropy_gathers_at_the_label():
    G, V = 3, 10
    w = np.exp(-np.arange(G) / G)
    uni = np.zeros((1, G, V), np.float32)
    lab = np.array([[2, 7, 0]], np.int32)
    r = oracle.draft_loss(T=1.0, draft_logits=uni, target_logits=uni, labels=lab,
                          conf_logits=np.zeros((1, G), np.float32))
    assert abs(r.parts[0, 0] - np.log(V) * w.sum()) < 1e-12
    onehot = np.full((1, G, V), -1e4, np.float32)
    for j, x in enumerate(lab[0]):
        onehot[0, j, x] = 0.0
    r = oracle.draft_loss(T=1.0, draft_logits=onehot, target_logits=onehot, labels=lab,
                          conf_logits=np.zeros((1, G), np.float32))
    assert abs(r.parts[0, 0]) < 1e-12


def test_alpha_defaults_combine_the_parts():
    zd, zt, lab, cf = inputs(3, 7, 50, seed=8)
    r = oracle.draft_loss(T=1.0, draft_logits=zd, target_logits=zt, labels=lab, conf_logits=cf)
    assert np.allclose(r.loss, r.parts @ np.array(printed("alpha")), rtol=0, atol=1e-12)


def test_disjoint_supports():
    G, V = 2, 4
    big = -1e4
    zd = np.array([[[0, 0, big, big]] * G], np.float32)
    zt = np.array([[[big, big, 0, 0]] * G], np.float32)
    cf = np.array([[0.3, -0.8]], np.float32)
    r = oracle.draft_loss(T=1.0, draft_logits=zd, target_logits=zt, labels=np.zeros((1, G), np.int32),
                          conf_logits=cf)
    w = np.exp(-np.arange(G) / G)
    assert abs(r.parts[0, 1] - 2 * w.sum()) < 1e-12        # ||p - q||_1 = 2 at every position
    c = 1 / (1 + np.exp(-cf[0].astype(np.float64)))
    assert abs(r.parts[0, 2] - (-(w * np.log(1 - c)).sum())) < 1e-9   # c* = 0
    assert np.allclose(r.grad_conf[0], w * c)                         # a_conf w (c - 0)


def test_invalid_label():
    zd, zt, lab, cf = inputs(2, 2, 6, seed=1)
    lab[1, 1] = 6
    r = oracle.draft_loss(T=1.0, draft_logits=zd, target_logits=zt, labels=lab, conf_logits=cf)
    assert r.status == 1 and np.isnan(r.loss[1]) and not np.isnan(r.loss[0])


def test_confidence_label_one_hot_against_uniform():
    # Eq 8 inside L_conf at a value strictly between 0 and 1: a one-hot draft against a uniform
    # target has c* = 1/V ("DSpark -- paper verification", delta table D7), so with the
    # confidence logit l (c = sigmoid(l) != 1/2):
    #   L_conf = -w [ (1/V) ln c + (1 - 1/V) ln(1 - c) ],  dL/dl = a_conf w (c - 1/V)
    G, V = 3, 8
    big = -1e4
    zd = np.full((1, G, V), big, np.float32)
    zd[0, :, 5] = 0.0
    zt = np.zeros((1, G, V), np.float32)
    cf = np.array([[1.0, -0.5, 2.0]], np.float32)
    r = oracle.draft_loss(T=1.0, draft_logits=zd, target_logits=zt, labels=np.zeros((1, G), np.int32),
                          conf_logits=cf, alpha=(0.0, 0.0, 1.0))
    w = np.exp(-np.arange(G) / G)
    c = 1 / (1 + np.exp(-cf[0].astype(np.float64)))
    cs = 1.0 / V
    want = -(w * (cs * np.log(c) + (1 - cs) * np.log(1 - c))).sum()
    assert abs(r.parts[0, 2] - want) < 1e-9
    assert np.allclose(r.grad_conf[0], w * (c - cs), rtol=0, atol=1e-12)
