"""Pins of the oracle's speculative verification (the accept/reject rule).

"Phase-Conditioned Speculative Decoding" section 3 identifies Eq 8's c* = 1 - TV(p, q) with
the single-step acceptance probability of the standard accept/reject rule (Leviathan, Kalman,
Matias, ICML 2023), and its prefix survival S_k = prod_{i<=k} c_i with the chance that the
first k positions survive.  "DSpark：既要猜得连贯…" ("Why DSpark?") describes the round: the
matching prefix is accepted, the round stops at the first rejection, and the final
distribution stays the target's.  These tests check the oracle against those facts, using
draft tokens drawn by numpy (independent of the oracle's generator):

* the output token is distributed exactly as q (the rule's defining property);
* the acceptance frequency is sum_v min(p_v, q_v) = c*;
* the exact joint law of (n, tokens) at gamma = 2, enumerated by brute force;
* P(n >= k) = prod_{j<k} c*_j for position-wise independent blocks;
* special cases: p = q accepts everything, disjoint supports reject at once, a point-mass
  draft is accepted with probability q(x).
"""
import itertools

import numpy as np
import pytest
from scipy import stats

from oracle import oracle


def softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def run(zd_rows, zt_rows, N, seed, rng, T=1.0):
    """N requests sharing per-position logits; draft tokens drawn from p by numpy."""
    gamma, V = zd_rows.shape
    zd = np.ascontiguousarray(np.broadcast_to(zd_rows, (N, gamma, V)), dtype=np.float32)
    zt = np.ascontiguousarray(np.broadcast_to(zt_rows, (N, gamma + 1, V)), dtype=np.float32)
    x = np.stack([rng.choice(V, size=N, p=softmax(zd_rows[j].astype(np.float64) / T))
                  for j in range(gamma)], axis=1).astype(np.int32)
    r = oracle.verify(gamma=gamma, T=T, seed=seed, draft_logits=zd, target_logits=zt,
                      draft_tokens=x)
    assert r.status == 0
    return r, x


def chi2_ok(counts, probs, min_p=1e-3):
    probs = np.asarray(probs, dtype=np.float64)
    keep = probs > 0
    assert counts[~keep].sum() == 0, "an outcome of probability 0 occurred"
    n = counts.sum()
    exp = n * probs[keep]
    chi2 = ((counts[keep] - exp) ** 2 / exp).sum()
    pval = stats.chi2.sf(chi2, keep.sum() - 1)
    sigma = np.sqrt(n * probs[keep] * (1 - probs[keep]))
    assert np.all(np.abs(counts[keep] - exp) < 5 * sigma + 1), (counts, exp)
    assert pval > min_p, pval


def test_output_token_is_distributed_as_target():
    rng = np.random.default_rng(1)
    V = 6
    zd = np.array([[1.2, 0.3, -0.5, 2.0, 0.0, -1.0]], dtype=np.float32)
    zt = np.array([[0.1, 1.5, 0.7, -0.3, 1.0, 0.2], [0.0] * V], dtype=np.float32)
    N = 200_000
    r, x = run(zd, zt, N, seed=11, rng=rng)
    p, q = softmax(zd[0].astype(np.float64)), softmax(zt[0].astype(np.float64))
    chi2_ok(np.bincount(r.tokens[:, 0], minlength=V), q)
    acc = (r.n_accepted == 1).mean()
    cstar = np.minimum(p, q).sum()
    assert abs(acc - cstar) < 5 * np.sqrt(cstar * (1 - cstar) / N), (acc, cstar)
    # accepted tokens are the drafted ones; a rejection replaces the token
    assert np.all(r.tokens[r.n_accepted == 1, 0] == x[r.n_accepted == 1, 0])


def test_temperature_scales_both_distributions():
    rng = np.random.default_rng(2)
    zd = np.array([[2.0, 0.0, -1.0, 1.0]], dtype=np.float32)
    zt = np.array([[0.0, 1.0, 1.5, -2.0], [0.0] * 4], dtype=np.float32)
    T = 0.7
    r, _ = run(zd, zt, 150_000, seed=5, rng=rng, T=T)
    q = softmax(zt[0].astype(np.float64) / T)
    chi2_ok(np.bincount(r.tokens[:, 0], minlength=4), q)


def exact_joint(P, Q):
    """Exact law of (n, output tokens) for gamma = 2 with position-wise fixed p_j, q_j."""
    V = P.shape[1]
    alpha = [np.minimum(1.0, Q[j] / P[j]) for j in range(2)]
    resid = []
    for j in range(2):
        w = np.maximum(0.0, Q[j] - P[j])
        resid.append(w / w.sum() if w.sum() > 0 else Q[j])
    law = {}
    for y in range(V):  # rejected at position 0
        law[(0, y)] = sum(P[0][x] * (1 - alpha[0][x]) for x in range(V)) * resid[0][y]
    for x1, y in itertools.product(range(V), range(V)):  # accepted x1, rejected at 1
        law[(1, x1, y)] = (P[0][x1] * alpha[0][x1]
                           * sum(P[1][x] * (1 - alpha[1][x]) for x in range(V)) * resid[1][y])
    for x1, x2, y in itertools.product(range(V), range(V), range(V)):  # both accepted + bonus
        law[(2, x1, x2, y)] = P[0][x1] * alpha[0][x1] * P[1][x2] * alpha[1][x2] * Q[2][y]
    return law


def test_joint_law_brute_force_gamma2():
    rng = np.random.default_rng(3)
    V = 4
    zd = np.array([[1.0, 0.2, -0.4, 0.5], [-0.3, 0.9, 0.1, 0.0]], dtype=np.float32)
    zt = np.array([[0.4, 0.8, -0.2, 0.1], [0.6, 0.0, 0.7, -0.5], [0.3, -0.2, 0.9, 0.0]],
                  dtype=np.float32)
    P = np.array([softmax(zd[j].astype(np.float64)) for j in range(2)])
    Q = np.array([softmax(zt[j].astype(np.float64)) for j in range(3)])
    law = exact_joint(P, Q)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    N = 400_000
    r, _ = run(zd, zt, N, seed=21, rng=rng)
    keys = list(law)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys), dtype=np.int64)
    for n, row in zip(r.n_accepted, r.tokens):
        counts[index[(int(n),) + tuple(int(t) for t in row[:n + 1])]] += 1
    chi2_ok(counts, np.array([law[k] for k in keys]))


def test_prefix_survival_is_product_of_cstar():
    rng = np.random.default_rng(4)
    gamma, V = 3, 5
    zd = rng.normal(0, 1.0, (gamma, V)).astype(np.float32)
    zt = np.concatenate([zd + rng.normal(0, 0.8, (gamma, V)), rng.normal(0, 1, (1, V))]).astype(np.float32)
    N = 200_000
    r, _ = run(zd, zt, N, seed=9, rng=rng)
    cstar = [np.minimum(softmax(zd[j].astype(np.float64)), softmax(zt[j].astype(np.float64))).sum()
             for j in range(gamma)]
    for k in range(1, gamma + 1):
        S = float(np.prod(cstar[:k]))
        f = (r.n_accepted >= k).mean()
        assert abs(f - S) < 5 * np.sqrt(S * (1 - S) / N), (k, f, S)
    # the margins are tested exactly where the rule looked: positions < n accepted, n rejected
    for n, m in zip(r.n_accepted[:2000], r.margin[:2000]):
        assert np.all(m[:n] > 0) and (n == gamma or m[n] <= 0) and np.all(np.isnan(m[n + 1:]))


def test_identical_distributions_accept_everything():
    rng = np.random.default_rng(5)
    V = 5
    zd = rng.normal(0, 1, (3, V)).astype(np.float32)
    bonus = np.array([[0.5, -1.0, 0.2, 1.1, 0.0]], dtype=np.float32)
    zt = np.concatenate([zd, bonus])
    r, x = run(zd, zt, 60_000, seed=13, rng=rng)
    assert np.all(r.n_accepted == 3)
    assert np.array_equal(r.tokens[:, :3], x)
    chi2_ok(np.bincount(r.tokens[:, 3], minlength=V), softmax(bonus[0].astype(np.float64)))


def test_disjoint_supports_reject_at_once():
    rng = np.random.default_rng(6)
    big = -1.0e4
    zd = np.array([[0.0, 0.3, big, big], [0.0, 0.0, 0.0, 0.0]], dtype=np.float32)
    zt = np.array([[big, big, 0.4, -0.2], [0.0] * 4, [0.0] * 4], dtype=np.float32)
    r, _ = run(zd, zt, 60_000, seed=17, rng=rng)
    assert np.all(r.n_accepted == 0)
    assert np.all(r.tokens[:, 1:] == -1)
    chi2_ok(np.bincount(r.tokens[:, 0], minlength=4), softmax(zt[0].astype(np.float64)))


def test_point_mass_draft_accepts_with_target_mass():
    # "Phase-Conditioned Speculative Decoding" Prop 1: a deterministic drafter's acceptance
    # rate is the target's mass on the drafted token
    rng = np.random.default_rng(7)
    zd = np.array([[-1.0e4, -1.0e4, 0.0, -1.0e4]], dtype=np.float32)
    zt = np.array([[0.2, -0.5, 0.9, 0.1], [0.0] * 4], dtype=np.float32)
    N = 200_000
    r, x = run(zd, zt, N, seed=23, rng=rng)
    assert np.all(x == 2)
    qx = softmax(zt[0].astype(np.float64))[2]
    f = (r.n_accepted == 1).mean()
    assert abs(f - qx) < 5 * np.sqrt(qx * (1 - qx) / N)


def test_invalid_draft_token_is_reported():
    zd = np.zeros((3, 2, 8), dtype=np.float32)
    zt = np.zeros((3, 3, 8), dtype=np.float32)
    x = np.array([[0, 1], [2, 8], [3, 4]], dtype=np.int32)
    r = oracle.verify(gamma=2, T=1.0, seed=1, draft_logits=zd, target_logits=zt, draft_tokens=x)
    assert r.status == 1
    assert r.n_accepted[1] == -1 and np.all(r.tokens[1] == -1)
    assert r.n_accepted[0] == 2 and r.n_accepted[2] == 2  # p = q: everything accepted


@pytest.mark.parametrize("seed", [0, 1])
def test_noise_streams_are_distinct(seed):
    # acceptance uniforms and correction noise come from separate Philox streams: with p = q
    # (everything accepted) the bonus still varies with the request index
    zd = np.zeros((64, 1, 16), dtype=np.float32)
    zt = np.zeros((64, 2, 16), dtype=np.float32)
    x = np.zeros((64, 1), dtype=np.int32)
    r = oracle.verify(gamma=1, T=1.0, seed=seed, draft_logits=zd, target_logits=zt, draft_tokens=x)
    assert np.all(r.n_accepted == 1)
    assert len(set(r.tokens[:, 1].tolist())) > 8
