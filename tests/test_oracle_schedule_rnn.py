"""Pins for the oracle's prefix scheduler and RNN head.

Scheduler ("DSpark: 既要猜得连贯..." design section; "Phase-Conditioned Speculative Decoding"
section 3, Theta = tau * SPS): brute force over every legal choice of verify lengths on small
batches, the constant-capacity and collapsing-capacity limits, and the expected accepted
length tau(a, gamma) = (1 - a^(gamma+1)) / (1 - a) of i.i.d. acceptance (same page, section 6).

RNN head (Eq 6, "DSpark -- paper verification" section 1 and delta table D8): special weights
that reduce the recurrence to closed forms -- zero projection (s stays 0, no bias), an output
block reading only the embedding (a Markov head with a transformed table), a saturated-open
gate (s frozen at s_0) and a saturated-closed gate (s_k = tanh(W_c z_k), which makes B_k depend
on x_{k-2} through s_{k-1}).
"""
import itertools

import numpy as np
import pytest


def _random_S(rng, B, G):
    c = rng.uniform(0.05, 0.99, size=(B, G))
    return np.cumprod(c, axis=1).astype(np.float32)


def _brute(S, sps):
    B, G = S.shape
    best, arg = -1.0, None
    S64 = S.astype(np.float64)
    for ls in itertools.product(range(G + 1), repeat=B):
        n = sum(ls) + B
        tau = B + sum(S64[b, :l].sum() for b, l in enumerate(ls))
        th = sps[n] * tau
        if th > best + 1e-12 * abs(best):
            best, arg = th, ls
    return np.array(arg), best


@pytest.mark.parametrize("B,G", [(1, 3), (2, 3), (3, 2), (4, 3), (3, 1)])
def test_schedule_brute_force(oracle_mod, B, G):
    rng = np.random.default_rng(B * 10 + G)
    for trial in range(20):
        S = _random_S(rng, B, G)
        n = np.arange(B * (G + 1) + 1)
        sps = 1000.0 / (1.0 + n / rng.uniform(0.5, 8.0)) ** rng.uniform(0.5, 2.0)
        ln, theta, st = oracle_mod.prefix_schedule(S, sps)
        ref_l, ref_theta = _brute(S, sps)
        assert st == 0
        assert abs(theta - ref_theta) <= 1e-9 * ref_theta
        assert np.array_equal(ln, ref_l), (S, sps, ln, ref_l)


def test_schedule_limits(oracle_mod):
    rng = np.random.default_rng(3)
    B, G = 16, 7
    S = _random_S(rng, B, G)
    ln, _, _ = oracle_mod.prefix_schedule(S, np.full(B * (G + 1) + 1, 5.0))
    assert np.all(ln == G)                     # free capacity: verify every positive-S token
    sps = np.zeros(B * (G + 1) + 1)
    sps[: B + 1] = 1.0                         # capacity collapses beyond the bonus tokens
    ln, theta, _ = oracle_mod.prefix_schedule(S, sps)
    assert np.all(ln == 0) and theta == B


@pytest.mark.parametrize("a", [0.3, 0.8, 0.95])
def test_schedule_tau_closed_form(oracle_mod, a):
    B, G = 5, 7
    S = np.tile(np.cumprod(np.full(G, a)), (B, 1)).astype(np.float32)
    ln, theta, _ = oracle_mod.prefix_schedule(S, np.ones(B * (G + 1) + 1))
    assert np.all(ln == G)
    tau = (1 - a ** (G + 1)) / (1 - a)          # i.i.d. expected accepted length incl. bonus
    # S is fp32 and the sums are taken in 2^-32 fixed point
    assert abs(theta / B - tau) < G * (2e-7 + 2**-32)


def test_schedule_rejects_increasing_or_out_of_range(oracle_mod):
    S = np.array([[0.5, 0.6]], np.float32)
    assert oracle_mod.prefix_schedule(S, np.ones(4))[2] == 1
    assert oracle_mod.prefix_schedule(np.array([[1.5, 0.2]], np.float32), np.ones(4))[2] == 1


def test_schedule_prefixes_are_contiguous(oracle_mod):
    rng = np.random.default_rng(9)
    B, G = 64, 7
    S = _random_S(rng, B, G)
    S[3] = S[3, 0]          # equal values along a block: ties must break towards smaller k
    n = np.arange(B * (G + 1) + 1)
    ln, theta, _ = oracle_mod.prefix_schedule(S, 2000.0 / (1 + n / 200.0))
    # recompute Theta from the returned lengths and check it is what the scan reported
    tau = B + sum(float(S[b, :l].astype(np.float64).sum()) for b, l in enumerate(ln))
    sps = 2000.0 / (1 + (ln.sum() + B) / 200.0)
    assert abs(sps * tau - theta) < 1e-9 * theta
    assert 0 < ln.sum() < B * G


# ------------------------------------------------------------------------------ RNN head (Eq 6)

def _rnn_case(seed=0, B=2, G=4, V=24, r=3, d=4):
    rng = np.random.default_rng(seed)
    return dict(B=B, gamma=G, V=V, r=r, d=d, W1=rng.standard_normal((V, r)),
                W2=rng.standard_normal((V, r)), U=rng.standard_normal((B, G, V)),
                h=rng.standard_normal((B, G, d)), x0=rng.integers(0, V, B)), rng


def _run(oracle_mod, case, Wj, **kw):
    return oracle_mod.draft(head=1, T=1.0, seed=3, Wj=Wj, want_z=True, **case, **kw)


def test_rnn_zero_projection(oracle_mod):
    case, _ = _rnn_case(0)
    r, d = case["r"], case["d"]
    res = _run(oracle_mod, case, np.zeros((3 * r, 2 * r + d)))
    assert np.array_equal(res.z, case["U"]) and np.all(res.s_final == 0)


def test_rnn_output_block_is_markov_with_transformed_table(oracle_mod):
    case, rng = _rnn_case(1)
    r, d = case["r"], case["d"]
    Wj = np.zeros((3 * r, 2 * r + d))
    Woe = rng.standard_normal((r, r))
    Wj[2 * r:, r:2 * r] = Woe                      # output rows read only W1[x_{k-1}]
    res = _run(oracle_mod, case, Wj)
    W1t = np.tanh(case["W1"] @ Woe.T)
    mk = oracle_mod.draft(head=0, T=1.0, seed=3, want_z=True, **{**case, "W1": W1t})
    assert np.array_equal(res.tokens, mk.tokens)
    np.testing.assert_allclose(res.z, mk.z, rtol=0, atol=1e-12)


def test_rnn_open_gate_freezes_state(oracle_mod):
    case, rng = _rnn_case(2)
    r, d = case["r"], case["d"]
    case["h"][..., 0] = 1.0                        # a constant feature in h
    Wj = np.zeros((3 * r, 2 * r + d))
    Wj[:r, 2 * r] = 60.0                           # gate rows: sigmoid(60) == 1 in fp64
    Wj[r:2 * r, :] = rng.standard_normal((r, 2 * r + d))   # any candidate: must be ignored
    Wos = rng.standard_normal((r, r))
    Wj[2 * r:, :r] = Wos                           # output rows read only s_{k-1}
    s0 = rng.standard_normal((case["B"], r))
    res = _run(oracle_mod, case, Wj, s0=s0)
    assert np.array_equal(res.s_final, s0)
    for b in range(case["B"]):
        bias = case["W2"] @ np.tanh(Wos @ s0[b])
        np.testing.assert_allclose(res.z[b] - case["U"][b], np.tile(bias, (case["gamma"], 1)),
                                   rtol=0, atol=1e-12)


def test_rnn_closed_gate_uses_previous_state(oracle_mod):
    case, rng = _rnn_case(3, G=5)
    r, d = case["r"], case["d"]
    case["h"][..., 0] = 1.0
    Wj = np.zeros((3 * r, 2 * r + d))
    Wj[:r, 2 * r] = -60.0                          # gate closed: s_k = tanh(W_c z_k)
    Wce = rng.standard_normal((r, r))
    Wj[r:2 * r, r:2 * r] = Wce                     # candidate reads only W1[x_{k-1}]
    Wos = rng.standard_normal((r, r))
    Wj[2 * r:, :r] = Wos                           # output reads only s_{k-1}
    B, G = case["B"], case["gamma"]
    forced = rng.integers(0, case["V"], (B, G)).astype(np.int32)
    res = _run(oracle_mod, case, Wj, forced=forced)
    for b in range(B):
        cond = np.concatenate([[case["x0"][b]], forced[b, :-1]])   # x_{k-1} for k = 1..G
        s_prev = np.zeros(r)
        for k in range(G):
            bias = case["W2"] @ np.tanh(Wos @ s_prev)              # B_k from s_{k-1}
            np.testing.assert_allclose(res.z[b, k] - case["U"][b, k], bias, rtol=0, atol=1e-12)
            s_prev = np.tanh(Wce @ case["W1"][cond[k]])
        np.testing.assert_allclose(res.s_final[b], s_prev, rtol=0, atol=1e-14)
