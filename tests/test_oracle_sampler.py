"""Pins for the oracle's counter-based generator, Gumbel-max sampler and Eq 4/5 logits.

Nothing here compares the oracle with itself: the generator is checked against Triton's
independent Philox4x32-10 (run in its CPU interpreter) and against distribution statistics; the
sampler against the exact block distribution enumerated by brute force; the Markov bias against
the dense V x V transition table W1 W2^T (a numpy matmul), the lookup the pages describe as the
memory-hungry equivalent of the low-rank form ("DSpark: Wait It's All Autoregressive?", "How the
Markov sampler works").
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import log_softmax, softmax

pytestmark = pytest.mark.filterwarnings("ignore")


# ---------------------------------------------------------------- Philox4x32-10 and uniforms

def _triton_philox(seeds, c0, c1, c2, c3):
    """Triton's own Philox4x32-10, executed by its CPU interpreter."""
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    import torch
    import triton.language as tl

    @triton.jit
    def kern(seed_ptr, c0p, c1p, c2p, c3p, out_ptr, N: tl.constexpr):
        i = tl.arange(0, N)
        seed = tl.load(seed_ptr + i)
        a, b, c, d = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i), tl.load(c2p + i),
                               tl.load(c3p + i))
        tl.store(out_ptr + i * 4 + 0, a)
        tl.store(out_ptr + i * 4 + 1, b)
        tl.store(out_ptr + i * 4 + 2, c)
        tl.store(out_ptr + i * 4 + 3, d)

    n = len(seeds)
    t = lambda a, dt: torch.tensor(np.asarray(a).astype(dt).view(
        np.int64 if dt == np.uint64 else np.int32))
    out = torch.zeros(n * 4, dtype=torch.int32)
    kern[(1,)](t(seeds, np.uint64), t(c0, np.uint32), t(c1, np.uint32), t(c2, np.uint32),
               t(c3, np.uint32), out, N=n)
    return out.numpy().view(np.uint32).reshape(n, 4)


def test_philox_matches_independent_implementation(oracle_mod):
    rng = np.random.default_rng(1234)
    n = 64
    seeds = rng.integers(0, 2**64, size=n, dtype=np.uint64)
    seeds[0] = 0
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    ctr[1] = 0xFFFFFFFF
    ref = _triton_philox(seeds, ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3])
    for i in range(n):
        key = [int(seeds[i]) & 0xFFFFFFFF, int(seeds[i]) >> 32]
        got = oracle_mod.philox4x32_10(ctr[i], key)
        assert np.array_equal(got, ref[i]), (i, got, ref[i])


def test_uniform_grid_and_range(oracle_mod):
    # u = (2m + 1) 2^-24 with m the top 23 bits of one Philox word: never 0, never 1.
    for (seed, b, k, v) in [(0, 0, 1, 0), (1, 3, 7, 151935), (2**63 + 5, 511, 16, 262143)]:
        u = oracle_mod.uniform(seed, b, k, v)
        m2 = u * 2**24
        assert 0.0 < u < 1.0 and m2 == int(m2) and int(m2) % 2 == 1


def test_uniform_distribution_ks(oracle_mod):
    us = np.array([oracle_mod.uniform(7, b, k, v)
                   for b in range(4) for k in range(1, 4) for v in range(2000)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    # neighbouring counters and lanes must not be correlated
    assert abs(np.corrcoef(us[:-1], us[1:])[0, 1]) < 0.03


def test_gumbel_bounds_and_moments(oracle_mod):
    g = np.array([oracle_mod.gumbel(3, 1, 2, v) for v in range(20000)])
    gmax = -math.log(-math.log(1 - 2.0**-24))   # largest value the 23-bit grid can produce
    assert g.max() <= gmax + 1e-12 and g.min() >= -math.log(-math.log(2.0**-24)) - 1e-12
    assert abs(g.mean() - np.euler_gamma) < 0.03          # Gumbel(0,1) mean
    assert abs(g.var() - math.pi**2 / 6) < 0.08


# ---------------------------------------------------------------- tiny Markov problem helpers

def _tiny(V=8, r=3, gamma=3, B=1, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    W1 = (rng.standard_normal((V, r)) * scale).astype(np.float64)
    W2 = (rng.standard_normal((V, r)) * scale).astype(np.float64)
    Urow = rng.standard_normal((gamma, V)).astype(np.float64)
    U = np.broadcast_to(Urow, (B, gamma, V)).copy()
    return W1, W2, U


def test_bias_equals_dense_transition_table(oracle_mod):
    V, r, gamma, B = 16, 4, 4, 3
    W1, W2, U = _tiny(V, r, gamma, B, seed=1)
    x0 = np.array([0, 5, 15], dtype=np.int32)
    res = oracle_mod.draft(head=0, B=B, gamma=gamma, V=V, r=r, d=0, T=1.0, seed=9, W1=W1,
                           W2=W2, U=U, x0=x0, want_z=True)
    table = W1 @ W2.T                         # dense V x V transition table
    for b in range(B):
        prev = x0[b]
        for k in range(gamma):
            np.testing.assert_allclose(res.z[b, k], U[b, k] + table[prev], rtol=0, atol=1e-12)
            prev = res.tokens[b, k]           # step k+1 conditions on the sampled x_k


def test_zero_embedding_gives_parallel_sampling(oracle_mod):
    # W1 = 0 => B_k = 0 => p_k = softmax(U_k) whatever the prefix: pure parallel drafting.
    V, r, gamma, B = 32, 4, 5, 2
    _, W2, U = _tiny(V, r, gamma, B, seed=2)
    res = oracle_mod.draft(head=0, B=B, gamma=gamma, V=V, r=r, d=0, T=0.7, seed=1,
                           W1=np.zeros((V, r)), W2=W2, U=U, x0=np.array([1, 2]), want_z=True)
    assert np.array_equal(res.z, U)
    np.testing.assert_allclose(res.lse, np.log(np.exp(U / 0.7).sum(-1)), rtol=0, atol=1e-12)


def test_lse_against_long_double(oracle_mod):
    V, r, gamma = 50, 4, 3
    W1, W2, U = _tiny(V, r, gamma, 1, seed=3, scale=2.0)
    res = oracle_mod.draft(head=0, B=1, gamma=gamma, V=V, r=r, d=0, T=1.3, seed=2, W1=W1,
                           W2=W2, U=U, x0=np.array([7]), want_z=True)
    for k in range(gamma):
        y = res.z[0, k].astype(np.longdouble) / np.longdouble(1.3)
        ref = float(np.log(np.sum(np.exp(y))))
        assert abs(res.lse[0, k] - ref) < 1e-12


def test_cold_temperature_is_argmax(oracle_mod):
    # |g| <= 16.64 on the 2^-24 grid, so at T = 1e-3 the noise moves scores by < 0.017 / T...
    # in units of z it is below 0.017: the sample must be argmax z whenever the gap is larger.
    V, r, gamma, B = 64, 4, 4, 8
    W1, W2, U = _tiny(V, r, gamma, B, seed=4, scale=1.0)
    U = U + np.random.default_rng(5).standard_normal(U.shape) * 3
    res = oracle_mod.draft(head=0, B=B, gamma=gamma, V=V, r=r, d=0, T=1e-3, seed=3, W1=W1,
                           W2=W2, U=U, x0=np.arange(B), want_z=True)
    checked = 0
    for b in range(B):
        for k in range(gamma):
            z = np.sort(res.z[b, k])
            if z[-1] - z[-2] > 0.04:
                assert res.tokens[b, k] == int(np.argmax(res.z[b, k]))
                checked += 1
    assert checked > B * gamma // 2


def test_gumbel_argmax_matches_scores(oracle_mod):
    V, r, gamma = 40, 3, 3
    W1, W2, U = _tiny(V, r, gamma, 1, seed=6)
    seed, T = 11, 0.9
    res = oracle_mod.draft(head=0, B=1, gamma=gamma, V=V, r=r, d=0, T=T, seed=seed, W1=W1,
                           W2=W2, U=U, x0=np.array([3]), want_z=True)
    for k in range(gamma):
        sc = res.z[0, k] / T + np.array([oracle_mod.gumbel(seed, 0, k + 1, v) for v in range(V)])
        order = np.argsort(-sc, kind="stable")
        assert res.tokens[0, k] == order[0] and res.tokens2[0, k] == order[1]
        assert res.best[0, k] == sc[order[0]] and res.best2[0, k] == sc[order[1]]


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_block_distribution_brute_force(oracle_mod, T):
    """Left-to-right Gumbel-max sampling reproduces P(X|x0) = prod_k p_k (Eq 4) exactly:
    enumerate all V^gamma = 512 blocks and compare with 2^18 sampled requests."""
    V, r, gamma, n = 8, 3, 3, 1 << 18
    W1, W2, U = _tiny(V, r, gamma, 1, seed=7, scale=0.9)
    x0 = 5
    # exact block probabilities, written from Eq 4 / Eq 5 with log-softmax
    P = np.zeros((V,) * gamma)
    for blk in itertools.product(range(V), repeat=gamma):
        prev, lp = x0, 0.0
        for k, x in enumerate(blk):
            z = U[0, k] + W1[prev] @ W2.T
            lp += log_softmax(z / T)[x]
            prev = x
        P[blk] = math.exp(lp)
    assert abs(P.sum() - 1) < 1e-12
    Ub = np.broadcast_to(U, (n, gamma, V)).copy()
    res = oracle_mod.draft(head=0, B=n, gamma=gamma, V=V, r=r, d=0, T=T, seed=2024, W1=W1,
                           W2=W2, U=Ub, x0=np.full(n, x0), nthreads=os.cpu_count())
    idx = np.ravel_multi_index(res.tokens.T, (V,) * gamma)
    counts = np.bincount(idx, minlength=V**gamma).astype(np.float64)
    expected = P.ravel() * n
    keep = expected >= 5
    chi2 = (((counts - expected) ** 2)[keep] / expected[keep]).sum()
    pval = stats.chi2.sf(chi2, keep.sum() - 1)
    assert pval > 1e-4, (chi2, keep.sum(), pval)
    sigma = np.sqrt(P.ravel() * (1 - P.ravel()) / n)
    assert np.all(np.abs(counts / n - P.ravel()) < 5 * sigma + 1e-5)
