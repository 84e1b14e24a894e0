"""Pins of the oracle's sequential temperature scaling (STS) of the confidence head.

"Phase-Conditioned Speculative Decoding" section 3: the head's output is calibrated afterwards
by temperature scaling that minimises the expected calibration error of the cumulative
product, one position at a time; "DSpark -- paper verification" (delta table D13): a
left-to-right 1-D grid search with the prefix held fixed.  The pins:

* recovery: data drawn calibrated at known per-position temperatures (each position survives
  with probability sigmoid(l / tau*) given that the prefix survived) give back tau* to the grid
  step, from logits that are miscalibrated at tau = 1;
* the ECE's closed form on hand examples (constant predictions; perfect separation);
* with the identity temperature in the grid, the first position's ECE never gets worse;
* a grid of one entry returns that entry; invalid inputs are reported.
"""
import numpy as np
import pytest

from oracle import oracle


def calibrated_sample(N, taus, seed):
    rng = np.random.default_rng(seed)
    gamma = len(taus)
    conf = rng.normal(1.5, 2.0, (N, gamma)).astype(np.float32)
    acc = np.zeros(N, np.int32)
    alive = np.ones(N, bool)
    for k in range(gamma):
        c = 1 / (1 + np.exp(-conf[:, k].astype(np.float64) / taus[k]))
        survive = alive & (rng.random(N) < c)
        acc += survive
        alive = survive
    return conf, acc


def test_recovers_known_temperatures():
    taus = [1.6, 0.7, 2.5, 1.0]
    conf, acc = calibrated_sample(400_000, taus, seed=1)
    grid = np.round(np.arange(0.3, 3.01, 0.1), 2).astype(np.float32)
    tau, ece, eg, st = oracle.sts(conf, acc, grid)
    assert st == 0
    assert np.allclose(tau, taus, atol=0.11), tau
    assert np.all(ece < 0.01)
    raw = eg[:, np.argmin(np.abs(grid - 1.0))]  # ECE at tau = 1 given the chosen prefix
    assert raw[0] > 5 * ece[0]  # the raw head is visibly miscalibrated at position 1


def test_ece_closed_forms():
    N = 1000
    conf = np.full((N, 1), np.log(0.7 / 0.3), np.float32)  # sigmoid = 0.7 at tau = 1
    acc = np.zeros(N, np.int32)
    acc[:700] = 1
    tau, ece, eg, st = oracle.sts(conf, acc, np.array([1.0], np.float32))
    assert abs(ece[0]) < 1e-6  # 70% positives at confidence 0.7
    acc[:] = 1
    tau, ece, eg, st = oracle.sts(conf, acc, np.array([1.0], np.float32))
    assert abs(ece[0] - 0.3) < 1e-6
    # perfect separation: half at confidence 0.95 all survive, half at 0.05 none survive
    conf2 = np.concatenate([np.full(500, np.log(19.0)), np.full(500, -np.log(19.0))])[:, None].astype(np.float32)
    acc2 = np.concatenate([np.ones(500), np.zeros(500)]).astype(np.int32)
    tau, ece, eg, st = oracle.sts(conf2, acc2, np.array([1.0], np.float32), bins=10)
    assert abs(ece[0] - 0.05) < 1e-6


def test_identity_in_grid_never_worsens_position_one():
    rng = np.random.default_rng(3)
    conf = rng.normal(0, 3, (5000, 3)).astype(np.float32)
    acc = rng.integers(0, 4, 5000).astype(np.int32)
    grid = np.array([0.5, 1.0, 2.0, 4.0], np.float32)
    tau, ece, eg, st = oracle.sts(conf, acc, grid)
    assert ece[0] <= eg[0, 1] + 1e-15
    assert ece[0] == eg[0].min()


def test_single_grid_entry_and_ties_to_first():
    rng = np.random.default_rng(4)
    conf = rng.normal(0, 1, (100, 2)).astype(np.float32)
    acc = rng.integers(0, 3, 100).astype(np.int32)
    tau, ece, eg, st = oracle.sts(conf, acc, np.array([0.8], np.float32))
    assert np.all(tau == np.float32(0.8))
    tau, ece, eg, st = oracle.sts(conf, acc, np.array([0.8, 0.8], np.float32))
    assert np.all(tau == np.float32(0.8)) and np.all(eg[:, 0] == eg[:, 1])


def test_invalid_inputs():
    conf = np.zeros((4, 2), np.float32)
    assert oracle.sts(conf, np.array([0, 1, 3, 2], np.int32), np.array([1.0], np.float32))[3] == 1
    assert oracle.sts(conf, np.array([0, 1, 2, 2], np.int32), np.array([0.0], np.float32))[3] == 1
