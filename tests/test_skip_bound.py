"""The tensor-core sampler's exact skip test, emulated in fp32 on the CPU.

For an entry with uniform u (from the Philox word `bits`, u = (2 (bits >> 9) + 1) 2^-24) and
w = 1 - u, the kernel forms f = bits of 0x3F800000 | (bits >> 9) read as a float (one funnel
shift; f = 2 - 2^-24 - w), P = pe * Cp with pe = 2^(y2 - ref) and Cp = 1.002 * 2^(ref - best2)
(so P is the computed 1.002 exp(y - best)), X = fl(2 - P) in one fma, and skips the entry when
f < X.  The claim: a skipped entry satisfies w >= 1.001 exp(y - best) and so cannot beat the
running best (-ln u >= w).  Here the same fp32 steps run in numpy on entries spread around the
threshold (including u close to 1, where the Gumbel noise is largest) and every skipped entry is
checked against its exact perturbed score in fp64.  The 2^x steps are taken exact; the
kernel's ex2.approx error (about 2^-22 relative) is far inside the 0.1% margin of the bound.
"""
import numpy as np

LOG2E = 1.4426950408889634


def _skip_case(seed, n=2_000_000):
    rng = np.random.default_rng(seed)
    f32 = np.float32
    T = rng.choice([1.0, 0.7, 1.3], n)
    s2 = ((f32(1.0) / T.astype(f32)).astype(f32) * f32(LOG2E)).astype(f32)
    z = rng.normal(0, 3, n).astype(f32)
    ref = ((z + rng.normal(0, 5, n)).astype(f32) * s2).astype(f32)       # reference point
    best2 = (z * s2 + rng.uniform(-30, 8, n)).astype(f32)                # running best, log2
    j = rng.integers(0, 2**23, n, dtype=np.int64)
    tail = rng.random(n) < 0.5                                          # u near 1: large noise
    j[tail] = 2**23 - 1 - rng.integers(0, 2**12, tail.sum())
    bits = (j << 9) | rng.integers(0, 512, n)
    u = (2 * j + 1) * 2.0**-24
    w = 1 - u
    t = (z.astype(np.float64) * s2 - ref).astype(f32)                    # fma: one rounding
    pe = np.exp2(t.astype(np.float64)).astype(f32)
    cp = (f32(1.002) * np.exp2((ref - best2).astype(np.float64)).astype(f32)).astype(f32)
    X = (2.0 - pe.astype(np.float64) * cp.astype(np.float64)).astype(f32)  # fma: one rounding
    f = (0x3F800000 | (bits >> 9)).astype(np.uint32).view(np.float32)
    skipped = ~(f >= X)
    y = z.astype(np.float64) * s2.astype(np.float64) / LOG2E             # natural units
    best = best2.astype(np.float64) / LOG2E
    score = y - np.log(-np.log(u))
    return skipped, w, y, best, score


def test_skipped_entries_cannot_win():
    for seed in (1, 2, 3):
        skipped, w, y, best, score = _skip_case(seed)
        assert skipped.mean() > 0.05                        # the case exercises the skip
        assert not np.any(skipped & (score >= best - 1e-4))
        assert not np.any(skipped & (w < 1.001 * np.exp(y - best)))


def test_funnel_shift_float_is_the_uniform():
    # f = 0x3F800000 | (bits >> 9) as a float equals 1 + u - 2^-24 exactly
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2**32, 100_000, dtype=np.uint64)
    f = (0x3F800000 | (bits >> 9)).astype(np.uint32).view(np.float32).astype(np.float64)
    u = (2.0 * (bits >> 9).astype(np.float64) + 1.0) * 2.0**-24
    assert np.array_equal(f, 1.0 + u - 2.0**-24)
