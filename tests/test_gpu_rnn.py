"""GPU parity of the RNN-head draft (Eq 6) against the fp64 oracle.

The sequential update runs in fp32 on the CUDA cores, the h_k columns of the joint projection
come from the tensor-core pre-pass GEMM, and the bias product uses fp32 a_k = tanh(o_k) on the
CUDA cores, or a bf16 high/low split of a_k on the tensor cores (larger batches, and small ones
on the vocabulary-major tensor-core variant).  Same rules as
the Markov tests: tokens bit-exact up to counted near-ties, floats (and the final state) within
2e-3.
"""
import numpy as np
import pytest

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

RNN = inputs.WORKLOADS["rnn_head"]


SMALL_PATHS = [("cuda-core", 0), ("tensor-vocab", 2)]


@pytest.mark.parametrize("name,code", SMALL_PATHS)
@pytest.mark.parametrize("B", [1, 3])
def test_rnn_small_batch(monkeypatch, name, code, B):
    wl = RNN.with_(B=B, V=12000, d=128, seed=100 + B)
    monkeypatch.setenv("DSPARK_DRAFT_PATH", name)
    assert ds.draft_path(1, B, wl.V, wl.r) == code
    parity.run_case(wl, ds=ds, s0_scale=0.5)


@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_rnn_small_batch_rank64_target(monkeypatch, name, code):
    wl = RNN.with_(B=2, V=8008, r=64, d=64, seed=104)
    monkeypatch.setenv("DSPARK_DRAFT_PATH", name)
    assert ds.draft_path(1, wl.B, wl.V, wl.r) == code
    parity.run_case(wl, ds=ds, target_noise=1.0)


@pytest.mark.parametrize("lay", ["vr", "rv"])
@pytest.mark.parametrize("B", [8, 64])
def test_rnn_tensor_core(B, lay):
    wl = RNN.with_(B=B, V=10000, d=256, seed=110 + B)
    assert ds.draft_path(1, B, wl.V, wl.r) == 1
    parity.run_case(wl, ds=ds, s0_scale=0.5, w2_layout=lay)


@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_rnn_small_batch_w2_rv(monkeypatch, name, code):
    # W2 as [r][V] on the small-batch kernels (read through the transposed copy)
    wl = RNN.with_(B=2, V=12000, d=128, seed=106)
    monkeypatch.setenv("DSPARK_DRAFT_PATH", name)
    assert ds.draft_path(1, wl.B, wl.V, wl.r) == code
    parity.run_case(wl, ds=ds, s0_scale=0.5, w2_layout="rv")


def test_rnn_tensor_core_two_chunks_target():
    parity.run_case(RNN.with_(B=130, V=9000, d=128, seed=120), ds=ds, target_noise=1.0,
                    want_logits=False)


@pytest.mark.slow
def test_rnn_head_full_sampled_rows():
    # 32 of the 128 requests (tokens, lse, c, S and the final state), z element-wise on two
    rng = np.random.default_rng(5)
    rows = sorted({0, 127, *rng.choice(np.arange(1, 127), size=30, replace=False).tolist()})
    for lay in ("vr", "rv"):
        ties, _ = parity.run_case(RNN, ds=ds, rows=rows, z_rows=[rows[0], rows[-1]], w2_layout=lay)
        assert ties <= 2
