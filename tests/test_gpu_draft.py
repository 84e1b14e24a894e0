"""GPU parity of the draft calls against the fp64 oracle, through the C ABI.

Each case runs the library free-running and teacher-forced on the oracle's tokens, checks
tokens bit-exact up to counted near-ties, and every float output within 2e-3 absolute.
Cases span several vocab slices per block and a ragged tail, both dtypes, the degenerate
shapes (B = 1, gamma = 1, vocab smaller than the grid's slices), the 16-byte-misaligned U
row path, forced tokens, a target for Eq 8, and the full latency-regime workload.
"""
import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

TINY = inputs.WORKLOADS["tiny_markov"]


def _run_case(wl, **kw):
    return parity.run_case(wl, ds=ds, **kw)


# bf16 cases with B <= 4 run on both small-batch kernels: CUDA-core dot products (path 0) and
# the tensor-core bias product with vocabulary rows on M (path 2)
SMALL_PATHS = [("cuda-core", 0), ("tensor-vocab", 2)]


def _use_path(monkeypatch, name, code, wl, head=0):
    monkeypatch.setenv("DSPARK_DRAFT_PATH", name)
    assert ds.draft_path(head, wl.B, wl.V, wl.r, wl.dtype == "bf16") == code


# W2 as the pages write it ([r][V]) or as a linear layer's weight ([V][r]); the small-batch
# kernels read the [r][V] form through a transposed copy in the workspace
LAYOUTS = ["vr", "rv"]


@pytest.mark.parametrize("lay", LAYOUTS)
def test_tiny_markov_workload(lay):
    _run_case(TINY, w2_layout=lay)


@pytest.mark.parametrize("B", [1, 2, 3])
def test_tiny_batches(B):
    _run_case(TINY.with_(B=B, seed=10 + B))


@pytest.mark.parametrize("gamma", [1, 15, 16])
def test_block_sizes(gamma):
    _run_case(TINY.with_(gamma=gamma, seed=20 + gamma))


@pytest.mark.parametrize("lay", LAYOUTS)
def test_temperature_and_target_fp32(lay):
    _run_case(TINY.with_(T=0.7, seed=31), target_noise=1.0, w2_layout=lay)


def test_ragged_vocab_unaligned_rows():
    # V * 4 bytes is not a multiple of 16: U rows are fetched with plain loads
    _run_case(TINY.with_(V=1001, seed=32), target_noise=0.5)


def test_vocab_smaller_than_grid():
    # most blocks own an empty slice
    _run_case(TINY.with_(V=40, B=2, seed=33), target_noise=1.0)


@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_bf16_small_with_target(monkeypatch, name, code):
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=20008, d=512, B=3, seed=34)
    _use_path(monkeypatch, name, code, wl)
    _run_case(wl, target_noise=1.0)


@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("name,code", SMALL_PATHS)
@pytest.mark.parametrize("B", [1, 2, 4])
def test_bf16_batches_both_paths(monkeypatch, name, code, B, lay):
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=30000, d=256, B=B, seed=50 + B)
    _use_path(monkeypatch, name, code, wl)
    _run_case(wl, w2_layout=lay)


@pytest.mark.parametrize("V", [1000, 130, 40])
def test_tensor_vocab_partial_tiles(monkeypatch, V):
    # slices of a few rows: one partial 128-row tile per block, or none at all
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=V, d=64, B=2, seed=60 + V)
    _use_path(monkeypatch, "tensor-vocab", 2, wl)
    _run_case(wl, target_noise=1.0)


@pytest.mark.parametrize("r", [64, 128, 192])
def test_tensor_vocab_ranks(monkeypatch, r):
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=50000, r=r, d=64, B=3, seed=70 + r)
    _use_path(monkeypatch, "tensor-vocab", 2, wl)
    _run_case(wl, target_noise=0.5)


def test_bf16_rank_512():
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=12000, r=512, d=64, B=2, seed=35)
    _run_case(wl)


@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_ring_reuse_more_stages_than_slots(monkeypatch, name, code):
    # every block streams more W2 stages than the ring has slots, so slots are reused within a
    # step and warps reach a slot before its previous use completes
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=80000, d=128, B=1, seed=36)
    _use_path(monkeypatch, name, code, wl)
    _run_case(wl, want_logits=False)
    _run_case(wl.with_(B=2, seed=37), want_logits=False)


@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_qwen3_4b_vocab_small_hidden(monkeypatch, name, code):
    # the full vocabulary: every slab kind of the tensor-core variant (TMEM, resident, streamed)
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(d=256, seed=38)
    _use_path(monkeypatch, name, code, wl)
    _run_case(wl, want_logits=False)


@pytest.mark.slow
@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_qwen3_4b_markov_full(monkeypatch, name, code, lay):
    wl = inputs.WORKLOADS["qwen3_4b_markov"]
    _use_path(monkeypatch, name, code, wl)
    ties, _ = _run_case(wl, want_logits=False, w2_layout=lay)
    assert ties <= 1


def test_invalid_anchor_sets_status():
    wl = TINY.with_(seed=40)
    t = parity.to_dev(inputs.generate(wl))
    x0 = t["x0"].clone()
    x0[1] = wl.V
    ws = ds.Workspace(0, wl.B, wl.gamma, wl.V, wl.r, wl.d)
    out = ds.markov_draft(t["W1"], t["W2"], t["U"], x0, h=t["h"], w=t["w"], seed=wl.seed,
                          workspace=ws)
    assert ws.status() == 1                      # DSPARK_ERR_INVALID, then reset
    tok = out.tokens.cpu().numpy()
    assert np.all(tok[1] == -1) and np.all(tok[[0, 2, 3]] >= 0)
    assert np.all(np.isnan(out.c.cpu().numpy()[1]))
    # the workspace is clean again: the next call succeeds
    out2 = ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], seed=wl.seed, workspace=ws)
    assert ws.status() == 0 and np.all(out2.tokens.cpu().numpy() >= 0)


def test_repeat_runs_are_bit_identical():
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=50000, d=256, B=4, seed=41)
    t = parity.to_dev(inputs.generate(wl.with_(target_noise=1.0)))
    ws = ds.Workspace(0, wl.B, wl.gamma, wl.V, wl.r, wl.d, target=True)
    runs = [ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], h=t["h"], w=t["w"],
                            target=t["target"], seed=7, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in runs[1:]:
        for f in ("tokens", "lse", "c", "S", "cstar", "l1"):
            assert torch.equal(getattr(o, f), getattr(runs[0], f)), f


@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_draft_captured_in_cuda_graph(monkeypatch, name, code):
    # the call is stream-ordered and capturable: a graph replay gives the direct call's results
    wl = inputs.WORKLOADS["qwen3_4b_markov"].with_(V=20008, d=256, B=2, seed=90)
    _use_path(monkeypatch, name, code, wl)
    t = parity.to_dev(inputs.generate(wl))
    plan = ds.DraftPlan(0, t["W1"], t["W2"], t["U"], t["x0"], T=wl.T, seed=wl.seed, h=t["h"],
                        w=t["w"], Wj=None, target=None, forced=None, s0=None, want_logits=False,
                        workspace=None, stream=None)
    ref = plan.run()
    ref = {k: getattr(ref, k).clone() for k in ("tokens", "lse", "c", "S")}
    torch.cuda.synchronize()
    for k in ref:
        getattr(plan.out, k).zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run(torch.cuda.current_stream())
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert plan.workspace.status() == 0
    for k, v in ref.items():
        assert torch.equal(getattr(plan.out, k), v), k
