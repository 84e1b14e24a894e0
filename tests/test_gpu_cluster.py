"""The small-batch draft kernels (paths 0 and 2) in thread-block clusters, against the oracle.

The blocks of a cluster hand their per-step argmax key and (max, sum-exp) partials to the
cluster's first block through distributed shared memory; that block merges them and publishes
one slot per cluster, which every block then polls.  Each cluster size the library accepts on
this GPU (DSPARK_CLUSTER = 1, 2, 4, 8; 1 is the plain per-block merge) must give the oracle's
tokens (bit-exact up to counted near-ties) and floats within 2e-3, on both kernels, with and
without a target (whose Eq 8 pass needs the merged normalisers right after each step), with
blocks that own no vocabulary, and through the bounded-wait failure path.
"""
import time

import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 4, 8]
SMALL_PATHS = [("cuda-core", 0), ("tensor-vocab", 2)]
QWEN = inputs.WORKLOADS["qwen3_4b_markov"]


def _use(monkeypatch, size, name, code, wl, head=0):
    monkeypatch.setenv("DSPARK_DRAFT_PATH", name)
    monkeypatch.setenv("DSPARK_CLUSTER", str(size))
    assert ds.draft_path(head, wl.B, wl.V, wl.r, wl.dtype == "bf16") == code
    got = ds.draft_cluster(head, wl.B, wl.V, wl.r, wl.dtype == "bf16")
    if got < 0:
        pytest.skip(f"clusters of {size} blocks do not tile this GPU's SMs")
    assert got == size


def test_cluster_query(monkeypatch):
    monkeypatch.delenv("DSPARK_DRAFT_PATH", raising=False)
    monkeypatch.delenv("DSPARK_CLUSTER", raising=False)
    assert ds.draft_cluster(0, 1, QWEN.V, QWEN.r, True) == 1  # no clusters unless asked
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fits = []
    for c in (2, 4, 8):
        monkeypatch.setenv("DSPARK_CLUSTER", str(c))
        got = ds.draft_cluster(0, 1, QWEN.V, QWEN.r, True)
        assert got in (c, -1)
        if got == c:
            assert sms % c == 0
            fits.append(c)
    assert ds.draft_cluster(0, 512, 262144, 256, True) == 1  # the tensor-core path: no clusters
    print(f"cluster sizes that tile the {sms} SMs: {fits}")


@pytest.mark.parametrize("size", SIZES)
@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_cluster_sizes_bf16(monkeypatch, size, name, code):
    wl = QWEN.with_(V=30000, d=256, B=3 if code == 2 else 1, seed=400 + size)
    _use(monkeypatch, size, name, code, wl)
    parity.run_case(wl, ds=ds)


@pytest.mark.parametrize("size", SIZES)
@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_cluster_sizes_with_target(monkeypatch, size, name, code):
    wl = QWEN.with_(V=20008, d=512, B=4, T=0.8, seed=410 + size)
    _use(monkeypatch, size, name, code, wl)
    parity.run_case(wl, ds=ds, target_noise=1.0)


@pytest.mark.parametrize("size", SIZES)
def test_cluster_sizes_fp32_empty_blocks(monkeypatch, size):
    # V = 40: most blocks, and whole clusters, own no vocabulary
    wl = inputs.WORKLOADS["tiny_markov"].with_(V=40, B=2, seed=420 + size)
    _use(monkeypatch, size, "cuda-core", 0, wl)
    parity.run_case(wl, ds=ds, target_noise=1.0)


@pytest.mark.parametrize("size", [2, 8])
def test_cluster_rnn_head(monkeypatch, size):
    wl = inputs.WORKLOADS["rnn_head"].with_(B=2, V=20000, d=256, seed=430 + size)
    _use(monkeypatch, size, "cuda-core", 0, wl, head=1)
    parity.run_case(wl, ds=ds, target_noise=1.0)


@pytest.mark.parametrize("size", [2, 8])
@pytest.mark.parametrize("name,code", SMALL_PATHS)
def test_cluster_timeout_unwinds(monkeypatch, size, name, code):
    # the per-step wait made to time out: every block of every cluster must leave (the exit
    # waits for the cluster's blocks) and the next call must be clean
    wl = QWEN.with_(B=2, V=20000, d=256, seed=440 + size)
    _use(monkeypatch, size, name, code, wl)
    host = inputs.generate(wl)
    t = parity.to_dev(host)
    ws = ds.Workspace(0, wl.B, wl.gamma, wl.V, wl.r, wl.d)

    def call():
        return ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], T=wl.T, seed=wl.seed,
                               h=t["h"], w=t["w"], workspace=ws)

    call()
    assert ws.status() == 0
    monkeypatch.setenv("DSPARK_TEST_STUCK_WAIT", "grid")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    call()
    status = ws.status()
    elapsed = time.perf_counter() - t0
    assert status == 4 and elapsed < 0.5, (status, elapsed)
    monkeypatch.delenv("DSPARK_TEST_STUCK_WAIT")
    o = parity.oracle_draft(wl, host)
    out = call()
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert parity.check_tokens_free(out.tokens.cpu().numpy(), o) <= 1
