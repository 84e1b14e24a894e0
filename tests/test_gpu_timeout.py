"""The draft kernels' timeout path, exercised on the GPU without faulting or hanging it.

Every wait between thread blocks and every mbarrier wait in the draft kernels is bounded; when a
bound runs out the kernel records DSPARK_ERR_TIMEOUT, stops its producer (which waits for its
own bulk copies to land), lets the MMA thread finish its issued MMAs, frees TMEM and returns.
The test hook DSPARK_TEST_STUCK_WAIT (read by the library at every draft call) makes one named
wait wait for a signal that never comes, with a 20 us limit:

  grid  the per-step wait between thread blocks (one more arrival than there are blocks, or a
        key tag no block publishes);
  mbar  an mbarrier wait of the epilogue / consumer warps (on a barrier no thread arrives on).

For each draft kernel (CUDA-core, tensor cores with the vocabulary on M, tensor cores with the
requests on M) and each wait, the call must report DSPARK_ERR_TIMEOUT through
dspark_get_status, return within a fraction of the ordinary one-second bound, and leave the
workspace reset: the next call on the same workspace, without the hook, matches the oracle
(tokens bit-exact up to counted near-ties, floats within 2e-3).
"""
import time

import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

BASE = inputs.WORKLOADS["qwen3_4b_markov"]
PATHS = {
    # name: (DSPARK_DRAFT_PATH, path code, workload)
    "cuda-core": ("cuda-core", 0, BASE.with_(B=1, V=20000, d=256, seed=300)),
    "tensor-vocab": ("tensor-vocab", 2, BASE.with_(B=4, V=20000, d=256, seed=301)),
    "tensor": ("tensor", 1, BASE.with_(B=130, V=20000, d=256, seed=302)),
}


@pytest.mark.parametrize("wait", ["grid", "mbar"])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_stuck_wait_times_out_and_workspace_recovers(monkeypatch, path, wait):
    env, code, wl = PATHS[path]
    monkeypatch.setenv("DSPARK_DRAFT_PATH", env)
    assert ds.draft_path(0, wl.B, wl.V, wl.r, True) == code
    host = inputs.generate(wl)
    t = parity.to_dev(host)
    ws = ds.Workspace(0, wl.B, wl.gamma, wl.V, wl.r, wl.d)

    def call():
        return ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], T=wl.T, seed=wl.seed,
                               h=t["h"], w=t["w"], workspace=ws)

    call()  # warm-up: module load, attribute set-up
    assert ws.status() == 0
    monkeypatch.setenv("DSPARK_TEST_STUCK_WAIT", wait)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    call()
    status = ws.status()  # synchronises, reads and resets the workspace
    elapsed = time.perf_counter() - t0
    assert status == 4, f"expected DSPARK_ERR_TIMEOUT, got {status}"
    assert elapsed < 0.5, f"the timed-out call took {elapsed:.3f} s"
    monkeypatch.delenv("DSPARK_TEST_STUCK_WAIT")

    o = parity.oracle_draft(wl, host)
    out = call()
    torch.cuda.synchronize()
    assert ws.status() == 0
    ties = parity.check_tokens_free(out.tokens.cpu().numpy(), o)
    errs = {k: parity.close(k, getattr(out, k).cpu().numpy(), getattr(o, k))
            for k in ("lse", "c", "S")}
    assert ties <= 1, ties
    print(f"{path} {wait}: timed out in {elapsed * 1e3:.1f} ms; next call near-ties {ties}, {errs}")
