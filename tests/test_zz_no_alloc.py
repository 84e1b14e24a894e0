"""The allocation-free Markov draft (dspark_markov_draft_noalloc), through the C ABI.

Some callers cannot obtain device memory at drafting time: plugins that live inside another
framework's memory pool, serving engines that forbid allocation on their decode path, and code
that is only handed pre-allocated inputs and outputs.  They call the entry point that keeps its
scratch in an array built into the library.  For each case this test makes two calls in a row
of that entry point (the second runs on the scratch the first left behind) and checks each one:

  * against the fp64 oracle on the same inputs: tokens bit-exact up to counted near-ties,
    lse / c / S / c* / l1 within the 2e-3 tolerance of the other parity tests (teacher-forced on
    the oracle's tokens, plus a free-running call for the tokens);
  * against dspark_markov_draft with its own workspace: the same tokens, floats within 2e-3;
  * a clean device status, read from the optional status word the entry point writes.

The cases cover the three small-batch kernels the entry point can reach: the CUDA-core path
with fp32 and with bf16 weights, and the bf16 tensor-core path with the vocabulary on M (B = 4).

The file is named so that pytest collects it last: in a run that stops at the first failure
(``-x``), every other GPU test has then already run.  It relies on nothing the other tests leave
behind and passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import _lib, inputs
from tests import parity

pytestmark = pytest.mark.gpu

TOL = parity.TOL

CASES = {
    # name: (workload, kernel path the entry point takes)
    "f32_cuda_core": (inputs.WORKLOADS["tiny_markov"].with_(seed=200), 0),
    "bf16_cuda_core_target": (inputs.WORKLOADS["qwen3_4b_markov"].with_(
        V=30000, d=512, seed=201, target_noise=1.0), 0),
    "bf16_tensor_vocab_B4": (inputs.WORKLOADS["qwen3_4b_markov"].with_(
        B=4, V=30000, d=512, seed=202, target_noise=1.0), 2),
}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, wl, t, forced, status):
    B, G = wl.B, wl.gamma
    tgt = t.get("target") is not None
    out = {k: torch.full((B, G), float("nan"), device="cuda")
           for k in ("lse", "c", "S") + (("cstar", "l1") if tgt else ())}
    out["tokens"] = torch.full((B, G), -7, dtype=torch.int32, device="cuda")
    dt = 1 if wl.dtype == "bf16" else 0
    code = lib.dspark_markov_draft_noalloc(
        wl.B, wl.gamma, wl.V, wl.r, wl.d, float(wl.T), wl.seed, dt, _p(t["W1"]), _p(t["W2"]),
        _p(t["w"]), dt, _p(t["U"]), _p(t["h"]), _p(t["x0"]), _p(forced), _p(t.get("target")),
        _p(out["tokens"]), _p(out["lse"]), _p(out["c"]), _p(out["S"]), _p(out.get("cstar")),
        _p(out.get("l1")), None, _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, lib.dspark_last_error()
    return out


class _Out:
    """The entry point's outputs in the shape parity.compare_floats reads."""

    def __init__(self, d):
        self.lse, self.c, self.S = d["lse"], d["c"], d["S"]
        self.cstar, self.l1 = d.get("cstar"), d.get("l1")
        self.logits = self.s_out = None


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_oracle_and_workspace_draft_twice(case):
    wl, path = CASES[case]
    tgt = wl.target_noise is not None
    lib = _lib.load()
    assert lib.dspark_workspace_bytes(0, wl.B, wl.gamma, wl.V, wl.r, wl.d, 1 if tgt else 0) <= 1 << 20
    assert ds.draft_path(0, wl.B, wl.V, wl.r, wl.dtype == "bf16") == path
    host = inputs.generate(wl)
    t = parity.to_dev(host)
    o = parity.oracle_draft(wl, host)
    assert o.status == 0
    forced = torch.from_numpy(o.tokens.astype(np.int32)).cuda()
    ref = ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], T=wl.T, seed=wl.seed, h=t["h"],
                          w=t["w"], target=t.get("target"))
    ref_tf = ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], T=wl.T, seed=wl.seed, h=t["h"],
                             w=t["w"], target=t.get("target"), forced=forced)
    torch.cuda.synchronize()
    for call in range(2):
        status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        free = _noalloc(lib, wl, t, None, status[0:1])
        tf = _noalloc(lib, wl, t, forced, status[1:2])
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0], f"call {call}: device status {status.tolist()}"
        # against the oracle
        parity.check_tokens_free(free["tokens"].cpu().numpy(), o)
        parity.check_tokens_forced(tf["tokens"].cpu().numpy(), o)
        parity.compare_floats(_Out(tf), o, logits=False)
        # against the workspace entry point
        assert torch.equal(free["tokens"], ref.tokens), f"call {call}: tokens differ"
        assert torch.equal(tf["tokens"], ref_tf.tokens), f"call {call}: forced tokens differ"
        for k in free:
            if k == "tokens":
                continue
            err = (tf[k] - getattr(ref_tf, k)).abs().max().item()
            assert err <= TOL, f"call {call}: {k} differs from the workspace draft by {err}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    p = ctypes.c_void_p(256)
    # B = 512 needs far more than the built-in 1 MiB of scratch
    code = lib.dspark_markov_draft_noalloc(512, 7, 262144, 256, 0, 1.0, 0, 1, p, p, None, 1, p,
                                           None, p, None, None, p, p, None, None, None, None,
                                           None, None, None)
    assert code == 2 and b"built-in" in lib.dspark_last_error()
