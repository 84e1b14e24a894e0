"""The allocation-free Markov draft (dspark_markov_draft_noalloc) against the ordinary one.

Callers that cannot obtain device memory at drafting time -- plugins living inside another
framework's memory pool, serving engines that forbid allocation on the decode path, code that
is only handed pre-allocated inputs and outputs -- use the entry point that keeps its scratch in
an array built into the library.  This checks, through the C ABI, that two calls in a row of that
entry point give the same results as dspark_markov_draft with its own workspace: tokens equal,
floats within the 2e-3 tolerance the parity tests use, and a clean device status each time
(the second call runs on the scratch the first one left behind).  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, wl, t, out, status):
    code = lib.dspark_markov_draft_noalloc(
        wl.B, wl.gamma, wl.V, wl.r, wl.d, float(wl.T), wl.seed,
        1 if wl.dtype == "bf16" else 0, _p(t["W1"]), _p(t["W2"]), _p(t["w"]),
        1 if wl.dtype == "bf16" else 0, _p(t["U"]), _p(t["h"]), _p(t["x0"]), None,
        _p(t.get("target")), _p(out["tokens"]), _p(out["lse"]), _p(out["c"]), _p(out["S"]),
        _p(out.get("cstar")), _p(out.get("l1")), None, _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, lib.dspark_last_error()


@pytest.mark.parametrize("name,target", [("tiny_markov", False), ("qwen3_4b_markov", True)])
def test_noalloc_matches_workspace_draft_twice(name, target):
    wl = inputs.WORKLOADS[name].with_(seed=200)
    if name == "qwen3_4b_markov":
        wl = wl.with_(V=30000, d=512)
    if target:
        wl = wl.with_(target_noise=1.0)
    t = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in inputs.generate(wl).items()}
    ref = ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], T=wl.T, seed=wl.seed, h=t["h"],
                          w=t["w"], target=t.get("target"))
    lib = _lib.load()
    B, G = wl.B, wl.gamma
    for call in range(2):
        out = {k: torch.full((B, G), float("nan"), device="cuda")
               for k in ("lse", "c", "S") + (("cstar", "l1") if target else ())}
        out["tokens"] = torch.full((B, G), -7, dtype=torch.int32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        _noalloc(lib, wl, t, out, status)
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status {status.item()}"
        assert torch.equal(out["tokens"], ref.tokens), f"call {call}: tokens differ"
        for k in out:
            if k == "tokens":
                continue
            err = (out[k] - getattr(ref, k)).abs().max().item()
            assert err <= TOL, f"call {call}: {k} differs by {err}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    p = ctypes.c_void_p(256)
    # B = 512 needs far more than the built-in 1 MiB of scratch
    code = lib.dspark_markov_draft_noalloc(512, 7, 262144, 256, 0, 1.0, 0, 1, p, p, None, 1, p,
                                           None, p, None, None, p, p, None, None, None, None,
                                           None, None, None)
    assert code == 2 and b"built-in" in lib.dspark_last_error()
