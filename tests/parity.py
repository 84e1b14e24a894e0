"""GPU-vs-oracle comparison rules for the draft calls.

Tokens: bit-exact, except where the oracle's own fp64 perturbed scores of the two candidates
differ by less than TIE (a near-tie: fp32 and fp64 may legitimately rank them differently);
near-ties are counted and returned.  The free-running comparison stops at a row's first
near-tie (the rows then condition on different tokens); the teacher-forced comparison (both
sides conditioned on the oracle's tokens) judges every position on its own.
Floats (logits z, lse, c, S, c*, l1): absolute difference <= TOL (fp32 accumulation against
fp64).
"""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import oracle
from semi_autoregressive_drafting_gb300 import inputs

TOL = 2e-3
TIE = 1e-4


def host_inputs(wl: inputs.Workload):
    return inputs.generate(wl)


def to_dev(t, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def oracle_draft(wl, t, rows=None, forced=None, want_z=False):
    O = inputs.to_oracle
    return oracle.draft(
        head=0 if wl.head == "markov" else 1, B=wl.B, gamma=wl.gamma, V=wl.V, r=wl.r, d=wl.d,
        T=wl.T, seed=wl.seed, W1=O(t["W1"]), W2=O(t["W2"]), Wj=O(t.get("Wj")), U=O(t["U"]),
        x0=O(t["x0"]), h=O(t["h"]), w=O(t["w"]), target=O(t.get("target")),
        s0=None if t.get("s0") is None else O(t["s0"]).astype(np.float64),
        forced=None if forced is None else np.asarray(forced, dtype=np.int32),
        rows=rows, want_z=want_z, nthreads=os.cpu_count() or 1)


def check_tokens_free(gpu_tok: np.ndarray, o) -> int:
    """Free-running rows: equal up to the first near-tie of each row."""
    ties = 0
    for i in range(gpu_tok.shape[0]):
        for k in range(gpu_tok.shape[1]):
            if gpu_tok[i, k] == o.tokens[i, k]:
                continue
            gap = o.best[i, k] - o.best2[i, k]
            assert gpu_tok[i, k] == o.tokens2[i, k] and gap < TIE, (
                f"row {i} step {k}: gpu {gpu_tok[i, k]} oracle {o.tokens[i, k]} "
                f"(runner-up {o.tokens2[i, k]}, gap {gap:.3g})")
            ties += 1
            break
    return ties


def check_tokens_forced(gpu_tok: np.ndarray, o) -> int:
    """Teacher-forced rows: every position equal or a near-tie."""
    ties = 0
    bad = np.argwhere(gpu_tok != o.tokens)
    for i, k in bad:
        gap = o.best[i, k] - o.best2[i, k]
        assert gpu_tok[i, k] == o.tokens2[i, k] and gap < TIE, (
            f"row {i} step {k}: gpu {gpu_tok[i, k]} oracle {o.tokens[i, k]} "
            f"(runner-up {o.tokens2[i, k]}, gap {gap:.3g})")
        ties += 1
    return ties


def close(name, gpu, ref, tol=TOL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    worst = float(np.nanmax(err)) if err.size else 0.0
    assert np.array_equal(np.isnan(gpu), np.isnan(ref)), f"{name}: NaN pattern differs"
    assert worst <= tol, f"{name}: max |gpu - oracle| = {worst:.3g} > {tol}"
    return worst


def _rows(a, rows):
    """The selected request rows of a GPU output, taken on the device before the copy."""
    if rows is None:
        return a.cpu().numpy()
    return a[torch.as_tensor(rows, device=a.device)].cpu().numpy()


def compare_floats(out, o, rows=None, logits=True, z_rows=None):
    """Floats within TOL.  z_rows (a subset of rows) limits the element-wise logits comparison
    to those requests."""
    sel = lambda a: _rows(a, rows)
    errs = {"lse": close("lse", sel(out.lse), o.lse)}
    if o.c is not None and out.c is not None:
        errs["c"] = close("c", sel(out.c), o.c)
        errs["S"] = close("S", sel(out.S), o.S)
    if o.cstar is not None and out.cstar is not None:
        errs["cstar"] = close("cstar", sel(out.cstar), o.cstar)
        errs["l1"] = close("l1", sel(out.l1), o.l1)
    if logits and o.z is not None and out.logits is not None:
        if z_rows is None:
            errs["logits"] = close("logits", sel(out.logits), o.z)
        else:
            pos = [list(rows).index(r) for r in z_rows] if rows is not None else list(z_rows)
            errs["logits"] = close("logits", _rows(out.logits, z_rows), o.z[pos])
    if o.s_final is not None and out.s_out is not None:
        errs["s_out"] = close("s_out", sel(out.s_out), o.s_final)
    return errs


def run_case(wl, *, target_noise=None, want_logits=True, rows=None, check_free=True, ds=None,
             s0_scale=None, z_rows=None, w2_layout="vr"):
    """Free-running and teacher-forced GPU draft against the oracle on the same inputs.
    z_rows (a subset of rows): compare the logits z element-wise on those requests only.
    w2_layout "rv": the library gets W2 as [r][V] (the oracle keeps its [V][r] copy)."""
    if z_rows is not None:
        want_logits = True
    if target_noise is not None:
        wl = wl.with_(target_noise=target_noise)
    t = inputs.generate(wl)
    rnn = wl.head == "rnn"
    if rnn and s0_scale is not None:
        g = torch.Generator().manual_seed(wl.seed + 1000)
        t["s0"] = torch.randn(wl.B, wl.r, generator=g) * s0_scale
    d = to_dev(t)
    o = oracle_draft(wl, t, rows=rows, want_z=want_logits)
    assert o.status == 0
    has_t = d.get("target") is not None
    if w2_layout == "rv":
        d["W2"] = d["W2"].t().contiguous()
    ws = ds.Workspace(1 if rnn else 0, wl.B, wl.gamma, wl.V, wl.r, wl.d, target=has_t,
                      w2_layout=w2_layout)
    kw = dict(T=wl.T, seed=wl.seed, w=d["w"], target=d.get("target"), workspace=ws,
              w2_layout=w2_layout)
    if rnn:
        call = lambda **k: ds.rnn_draft(d["W1"], d["W2"], d["Wj"], d["U"], d["h"], d["x0"],
                                        s0=d.get("s0"), **kw, **k)
    else:
        call = lambda **k: ds.markov_draft(d["W1"], d["W2"], d["U"], d["x0"], h=d["h"], **kw, **k)
    ties = 0
    if check_free:
        free = call()
        torch.cuda.synchronize()
        assert ws.status() == 0
        ties += check_tokens_free(_rows(free.tokens, rows), o)
    forced = np.zeros((wl.B, wl.gamma), np.int32)
    forced[rows if rows is not None else slice(None)] = o.tokens
    tf = call(forced=torch.from_numpy(forced).cuda(), want_logits=want_logits)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ties += check_tokens_forced(_rows(tf.tokens, rows), o)
    errs = compare_floats(tf, o, rows=rows, logits=want_logits, z_rows=z_rows)
    print(f"{wl.name} B={wl.B} V={wl.V} r={wl.r} W2 {w2_layout}: near-ties {ties}, max errors {errs}")
    return ties, errs
