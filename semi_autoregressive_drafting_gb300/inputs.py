"""Seeded synthetic inputs for the draft-sampling path.

This module only draws random tensors with the shapes and value distributions of the five
workloads below; it holds none of the method's arithmetic.  The tests and the benchmark feed
the same bytes to the CUDA library and to the CPU oracle.

Workloads (the drafter models of the DSpark pages: Qwen3 vocabularies of 151936 entries,
block size gamma = 7, Markov rank r = 256; the 262144-entry vocabulary is the high-concurrency
shape):

=========================  ====  =====  ======  ===  ====  =====================================
name                       B     gamma  V       r    d     notes
=========================  ====  =====  ======  ===  ====  =====================================
tiny_markov                4     7      4096    64   256   all fp32; U~N(0,2^2), W~N(0,0.05^2)
qwen3_4b_markov            1     7      151936  256  2560  bf16; U~N(0,3^2), W,w~N(0,0.02^2)
qwen3_8b_labels            64    7      151936  256  4096  + fp32 target = U + N(0,1) noise
high_concurrency_sched     512   7      262144  256  3840  + steps/s table 2000/(1+n/4096)
rnn_head                   128   7      151936  256  5120  RNN head, Wj [3r][2r+d] ~N(0,0.02^2)
=========================  ====  =====  ======  ===  ====  =====================================

h ~ N(0, 1) everywhere, anchors x0 uniform in [0, V), T = 1.0.  Seeds are 0..4 in table order.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    head: str            # "markov" or "rnn"
    B: int
    gamma: int
    V: int
    r: int
    d: int
    dtype: str           # "f32" or "bf16" for weights, U and h
    U_std: float
    W_std: float
    w_std: float
    h_std: float = 1.0
    T: float = 1.0
    seed: int = 0
    target_noise: float | None = None   # target = U + N(0, noise^2) in fp32 when set
    sched: bool = False                 # emit the steps/s table for the prefix scheduler

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_markov", "markov", 4, 7, 4096, 64, 256, "f32", 2.0, 0.05, 0.05, seed=0),
        Workload("qwen3_4b_markov", "markov", 1, 7, 151936, 256, 2560, "bf16", 3.0, 0.02, 0.02,
                 seed=1),
        Workload("qwen3_8b_labels", "markov", 64, 7, 151936, 256, 4096, "bf16", 3.0, 0.02, 0.02,
                 seed=2, target_noise=1.0),
        Workload("high_concurrency_sched", "markov", 512, 7, 262144, 256, 3840, "bf16", 3.0,
                 0.02, 0.02, seed=3, sched=True),
        Workload("rnn_head", "rnn", 128, 7, 151936, 256, 5120, "bf16", 3.0, 0.02, 0.02, seed=4),
    ]
}


def sps_table(B: int, gamma: int) -> torch.Tensor:
    """Synthetic verify-engine capacity: steps/s at n verify tokens, n = 0..B*(gamma+1)."""
    n = torch.arange(B * (gamma + 1) + 1, dtype=torch.float64)
    return 2000.0 / (1.0 + n / 4096.0)


def _randn(g: torch.Generator, shape, std: float, dtype: torch.dtype, chunk: int = 1 << 24):
    """N(0, std^2) draws, generated in fp32 in chunks (bounded host memory), cast to dtype."""
    numel = int(np.prod(shape))
    out = torch.empty(numel, dtype=dtype)
    for s in range(0, numel, chunk):
        e = min(numel, s + chunk)
        out[s:e] = (torch.randn(e - s, generator=g, dtype=torch.float32) * std).to(dtype)
    return out.view(*shape)


def generate(wl: Workload) -> dict:
    """Host (CPU) tensors for one workload.  Same seed, same bytes, on every machine."""
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    B, G, V, r, d = wl.B, wl.gamma, wl.V, wl.r, wl.d
    t = {}
    t["W1"] = _randn(g, (V, r), wl.W_std, dt)
    t["W2"] = _randn(g, (V, r), wl.W_std, dt)
    t["Wj"] = _randn(g, (3 * r, 2 * r + d), wl.W_std, dt) if wl.head == "rnn" else None
    t["w"] = _randn(g, (d + r,), wl.w_std, dt)
    t["U"] = _randn(g, (B, G, V), wl.U_std, dt)
    t["h"] = _randn(g, (B, G, d), wl.h_std, dt)
    t["x0"] = torch.randint(0, V, (B,), generator=g, dtype=torch.int32)
    if wl.target_noise is not None:
        t["target"] = t["U"].float() + _randn(g, (B, G, V), wl.target_noise, torch.float32)
    else:
        t["target"] = None
    t["sps"] = sps_table(B, G) if wl.sched else None
    return t


def to_oracle(x: torch.Tensor | None):
    """numpy view of a host tensor in the oracle's convention (bf16 as raw uint16)."""
    if x is None:
        return None
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


def verify_inputs(B: int, gamma: int, V: int, *, seed: int, logit_std: float = 3.0,
                  target_noise: float = 1.0, tokens: str = "uniform") -> dict:
    """Host tensors for the verify step: draft logits [B, gamma, V] ~ N(0, logit_std^2) fp32,
    target logits [B, gamma + 1, V] fp32 (the first gamma rows = draft + N(0, target_noise^2),
    the bonus row ~ N(0, logit_std^2)), and drafted tokens [B, gamma] int32: uniform in [0, V)
    ("uniform") or each row's largest draft logit ("argmax", a high-acceptance stand-in)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    zd = _randn(g, (B, gamma, V), logit_std, torch.float32)
    zt = torch.empty(B, gamma + 1, V, dtype=torch.float32)
    zt[:, :gamma] = zd + _randn(g, (B, gamma, V), target_noise, torch.float32)
    zt[:, gamma] = _randn(g, (B, V), logit_std, torch.float32)
    if tokens == "uniform":
        x = torch.randint(0, V, (B, gamma), generator=g, dtype=torch.int32)
    elif tokens == "argmax":
        x = zd.argmax(dim=2).to(torch.int32)
    else:
        raise ValueError(tokens)
    return {"draft_logits": zd, "target_logits": zt.contiguous(), "draft_tokens": x}
