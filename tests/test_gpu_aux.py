"""GPU parity of the per-round kernels against the oracle: teacher-forced confidence (Eq 7,
S_k), the Eq 8 label on independent rows, and the prefix scheduler (bit-exact lengths and
Theta on the same S input)."""
import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from oracle import oracle
from semi_autoregressive_drafting_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_markov", "qwen3_4b_markov"])
def test_confidence(name):
    wl = inputs.WORKLOADS[name].with_(B=8, V=3000, seed=50)
    t = inputs.generate(wl)
    g = torch.Generator().manual_seed(1)
    tokens = torch.randint(0, wl.V, (wl.B, wl.gamma), generator=g, dtype=torch.int32)
    O = inputs.to_oracle
    c_ref, S_ref, st = oracle.confidence(B=wl.B, gamma=wl.gamma, V=wl.V, r=wl.r, d=wl.d,
                                         W1=O(t["W1"]), h=O(t["h"]), w=O(t["w"]), x0=O(t["x0"]),
                                         tokens=tokens.numpy())
    d = parity.to_dev(t)
    c, S = ds.confidence(d["W1"], d["w"], d["h"], d["x0"], tokens.cuda())
    parity.close("c", c.cpu().numpy(), c_ref)
    parity.close("S", S.cpu().numpy(), S_ref)
    assert np.all(np.diff(S.cpu().numpy(), axis=1) <= 0)


def test_confidence_bad_token_is_nan():
    wl = inputs.WORKLOADS["tiny_markov"].with_(seed=51)
    d = parity.to_dev(inputs.generate(wl))
    tokens = torch.zeros(wl.B, wl.gamma, dtype=torch.int32, device="cuda")
    tokens[2, 3] = wl.V
    c, S = ds.confidence(d["W1"], d["w"], d["h"], d["x0"], tokens)
    c = c.cpu().numpy()
    assert np.all(np.isnan(c[2, 4:])) and not np.any(np.isnan(c[2, :4]))
    assert not np.any(np.isnan(np.delete(c, 2, axis=0)))


@pytest.mark.parametrize("N,V,T", [(5, 7, 1.0), (33, 4096, 0.8), (4, 151936, 1.0)])
def test_tv_label(N, V, T):
    g = torch.Generator().manual_seed(V)
    dl = torch.randn(N, V, generator=g) * 3
    tl = dl + torch.randn(N, V, generator=g)
    dl[0] = 0.0
    tl[0] = 0.0                        # identical rows: c* = 1
    cs_ref, l1_ref = oracle.tv_label(dl.numpy(), tl.numpy(), T=T)
    cs, l1 = ds.tv_label(dl.cuda(), tl.cuda(), T=T)
    parity.close("cstar", cs.cpu().numpy(), cs_ref)
    parity.close("l1", l1.cpu().numpy(), l1_ref)
    assert abs(cs[0].item() - 1.0) < 1e-6


@pytest.mark.parametrize("B,G", [(1, 1), (3, 7), (64, 7), (512, 7), (128, 15), (1000, 16)])
def test_prefix_schedule_bit_exact(B, G):
    rng = np.random.default_rng(B * 31 + G)
    c = rng.uniform(0.02, 0.999, (B, G))
    S = np.cumprod(c, axis=1).astype(np.float32)
    S[0] = S[0, 0]                     # equal values inside a row: ties to smaller k
    sps = inputs.sps_table(B, G).numpy()
    ln_ref, th_ref, st = oracle.prefix_schedule(S, sps)
    assert st == 0
    ln, th = ds.prefix_schedule(torch.from_numpy(S).cuda(), torch.from_numpy(sps).cuda())
    assert np.array_equal(ln.cpu().numpy(), ln_ref)
    assert th.item() == th_ref          # bit-exact


@pytest.mark.parametrize("B,G", [(512, 7), (40, 3), (2048, 8)])
def test_prefix_schedule_ties_bit_exact(B, G):
    # S on a coarse grid: many equal values across requests and positions, so the order of
    # equal keys (position, then request) decides which prefixes are taken
    rng = np.random.default_rng(B + 7 * G)
    c = rng.choice([0.5, 0.75, 1.0], size=(B, G))
    S = np.cumprod(c, axis=1).astype(np.float32)
    sps = inputs.sps_table(B, G).numpy()
    ln_ref, th_ref, st = oracle.prefix_schedule(S, sps)
    assert st == 0
    ln, th = ds.prefix_schedule(torch.from_numpy(S).cuda(), torch.from_numpy(sps).cuda())
    assert np.array_equal(ln.cpu().numpy(), ln_ref)
    assert th.item() == th_ref


def test_prefix_schedule_rejects_increasing_S():
    S = torch.tensor([[0.5, 0.6], [0.4, 0.3]], device="cuda")
    sps = torch.ones(7, dtype=torch.float64, device="cuda")
    ln, th = ds.prefix_schedule(S, sps)
    assert np.all(ln.cpu().numpy() == -1) and np.isnan(th.item())
