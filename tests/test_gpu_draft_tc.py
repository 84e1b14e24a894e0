"""GPU parity of the tensor-core draft path (bf16 weights, B > 4) against the fp64 oracle.

Same rules as the small-batch tests: tokens bit-exact up to counted near-ties, floats within
2e-3.  Cases cover one and several 128-request chunks, ragged vocabularies (a partial last
tile, slices of unequal tile counts), ranks that are not a multiple of the 64-wide K slab,
the Eq 8 target path, and the full Qwen3-8B-with-labels and
high-concurrency workloads on sampled requests.
"""
import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from semi_autoregressive_drafting_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

BASE = inputs.WORKLOADS["qwen3_4b_markov"]


def _run(wl, **kw):
    assert ds.draft_path(0, wl.B, wl.V, wl.r, wl.dtype == "bf16") == 1
    return parity.run_case(wl, ds=ds, **kw)


# W2 as the pages write it ([r][V], an MN-major operand) or as a linear layer's weight ([V][r],
# K-major); [r][V] needs V a multiple of 8 on this path, so its ragged cases use V = 20008
LAYOUTS = ["vr", "rv"]


@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("B", [5, 8, 64])
def test_tc_small_vocab(B, lay):
    _run(BASE.with_(B=B, V=9000, d=256, seed=60 + B), w2_layout=lay)


@pytest.mark.parametrize("lay,V", [("vr", 20001), ("rv", 20008)])
def test_tc_two_chunks_ragged_vocab(lay, V):
    _run(BASE.with_(B=130, V=V, d=128, seed=70), want_logits=False, w2_layout=lay)


@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("r", [64, 192, 512])
def test_tc_ranks(r, lay):
    _run(BASE.with_(B=16, V=12000, r=r, d=64, seed=80 + r // 64), w2_layout=lay)


@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("r", [64, 192, 512])
def test_tc_unpacked_ranks(r, lay):
    # more than 64 requests: unpacked tiles, one to eight 64-wide K blocks per A slab
    _run(BASE.with_(B=80, V=12000, r=r, d=64, seed=84 + r // 64), w2_layout=lay)


@pytest.mark.parametrize("lay", LAYOUTS)
def test_tc_unpacked_target_labels(lay):
    _run(BASE.with_(B=96, V=30000, d=256, T=0.8, seed=92), target_noise=1.0, w2_layout=lay)


@pytest.mark.parametrize("lay", LAYOUTS)
def test_tc_target_labels(lay):
    _run(BASE.with_(B=24, V=30000, d=256, T=0.8, seed=90), target_noise=1.0, w2_layout=lay)


def test_tc_rv_needs_16_byte_rows():
    # [r][V] with V not a multiple of 8 cannot be tiled by TMA: rejected on the host
    wl = BASE.with_(B=8, V=9001, d=64, seed=95)
    t = parity.to_dev(inputs.generate(wl))
    with pytest.raises(ds._lib.DsparkError, match="multiple of 8"):
        ds.markov_draft(t["W1"], t["W2"].t().contiguous(), t["U"], t["x0"], h=t["h"], w=t["w"],
                        w2_layout="rv")


def test_tc_invalid_anchor_and_repeatability():
    wl = BASE.with_(B=12, V=5000, d=64, seed=91)
    t = parity.to_dev(inputs.generate(wl))
    x0 = t["x0"].clone()
    x0[5] = -3
    ws = ds.Workspace(0, wl.B, wl.gamma, wl.V, wl.r, wl.d)
    out = ds.markov_draft(t["W1"], t["W2"], t["U"], x0, h=t["h"], w=t["w"], seed=3, workspace=ws)
    assert ws.status() == 1
    tok = out.tokens.cpu().numpy()
    assert np.all(tok[5] == -1) and np.all(np.delete(tok, 5, axis=0) >= 0)
    a = ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], h=t["h"], w=t["w"], seed=3, workspace=ws)
    b = ds.markov_draft(t["W1"], t["W2"], t["U"], t["x0"], h=t["h"], w=t["w"], seed=3, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    for f in ("tokens", "lse", "c", "S"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def sampled_rows(B, n=32, seed=0):
    """n distinct requests of B: the first and last, the rest drawn at random (sorted)."""
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, B - 1), size=min(n, B) - 2, replace=False)
    return sorted({0, B - 1, *mid.tolist()})


@pytest.mark.slow
@pytest.mark.parametrize("lay", LAYOUTS)
def test_qwen3_8b_labels_full_sampled_rows(lay):
    # the whole workload on the GPU, in the configuration the benchmark times; 32 of its 64
    # requests compared with the oracle (tokens, lse, c, S, c*, l1), z element-wise on two
    wl = inputs.WORKLOADS["qwen3_8b_labels"]
    rows = sampled_rows(wl.B, seed=3)
    ties, _ = _run(wl, rows=rows, z_rows=[rows[0], rows[-1]], w2_layout=lay)
    assert ties <= 2


@pytest.mark.slow
@pytest.mark.parametrize("lay", LAYOUTS)
def test_high_concurrency_full_sampled_rows(lay):
    # 32 of the 512 requests (all four 128-request chunks), z element-wise on two
    wl = inputs.WORKLOADS["high_concurrency_sched"]
    rows = sampled_rows(wl.B, seed=4)
    assert len({r // 128 for r in rows}) == 4
    ties, _ = _run(wl, rows=rows, z_rows=[rows[1], rows[-1]], w2_layout=lay)
    assert ties <= 2


@pytest.mark.parametrize("B,G", [(64, 15), (130, 15)])
def test_tc_gamma15(B, G):
    # the longer draft length the pages also evaluate ("DSpark：既要猜得连贯…", Results: gamma 15)
    _run(BASE.with_(B=B, gamma=G, V=12000, d=128, seed=110 + B), want_logits=False,
         target_noise=1.0 if B == 64 else None)


@pytest.mark.parametrize("B,V,lay", [(37, 40000, "vr"), (64, 38537, "vr"), (6, 2000, "vr"),
                                     (37, 40000, "rv"), (64, 38536, "rv")])
def test_tc_paired_tiles(B, V, lay):
    # at most 64 requests: vocabulary tiles go in pairs (lanes 64-127 hold the second tile);
    # blocks with an odd tile count end with a single-tile round
    _run(BASE.with_(B=B, V=V, d=128, seed=100 + B), target_noise=0.5 if B == 37 else None,
         w2_layout=lay)
