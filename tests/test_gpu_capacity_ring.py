"""The scheduler's two-step-delayed capacity input, run on the GPU.

"DSpark：既要猜得连贯…" (设计) says the production prefix scheduler reads a capacity estimate
(steps/s at n verify tokens) that is two steps old, so that scheduling can run ahead
asynchronously and inside CUDA Graphs.  Here every step t draws a fresh prefix-survival matrix
S_t and a fresh steps/s table sps_t; ``CapacityRing.advance(sps_t)`` records the table and puts
the one from step t - 2 in its fixed ``table`` buffer, and ``prefix_schedule`` reads that buffer.
The lengths and Theta must equal, bit for bit, the oracle's schedule of S_t on sps_{t-2} (on
the initial table while t < 2).  The tables are drawn so that the delay changes the schedule:
the oracle's schedule on sps_{t-1} or sps_t differs from it at some step.
"""
import numpy as np
import pytest
import torch

import semi_autoregressive_drafting_gb300 as ds
from oracle import oracle
from semi_autoregressive_drafting_gb300 import inputs

pytestmark = pytest.mark.gpu

STEPS = 8
DELAY = 2


def _steps(B, G, seed):
    """Per step: S_t [B][G] fp32 (non-increasing rows) and sps_t [B(G+1)+1] fp64."""
    rng = np.random.default_rng(seed)
    n = np.arange(B * (G + 1) + 1, dtype=np.float64)
    out = []
    for t in range(STEPS):
        c = rng.uniform(0.3, 0.995, (B, G))
        S = np.cumprod(c, axis=1).astype(np.float32)
        # the engine's capacity knee moves from step to step (a load change)
        knee = B * (G + 1) * rng.uniform(0.05, 0.6)
        sps = 2000.0 / (1.0 + n / knee)
        out.append((S, sps))
    return out


def _expected(steps, init):
    exp, other = [], []
    for t, (S, _) in enumerate(steps):
        table = steps[t - DELAY][1] if t >= DELAY else init
        ln, th, st = oracle.prefix_schedule(S, table)
        assert st == 0
        exp.append((ln, th))
        # the schedule the same S would get from a table that is not delayed by two steps
        wrong = steps[t - 1][1] if t >= 1 else steps[t][1]
        other.append(oracle.prefix_schedule(S, wrong)[:2])
    return exp, other


@pytest.mark.parametrize("B,G", [(64, 7), (512, 7), (96, 15)])
def test_schedule_reads_the_table_from_two_steps_back(B, G):
    steps = _steps(B, G, seed=B + G)
    init = inputs.sps_table(B, G).numpy()
    exp, other = _expected(steps, init)
    assert any(not np.array_equal(e[0], o[0]) for e, o in zip(exp, other)), \
        "inputs do not discriminate the delay"
    ring = ds.CapacityRing(torch.from_numpy(init).cuda(), delay=DELAY)
    for t, (S, sps) in enumerate(steps):
        table = ring.advance(torch.from_numpy(sps).cuda())
        ln, th = ds.prefix_schedule(torch.from_numpy(S).cuda(), table)
        assert np.array_equal(ln.cpu().numpy(), exp[t][0]), f"step {t}: lengths differ"
        assert th.item() == exp[t][1], f"step {t}: Theta differs"


def test_schedule_replayed_from_a_cuda_graph():
    # the scheduler call is captured once, reading the ring's fixed table buffer and a fixed S
    # buffer; each step refreshes S, advances the ring (stream-ordered copies) and replays it
    B, G = 128, 7
    steps = _steps(B, G, seed=7)
    init = inputs.sps_table(B, G).numpy()
    exp, _ = _expected(steps, init)
    ring = ds.CapacityRing(torch.from_numpy(init).cuda(), delay=DELAY)
    S_buf = torch.from_numpy(steps[0][0]).cuda()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        ds.prefix_schedule(S_buf, ring.table, stream=stream)  # warm-up outside the capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ln_g, th_g = ds.prefix_schedule(S_buf, ring.table, stream=stream)
    for t, (S, sps) in enumerate(steps):
        with torch.cuda.stream(stream):
            S_buf.copy_(torch.from_numpy(S), non_blocking=False)
            ring.advance(torch.from_numpy(sps).cuda())
            graph.replay()
        stream.synchronize()
        assert np.array_equal(ln_g.cpu().numpy(), exp[t][0]), f"step {t}: lengths differ"
        assert th_g.item() == exp[t][1], f"step {t}: Theta differs"
