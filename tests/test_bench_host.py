"""Host-side arithmetic of bench.py: the algorithmic bytes behind every roofline fraction, and
the DRAM-traffic records (no GPU)."""
import os
import re

import pytest

import bench
from semi_autoregressive_drafting_gb300 import inputs

# MB per draft step: W2 once, U_k once, the target once (labelled workload), the gathered W1
# rows and h_k, and Wj for the RNN head
PER_STEP_MB = {"tiny_markov": 1.12, "qwen3_4b_markov": 78.10, "qwen3_8b_labels": 136.69,
               "high_concurrency_sched": 406.85, "rnn_head": 126.72}


@pytest.mark.parametrize("name", sorted(PER_STEP_MB))
def test_algorithmic_bytes_per_step(name):
    wl = inputs.WORKLOADS[name]
    per_block = bench.algorithmic_bytes(wl)
    assert per_block / wl.gamma / 1e6 == pytest.approx(PER_STEP_MB[name], abs=0.01)


def test_qwen3_4b_bytes_by_hand():
    wl = inputs.WORKLOADS["qwen3_4b_markov"]
    V, r, d, G = 151936, 256, 2560, 7
    assert (wl.V, wl.r, wl.d, wl.gamma, wl.B, wl.dtype) == (V, r, d, G, 1, "bf16")
    step = V * r * 2 + V * 2 + r * 2 + d * 2  # W2, U_k, one W1 row, h_k (bf16)
    assert bench.algorithmic_bytes(wl) == G * step + (d + r) * 2  # + the confidence weight w


def test_traffic_records_name_existing_sources():
    csrc = os.path.join(bench.ROOT, "semi_autoregressive_drafting_gb300", "csrc")
    for key, (src, sha, nbytes) in bench.TRAFFIC.items():
        assert os.path.exists(os.path.join(csrc, src)), key
        assert re.fullmatch(r"[0-9a-f]{16}", sha), key
        assert isinstance(nbytes, int) and nbytes > 0, key
        assert key.split()[-1] in inputs.WORKLOADS, key
