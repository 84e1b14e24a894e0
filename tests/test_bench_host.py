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


def test_default_workload_is_the_largest_single_gpu_config():
    # the high-concurrency tensor-core regime: B = 512, V = 262144
    args = bench.build_parser().parse_args([])
    wl = inputs.WORKLOADS[args.workload]
    assert args.workload == "high_concurrency_sched"
    assert (wl.B, wl.gamma, wl.V, wl.r) == (512, 7, 262144, 256)
    assert all(bench.algorithmic_bytes(w) <= bench.algorithmic_bytes(wl)
               for w in inputs.WORKLOADS.values())


def test_algorithmic_flops_by_hand():
    wl = inputs.WORKLOADS["high_concurrency_sched"]
    assert bench.algorithmic_flops(wl) == 2 * 512 * 256 * 262144 * 7  # 481 GFLOP per block
    rnn = inputs.WORKLOADS["rnn_head"]
    B, r, V, d, G = 128, 256, 151936, 5120, 7
    assert bench.algorithmic_flops(rnn) == G * (2 * B * r * V + 2 * B * 3 * r * (2 * r + d))


def test_every_workload_names_its_limiter():
    for name in inputs.WORKLOADS:
        assert bench.LIMITER.get(name), name


def test_clock_summary_from_nvml_samples():
    c = bench.ClockSampler(0)
    c.samples = [(2070.0, 0), (2055.0, 0x4), (2070.0, 0x1)]
    c.smax = 2070.0
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]  # idle (0x1) is not a throttle reason


def test_shape_override_renames_and_resizes():
    wl = bench.override_shape(inputs.WORKLOADS["high_concurrency_sched"], "V=65536,d=512")
    assert (wl.B, wl.V, wl.d, wl.r) == (512, 65536, 512, 256)
    assert wl.name == "high_concurrency_sched[V=65536,d=512]"
    assert wl.name not in bench.TRAFFIC  # a resized case carries no traffic record
    assert bench.override_shape(wl, "") is wl
    with pytest.raises(SystemExit):
        bench.override_shape(wl, "T=2")
