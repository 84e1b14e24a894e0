#!/usr/bin/env python3
"""Benchmark of libdspark's draft-sampling hot path on GB300.

One step = one draft block (all gamma positions) of the workload: W1 gather, bias product,
logits, temperature softmax normaliser, Philox Gumbel-max sampling, Eq 7 confidence and the
prefix survival, all in libdspark's kernels.  The default workload is the largest one that
fits one GPU, the high-concurrency tensor-core regime (B=512, gamma=7, V=262144, r=256,
d=3840, bf16); ``--workload`` picks another (qwen3_4b_markov is the B=1 latency regime).  The
metric is draft tokens/s (B * gamma per block), plus the achieved HBM bandwidth of the draft
call against the measured copy bandwidth and, on the tensor-core paths, the bias product's
bf16 throughput against the measured cuBLAS burst peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload W]

With N > 1 (torchrun), every rank drafts its own independent requests (weak scaling, no
collective on the data path); value = all ranks' tokens / the slowest rank's time.
``--impl reference`` times the CPU oracle (the plain fp64 restatement of the pages' equations)
on the host cores, one draft position over the full vocabulary per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft tokens/sec (B×γ per block) and achieved HBM GB/s vs roofline, 1 GB300"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20   # > 129 MB L2: every timed block starts with a cold L2

# ncu DRAM traffic (read + write bytes) of one draft-kernel launch per workload: the kernel's
# source file, the sha256 prefix of the source it was measured on, and the bytes.  A workload
# without a capture, or whose kernel changed since, reports null.
TRAFFIC = {
    "qwen3_4b_markov": ("draft_cc.cu", "cb8724e6c2d82289", 81708288),           # 80.61 + 1.10 MB
    "tiny_markov": ("draft_cc.cu", "cb8724e6c2d82289", 2332160),                # 2.33 + 0 MB
    "high_concurrency_sched": ("draft_tc.cu", "ec52e23d3affb2df", 2411139584),  # 2407 + 4.2 MB
    # draft_tc_kernel alone; the target's normalisers (272.4 MB) are a launch before it
    "qwen3_8b_labels": ("draft_tc.cu", "ec52e23d3affb2df", 628756992),         # 607.2 + 21.5 MB
    "rnn_head": ("draft_tc.cu", "ec52e23d3affb2df", 528002048),                 # 523.2 + 4.8 MB
    # the three verify kernels of one call (bench.py --op verify)
    "verify qwen3_8b_labels": ("verify.cu", "c5b18516acacc741", 661831424),
    # the four loss kernels of one call (bench.py --op loss)
    "loss qwen3_8b_labels": ("loss.cu", "4c19b76551491e6e", 1871557376),
}


def ranks_max(dist, values, device="cuda"):
    """Each timing's maximum over the ranks (the slowest replica sets the job's time); the
    values unchanged on one process (dist None)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput: every rank processes units_per_rank units per step of ms."""
    return world * units_per_rank / (ms * 1e-3)


def _sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def algorithmic_bytes(wl) -> int:
    """What one block must move: per step W2 once, U_k once, the target once, the gathered W1
    rows and h_k; once per block the confidence weight w; outputs are negligible."""
    es_w = 4 if wl.dtype == "f32" else 2
    es_u = es_w
    per_step = wl.V * wl.r * es_w + wl.B * wl.V * es_u + wl.B * wl.r * es_w + wl.B * wl.d * es_u
    if wl.target_noise is not None:
        per_step += wl.B * wl.V * 4
    if wl.head == "rnn":
        per_step += 3 * wl.r * (2 * wl.r + wl.d) * es_w
    return wl.gamma * per_step + (wl.d + wl.r) * es_w


def packed(specs, device):
    """One buffer holding the arrays (name, shape, dtype) at 256-byte aligned offsets, pinned
    when on the host; returns the flat uint8 buffer and the named views."""
    import torch

    offs, o = {}, 0
    for name, shape, dt in specs:
        n = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
        offs[name] = (o, n)
        o = (o + n + 255) // 256 * 256
    buf = (torch.empty(o, dtype=torch.uint8, pin_memory=True) if device == "cpu"
           else torch.empty(o, dtype=torch.uint8, device=device))
    views = {name: buf[a:a + n].view(dt).view(shape)
             for (name, shape, dt), (a, n) in zip(specs, offs.values())}
    return buf, views


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_tensor_peak():
    """Measured dense bf16 throughput (cuBLAS burst: the draft call is timed on its own)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        if "bf16_tflops" in j:
            return float(j["bf16_tflops"]), "measured cuBLAS bf16 burst"
    return 1900.0, "fallback bf16 burst"


def algorithmic_flops(wl) -> int:
    """Dense multiply-adds of one block, 2 flops each: the bias product e W2^T (B x r x V per
    step) and, for the RNN head, the joint projection Wj z_k (B x 3r x (2r + d) per step)."""
    per_step = 2 * wl.B * wl.r * wl.V
    if wl.head == "rnn":
        per_step += 2 * wl.B * 3 * wl.r * (2 * wl.r + wl.d)
    return wl.gamma * per_step


# What limits each workload's draft call, from its ncu captures (profiles/).  The roofline's
# "bound" is the roof the call's arithmetic intensity puts it under (HBM for every workload:
# the B = 512 bias product has about 169 flop/B against a ridge near 285); "limiter" names what
# the counters show actually sets the time.
LIMITER = {
    "qwen3_4b_markov": "latency of the gamma - 1 sequential grid steps: W2 stays in TMEM and L2 "
                       "across steps, so DRAM moves about 0.15x the algorithmic bytes "
                       "(profiles/draft_cc_qwen3_4b_markov.md)",
    "high_concurrency_sched": "instruction issue in the epilogue: Philox noise, the normaliser "
                              "and the exact skip test for every (request, vocabulary entry) "
                              "(profiles/draft_tc_high_concurrency_sched.md)",
    "qwen3_8b_labels": "instruction issue in the epilogue plus the Eq 8 second pass "
                       "(profiles/draft_tc_qwen3_8b_labels.md)",
    "rnn_head": "instruction issue in the epilogue and the request owners' recurrent update "
                "(profiles/draft_tc_rnn_head.md)",
    "tiny_markov": "launch and grid-step latency (1.1 MB per step)",
}


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, sampled while the timed region
    runs.  NVML's read-only queries are polled every 2 ms from a host thread (a timed region of a
    few tens of milliseconds still gets samples); without NVML, nvidia-smi every 200 ms.  The
    first sample is taken before __enter__ returns, so the samples cover the whole region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.index = index
        self.period = period_s
        self.proc = None
        self.lines = []
        self.samples = []      # (sm_mhz, reason bits) from NVML
        self.smax = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None

    # ---- NVML (libnvidia-ml, part of the driver), read-only queries
    def _nvml_open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None
        dev = ctypes.c_void_p()
        handle_ok = False
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.index).uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            handle_ok = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(dev)) == 0
        except Exception:
            handle_ok = False
        if not handle_ok and nv.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(dev)) != 0:
            return None
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.smax = float(mx.value)
        return nv, dev, reasons_fn

    def _nvml_sample(self, nv, dev, reasons_fn):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk)) != 0:
            return
        if reasons_fn(dev, ctypes.byref(rs)) != 0:
            rs.value = 0
        self.samples.append((float(clk.value), int(rs.value)))

    def _nvml_loop(self, h):
        while not self._stop.is_set():
            self._nvml_sample(*h)
            time.sleep(self.period)

    def __enter__(self):
        h = None
        try:
            h = self._nvml_open()
        except (OSError, AttributeError):
            h = None
        if h is not None:
            self.source = f"nvml every {self.period * 1e3:.0f} ms"
            self._nvml_sample(*h)
            self._thread = threading.Thread(target=self._nvml_loop, args=(h,), daemon=True)
            self._thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thread = threading.Thread(target=self._read, daemon=True)
            self._thread.start()
            self.source = "nvidia-smi every 200 ms"
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], self.smax, set()
        for mhz, bits in self.samples:
            sm.append(mhz)
            for bit, name in self.REASONS.items():
                if bits & bit:
                    reasons.add(name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


REFERENCE_BUDGET_S = 150.0  # the whole reference run (warm-up and timed steps) stays within this


def run_reference(args, wl):
    """CPU oracle, one draft position over the full vocabulary per step, for all B requests, or
    for the first Bs of them when all B would not let --steps K --warmup W finish within
    REFERENCE_BUDGET_S (sized from one probe step; the rate is per request, so it compares)."""
    import numpy as np

    from oracle import oracle
    from semi_autoregressive_drafting_gb300 import inputs

    t = inputs.generate(wl)
    O = inputs.to_oracle
    cores = os.cpu_count() or 1
    U = O(t["U"])
    h = O(t["h"])
    x0 = O(t["x0"])
    W1, W2, Wj, w = O(t["W1"]), O(t["W2"]), O(t.get("Wj")), O(t["w"])
    sps = t["sps"].numpy() if t["sps"] is not None else None

    cs = []

    def one(k, nb):
        o = oracle.draft(head=0 if wl.head == "markov" else 1, B=nb, gamma=1, V=wl.V,
                         r=wl.r, d=wl.d, T=wl.T, seed=wl.seed, W1=W1, W2=W2, Wj=Wj,
                         U=np.ascontiguousarray(U[:nb, k:k + 1]), x0=np.ascontiguousarray(x0[:nb]),
                         h=np.ascontiguousarray(h[:nb, k:k + 1]), w=w, nthreads=cores)
        if sps is not None:  # the prefix schedule once gamma positions are in
            cs.append(o.c[:, 0])
            if len(cs) == wl.gamma:
                oracle.prefix_schedule(np.cumprod(np.stack(cs, 1), 1), sps)
                cs.clear()

    t0 = time.perf_counter()
    one(0, wl.B)  # probe step (also the first warm-up)
    per_req = (time.perf_counter() - t0) / wl.B
    nsteps = args.steps + max(0, args.warmup - 1)
    nb = int(max(1, min(wl.B, REFERENCE_BUDGET_S / max(nsteps, 1) / max(per_req, 1e-9))))
    for i in range(1, args.warmup):
        one(i % wl.gamma, nb)
    cs.clear()
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i % wl.gamma, nb)
    dt = time.perf_counter() - t0
    value = nb * args.steps / dt
    sample = (f"one draft position over the full vocabulary per step, for {nb} of the "
              f"{wl.B} requests" + (", the prefix schedule every gamma steps" if sps is not None else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "B": wl.B, "gamma": wl.gamma,
                                        "V": wl.V, "r": wl.r, "d": wl.d, "T": wl.T},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def cpu_baseline(wl, seconds: float = 15.0):
    """The oracle as it stands on the host cores, on whole draft positions of the workload."""
    import numpy as np

    from oracle import oracle
    from semi_autoregressive_drafting_gb300 import inputs

    t = inputs.generate(wl)
    O = inputs.to_oracle
    cores = os.cpu_count() or 1
    U, h = O(t["U"]), O(t["h"])
    n, nsched, cs, t0 = 0, 0, [], time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        k = n % wl.gamma
        o = oracle.draft(head=0 if wl.head == "markov" else 1, B=wl.B, gamma=1, V=wl.V, r=wl.r,
                         d=wl.d, T=wl.T, seed=wl.seed, W1=O(t["W1"]), W2=O(t["W2"]),
                         Wj=O(t.get("Wj")), U=np.ascontiguousarray(U[:, k:k + 1]),
                         x0=O(t["x0"]), h=np.ascontiguousarray(h[:, k:k + 1]), w=O(t["w"]),
                         nthreads=cores)
        n += 1
        if t["sps"] is not None:  # the block's prefix schedule, on the sampled positions' c
            cs.append(o.c[:, 0])
            if len(cs) == wl.gamma:
                oracle.prefix_schedule(np.cumprod(np.stack(cs, 1), 1), t["sps"].numpy())
                cs, nsched = [], nsched + 1
    dt = time.perf_counter() - t0
    sched = f", {nsched} prefix schedules" if t["sps"] is not None else ""
    return {"value": wl.B * n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} draft positions x B={wl.B} over the full vocabulary{sched} ({dt:.1f} s)"}

VERIFY_METRIC = "verified draft blocks/sec (B per call) and achieved HBM GB/s vs roofline, 1 GB300"


def run_verify(args, wl, rank, world, local_rank):
    """The speculative verify step on fp32 draft and target logits of the workload's shape."""
    import torch

    import semi_autoregressive_drafting_gb300 as ds
    from semi_autoregressive_drafting_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    B, G, V = wl.B, wl.gamma, wl.V
    host = inputs.verify_inputs(B, G, V, seed=wl.seed + 100 * rank, tokens="argmax")
    dev = {k: v.cuda() for k, v in host.items()}
    ws = ds.VerifyWorkspace(B, G, V)
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    toks = torch.empty(B, G + 1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def call(d):
        ds.verify(d["draft_logits"], d["target_logits"], d["draft_tokens"], T=wl.T, seed=wl.seed,
                  workspace=ws, stream=stream, out=(n, toks))

    for _ in range(args.warmup):
        flush.zero_()
        call(dev)
    torch.cuda.synchronize()
    assert ws.status() == 0, "verify reported a device error during warm-up"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            call(dev)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = sum(times) / len(times)
    assert ws.status() == 0, "verify reported a device error"
    # end to end: the logits and tokens copied in from pinned host memory, results copied out
    hin = {k: v.pin_memory() for k, v in host.items()}
    din = {k: torch.empty_like(v) for k, v in dev.items()}
    hn = torch.empty(B, dtype=torch.int32).pin_memory()
    ht = torch.empty(B, G + 1, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = hn.numel() * 4 + ht.numel() * 4

    def e2e_step():
        for k in din:
            din[k].copy_(hin[k], non_blocking=True)
        call(din)
        hn.copy_(n, non_blocking=True)
        ht.copy_(toks, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = min(args.steps, 50)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for _ in range(e2e_steps):
        flush.zero_()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= e2e_steps
    ms, e2e_ms = ranks_max(dist, [ms, e2e_ms])
    if rank == 0:
        peak, peak_kind = load_peaks()
        # what the step must move: every draft row and every target row once (the
        # normalisers), and the one drawn row per request (draft and target) again
        alg = (B * G * V + B * (G + 1) * V) * 4 + B * 2 * V * 4 + B * G * 4
        achieved = alg / (ms * 1e-3) / 1e9
        cap = TRAFFIC.get("verify " + wl.name)
        src = cap and os.path.join(ROOT, "semi_autoregressive_drafting_gb300", "csrc", cap[0])
        traffic = cap[2] if cap and _sha(src) == cap[1] else None
        line = {
            "metric": VERIFY_METRIC, "value": job_rate(world, B, ms), "unit": "blocks/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"verify {wl.name}", "B": B, "gamma": G, "V": V, "T": wl.T,
                       "tokens": "largest draft logit per position",
                       "l2": "flushed between timed calls (512 MB write)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": f"{peak_kind} copy bandwidth",
                         "algorithmic_bytes_per_launch": alg,
                         "kernel": "verify_part_kernel + verify_decide_kernel + verify_draw_kernel"},
            "e2e": {"value": job_rate(world, B, e2e_ms), "unit": "blocks/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 3 * args.steps,
            "clocks": clk.summary(),
            "ms_per_step_min": min(times), "ms_per_step_median": statistics.median(times),
            "accepted_mean": float(n.float().mean()),
        }
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


LOSS_METRIC = "loss+gradient draft blocks/sec (B per call) and achieved HBM GB/s vs roofline, 1 GB300"


def run_loss(args, wl, rank, world, local_rank):
    """Eqs 9-12 and their gradients on fp32 draft and target logits of the workload's shape."""
    import torch

    import semi_autoregressive_drafting_gb300 as ds

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    B, G, V = wl.B, wl.gamma, wl.V
    g = torch.Generator().manual_seed(wl.seed + 100 * rank)
    host = {"zd": torch.randn(B, G, V, generator=g) * wl.U_std}
    host["zt"] = host["zd"] + torch.randn(B, G, V, generator=g)
    host["lab"] = torch.randint(0, V, (B, G), generator=g, dtype=torch.int32)
    host["cf"] = torch.randn(B, G, generator=g)
    dev = {k: v.cuda() for k, v in host.items()}
    lib = ds._lib.load()
    ws = ds.LossWorkspace(B, G, V)
    loss = torch.empty(B, device="cuda")
    parts = torch.empty(B, 3, device="cuda")
    gz = torch.empty(B, G, V, device="cuda")
    gc = torch.empty(B, G, device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def call(d):
        code = lib.dspark_draft_loss(B, G, V, float(wl.T), d["zd"].data_ptr(), d["zt"].data_ptr(),
                                     d["lab"].data_ptr(), d["cf"].data_ptr(), 0.1, 0.9, 1.0,
                                     loss.data_ptr(), parts.data_ptr(), gz.data_ptr(),
                                     gc.data_ptr(), ws.buf.data_ptr(), ws.nbytes, stream.cuda_stream)
        assert code == 0, ds._lib.load().dspark_last_error()

    for _ in range(args.warmup):
        flush.zero_()
        call(dev)
    torch.cuda.synchronize()
    assert ws.status() == 0, "loss reported a device error during warm-up"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            call(dev)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = sum(times) / len(times)
    assert ws.status() == 0, "loss reported a device error"
    # end to end: logits, labels and confidence logits in from pinned host memory; the losses,
    # their parts and both gradients out
    hin = {k: v.pin_memory() for k, v in host.items()}
    din = {k: torch.empty_like(v) for k, v in dev.items()}
    hout = [torch.empty_like(t, device="cpu").pin_memory() for t in (loss, parts, gz, gc)]
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = sum(t.numel() * 4 for t in hout)

    def e2e_step():
        for k in din:
            din[k].copy_(hin[k], non_blocking=True)
        call(din)
        for h, t in zip(hout, (loss, parts, gz, gc)):
            h.copy_(t, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = min(args.steps, 30)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for _ in range(e2e_steps):
        flush.zero_()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= e2e_steps
    ms, e2e_ms = ranks_max(dist, [ms, e2e_ms])
    if rank == 0:
        peak, peak_kind = load_peaks()
        # the least the step must move: both logit arrays read once, the logit gradient written once
        alg = 3 * B * G * V * 4 + B * G * 4 * 3
        achieved = alg / (ms * 1e-3) / 1e9
        cap = TRAFFIC.get("loss " + wl.name)
        src = cap and os.path.join(ROOT, "semi_autoregressive_drafting_gb300", "csrc", cap[0])
        traffic = cap[2] if cap and _sha(src) == cap[1] else None
        line = {
            "metric": LOSS_METRIC, "value": job_rate(world, B, ms), "unit": "blocks/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"loss {wl.name}", "B": B, "gamma": G, "V": V, "T": wl.T,
                       "alpha": [0.1, 0.9, 1.0],
                       "l2": "flushed between timed calls (512 MB write)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": f"{peak_kind} copy bandwidth",
                         "algorithmic_bytes_per_launch": alg,
                         "kernel": "loss_part + loss_stat + loss_grad + loss_final"},
            "e2e": {"value": job_rate(world, B, e2e_ms), "unit": "blocks/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": ds.draft_loss_launches(B, G, V, True) * args.steps,
            "clocks": clk.summary(),
            "ms_per_step_min": min(times), "ms_per_step_median": statistics.median(times),
        }
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def build_parser():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="high_concurrency_sched")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--w2-layout", choices=["vr", "rv"], default="vr",
                    help="W2 as a linear layer's [V][r] weight (vr) or as the pages write it, "
                         "[r][V] (rv)")
    ap.add_argument("--op", choices=["draft", "verify", "loss"], default="draft",
                    help="draft: the draft block (default); verify: the speculative accept/reject "
                         "step on the workload's B, gamma, V; loss: the training losses (Eqs 9-12) "
                         "and their gradients on that shape")
    ap.add_argument("--shape", default="",
                    help="comma-separated overrides of the workload's sizes, e.g. "
                         "'V=65536,d=512': a smaller case of the same kernels for counter "
                         "captures; the workload name then carries the overrides")
    return ap


def override_shape(wl, spec):
    """The workload with the sizes in `spec` ('B=512,V=65536') replaced; its name records them."""
    if not spec:
        return wl
    kw = {}
    for item in spec.split(","):
        key, _, val = item.partition("=")
        if key not in ("B", "gamma", "V", "r", "d"):
            raise SystemExit(f"--shape: unknown size {key!r} (B, gamma, V, r, d)")
        kw[key] = int(val)
    return wl.with_(name=f"{wl.name}[{spec}]", **kw)


def main():
    args = build_parser().parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from semi_autoregressive_drafting_gb300 import inputs
    wl = override_shape(inputs.WORKLOADS[args.workload], args.shape)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return
    if args.op == "verify":
        run_verify(args, wl, rank, world, local_rank)
        return
    if args.op == "loss":
        run_loss(args, wl, rank, world, local_rank)
        return

    import torch

    import semi_autoregressive_drafting_gb300 as ds

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    host = inputs.generate(wl)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    if args.w2_layout == "rv":
        dev["W2"] = dev["W2"].t().contiguous()
    ws = ds.Workspace(0 if wl.head == "markov" else 1, wl.B, wl.gamma, wl.V, wl.r, wl.d,
                      target=wl.target_noise is not None, w2_layout=args.w2_layout)
    stream = torch.cuda.current_stream()
    B, G = wl.B, wl.gamma

    def plan(U, h, x0, target, out=None):
        return ds.DraftPlan(0 if wl.head == "markov" else 1, dev["W1"], dev["W2"], U, x0, T=wl.T,
                            seed=wl.seed, h=h, w=dev["w"], Wj=dev.get("Wj"), target=target,
                            forced=None, s0=None, want_logits=False, workspace=ws, stream=stream,
                            out=out, w2_layout=args.w2_layout)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    resident = plan(dev["U"], dev["h"], dev["x0"], dev.get("target"))
    # the batch prefix scheduler (the last step of the hot path) when the workload carries a
    # steps/s table: the verify lengths from the block's S, in the timed step
    conf = dev["h"] is not None and dev["w"] is not None
    sched = conf and dev.get("sps") is not None
    sl = torch.empty(B, dtype=torch.int32, device="cuda")
    sth = torch.empty(1, dtype=torch.float64, device="cuda")

    def schedule(p, s, out):
        if sched:
            ds.prefix_schedule(p.out.S, dev["sps"], stream=s, out=out)

    for _ in range(args.warmup):
        flush.zero_()
        resident.run()
        schedule(resident, stream, (sl, sth))
    torch.cuda.synchronize()
    assert ws.status() == 0, "draft kernel reported a device error during warm-up"

    # ---- device-resident timing: CUDA events around each step (the draft call, then the
    # scheduler when there is one, with one more event between them for the draft's own
    # roofline); L2 flushed between steps
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3 if sched else 2))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            resident.run()
            if sched:
                ev[i][1].record(stream)
                schedule(resident, stream, (sl, sth))
            ev[i][-1].record(stream)
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    times = [e[0].elapsed_time(e[-1]) for e in ev]   # ms per step (block, and schedule)
    ms_step = sum(times) / len(times)
    ms_draft = sum(e[0].elapsed_time(e[1]) for e in ev) / len(ev)  # the draft call alone
    assert ws.status() == 0, "draft kernel reported a device error"
    sched_ok = (not sched) or bool(((sl >= 0) & (sl <= G)).all())

    # ---- end to end through the public API: pinned host inputs in, results out, every step.
    # The step's inputs (U, h, x0 and the target) sit in one pinned host buffer and the results
    # (tokens, lse, c, S, c*, l1) in one device buffer, each array at a 256-byte aligned offset
    # (the draft call takes any aligned device pointers), so a step is one copy in, the draft
    # call and one copy out.  The weights stay resident on the device.
    names = ["U", "h", "x0"] + (["target"] if host.get("target") is not None else [])
    in_specs = [(k, tuple(host[k].shape), host[k].dtype) for k in names]
    hin_buf, hin = packed(in_specs, "cpu")
    din_buf, din = packed(in_specs, "cuda")
    for k in names:
        hin[k].copy_(host[k])
    out_specs = [("tokens", (B, G), torch.int32), ("lse", (B, G), torch.float32)]
    if conf:
        out_specs += [("c", (B, G), torch.float32), ("S", (B, G), torch.float32)]
    if host.get("target") is not None:
        out_specs += [("cstar", (B, G), torch.float32), ("l1", (B, G), torch.float32)]
    if sched:
        out_specs += [("len", (B,), torch.int32), ("theta", (1,), torch.float64)]
    dout_buf, dout = packed(out_specs, "cuda")
    hout_buf, hout = packed(out_specs, "cpu")
    staged = plan(din["U"], din["h"], din["x0"], din.get("target"), out=dout)
    o = staged.out
    h2d = hin_buf.numel()
    d2h = hout_buf.numel()
    e2e_steps = min(args.steps, 200)

    def e2e_step(s):
        din_buf.copy_(hin_buf, non_blocking=True)
        staged.run(s)
        schedule(staged, s, (dout["len"], dout["theta"]) if sched else None)
        hout_buf.copy_(dout_buf, non_blocking=True)

    for _ in range(3):
        e2e_step(stream)
    torch.cuda.synchronize()
    # the step (input copy, the draft call, result copy) is captured once in a CUDA graph and
    # replayed: one launch per step, so the host's issue time does not stretch the step
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            e2e_step(torch.cuda.current_stream())
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    except RuntimeError:
        graph = None
        torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for i in range(e2e_steps):
        flush.zero_()
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            e2e_step(stream)
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= e2e_steps
    res_ok = bool((hout["tokens"] >= 0).all()) and torch.equal(hout["tokens"].cuda(), o.tokens)
    assert ws.status() == 0, "draft kernel reported a device error (end-to-end loop)"

    # ---- max over ranks
    ms_step, ms_draft, e2e_ms = ranks_max(dist, [ms_step, ms_draft, e2e_ms])
    value = job_rate(world, B * G, ms_step)
    e2e_value = job_rate(world, B * G, e2e_ms)

    if rank == 0:
        peak, peak_kind = load_peaks()
        alg = algorithmic_bytes(wl)
        achieved = alg / (ms_draft * 1e-3) / 1e9
        cap = TRAFFIC.get(wl.name)
        src = cap and os.path.join(ROOT, "semi_autoregressive_drafting_gb300", "csrc", cap[0])
        traffic = cap[2] if cap and _sha(src) == cap[1] else None
        head = 0 if wl.head == "markov" else 1
        launches = ds.draft_launches(head, B, wl.V, wl.r, wl.dtype == "bf16")
        path = ds.draft_path(head, B, wl.V, wl.r, wl.dtype == "bf16")
        if path == 1 and wl.target_noise is not None:
            launches += 1  # the target's normalisers, before the draft
        if path in (0, 2) and args.w2_layout == "rv":
            launches += 1  # W2's transpose for the small-batch kernels
        kernel_name = "draft_tc_kernel" if path == 1 else "draft_cc_kernel"
        # achieved covers the whole draft call: with launches before the draft kernel (the RNN
        # head's h-part GEMM, the target's normalisers) their time is in ms_draft too; the
        # scheduler after it is timed in the step but not in the roofline
        scope = "one launch" if launches == 1 else f"whole draft call, {launches} launches"
        step_launches = launches + (1 if sched else 0)
        path_name = {0: "cuda-core", 1: "tcgen05, requests on M",
                     2: "tcgen05, vocabulary on M"}.get(path, "none")
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_kind": f"{peak_kind} copy bandwidth",
                "algorithmic_bytes_per_launch": alg,
                "kernel": kernel_name, "scope": scope,
                "traffic_scope": f"{kernel_name}, one launch"}
        if traffic is not None:
            # the bytes that actually crossed HBM (ncu) over the same time: below the
            # algorithmic fraction when the kernel keeps data on chip across steps
            roof["dram_frac"] = traffic / (ms_draft * 1e-3) / 1e9 / peak
        if path in (1, 2):
            tpeak, tkind = load_tensor_peak()
            flops = algorithmic_flops(wl)
            tach = flops / (ms_draft * 1e-3) / 1e12
            roof["tensor"] = {"achieved": tach, "peak": tpeak, "unit": "TFLOP/s",
                              "frac": tach / tpeak, "peak_kind": tkind,
                              "algorithmic_flops_per_launch": flops}
        roof["limiter"] = LIMITER.get(wl.name, "not profiled")
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "gamma": G, "V": wl.V, "r": wl.r, "d": wl.d,
                       "T": wl.T, "l2": "flushed between timed blocks (512 MB write)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "path": path_name, "w2_layout": args.w2_layout,
                       "step": "draft block + prefix scheduler" if sched else "draft block",
                       "draft_ms": ms_draft, "schedule_ok": sched_ok},
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "cuda_graph": graph is not None, "results_copied": res_ok},
            "gpu_launches": step_launches * args.steps,
            "clocks": clk.summary(),
            "wall_s": wall,
            "ms_per_step_min": min(times), "ms_per_step_median": statistics.median(times),
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
