"""Benchmark: fused attention-KL forward + P2-side backward at 64K context x
32 heads (d = 128, causal, bf16), one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

A step is one pass of the whole path over one batch: streamkl_fwd (KL, LSE1,
LSE2) then streamkl_bwd in the standard-distillation mode (dQ2, dK2, fused
with atomics).  value = algorithmic TFLOP/s of the step: 2(d1+d2) flops per
unmasked (query, key) pair forward, 2(d1+d2) + 4 d2 backward.  Inputs
(2.15 GB) are larger than L2, so no flush is needed between steps.  Under
torchrun every rank runs its own batch (weak scaling, no collective on the
data path); the reported time is the max over ranks.

--impl reference times the float64 CPU oracle (the reference arm for this
method) on a bounded sample of the same workload.
"""

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_distillation_kl_gb300.workloads import WORKLOADS, generate, generate_dkl  # noqa: E402

W = WORKLOADS["c4"]
METRIC = "fused attn-KL fwd+bwd TFLOP/s at 64K ctx x 32 heads (d=128, causal, P2-side grad)"
UNIT = "TFLOP/s"

# DRAM bytes per launch of the dominant kernel from one ncu capture, valid
# only while its source is unchanged (sha256 of the file it lives in).
TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one full-size launch
    "bwd_fused": {"bytes": 3294571264 + 2136466432, "src_sha": "cdaacbf38a1b7730"},
    "fwd": {"bytes": 2160437760 + 28472320, "src_sha": "f0ca1b124adb173a"},
}


def rank_workload(w, rank):
    """Each rank runs its own batch of the same shape (weak scaling): same
    workload, seed offset by the rank, so no two ranks process the same data."""
    return w.with_(seed=w.seed + 1000 * rank)


def max_over_ranks(x, world, device):
    """The slowest rank's time defines the job's time."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank, ms_per_step):
    """Whole-job throughput: the work of every rank over the slowest time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def flops(w):
    p = w.pairs
    return 2 * (w.d1 + w.d2) * p, (2 * (w.d1 + w.d2) + 4 * w.d2) * p


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


class Clocks:
    """Samples SM clocks and throttle reasons while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=10)
            self.t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


KERNEL_SOURCES = {"bwd_fused": ["bwd.cu", "bwd_common.cuh", "ptx.cuh", "kernels.cuh", "tiles.cuh"],
                  "fwd": ["fwd_kernel.cuh", "ptx.cuh", "kernels.cuh", "tiles.cuh"]}


def src_sha(kernel):
    """Hash of the sources a kernel is compiled from (its .cu and the headers
    it includes): recorded traffic is only reported for the same sources."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "attention_distillation_kl_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def cpu_sample(rows):
    """The oracle, as it stands, on the last `rows` query rows of one head of
    the workload (each sees ~64K keys): forward plus P2-side backward.  The
    causal sub-problem (rows x all keys, bottom-right aligned) is exactly
    those rows of the full problem."""
    import oracle
    from attention_distillation_kl_gb300.workloads import generate_head, to_f64
    q1, k1, q2, k2 = [to_f64(t) for t in generate_head(W, 0, 0)]
    q1, q2 = q1[-rows:], q2[-rows:]
    t0 = time.perf_counter()
    oracle.forward_head(q1, k1, q2, k2, W.scale, True)
    oracle.backward_head(q1, k1, q2, k2, W.scale, True, np.ones(rows), oracle.MODE_P2)
    dt = time.perf_counter() - t0
    nk = W.NK
    pairs = rows * (nk - rows) + rows * (rows + 1) // 2
    fl = (2 * (W.d1 + W.d2) + 2 * (W.d1 + W.d2) + 4 * W.d2) * pairs
    return fl / dt / 1e12, dt


def run_reference(args, rank):
    if rank != 0:
        return
    rows = 512
    for _ in range(args.warmup):
        cpu_sample(rows)
    vals, dts = [], []
    for _ in range(args.steps):
        v, dt = cpu_sample(rows)
        vals.append(v)
        dts.append(dt)
    value = float(np.median(vals))
    cores = len(os.sched_getaffinity(0))
    sample = f"last {rows} query rows of head (0,0) of the 64K x 32-head workload, fwd + P2 bwd, float64 numpy"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.median(dts)) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded normal, perturbed student)",
        "config": {"workload": "c4: B=1 H=32 NQ=NK=65536 d1=d2=128 causal bf16 inputs", "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def ex2_rate(skl):
    out = torch.empty(1, device="cuda")
    blocks, iters = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count * 8, 4096
    skl.streamkl_probe_ex2(out, blocks, iters)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = None
    for _ in range(3):
        e0.record()
        skl.streamkl_probe_ex2(out, blocks, iters)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3
        best = t if best is None else min(best, t)
    return blocks * 256 * iters * 8 / best


def timed(fn, stream, reps=4):
    """Median CUDA-event time (ms) of fn on `stream` over `reps` calls, after
    one warm-up call."""
    fn()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return float(np.median(ts))


def oracle_seconds(w, rows, modes):
    """The float64 oracle, as it stands, on head (0, 0) of workload w: the
    whole head when rows is None, else its last `rows` query rows (for a
    causal problem the rows x all-keys sub-problem, bottom-right aligned, is
    exactly those rows); forward plus one backward per mode in `modes`.
    Returns (seconds for all B*H heads, extrapolated by unmasked pairs when
    sampled; the sample's own seconds; its pairs)."""
    import oracle
    from attention_distillation_kl_gb300.workloads import generate_head, to_f64
    q1, k1, q2, k2 = [to_f64(t) for t in generate_head(w, 0, 0)]
    n = w.NQ if rows is None else min(rows, w.NQ)
    q1, q2 = q1[-n:], q2[-n:]
    t0 = time.perf_counter()
    oracle.forward_head(q1, k1, q2, k2, w.scale, w.causal)
    for m in modes:
        oracle.backward_head(q1, k1, q2, k2, w.scale, w.causal, np.ones(n), m)
    dt = time.perf_counter() - t0
    off = w.NK - w.NQ
    if w.causal:  # rows NQ - n .. NQ - 1 see i + off + 1 keys each
        pairs = sum(i + off + 1 for i in range(w.NQ - n, w.NQ))
    else:
        pairs = n * w.NK
    return dt * w.pairs / pairs, dt, pairs


def config_report(skl, stream, sustained, rate, with_oracle):
    """Every named workload besides the headline one: forward and backward
    times, algorithmic TFLOP/s (2(d1+d2) flops per unmasked pair forward,
    + 4 d_g backward) and the fraction of the roofline (the slower of the
    sustained tensor peak and the measured ex2 rate; 2 ex2 per pair forward
    and in mode P2, 1 in mode P1), with the oracle's time on the host."""
    import oracle
    out = {}
    plan = [("pr1", ("p2", "p1"), None), ("c2", ("p2",), 256), ("c3", ("p2", "p1"), 128), ("c5", ("p2",), 32)]
    for name, modes, rows in plan:
        w = WORKLOADS[name]
        dev = [t.cuda() for t in generate(w)]
        kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
        dkl = torch.ones_like(kl)
        p = w.pairs
        f_fwd = 2 * (w.d1 + w.d2) * p
        r = {"workload": f"{name}: B={w.B} H={w.H} NQ={w.NQ} NK={w.NK} d1={w.d1} d2={w.d2} "
                         f"{'causal' if w.causal else 'non-causal'}", "pairs": p}
        r["fwd_ms"] = timed(lambda: skl.streamkl_fwd(*dev, w.scale, w.causal, kl, l1, l2), stream)
        r["fwd_tflops"] = f_fwd / (r["fwd_ms"] * 1e-3) / 1e12
        r["fwd_roofline_frac"] = max(f_fwd / (sustained * 1e12), 2 * p / rate) / (r["fwd_ms"] * 1e-3)
        for m in modes:
            mode = skl.STREAMKL_GRAD_P2 if m == "p2" else skl.STREAMKL_GRAD_P1
            dg = w.d2 if m == "p2" else w.d1
            dq = torch.empty(w.B, w.H, w.NQ, dg, device="cuda")
            dk = torch.empty(w.B, w.H, w.NK, dg, device="cuda")
            ms = timed(lambda: skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, mode, False, dq, dk), stream)
            f = (2 * (w.d1 + w.d2) + 4 * dg) * p
            r[f"bwd_{m}_ms"] = ms
            r[f"bwd_{m}_tflops"] = f / (ms * 1e-3) / 1e12
            r[f"bwd_{m}_roofline_frac"] = max(f / (sustained * 1e12), (2 if m == "p2" else 1) * p / rate) / (ms * 1e-3)
            del dq, dk
        if name == "c5":  # the key-split workload: forced and suggested split counts
            heur = skl.streamkl_suggest_splits(w.B, w.H, w.NQ, w.NK, w.causal)
            ws = torch.empty(skl.streamkl_fwd_splitk_workspace_bytes(w.B, w.H, w.NQ, max(8, heur)),
                             dtype=torch.uint8, device="cuda")
            r["suggested_splits"] = heur
            r["fwd_splitk8_ms"] = timed(lambda: skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, 8, ws, kl, l1, l2),
                                        stream)
            r["fwd_splitk_suggested_ms"] = timed(
                lambda: skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, heur, ws, kl, l1, l2), stream)
            del ws
        if with_oracle:
            omodes = [oracle.MODE_P2 if m == "p2" else oracle.MODE_P1 for m in modes]
            secs, dt, sp = oracle_seconds(w, rows, omodes)
            r["oracle_s"] = secs
            r["oracle_sample"] = ("all rows of head (0,0)" if rows is None else f"last {rows} rows of head (0,0)") + \
                (f", {dt:.2f} s for {sp} pairs" + ("" if rows is None and w.B * w.H == 1 else
                                                    f", scaled to {w.B * w.H} heads by pairs"))
        out[name] = r
        del dev, kl, l1, l2, dkl
        torch.cuda.empty_cache()
    return out


def key_split_shapes(skl, stream):
    """Short query blocks against long keys, where a CTA per query tile
    leaves most SMs idle: the plain forward against the key-split forward
    with the heuristic's split count and with fixed counts (B=1, H=4,
    NQ=256, NK=131072, d=128, causal and not)."""
    from attention_distillation_kl_gb300.workloads import Workload
    out = {}
    for causal in (True, False):
        w = Workload("short-q", 1, 4, 256, 131072, 128, 128, causal, 1 / np.sqrt(128), "independent", 0.0, 1.0, 1008)
        dev = [t.cuda() for t in generate(w)]
        kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
        heur = skl.streamkl_suggest_splits(w.B, w.H, w.NQ, w.NK, w.causal)
        ws = torch.empty(skl.streamkl_fwd_splitk_workspace_bytes(w.B, w.H, w.NQ, max(64, heur)), dtype=torch.uint8,
                         device="cuda")
        f = 2 * (w.d1 + w.d2) * w.pairs
        r = {"workload": f"B=1 H=4 NQ=256 NK=131072 d1=d2=128 {'causal' if causal else 'non-causal'}",
             "suggested_splits": heur}
        r["fwd_ms"] = timed(lambda: skl.streamkl_fwd(*dev, w.scale, w.causal, kl, l1, l2), stream)
        for sp in sorted({8, 32, heur}):
            r[f"fwd_splitk{sp}_ms"] = timed(
                lambda: skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, sp, ws, kl, l1, l2), stream)
        r["fwd_tflops"] = f / (r["fwd_ms"] * 1e-3) / 1e12
        r["fwd_splitk_suggested_tflops"] = f / (r[f"fwd_splitk{heur}_ms"] * 1e-3) / 1e12
        r["speedup_suggested_over_plain"] = r["fwd_ms"] / r[f"fwd_splitk{heur}_ms"]
        out["causal" if causal else "non_causal"] = r
        del dev, ws
        torch.cuda.empty_cache()
    return out


def wide_head_timing(skl, stream, sustained, rate):
    """Head dim 256 on both sides (16K tokens x 8 heads, causal): forward
    (K streamed in 64-column blocks) and the two-pass P2 backward."""
    from attention_distillation_kl_gb300.workloads import Workload
    w = Workload("wide256", 1, 8, 16384, 16384, 256, 256, True, 1 / 16.0, "perturbed", 0.3, 1.0, 1009)
    dev = [t.cuda() for t in generate(w)]
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    dkl = torch.ones_like(kl)
    dq = torch.empty(w.B, w.H, w.NQ, w.d2, device="cuda")
    dk = torch.empty(w.B, w.H, w.NK, w.d2, device="cuda")
    f_fwd, f_bwd = flops(w)
    r = {"workload": "B=1 H=8 NQ=NK=16384 d1=d2=256 causal"}
    r["fwd_ms"] = timed(lambda: skl.streamkl_fwd(*dev, w.scale, w.causal, kl, l1, l2), stream)
    r["bwd_p2_ms"] = timed(lambda: skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl,
                                                    skl.STREAMKL_GRAD_P2, False, dq, dk), stream)
    r["fwd_tflops"] = f_fwd / (r["fwd_ms"] * 1e-3) / 1e12
    r["bwd_p2_tflops"] = f_bwd / (r["bwd_p2_ms"] * 1e-3) / 1e12
    r["fwd_roofline_frac"] = max(f_fwd / (sustained * 1e12), 2 * w.pairs / rate) / (r["fwd_ms"] * 1e-3)
    r["bwd_p2_roofline_frac"] = max(f_bwd / (sustained * 1e12), 2 * w.pairs / rate) / (r["bwd_p2_ms"] * 1e-3)
    del dev, dq, dk
    torch.cuda.empty_cache()
    return r


def gqa_timing(skl, stream):
    """Grouped key heads: 32 query heads sharing 8 key heads on each side
    (16K tokens, d = 128, causal): forward, fused and deterministic P2
    backward (dK of each shared head summed over its 4 query heads)."""
    from attention_distillation_kl_gb300.workloads import Workload, generate_gqa
    w = Workload("gqa", 1, 32, 16384, 16384, 128, 128, True, 1 / np.sqrt(128), "independent", 0.0, 1.0, 1007)
    hk = 8
    dev = [t.cuda() for t in generate_gqa(w, hk, hk, sd=1.0)]
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, w.scale, w.causal)
    dkl = torch.ones_like(kl)
    dq = torch.empty(w.B, w.H, w.NQ, w.d2, device="cuda")
    dk = torch.empty(w.B, hk, w.NK, w.d2, device="cuda")
    f_fwd, f_bwd = flops(w)
    out = {"workload": f"B={w.B} H={w.H} HK1=HK2={hk} NQ=NK={w.NQ} d1=d2=128 causal"}
    out["fwd_ms"] = timed(lambda: skl.streamkl_fwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2), stream)
    out["bwd_p2_ms"] = timed(lambda: skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl,
                                                          skl.STREAMKL_GRAD_P2, False, dq, dk), stream)
    out["bwd_p2_det_ms"] = timed(lambda: skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl,
                                                              skl.STREAMKL_GRAD_P2, True, dq, dk), stream)
    out["fwd_tflops"] = f_fwd / (out["fwd_ms"] * 1e-3) / 1e12
    out["bwd_p2_tflops"] = f_bwd / (out["bwd_p2_ms"] * 1e-3) / 1e12
    del dev, dq, dk
    torch.cuda.empty_cache()
    return out


def both_sides_timing(skl, stream, d=64):
    """Both-sides backward in one pass (atomic and deterministic) against the
    two single-side passes, on a d1 = d2 = d problem (16K tokens x 32 heads,
    causal)."""
    from attention_distillation_kl_gb300.workloads import Workload
    w = Workload(f"both-d{d}", 1, 32, 16384, 16384, d, d, True, 1 / np.sqrt(d), "independent", 0.0, 1.0, 1006)
    dev = [t.cuda() for t in generate(w)]
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    dkl = torch.ones_like(kl)
    bufs = [torch.empty(w.B, w.H, n, d, device="cuda") for n in (w.NQ, w.NK, w.NQ, w.NK)]
    out = {"workload": f"B={w.B} H={w.H} NQ=NK={w.NQ} d1=d2={d} causal"}
    out["bwd_p2_ms"] = timed(lambda: skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl,
                                                      skl.STREAMKL_GRAD_P2, False, bufs[2], bufs[3]), stream)
    out["bwd_p1_ms"] = timed(lambda: skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl,
                                                      skl.STREAMKL_GRAD_P1, False, bufs[0], bufs[1]), stream)
    out["bwd_both_ms"] = timed(lambda: skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl,
                                                             False, *bufs), stream)
    out["bwd_both_det_ms"] = timed(lambda: skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl,
                                                                 True, *bufs), stream)
    # two S products and four gradient products, 2 d flops each per pair
    out["bwd_both_tflops"] = 12 * d * w.pairs / (out["bwd_both_ms"] * 1e-3) / 1e12
    del dev, bufs
    torch.cuda.empty_cache()
    return out


def gpu_numa(dev_id):
    """The GPU's PCI address, the host NUMA node sysfs gives for it and the
    CPUs local to it (empty when the system does not say)."""
    info = {"pci_bus_id": None, "numa_node": None, "local_cpus": None}
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(dev_id), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip()
        dom, rest = bus.split(":", 1)
        sys_id = f"{int(dom, 16):04x}:{rest}".lower()
        info["pci_bus_id"] = sys_id
        base = f"/sys/bus/pci/devices/{sys_id}"
        if os.path.exists(base + "/numa_node"):
            info["numa_node"] = int(open(base + "/numa_node").read().strip())
        if os.path.exists(base + "/local_cpulist"):
            info["local_cpus"] = open(base + "/local_cpulist").read().strip()
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    return info


def parse_cpulist(txt):
    cpus = set()
    for part in txt.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        elif part.strip():
            cpus.add(int(part))
    return cpus


def pages_by_node(ptr):
    """NUMA nodes of the pages of the mapping that holds host address ptr,
    from /proc/self/numa_maps ({"N0": pages, ...}; empty if unknown)."""
    try:
        best, fields = -1, []
        for line in open("/proc/self/numa_maps"):
            parts = line.split()
            start = int(parts[0], 16)
            if best < start <= ptr:
                best, fields = start, parts
        return {f.split("=")[0]: int(f.split("=")[1]) for f in fields if f[:1] == "N" and "=" in f}
    except (OSError, ValueError, IndexError):
        return {}


def run_mine(args, rank, world, local):
    import attention_distillation_kl_gb300 as skl  # raises if the CUDA library is missing
    torch.cuda.set_device(local)
    dev_id = torch.cuda.current_device()
    w = rank_workload(W, rank)  # each rank its own batch
    # Pinned host inputs on the memory node local to this GPU: run on its
    # local CPUs while the buffers are allocated and touched, so the pages
    # land there (first touch); then record where they actually are.
    numa = gpu_numa(dev_id)
    affinity0 = os.sched_getaffinity(0)
    if numa["local_cpus"]:
        local = parse_cpulist(numa["local_cpus"]) & affinity0
        if local:
            os.sched_setaffinity(0, local)
    host = [t.pin_memory() for t in generate(w)]
    numa["pinned_pages_by_node"] = pages_by_node(host[0].data_ptr())
    os.sched_setaffinity(0, affinity0)
    dkl_h = generate_dkl(w).pin_memory()
    dev = [t.cuda() for t in host]
    dkl = dkl_h.cuda()
    B, H, N = w.B, w.H, w.NQ
    kl = torch.empty(B, H, N, device="cuda")
    l1, l2 = torch.empty_like(kl), torch.empty_like(kl)
    dq = torch.empty(B, H, N, w.d2, device="cuda")
    dk = torch.empty(B, H, w.NK, w.d2, device="cuda")
    kl_h = torch.empty(B, H, N).pin_memory()
    f_fwd, f_bwd = flops(w)
    stream = torch.cuda.current_stream()

    def step(ev=None, inp=None, dkl_in=None):
        x = dev if inp is None else inp
        g = dkl if dkl_in is None else dkl_in
        if ev is not None:
            ev[0].record(stream)
        skl.streamkl_fwd(*x, w.scale, w.causal, kl, l1, l2)
        if ev is not None:
            ev[1].record(stream)
        skl.streamkl_bwd(*x, w.scale, w.causal, kl, l1, l2, g, skl.STREAMKL_GRAD_P2, False, dq, dk)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if skl.streamkl_get_device_status() != 0:
        raise RuntimeError("device status reported a timeout during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(dev_id) as clk:
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    total_ms = max_over_ranks(total_ms, world, "cuda")
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, f_fwd + f_bwd, ms_per_step)

    # End to end through the public API: every step copies its inputs from
    # pinned host memory and reads its KL back, inside the timed region.  The
    # inputs are double-buffered and copied on a second stream, so the copy
    # for step k+1 overlaps the kernels of step k (each buffer is refilled
    # only after the step that used it has finished).  The loop runs three
    # times and the median is reported: the host link is shared with the
    # machine's other GPUs, and its rate during each copy is recorded too.
    e2e_steps = max(3, min(args.steps, 6))
    sets = [(dev, dkl), ([torch.empty_like(t) for t in dev], torch.empty_like(dkl))]
    copy_stream = torch.cuda.Stream()
    in_bytes = sum(t.numel() * t.element_size() for t in host) + dkl_h.numel() * 4

    def e2e_loop():
        copied = [torch.cuda.Event() for _ in range(e2e_steps)]
        consumed = [torch.cuda.Event() for _ in range(e2e_steps)]
        c_on = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def issue_copy(j):
            with torch.cuda.stream(copy_stream):
                if j >= 2:
                    copy_stream.wait_event(consumed[j - 2])
                c_on[j][0].record(copy_stream)
                bufs, g = sets[j % 2]
                for d, h in zip(bufs, host):
                    d.copy_(h, non_blocking=True)
                g.copy_(dkl_h, non_blocking=True)
                c_on[j][1].record(copy_stream)
                copied[j].record(copy_stream)

        torch.cuda.synchronize()
        e0.record(stream)
        copy_stream.wait_event(e0)
        issue_copy(0)
        for k in range(e2e_steps):
            if k + 1 < e2e_steps:
                issue_copy(k + 1)
            stream.wait_event(copied[k])
            step(inp=sets[k % 2][0], dkl_in=sets[k % 2][1])
            consumed[k].record(stream)
            kl_h.copy_(kl, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        rates = [in_bytes / (c[0].elapsed_time(c[1]) * 1e-3) / 1e9 for c in c_on]
        return e0.elapsed_time(e1) / e2e_steps, rates

    loops = [e2e_loop() for _ in range(3)]
    e2e_runs = [ms for ms, _ in loops]
    e2e_ms = float(np.median(e2e_runs))
    h2d_in_loop = float(np.median([r for _, rates in loops for r in rates]))
    # the host-to-device rate on its own, after the loops (reported: it
    # bounds the pipelined loop once it is slower than the kernels)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(copy_stream)
    with torch.cuda.stream(copy_stream):
        for d, h in zip(sets[1][0], host):
            d.copy_(h, non_blocking=True)
    c1.record(copy_stream)
    torch.cuda.synchronize()
    h2d_ms = c0.elapsed_time(c1)
    e2e_ms = max_over_ranks(e2e_ms, world, "cuda")
    h2d = sum(t.numel() * t.element_size() for t in host) + dkl_h.numel() * 4
    d2h = kl_h.numel() * 4

    # mode P1 backward timed on its own (outside the step): the other gradient side, d1-wide
    dq1 = torch.empty(B, H, N, w.d1, device="cuda")
    dk1 = torch.empty(B, H, w.NK, w.d1, device="cuda")
    free0 = torch.cuda.mem_get_info()[0]
    p1_ms = []
    for k in range(4):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P1, False, dq1, dk1)
        b_.record(stream)
        torch.cuda.synchronize()
        if k > 0:  # the first is warm-up
            p1_ms.append(a.elapsed_time(b_))
    p1_ms = float(np.median(p1_ms))
    # the deterministic P2 backward (dQ on the per-row grid) on the same inputs
    det_ms = timed(lambda: skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P2, True,
                                            dq, dk), stream, reps=3)
    # the library holds no device memory across calls (the deterministic
    # backward's scratch block comes from the stream's pool and goes back to
    # it): device memory free before and after the calls must agree
    extra_bytes = free0 - torch.cuda.mem_get_info()[0]
    f_p1 = (2 * (w.d1 + w.d2) + 4 * w.d1) * w.pairs

    rate = ex2_rate(skl)
    burst, sustained, _hbm, src = peaks()
    # every other named workload, the short-query key-split shapes, head dim
    # 256, both-sides and grouped-key-head calls: each timed on its own after
    # the step loop (single-GPU runs only; the oracle times need the host)
    extras = rank == 0 and world == 1 and not args.no_cpu_baseline
    configs = config_report(skl, stream, sustained, rate, with_oracle=True) if extras else None
    short = key_split_shapes(skl, stream) if extras else None
    wide = wide_head_timing(skl, stream, sustained, rate) if extras else None
    both = both_sides_timing(skl, stream) if extras else None
    both32 = both_sides_timing(skl, stream, 32) if extras else None
    gqa = gqa_timing(skl, stream) if extras else None
    pairs = w.pairs
    # roofline time of each kernel: the slower of the tensor pipe and the ex2 unit
    t_fwd = max(f_fwd / (sustained * 1e12), 2 * pairs / rate)
    t_bwd = max(f_bwd / (sustained * 1e12), 2 * pairs / rate)
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    dom = "bwd" if bwd_ms >= fwd_ms else "fwd"
    kname = "bwd_fused" if dom == "bwd" else "fwd"
    tr = TRAFFIC.get(kname)
    traffic = None
    if tr and tr["src_sha"] == src_sha(kname):
        traffic = tr["bytes"]
    if skl.streamkl_get_device_status() != 0:
        raise RuntimeError("device status reported a timeout")

    out = None
    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal, perturbed student)",
            "config": {"workload": (f"{w.name}: B={w.B} H={w.H} NQ={w.NQ} NK={w.NK} d1={w.d1} d2={w.d2} "
                                    f"{'causal' if w.causal else 'non-causal'}, fwd + P2-side bwd (fused)"),
                       "global_batch": world * w.B, "seq_len": w.NQ, "heads": w.H,
                       "parallelism": f"replicas{world}",
                       "l2": "inputs (2.15 GB) larger than L2, no flush"},
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "fwd_roofline_frac": t_fwd / (fwd_ms * 1e-3), "bwd_roofline_frac": t_bwd / (bwd_ms * 1e-3),
            "bwd_p1_ms": p1_ms, "bwd_p1_tflops": f_p1 / (p1_ms * 1e-3) / 1e12,
            "bwd_p1_roofline_frac": max(f_p1 / (sustained * 1e12), pairs / rate) / (p1_ms * 1e-3),
            "bwd_p2_deterministic_ms": det_ms, "bwd_p2_deterministic_over_fused": det_ms / bwd_ms,
            "extra_device_bytes": extra_bytes,
            "configs": configs,
            "key_split_short_queries": short,
            "wide_head_d256": wide,
            "both_sides_d64": both,
            "both_sides_d32": both32,
            "gqa_16k": gqa,
            "ex2_per_s": rate,
            "roofline": {"bound": "tensor", "achieved": bwd_tf if dom == "bwd" else fwd_tf,
                         "peak": sustained, "unit": "TFLOP/s",
                         "frac": (bwd_tf if dom == "bwd" else fwd_tf) / sustained,
                         "traffic": traffic, "kernel": f"bwd_fused_kernel<{w.d1},{w.d2},P2>" if dom == "bwd"
                         else f"fwd_kernel<{w.d1},{w.d2}>", "peak_source": f"{src} bf16 sustained",
                         "frac_of_burst": (bwd_tf if dom == "bwd" else fwd_tf) / burst},
            "e2e": {"value": job_tflops(world, f_fwd + f_bwd, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "loops": 3, "reported": "median loop",
                    "copies": "pinned host -> device on a second stream, double-buffered, overlapping "
                              "the previous step; KL read back every step",
                    "h2d_gbs_alone": sum(t.numel() * t.element_size() for t in host) / (h2d_ms * 1e-3) / 1e9,
                    "h2d_gbs_in_loop": h2d_in_loop, "loops_ms_per_step": e2e_runs,
                    "numa": numa},
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
        }
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="c4", choices=sorted(WORKLOADS),
                    help="profiling aid: run the same step on another named workload")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    global W
    if args.workload != "c4":
        W = WORKLOADS[args.workload]
        args.no_cpu_baseline = True
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    out = run_mine(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt = cpu_sample(3072)
        out["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                               "sample": "last 3072 query rows of head (0,0) of the 64K x 32-head workload, "
                                         f"fwd + P2 bwd, float64 numpy ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
