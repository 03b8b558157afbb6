#!/usr/bin/env python3
"""Benchmark of the content-dependent block-sparse attention forward.

One step = one forward (block mean-pool -> coarse scoring + top-k -> fine
attention over the selected blocks), replayed as one captured CUDA graph of
``bsa_forward_ex`` (``--no-graph``: one direct call) on the 32k-token workload:
bh = 8 heads, n = 32768, d = 64, bf16, key block 64, top-16, planted block
centres; inputs resident in HBM, L2 flushed (a 256 MiB write) before every
timed step.  Prints ONE JSON line (rank 0):

  value      effective TFLOP/s over all ranks (selected FLOPs only, page
             "sparse-attention-triton-bench" convention: 87.24 GFLOP/forward)
  e2e        the same metric through the public API with host buffers:
             pinned-host -> device copies of Q, K, V and the device -> host
             copy of O inside every timed step
  roofline   the dominant kernel (fine attention), timed alone with CUDA
             events on its stream, against the measured bf16 tensor peak
  cpu_baseline  the fp64 oracle on a bounded row sample, host cores (rank 0)

``--impl reference`` times the oracle itself as the reference arm.
``--workload`` selects another workload: the selection-option, skewed-list
and smaller dynamic ones time the same forward; the sliding-window one times
the static-list fine stage alone.
Multi-GPU (torchrun): every rank runs its own independent problem (weak
scaling, no collective on the data path); the barrier and max-over-ranks
timing use torch.distributed.
"""
from __future__ import annotations

import argparse
import csv
import ctypes
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from content_dependent_block_gb300 import metrics  # noqa: E402

METRIC = "sparse-attn fwd ms & effective TFLOP/s at N=32k (1 GB300); % of roofline"
WORKLOAD = "dyn_n32768"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--backward", action="store_true",
                   help="time the fine stage's backward pass (bsa_fine_backward) over the "
                        "forward's lists instead of the forward; prints its own JSON line")
    p.add_argument("--no-graph", dest="graph", action="store_false",
                   help="call bsa_forward_ex for every forward instead of replaying one "
                        "captured CUDA graph (bsa_forward_graph_create / bsa_graph_launch)")
    p.add_argument("--profile-forwards", type=int, default=0, metavar="N",
                   help="run N untimed forwards of the workload and exit (a fixed launch "
                        "sequence for profilers: 6 kernels per forward); prints no JSON")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU seconds of the oracle sample")
    p.add_argument("--preroll-s", type=float, default=1.5,
                   help="seconds of untimed calls inside the clock-sampling window, "
                        "before the warm-up and the timed steps")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    return args


# ---------------------------------------------------------------- ranks
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def aggregate(dist, total_ms: float, units: float, device=None):
    """Max of the timed region and sum of the work over ranks."""
    if dist is None:
        return total_ms, units
    import torch
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = [r for r in csv.reader(io.StringIO(open(self.path).read())) if len(r) >= 9]
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def fp32_peak(peaks, sms: int) -> float:
    """FP32 FLOP/s derived from unit counts and clocks: SMs x 128 FP32
    lanes x 2 FLOP (one FMA) x the maximum SM clock."""
    return sms * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6


def roofline(f_mma: float, f_alu: float, nbytes: float, t_ms: float, peaks, sms: int,
             kernel: str, traffic, tc_key: str = "bf16_tflops"):
    """Roofline object of the scope table (d): the bound is
    t_roof = max(F_mma / P_tensor + F_alu / P_fp32, bytes / BW_hbm), with the
    measured tensor peak and HBM bandwidth and the derived FP32 peak.
    `achieved` is the algorithmic FLOPs over the measured time, `peak` the
    same FLOPs over t_roof, so that frac = achieved / peak = t_roof / t."""
    p_tc = peaks[tc_key] * 1e12
    p_fp32 = fp32_peak(peaks, sms)
    bw = peaks["hbm_gbs"] * 1e9
    t_mma, t_alu, t_hbm = f_mma / p_tc, f_alu / p_fp32, nbytes / bw
    t_roof = max(t_mma + t_alu, t_hbm)
    flops = f_mma + f_alu
    achieved = flops / (t_ms * 1e-3) / 1e12
    peak = flops / t_roof / 1e12
    if t_hbm >= t_mma + t_alu:
        bound = "hbm"
    elif t_mma >= t_alu:
        bound = "tensor"
    else:
        bound = "alu"
    return {"kernel": kernel, "bound": bound, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
            "t_roof_us": t_roof * 1e6, "launch_ms": t_ms,
            "terms_us": {"mma_at_tensor_peak": t_mma * 1e6, "softmax_at_fp32_peak": t_alu * 1e6,
                         "bytes_at_hbm_bw": t_hbm * 1e6},
            "algorithmic": {"mma_flops": f_mma, "alu_flops": f_alu, "unique_bytes": nbytes},
            "peaks": {"tensor_tflops": p_tc / 1e12, "tensor_source": f"{tc_key}, {peaks['source']}",
                      "fp32_tflops": p_fp32 / 1e12,
                      "fp32_source": f"{sms} SMs x 128 lanes x 2 x max clock (derived)",
                      "hbm_gbs": bw / 1e9, "hbm_source": f"hbm_gbs, {peaks['source']}"},
            "formula": "peak = F / max(F_mma/P_tensor + F_alu/P_fp32, bytes/BW_hbm)"}


def preroll(fn, seconds: float, sync):
    """Untimed calls for about `seconds` (so that clock samplers see the
    GPU under steady load before the timed region)."""
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds:
        for _ in range(8):
            fn()
        sync()
        n += 8
    return n


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was
    captured on this workload and the kernel's source has not changed since;
    else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    ent = table.get(kernel)
    if not ent or ent.get("workload") != workload:
        return None
    sources = ent.get("sources") or {ent["source"]: ent.get("source_sha")}
    for rel, want in sources.items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != want:
            return None
    return ent["bytes_per_launch"]


# ------------------------------------------------------------ CPU oracle
def select_args(w, device):
    """Selection-option keyword arguments of bsa.Forward for workload w."""
    import torch
    hk = torch.tensor(w.head_topk, dtype=torch.int32, device=device) if w.head_topk else None
    return dict(head_topk=hk, causal=w.causal, local_block=w.local_block)


def eligible_scores(w) -> int:
    """Coarse scores the selection needs: every block, or b <= i // B (causal)."""
    import numpy as np
    if not w.causal:
        return w.bh * w.n * w.nb
    return w.bh * int((np.arange(w.n) // w.key_block + 1).sum())


def admitted_pairs(idx, w, rows=None) -> int:
    """(query, key) pairs a selection admits: the valid keys of each listed
    block, only keys j <= i when causal.  idx is a torch tensor [bh, n, k] or
    a numpy array [len(rows), k] of the flat rows `rows`."""
    import numpy as np
    if rows is None:
        import torch
        b = idx.long()
        i = torch.arange(w.n, device=idx.device).view(1, w.n, 1)
        start = b * w.key_block
        keys = torch.clamp(w.n - start, max=w.key_block)
        if w.causal:
            keys = torch.minimum(keys, i - start + 1)
        return int((keys.clamp(min=0) * (b >= 0)).sum())
    b = idx.astype(np.int64)
    i = (rows % w.n)[:, None]
    start = b * w.key_block
    keys = np.minimum(w.n - start, w.key_block)
    if w.causal:
        keys = np.minimum(keys, i - start + 1)
    return int((np.clip(keys, 0, None) * (b >= 0)).sum())


def oracle_step(orc, w, t, rows):
    """The oracle's whole dynamic path for `rows`; returns its FLOPs."""
    import numpy as np
    kbar = orc.pool(t.k, w.key_block)
    s = orc.scores(t.q, kbar, rows)
    if w.has_options:
        hk = np.array(w.head_topk, dtype=np.int32) if w.head_topk else None
        idx = orc.select(s, rows, w.n, w.key_block, w.topk, head_k=hk, causal=w.causal,
                         local=w.local_block)
    else:
        idx, _ = orc.topk(s, w.topk)
    orc.fine(t.q, t.k, t.v, w.key_block, idx, rows, causal=w.causal)
    if not w.has_options:
        return rows.size * metrics.sparse_flops(w.n, w.bh, w.d, w.key_block, w.topk) / (w.n * w.bh)
    return (metrics.pairs_flops(admitted_pairs(idx, w, rows), w.d)
            + 2 * w.d * rows.size * eligible_scores(w) / (w.bh * w.n))


def oracle_sample(w, t, seconds: float):
    """Time the oracle's whole dynamic path on a row sample; returns
    (TFLOP/s, rows, seconds, cores, description)."""
    import numpy as np
    import oracle
    cores = oracle.num_threads()

    def run(nrows):
        rows = workloads.sample_rows(w.bh, w.n, max(1, nrows // w.bh), seed=7)
        t0 = time.perf_counter()
        fl = oracle_step(oracle, w, t, rows)
        return rows.size, time.perf_counter() - t0, fl

    r0, t0, _ = run(256 * w.bh)
    # bounded: at most 32768 rows per pass (the oracle keeps every row's
    # scores); passes repeat until about `seconds` of CPU time is spent
    nrows = int(min(w.bh * w.n, 32768, max(r0, r0 * seconds / max(t0, 1e-3))))
    r1 = t1 = f1 = 0
    passes = 0
    while passes == 0 or (t1 < seconds and passes < 64):
        r, dt, fl = run(nrows)
        r1 += r
        t1 += dt
        f1 += fl
        passes += 1
    tflops = f1 / t1 / 1e12
    desc = (f"{r1 // passes} of {w.bh * w.n} query rows (seeded sample) x {passes} passes, "
            f"full pool + scores + top-k + fine per row, fp64, {cores} threads")
    return tflops, r1 // passes, t1, cores, desc


def reference_arm(args, rank, world, w):
    """The oracle as the reference arm: each step a bounded row sample."""
    if rank != 0:
        return 0
    import oracle  # noqa: F401
    t = workloads.generate(w)
    cores = None
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    _, rows, secs, cores, desc = oracle_sample(w, t, budget)
    import oracle as orc
    times = []
    rws = workloads.sample_rows(w.bh, w.n, max(1, rows // w.bh), seed=7)
    flops = 0.0
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        fl = oracle_step(orc, w, t, rws)
        if it >= args.warmup:
            times.append(time.perf_counter() - t0)
            flops += fl
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rws.size} of {w.bh * w.n} query rows per step; " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def static_oracle_sample(w, t, seconds: float):
    """The oracle's static-pattern attention (plain masked definition: the
    sliding window or the local+global mask) on a seeded row sample,
    repeated until about `seconds` of CPU time; returns (TFLOP/s on admitted
    pairs, rows per pass, seconds, cores, description)."""
    import numpy as np
    import oracle
    cores = oracle.num_threads()
    if w.kind == "sliding":
        kind, kw, what = oracle.MASK_SLIDING, dict(W=w.sliding), "i-W < j <= i"
    else:
        kind, kw, what = oracle.MASK_LOCAL_GLOBAL, dict(w=w.window, s=w.stride), \
            f"|i-j| <= {w.window} or j % {w.stride} == 0"

    def keys_of(rows):
        i = rows % w.n
        if w.kind == "sliding":
            return int(np.minimum(i + 1, w.sliding).sum())
        j = np.arange(w.n)
        return int(sum(int(((np.abs(ii - j) <= w.window) | (j % w.stride == 0)).sum()) for ii in i))

    def run(count):
        rows = workloads.sample_rows(w.bh, w.n, max(1, count // w.bh), seed=7)
        t0 = time.perf_counter()
        oracle.masked(t.q, t.k, t.v, kind, rows, **kw)
        return rows.size, time.perf_counter() - t0, metrics.pairs_flops(keys_of(rows), w.d)

    r0, t0, _ = run(16 * w.bh)
    count = int(min(w.bh * w.n, 8192, max(r0, r0 * seconds / max(t0, 1e-3))))
    rows = secs = flops = 0
    passes = 0
    while passes == 0 or (secs < seconds and passes < 64):
        r, dt, fl = run(count)
        rows += r
        secs += dt
        flops += fl
        passes += 1
    desc = (f"{rows // passes} of {w.bh * w.n} query rows (seeded sample) x {passes} passes, "
            f"dense masked attention over {what} per row, fp64, {cores} threads")
    return flops / secs / 1e12, rows // passes, secs, cores, desc


def run_static(args, w, device, dist):
    """A static-pattern workload: one bsa_fine_attention call per step over
    the host-built block lists (bsa_static_blocks).  The sliding window runs
    on the tensors of the dynamic workload of the same shape (block key
    norms, the one-pass tensor-core kernel, the relaunch for flagged tiles);
    the local+global pattern is the fp32 16x16-tile workload of the
    yayme/CUDA-kernel README (CUDA-core kernel).  With --profile-forwards N,
    N untimed calls; else a timed run (clocks sampled around it, L2 flushed
    before every step) and one JSON line."""
    import torch
    from content_dependent_block_gb300 import bsa
    if w.kind == "sliding":
        base = next(x for x in workloads.WORKLOADS.values()
                    if x.kind == "dynamic" and (x.bh, x.n, x.d) == (w.bh, w.n, w.d))
        t = workloads.generate(base)
        q, k, v = (torch.from_numpy(getattr(t, x).view("int16")).view(torch.bfloat16).to(device)
                   for x in "qkv")
        m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=w.sliding)
        pairs = metrics.sliding_pairs(w.n, w.sliding) * w.bh
        elem, dtype, tc_key = 2, "bf16", "bf16_tflops"
        kernel = ("static fine stage: block key norms + one-pass tensor-core kernel "
                  "(+ the two-pass relaunch for flagged tiles)")
        metric = "static sliding-window fine stage, effective TFLOP/s on admitted pairs"
    else:
        t = workloads.generate(w)
        q, k, v = (torch.from_numpy(getattr(t, x)).to(device) for x in "qkv")
        m = bsa.mask_struct(bsa.MASK_LOCAL_GLOBAL, window=w.window, stride=w.stride)
        pairs = metrics.local_global_pairs(w.n, w.window, w.stride) * w.bh
        elem, dtype, tc_key = 4, "f32", "bf16_tflops"
        kernel = "static fine stage, fp32 on the CUDA cores (query-major kernel over the tile lists)"
        metric = "static local+global fine stage (fp32), effective TFLOP/s on admitted pairs"
    lst, _, _ = bsa.static_blocks(w.n, w.q_group, w.key_block, m)
    dl = torch.from_numpy(lst).to(device)
    out = torch.empty_like(q)

    def run():
        bsa.fine_attention(q, k, v, dl, key_block=w.key_block, q_group=w.q_group,
                           per_head=False, mask=m, out=out)

    if args.profile_forwards > 0:
        for _ in range(args.profile_forwards):
            run()
        torch.cuda.synchronize(device)
        status = bsa.device_status()
        if dist is not None:
            dist.destroy_process_group()
        return 0 if status == 0 else 1
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or 0) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else device.index
    with ClockSampler(gpu_index) as clocks:
        preroll(run, args.preroll_s, lambda: torch.cuda.synchronize(device))
        for _ in range(args.warmup):
            flush.fill_(1)
            run()
        torch.cuda.synchronize(device)
        evs = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(device)
    clk = clocks.summary()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    achieved = metrics.pairs_flops(pairs, w.d) / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    nbytes = metrics.unique_bytes(w.n, w.bh, w.d, elem)
    if w.kind == "sliding":
        rl = roofline(4 * w.d * pairs, 5 * pairs, nbytes, ms, peaks, sms, kernel,
                      kernel_traffic("fine_static_tc", w.name), tc_key)
    else:
        # fp32 throughout: every FLOP at the FP32 peak (no tensor term)
        rl = roofline(0, metrics.pairs_flops(pairs, w.d), nbytes, ms, peaks, sms, kernel, None,
                      tc_key)
    status = bsa.device_status()
    if dist is not None:
        dist.destroy_process_group()
    cfg = {"workload": w.name, "bh": w.bh, "n": w.n, "d": w.d, "key_block": w.key_block,
           "q_group": w.q_group, "dtype": w.dtype, "inputs": w.note,
           "timing": "median of CUDA-event times; L2 flushed (256 MiB write) before every step"}
    if w.kind == "sliding":
        cfg["sliding"] = w.sliding
    else:
        cfg.update(window=w.window, stride=w.stride)
    line = {
        "metric": metric, "value": achieved, "unit": "TFLOP/s",
        "roofline": rl,
        "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup, "n_gpus": 1,
        "higher_is_better": True, "dtype": dtype, "data": "synthetic", "config": cfg,
        "clocks": clk, "admitted_pairs": pairs, "device_status": status,
        # per call: sliding = block key norms, the one-pass kernel, the
        # relaunch for flagged tiles (plus a memset); fp32 = one kernel
        "gpu_launches": (3 if w.kind == "sliding" else 1) * args.steps}
    if not args.no_cpu_baseline:
        tf, rows, secs, cores, desc = static_oracle_sample(w, t, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": secs}
    print(json.dumps(line), flush=True)
    return 0 if status == 0 else 1


def run_backward(args, w, fwd, q, k, v, device, dist):
    """The fine stage's backward pass over the lists (and output) of one
    forward: bsa_fine_backward_lse timed alone, given the rows' log2-sum-exp
    that the forward saved (bsa_fine_attention_lse, untimed, as a training
    step keeps it), CUDA events, L2 flushed before every step, clocks sampled
    around the timed steps; one JSON line, which also reports the same steps
    through bsa_fine_backward (statistics recomputed by a forward pass).
    With 64-key blocks it runs on the tensor cores (bwd_tc_kernel in
    csrc/backward.cu); the roofline takes its contractions at the tensor
    peak, its softmax ops at the FP32 peak and its bytes at the HBM
    bandwidth."""
    import torch
    from content_dependent_block_gb300 import bsa
    gen = torch.Generator(device="cpu").manual_seed(1)
    dout = torch.randn(q.shape, generator=gen).to(torch.bfloat16).to(device)
    L = bsa.lib()
    ld = bsa.ListDesc(1, w.key_block, w.topk, 1)
    m = bsa.mask_struct(bsa.MASK_CAUSAL if w.causal else bsa.MASK_NONE)
    dq, dk, dv = (torch.empty(q.shape, dtype=torch.float32, device=device) for _ in range(3))
    ws_n = L.bsa_fine_backward_workspace_size(fwd.shape, ld)
    ws = bsa._workspace(ws_n, device)
    P = bsa._ptr
    # the rows' log2-sum-exp as the forward saves it (same lists, same output)
    _, lse = bsa.fine_attention_lse(q, k, v, fwd.idx.contiguous(), key_block=w.key_block,
                                    causal=w.causal)

    def step():
        bsa._check(L.bsa_fine_backward_lse(fwd.shape, P(q), P(k), P(v), P(fwd.out), P(dout),
                                           P(fwd.idx), ld, m, 0.0, P(lse), P(dq), P(dk), P(dv),
                                           P(ws), ws_n, bsa._stream()))

    def step_recompute():
        bsa._check(L.bsa_fine_backward(fwd.shape, P(q), P(k), P(v), P(fwd.out), P(dout),
                                       P(fwd.idx), ld, m, 0.0, P(dq), P(dk), P(dv), P(ws), ws_n,
                                       bsa._stream()))

    if args.profile_forwards > 0:
        # N untimed backward calls (a fixed launch sequence for profilers)
        for _ in range(args.profile_forwards):
            step()
        torch.cuda.synchronize(device)
        status = bsa.device_status()
        if dist is not None:
            dist.destroy_process_group()
        return 0 if status == 0 else 1
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or 0) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else device.index
    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(device)
        evs = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(device)
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    with ClockSampler(gpu_index) as clocks:
        preroll(step, args.preroll_s, lambda: torch.cuda.synchronize(device))
        ms = timed(step)
        ms_recompute = timed(step_recompute)
    clk = clocks.summary()
    pairs = admitted_pairs(fwd.idx, w)
    # per admitted (query, key) pair: q.k, dO.v, dQ, dK and dV updates (2d each,
    # tensor cores) + softmax ops
    flops = pairs * (10 * w.d + 5)
    peaks = measured_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    achieved = flops / (ms * 1e-3) / 1e12
    rl = roofline(10 * w.d * pairs, 5 * pairs, 5 * w.n * w.bh * w.d * 2 + 3 * w.n * w.bh * w.d * 4,
                  ms, peaks, sms, "fine-stage backward: one bsa_fine_backward_lse call (list "
                  "inversion, D = dO.O, tensor-core dQ/dK/dV kernel; the rows' log2-sum-exp saved by "
                  "the forward)", None)
    status = bsa.device_status()
    if dist is not None:
        dist.destroy_process_group()
    print(json.dumps({
        "metric": "fine-stage backward pass (dQ, dK, dV over the forward's lists), effective TFLOP/s",
        "value": achieved, "unit": "TFLOP/s", "ms_per_step": ms, "steps": args.steps,
        "warmup": args.warmup, "n_gpus": 1, "higher_is_better": True, "dtype": "bf16 in, fp32",
        "data": "synthetic", "config": config_of(w),
        "roofline": rl,
        "admitted_pairs": pairs, "flops_per_step": flops, "clocks": clk,
        "recompute_stats": {"call": "bsa_fine_backward (a forward pass recomputes the rows' "
                                    "log2-sum-exp)", "ms_per_step": ms_recompute},
        "device_status": status}), flush=True)
    return 0 if status == 0 else 1


def config_of(w):
    c = {"workload": w.name, "bh": w.bh, "n": w.n, "d": w.d, "key_block": w.key_block,
         "topk": w.topk, "dtype": w.dtype, "inputs": w.note,
         "l2": "flushed before every timed step (256 MiB write)",
         "parallelism": "independent problem per rank (weak)"}
    if w.has_options:
        c["select"] = {"causal": w.causal, "local_block": w.local_block,
                       "head_topk": list(w.head_topk) or None}
        c["flops"] = "counted from the selection: admitted (query, key) pairs x (4d+5) + eligible scores x 2d"
    return c


# ------------------------------------------------------------- GPU arm
def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, rank, world, w)

    import torch
    from content_dependent_block_gb300 import _build, bsa
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    if rank == 0:
        _build.build()
    barrier(dist, device)
    bsa.lib()

    if w.kind in ("sliding", "local_global"):
        return run_static(args, w, device, dist)
    t = workloads.generate(w, seed=w.seed + rank)
    torch.cuda.reset_peak_memory_stats(device)
    mem0 = torch.cuda.memory_allocated(device)
    q, k, v = (torch.from_numpy(getattr(t, x).view("int16")).view(torch.bfloat16).to(device)
               for x in "qkv")
    fwd = bsa.Forward(w.bh, w.n, w.d, w.key_block, w.topk, device=device, graph=args.graph,
                      **select_args(w, device))
    fwd(q, k, v)
    torch.cuda.synchronize(device)
    if args.backward:
        return run_backward(args, w, fwd, q, k, v, device, dist)
    if args.profile_forwards > 0:
        for _ in range(args.profile_forwards - 1):
            fwd(q, k, v)
        torch.cuda.synchronize(device)
        status = bsa.device_status()
        if dist is not None:
            dist.destroy_process_group()
        return 0 if status == 0 else 1
    peak_mb = (torch.cuda.max_memory_allocated(device) - mem0) / 2**20
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    flops = metrics.sparse_flops(w.n, w.bh, w.d, w.key_block, w.topk)
    fine_flops = metrics.pairs_flops(w.n * w.bh * min(w.topk, w.nb) * w.key_block, w.d)
    if w.has_options:
        # the selection decides the work: count it from the first forward's lists
        pairs, elig = admitted_pairs(fwd.idx, w), eligible_scores(w)
        fine_flops = metrics.pairs_flops(pairs, w.d)
        flops = fine_flops + 2 * w.d * elig

    def flush_l2():
        flush.fill_(1)

    def timed(fn, steps):
        evs = []
        for _ in range(steps):
            flush_l2()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(device)
        return [a.elapsed_time(b) for a, b in evs]

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    with ClockSampler(gpu_index) as clocks:
        preroll(lambda: fwd(q, k, v), args.preroll_s, lambda: torch.cuda.synchronize(device))
        for _ in range(args.warmup):
            flush_l2()
            fwd(q, k, v)
        torch.cuda.synchronize(device)
        barrier(dist, device)
        torch.cuda.synchronize(device)
        step_ms = timed(lambda: fwd(q, k, v), args.steps)
        torch.cuda.synchronize(device)
        barrier(dist, device)
        total_ms, total_flops = aggregate(dist, sum(step_ms), flops * args.steps, device)

        # stages, each timed alone on the launching stream
        kbar = torch.empty((w.bh, w.nb, w.d), dtype=torch.float32, device=device)
        idx = torch.empty((w.bh, w.n, w.topk), dtype=torch.int32, device=device)
        out = torch.empty_like(q)
        ws_c = bsa.lib().bsa_coarse_topk_workspace_size(fwd.shape, w.key_block, w.topk)
        ws_cb = bsa._workspace(ws_c, device)
        shp = fwd.shape
        L = bsa.lib()
        S = bsa._stream
        P = bsa._ptr

        def pool():
            bsa._check(L.bsa_pool_blocks(shp, P(k), w.key_block, P(kbar), S()))

        sel = None if fwd.sel is None else ctypes.byref(fwd.sel)

        def coarse():
            bsa._check(L.bsa_coarse_topk_ex(shp, P(q), P(kbar), w.key_block, w.topk, sel, P(idx),
                                            P(ws_cb), ws_c, S()))

        ld = bsa.ListDesc(1, w.key_block, w.topk, 1)
        msk = bsa.mask_struct(bsa.MASK_CAUSAL) if w.causal else bsa.mask_struct()
        ws_f = L.bsa_fine_attention_workspace_size(shp, ld, msk)
        ws_fb = bsa._workspace(ws_f, device)

        def fine():
            bsa._check(L.bsa_fine_attention(shp, P(q), P(k), P(v), P(idx), ld, msk, 0.0, P(out),
                                            P(ws_fb), ws_f, S()))

        stage_steps = max(3, min(args.steps, 20))
        pool_ms = statistics.mean(timed(pool, stage_steps))
        coarse_ms = statistics.mean(timed(coarse, stage_steps))
        fine_ms = statistics.mean(timed(fine, stage_steps))

        # end to end through the public API with host buffers
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        ho = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        dq, dk, dv = (torch.empty_like(x) for x in (q, k, v))

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            o = fwd(dq, dk, dv)
            ho.copy_(o, non_blocking=True)

        for _ in range(2):
            e2e_step()
        e2e_ms = timed(e2e_step, args.steps)
        e2e_total, _ = aggregate(dist, sum(e2e_ms), 0.0, device)
    clk = clocks.summary()

    status = bsa.device_status()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0 if status == 0 else 1

    ms = total_ms / args.steps
    value = total_flops / (total_ms * 1e-3) / 1e12
    peaks = measured_peaks()
    tc_peak = peaks["bf16_tflops"]
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    # the dominant unit: one bsa_fine_attention call (list inversion + the
    # fine kernel), timed alone; per admitted (query, key) pair 4d MMA FLOPs
    # (q.k and p.v) and 5 softmax ops, compulsory bytes Q, K, V in and O out
    fine_keys = fine_flops // (4 * w.d + 5)
    fine_rl = roofline(4 * w.d * fine_keys, 5 * fine_keys, metrics.unique_bytes(w.n, w.bh, w.d, 2),
                       fine_ms, peaks, sms,
                       "fine attention stage: one bsa_fine_attention call over the top-k list "
                       "(list inversion + fine_ws_kernel)",
                       kernel_traffic("fine_stage", w.name))
    cfg = config_of(w)
    cfg["launch"] = (f"one CUDA-graph replay per forward ({fwd.launches} kernels)" if args.graph
                     else f"one bsa_forward_ex call per forward ({fwd.launches} kernels)")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": fine_rl,
        "e2e": {"value": flops * world / (e2e_total / args.steps * 1e-3) / 1e12,
                "unit": "TFLOP/s", "ms_per_step": e2e_total / args.steps,
                "h2d_bytes_per_step": 3 * q.numel() * q.element_size(),
                "d2h_bytes_per_step": q.numel() * q.element_size()},
        "gpu_launches": fwd.launches * args.steps,
        "clocks": clk,
        "stages_ms": {"pool": pool_ms, "coarse_topk": coarse_ms, "fine": fine_ms},
        "peak_hbm_mb": peak_mb,
        "flops_per_forward": flops,
        "device_status": status,
    }
    # whole-forward roofline (scope table (d)): the slower of the contraction
    # FLOPs at the tensor peak plus the softmax ops at the FP32 peak, and the
    # compulsory bytes at the measured HBM bandwidth.  The FP32 peak is derived
    # from unit counts and clocks: SMs x 128 FP32 lanes x 2 FLOP x max clock.
    f_mma, f_alu = metrics.sparse_flops_split(w.n, w.bh, w.d, w.key_block, w.topk)
    if w.has_options:
        f_mma, f_alu = 4 * w.d * pairs + 2 * w.d * elig, 5 * pairs
    p_fp32 = fp32_peak(peaks, sms)
    bytes_fwd = metrics.unique_bytes(w.n, w.bh, w.d, 2)
    t_roof = max(f_mma / (tc_peak * 1e12) + f_alu / p_fp32, bytes_fwd / (peaks["hbm_gbs"] * 1e9))
    line["roofline_forward"] = {
        "t_roof_us": t_roof * 1e6, "ms_per_forward": ms, "frac": t_roof * 1e3 / ms,
        "mma_flops": f_mma, "softmax_flops": f_alu, "unique_bytes": bytes_fwd,
        "fp32_peak_tflops": p_fp32 / 1e12, "fp32_peak_source": f"{sms} SMs x 128 lanes x 2 x max clock",
        "formula": "max(F_mma/P_tc + F_alu/P_fp32, bytes/BW_hbm)"}
    if not args.no_cpu_baseline and world == 1:
        tf, rows, secs, cores, desc = oracle_sample(w, t, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": secs}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
