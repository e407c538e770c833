"""Benchmark of the fused attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line (rank 0).  A step is one pass of the hot path over one
batch of synthetic input already resident in HBM:
  * dense / causal / varlen workloads: one attention forward (attn_fwd or
    attn_fwd_varlen);
  * fp8: quantise + rotate Q, K, V (qkv_block_quant_hadamard), then the e4m3
    attention forward.
The default workload is bf16 non-causal B=4 H=16 N=8448 d=128 (inputs 553 MB,
larger than the 126 MB L2, so no flush is needed between steps).

value = attention FLOPs (4 B H N^2 d, halved when causal) of all ranks / max
over ranks of the device time of K steps (CUDA events on the launching stream,
barrier + synchronize on both sides).  `e2e` repeats the measurement through
the public API with the inputs copied from pinned host memory and O, lse
copied back inside the timed region: the host-buffer entry points for the
dense 16-bit workloads (attn_fwd_host) and the fp8 workload
(attn_fwd_fp8_host), which overlap the copies with the compute, and copies
around the device step for the others.  `--impl reference` times the fp64
CPU oracle on a bounded sample of the same workload instead.

The default line also carries an `fp8` block: the e4m3 workload (B=4 H=16
N=8192 d=128) with its attention kernel against the fp8 dense peak and its
quantise pre-step against HBM bandwidth.

`--gpus N` runs N replicas, one rank per GPU.  Under a launcher (WORLD_SIZE
set) N must equal the number of ranks; without one, the script starts N ranks
of itself under torch.distributed.run.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

NOMINAL_DENSE_TFLOPS = {"bf16": 2250.0, "fp16": 2250.0, "e4m3": 4500.0}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def get_workload(name: str):
    from datagen import workloads as W
    if name == "dense":
        return W.DENSE
    if name == "tiny":
        return W.TINY
    if name == "fp8":
        return W.FP8
    if name == "fp8_d64":
        return W.Workload("fp8 e4m3 non-causal B=4 H=16 N=8192 d=64, 0.1% outliers", "fp8",
                          4, 16, 8192, 64, False, 1003, outliers=True)
    if name == "varlen":
        return W.varlen_causal()
    if name == "gqa":
        return W.gqa_causal()
    if name in ("bwd", "bwd_causal"):
        return W.backward(name == "bwd_causal")
    if name == "paged":
        return W.paged_decode()
    if name.startswith("causal"):
        # causal:N:H:d
        _, N, H, d = name.split(":")
        N, H, d = int(N), int(H), int(d)
        return W.Workload(f"bf16 causal B={16384 // N} H={H} N={N} d={d}", "bf16",
                          16384 // N, H, N, d, True, 1004)
    raise SystemExit(f"unknown workload {name}")


def max_over_ranks(seconds: float, world: int, device) -> float:
    """The slowest rank's time: the job finishes when every replica has."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    tt = torch.tensor([seconds], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tflops(world: int, flops_per_rank_step: float, steps: int, seconds: float) -> float:
    """Whole-job throughput: every rank runs the full workload (replicas), so
    the job processes world * steps steps in the slowest rank's time."""
    return world * flops_per_rank_step * steps / seconds / 1e12


def rank_info():
    r = int(os.environ.get("RANK", "0"))
    w = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    return r, w, lr


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = set()
        for _, _, rest in rows:
            for nm, val in zip(names, rest[2:6]):
                if val.lower().startswith("active"):
                    seen.add(nm)
        load = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(seen), "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def build_step(w, dev):
    """Returns (step_fn, launches_per_step, e2e_fn, h2d_bytes, d2h_bytes, flops)."""
    import numpy as np
    import torch

    import attention_forward_softmax_gb300 as agb
    from datagen.workloads import make_inputs

    from datagen.workloads import PagedWorkload, make_paged_inputs
    if isinstance(w, PagedWorkload):
        x = make_paged_inputs(w)
        q = x["q"].to(dev)
        kc, vc = x["k_cache"].to(dev), x["v_cache"].to(dev)
        table = torch.from_numpy(x["block_table"]).to(dev)
        seql = torch.from_numpy(x["seqlens"]).to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Nq), device=dev, dtype=torch.float32)

        def step():
            agb.attn_fwd_paged(q, kc, vc, table, seql, max(w.lengths), causal=w.causal, out=o,
                               lse=lse)
        # the cache is state that stays in HBM; a decoding step brings the new
        # queries in and takes O and lse out
        hq = x["q"].pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        def e2e():
            q.copy_(hq, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        h2d = hq.numel() * hq.element_size()
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        return step, 2, e2e, h2d, d2h, w.flops(), step, None, (q, kc, vc, o)

    x = make_inputs(w)
    q, k, v = (x[n].to(dev) for n in "qkv")
    flops = w.flops()
    # the dense non-causal forward splits the last wave's tiles into key
    # halves when they would fill at most half of it: one merge launch more
    tiles = w.B * w.H * ((w.N + 255) // 256)
    grid = min(tiles, torch.cuda.get_device_properties(dev).multi_processor_count)
    rem = tiles % grid if grid else 0
    merge = int(not w.varlen and not w.causal and 0 < 2 * rem <= grid and w.N > 128
                and not (w.dtype == "fp8" and w.d != 128))
    if w.dtype == "fp8":
        signs = torch.from_numpy(x["signs"]).to(dev)
        qz = [torch.empty(q.shape, device=dev, dtype=torch.uint8) for _ in range(3)] + \
             [torch.empty((w.B, w.H, (w.N + 127) // 128), device=dev, dtype=torch.float32)
              for _ in range(3)]
        o = torch.empty(q.shape, device=dev, dtype=torch.bfloat16)
        lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)

        def step():
            q8, k8, v8, dq, dk, dv = agb.qkv_block_quant_hadamard(q, k, v, signs, outs=qz)
            agb.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=w.causal, out=o, lse=lse)
        launches = 2 + merge
        attn_only = (lambda: agb.attn_fwd_fp8(*qz, causal=w.causal, out=o, lse=lse))
        quant_only = (lambda: agb.qkv_block_quant_hadamard(q, k, v, signs, outs=qz))
    elif w.varlen:
        cu = torch.from_numpy(x["cu_seqlens"]).to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.H, w.tokens), device=dev, dtype=torch.float32)

        def step():
            agb.attn_fwd_varlen(q, k, v, cu, max(w.lengths), causal=w.causal, out=o, lse=lse)
        launches = 2   # tile-list builder + attention
        attn_only, quant_only = step, None
    elif w.name.startswith("bf16 backward"):
        # forward once outside the timed region; a step is the backward
        # (rowsum(dO O) pass, the main kernel, the dQ conversion)
        o, lse = agb.attn_fwd(q, k, v, causal=w.causal)
        from datagen.workloads import make_dout
        do = make_dout(w).to(dev)
        flops = 2.5 * w.flops()

        def step():
            agb.attn_bwd(q, k, v, o, lse, do, causal=w.causal)
        launches = 3
        attn_only, quant_only = step, None
    else:
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)

        def step():
            agb.attn_fwd(q, k, v, causal=w.causal, out=o, lse=lse)
        launches = 1 + merge
        attn_only, quant_only = step, None

    # end-to-end through the public API: pinned host inputs in, O and lse out
    hq, hk, hv = (x[n].pin_memory() for n in "qkv")
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    if (not w.varlen and w.dtype in ("bf16", "fp16") and w.Hkv in (None, w.H)
            and not w.name.startswith("bf16 backward")):
        # dense 16-bit: the host-buffer entry point, which overlaps the copies
        # of each chunk (batch entries, head groups at both ends) with the
        # compute of earlier chunks
        def e2e():
            agb.attn_fwd_host(hq, hk, hv, causal=w.causal, out=ho, lse=hl)
    elif w.dtype == "fp8" and not w.varlen:
        # the 8-bit path's host-buffer entry point: per chunk, bf16 in,
        # quantisation and the e4m3 forward on the device, bf16 out
        hsigns = torch.from_numpy(x["signs"]).pin_memory()

        def e2e():
            agb.attn_fwd_fp8_host(hq, hk, hv, signs=hsigns, causal=w.causal, out=ho, lse=hl)
    else:
        def e2e():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return step, launches, e2e, h2d, d2h, flops, attn_only, quant_only, (q, k, v, o)


def time_region(fn, steps, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def per_launch_ms(fn, steps, stream):
    """Average duration of fn's launches, CUDA events around each call."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def kernel_source_hash() -> str:
    import glob
    import hashlib
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "attention_forward_softmax_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def fp8_block(dev, stream, peaks, peak_kind, steps):
    """The 8-bit workload (e4m3, B=4 H=16 N=8192 d=128, 0.1% outliers) measured
    beside the default line: the e4m3 attention kernel alone (per-launch CUDA
    events) against the fp8 dense peak, the quantise pre-step against HBM
    bandwidth, and the whole step (pre-step + attention)."""
    import torch

    import attention_forward_softmax_gb300 as agb
    w = get_workload("fp8")
    step, _, _, _, _, flops, attn_only, quant_only, bufs = build_step(w, dev)
    for _ in range(5):
        step()
    torch.cuda.synchronize()
    agb.check_status()
    n = max(10, min(steps, 50))
    t_step = time_region(step, n, stream)
    attn_ms = per_launch_ms(attn_only, n, stream)
    q_ms = per_launch_ms(quant_only, n, stream)
    agb.check_status()
    peak = peaks["bf16_tflops"] * 2.0
    achieved = flops / (attn_ms / 1e3) / 1e12
    qb = 3 * (bufs[0].numel() * 2 + bufs[0].numel())   # read bf16, write e4m3
    return {"workload": w.name, "bound": "tensor", "unit": "TFLOP/s",
            "achieved": round(achieved, 2), "peak": round(peak, 1),
            "frac": round(achieved / peak, 4),
            "frac_of_nominal_dense": round(achieved / NOMINAL_DENSE_TFLOPS["e4m3"], 4),
            "peak_source": f"{peak_kind} bf16 burst x 2 (nominal fp8:bf16 ratio)",
            "kernel_ms": round(attn_ms, 4), "traffic": traffic_record("fp8"),
            "step_ms": round(t_step / n * 1e3, 4),
            "step_tflops": round(flops * n / t_step / 1e12, 2),
            "quant": {"bound": "hbm", "ms": round(q_ms, 4),
                      "achieved": round(qb / (q_ms / 1e3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                      "unit": "GB/s", "frac": round(qb / (q_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                      "algorithmic_bytes": qb}}


def traffic_record(workload: str):
    """DRAM bytes per launch from profiles/traffic.json, or None once the
    kernel sources differ from the ones the counters were taken on."""
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tr_path):
        return None
    with open(tr_path) as f:
        rec = json.load(f).get(workload)
    if rec and rec.get("source_sha") == kernel_source_hash():
        return rec["bytes"]
    return None


def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank, world, lrank = rank_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(lrank)
    dev = torch.device("cuda", lrank)
    import attention_forward_softmax_gb300 as agb
    agb.lib()

    w = get_workload(args.workload)
    step, launches, e2e, h2d, d2h, flops, attn_only, quant_only, bufs = build_step(w, dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    agb.check_status()

    barrier()
    with ClockSampler(lrank) as cs:
        t = time_region(step, args.steps, stream)
    barrier()
    agb.check_status()
    t = max_over_ranks(t, world, dev)

    # roofline leg: dominant kernel timed per launch on its own stream
    peaks, peak_kind = load_peaks()
    dtype = "e4m3" if w.dtype == "fp8" else w.dtype
    attn_ms = per_launch_ms(attn_only, max(10, min(args.steps, 50)), stream)
    from datagen.workloads import PagedWorkload
    paged = isinstance(w, PagedWorkload)
    if dtype == "e4m3":
        peak = peaks["bf16_tflops"] * 2.0          # fp8 dense = 2x bf16 (nominal ratio)
        peak_note = f"{peak_kind} bf16 burst x 2 (nominal fp8:bf16 ratio)"
    else:
        peak = peaks["bf16_tflops"]
        peak_note = f"{peak_kind} bf16 burst (cuBLAS)"
    achieved = flops / (attn_ms / 1e3) / 1e12
    traffic = traffic_record(args.workload)
    roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": peak_note, "kernel_ms": round(attn_ms, 4),
            "algorithmic_flops_per_launch": flops,
            "frac_of_nominal_dense": round(achieved / NOMINAL_DENSE_TFLOPS[dtype], 4)}
    if paged:
        # decoding reads every cached K and V row once: HBM-bound (the split
        # merge is included in the launch time)
        gbs = w.bytes() / (attn_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"{peak_kind} HBM copy bandwidth", "kernel_ms": round(attn_ms, 4),
                "algorithmic_bytes_per_launch": w.bytes()}
    # secondary roof: the exponential unit.  One exponential per (query,
    # allowed key) pair = flops / (4 d); the unit evaluates 32 per clock per SM
    # (ex2.approx.f32 or f16x2 pairs alike, measured on GB300), here at the
    # median SM clock sampled during the timed region.
    clk = cs.summary()
    sm_mhz = clk.get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    exps = flops / (4.0 * w.d)
    mufu_peak = 32.0 * n_sm * sm_mhz * 1e6
    roof["secondary"] = None if (paged or w.name.startswith("bf16 backward")) else {"bound": "mufu", "achieved": round(exps / (attn_ms / 1e3) / 1e12, 3),
                         "peak": round(mufu_peak / 1e12, 3), "unit": "Texp/s",
                         "frac": round(exps / (attn_ms / 1e3) / mufu_peak, 4),
                         "peak_source": f"32 exp2 per clock per SM x {n_sm} SMs x "
                                        f"{sm_mhz:.0f} MHz (median during the timed region)"}
    extra_fields = {}
    if quant_only is not None:
        q_ms = per_launch_ms(quant_only, 20, stream)
        qb = 3 * (bufs[0].numel() * 2 + bufs[0].numel())   # read bf16, write e4m3
        extra_fields["quant"] = {"bound": "hbm", "ms": round(q_ms, 4),
                                 "achieved": round(qb / (q_ms / 1e3) / 1e9, 1),
                                 "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": round(qb / (q_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                                 "algorithmic_bytes": qb}

    if args.workload == "dense" and not args.no_fp8:
        extra_fields["fp8"] = fp8_block(dev, stream, peaks, peak_kind, args.steps)

    # end to end through the public API (host buffers)
    for _ in range(2):
        e2e()
    torch.cuda.synchronize()
    barrier()
    te = time_region(e2e, max(5, args.steps // 10), stream)
    barrier()
    te = max_over_ranks(te, world, dev)
    e2e_steps = max(5, args.steps // 10)

    result = None
    if rank == 0 and paged:
        # decoding: whole-job bytes per second (every replica reads its cache)
        result = {
            "metric": "paged decode GB/s (cached K and V rows once, plus Q and O)",
            "value": round(world * w.bytes() * args.steps / t / 1e9, 1), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(t / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded N(0,1) cache, shuffled pages)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.Hkv, "d": w.d,
                       "Nq": w.Nq, "page_size": w.page_size, "causal": w.causal,
                       "l2": "cache larger than L2 (no flush)" if w.bytes() > 126e6
                       else "cache smaller than L2 (warm)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": None,
            "e2e": {"value": round(world * w.bytes() * e2e_steps / te / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(te / e2e_steps * 1e3, 4)},
            "gpu_launches": launches * args.steps, "clocks": cs.summary(),
            "tflops": round(world * flops * args.steps / t / 1e12, 2),
        }
    elif rank == 0:
        value = job_tflops(world, flops, args.steps, t)
        cpu = None if args.no_cpu_baseline else cpu_baseline(w, budget_s=args.cpu_seconds)
        bwd = w.name.startswith("bf16 backward")
        result = {
            "metric": ("attn bwd TFLOP/s (10*B*H*N^2*d, /2 causal)" if bwd else
                       "attn fwd TFLOP/s (4*B*H*N^2*d, /2 causal)"),
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(t / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": dtype, "data": "synthetic (seeded N(0,1)" +
            (", 0.1% N(0,100) outliers" if w.outliers else "") + ")",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "varlen": w.varlen,
                       **({"H_kv": w.Hkv} if w.Hkv else {}),
                       "l2": "inputs larger than L2 (no flush)"
                       if 3 * bufs[0].numel() * bufs[0].element_size() > 126e6
                       else "inputs smaller than L2 (cache warm)",
                       "parallelism": f"replicas x{world}"},
            "pct_of_dense_peak": round(100 * value / world / NOMINAL_DENSE_TFLOPS[dtype], 2),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": round(job_tflops(world, flops, e2e_steps, te), 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(te / e2e_steps * 1e3, 4)},
            "gpu_launches": launches * args.steps,
            "clocks": cs.summary(),
            **extra_fields,
        }
        if args.workload == "dense":
            result["baseline_context"] = ("661 TFLOP/s: FlashAttention-3 ablation, same shape, "
                                          "H100, 16-bit (another GPU; context only)")
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(w, nrows: int, seed: int = 7):
    """Seeded (token, head) rows of the workload and the inputs in fp64."""
    import numpy as np

    from datagen.workloads import make_inputs
    import torch
    x = make_inputs(w)
    q, k, v = (x[n].to(torch.float64).numpy() for n in "qkv")   # exact up-conversion, once
    if not w.varlen:
        q, k, v = (t.reshape(w.B * w.N, t.shape[2], w.d) for t in (q, k, v))
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, w.tokens, size=nrows)
    head = rng.integers(0, w.H, size=nrows).astype(np.int32)
    return q, k, v, x["cu_seqlens"], tok, head


def row_flops(w, cu, tok):
    """Attention FLOPs of the sampled query rows: 4 d per allowed key."""
    import numpy as np
    seq = np.searchsorted(cu, tok, side="right") - 1
    pos = tok - cu[seq]
    L = cu[seq + 1] - cu[seq]
    keys = (pos + 1) if w.causal else L
    return float(4.0 * w.d * keys.sum())


def calibrate(run, budget_s: float, n_max: int):
    """Grows the row count until one run takes >= 0.3 s, then runs once with
    the count sized for `budget_s`; returns (rows, seconds of that run)."""
    n = 64
    t0 = time.perf_counter()
    run(n)
    dt = time.perf_counter() - t0
    while dt < 0.3 and n < n_max:
        n = min(n_max, n * 4)
        t0 = time.perf_counter()
        run(n)
        dt = time.perf_counter() - t0
    n = max(1, min(n_max, int(n * budget_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    run(n)
    return n, time.perf_counter() - t0


def cpu_baseline(w, budget_s: float = 15.0, threads=None):
    """Times the oracle as it stands on this host's cores, on a bounded row
    sample sized to take about `budget_s` seconds."""
    import oracle
    threads = threads or oracle.default_threads()
    q, k, v, cu, tok, head = oracle_sample(w, 1 << 16)
    n, dt = calibrate(lambda m: oracle.attention_rows_gqa(q, k, v, cu, cu, w.scale, w.causal,
                                                          tok[:m], head[:m], threads),
                      budget_s, len(tok))
    flops = row_flops(w, cu, tok[:n])
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n} seeded (token, head) query rows of the same workload, all their keys, "
                      f"{dt:.1f} s, fp64 C, {threads} threads"}


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return None
    import oracle
    w = get_workload(args.workload)
    threads = oracle.default_threads()
    q, k, v, cu, tok, head = oracle_sample(w, 1 << 16)
    # size one step so that warmup + steps stay within a few minutes
    per_step_budget = args.ref_step_seconds or max(1.0, min(20.0,
                                                            150.0 / max(1, args.steps + args.warmup)))
    n, _ = calibrate(lambda m: oracle.attention_rows_gqa(q, k, v, cu, cu, w.scale, w.causal,
                                                         tok[:m], head[:m], threads),
                     per_step_budget, len(tok))
    for _ in range(max(0, args.warmup - 1)):
        oracle.attention_rows_gqa(q, k, v, cu, cu, w.scale, w.causal, tok[:n], head[:n], threads)
    times = []
    for s in range(args.steps):
        t0 = time.perf_counter()
        oracle.attention_rows_gqa(q, k, v, cu, cu, w.scale, w.causal, tok[:n], head[:n], threads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    flops = row_flops(w, cu, tok[:n])
    value = flops * args.steps / total / 1e12
    sample = (f"{n} seeded (token, head) query rows of the same workload per step, all their "
              f"keys, fp64 C oracle, {threads} threads")
    return {"metric": "attn fwd TFLOP/s (4*B*H*N^2*d, /2 causal)", "value": round(value, 6),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "varlen": w.varlen},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def relaunch_under_torchrun(args) -> int:
    """`--gpus N` without a launcher: start N ranks of this script under
    torch.distributed.run on this node and return its exit status."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr=127.0.0.1",
           f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dense",
                    help="dense | tiny | fp8 | fp8_d64 | varlen | gqa | paged | bwd | bwd_causal | "
                         "causal:N:H:d")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true",
                    help="omit the fp8 block of the default (dense) line")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="reference arm: oracle seconds per step (default: sized so the "
                         "whole run takes a few minutes)")
    args = ap.parse_args()
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        raise SystemExit(relaunch_under_torchrun(args))
    _, world, _ = rank_info()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but the launcher started {world} ranks")
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
