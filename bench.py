#!/usr/bin/env python
"""Throughput of the packed multi-adapter LoRA layer: forward + backward + AdamW per step.

Default workload: all seven projections of a Llama-3-8B decoder layer (q, k, v, o 4096 -> 4096 /
1024; gate, up 4096 -> 14336; down 14336 -> 4096), bf16 activations and weights, fp32 adapter
masters, 32 jobs with ranks in {8..128} and 1..8 sequences of 1024 tokens each (143,360 tokens
per step), every job training one adapter on every projection.  One step = the forward of every
projection (q .. down), the backward of every projection (down .. q) and the AdamW step of every
adapter, through mlora_forward / mlora_backward / mlora_adamw_ws, with inputs resident in HBM.
Prints one JSON line (rank 0).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]
  python bench.py --sweep        packed vs one plan per job vs a per-adapter PyTorch loop

--impl reference times the fp64 CPU oracle (the reference arm of this metric) on a bounded
sample of the same workload.  Under torchrun (N > 1) the pack's jobs are split across the ranks
(whole jobs, longest first onto the least-loaded rank, mlora_shard_jobs_multi); each rank trains
only its jobs, there is no collective on the data path, and the value is the whole pack's
tokens over the slowest rank's time (strong scaling: the pack is fixed as N grows).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed multi-LoRA fwd+bwd tokens/s and TFLOP/s per layer; % of bf16/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = "layer"
# a timed region longer than this runs into the part's power cap: GEMMs are rated against the
# sustained bf16 figure, shorter regions against the burst one
SUSTAINED_AFTER_MS = 1000.0


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


def workload(name):
    from adapter_gemm_packed_gb300 import workloads as W
    if name == "layer":
        return W.llama8b_layer_all()
    if name == "layer_eighth":
        return W.llama8b_layer_all(token_div=8)
    if name in W.CONFIGS:
        return W.CONFIGS[name]()
    if name.startswith("llama8b_layer_"):
        return W.llama8b_layer(int(name.rsplit("_", 1)[1]))
    raise SystemExit(f"unknown workload {name}")


def parts_of(wl):
    """The projections one step runs: the seven of a decoder layer, or the one workload."""
    return list(wl.parts) if hasattr(wl, "parts") else [wl]


def labels_of(wl):
    from adapter_gemm_packed_gb300 import workloads as W
    if hasattr(wl, "parts"):
        return [W.LLAMA8B_PROJ[i][0] for i in range(len(wl.parts))]
    return ["main"]


def _entries(wl):
    """(tokens, rank, output width of B) of every adapter (one per job, or one per job and
    projection of a shared-input pack)."""
    return list(zip(wl.entry_tokens, wl.ranks, wl.entry_width))


def flops_per_step(wl):
    # 4 N d_in d_out for the two base GEMMs, 6 n r (d_in + width) per adapter (shrink, expand,
    # dH, dB, dA, dX term); the zero padding and other projections' zero blocks are not counted
    if hasattr(wl, "parts"):
        return sum(flops_per_step(p) for p in wl.parts)
    return 4.0 * wl.N * wl.d_in * wl.d_out + sum(6.0 * n * r * (wl.d_in + w) for n, r, w in _entries(wl))


def kernel_flops(wl, kernel):
    """Algorithmic FLOPs of one launch of a tensor-core kernel."""
    if kernel == "fwd_gemm":
        return 2.0 * wl.N * wl.d_in * wl.d_out + sum(2.0 * n * r * w for n, r, w in _entries(wl))
    if kernel == "bwd_gemm":
        return 2.0 * wl.N * wl.d_in * wl.d_out + sum(2.0 * n * r * wl.d_in for n, r, w in _entries(wl))
    return None


def kernel_bytes(wl, kernel):
    """Algorithmic HBM bytes of one launch of a memory-bound kernel (bf16 activations)."""
    e = 2
    lora = sum(n * r for n, r, w in _entries(wl))
    sr = sum(wl.ranks)
    srw = sum(r * w for n, r, w in _entries(wl))
    params = sr * wl.d_in + srw
    if kernel == "shrink":
        return wl.N * wl.d_in * e + sr * wl.d_in * 2 + lora * 4
    if kernel == "dH":
        return wl.N * wl.d_out * e + srw * 2 + lora * 4
    if kernel == "dA":
        return wl.N * wl.d_in * e + lora * 2 + wl.d_in * sr * 4
    if kernel == "dB":
        return wl.N * wl.d_out * e + lora * 2 + srw * 4
    if kernel == "adamw":
        # p, g, m, v read and p, m, v written (28 B), plus the bf16 shadow copy of p (2 B) that the
        # step refreshes for the next forward
        return params * 30
    if kernel == "w4_expand":
        # codes (half a byte), scales (4 bytes per 64 weights) in; bf16 W^T out
        return wl.d_in * wl.d_out * (0.5 + 4 / 64 + 2)
    return None


def job_ranks(wl):
    """Each job's summed rank over the projections of a shared-input pack (its own rank otherwise)."""
    G = wl.n_groups
    return [sum(wl.ranks[j * G:(j + 1) * G]) for j in range(len(wl.n_tokens))]


def shard(wl, world):
    """Rank of every job of the pack: whole jobs, longest processing time first onto the
    least-loaded rank, a job's cost summed over the step's projections (mlora_shard_jobs_multi).
    Returns (rank_of_job, load per rank)."""
    from adapter_gemm_packed_gb300 import _mlora as M
    parts = parts_of(wl)
    probs = [M.mlora_problem(p.N, p.d_in, p.d_out, M.MLORA_BF16, M.MLORA_PLAN_HOST_ONLY) for p in parts]
    base = parts[0]
    segs = [M.mlora_segment(o, n, r, 1.0) for o, n, r in zip(base.offsets, base.n_tokens, job_ranks(base))]
    return M.mlora_shard_jobs_multi(probs, segs, world)


def jobs_of_rank(rank_of_job, rank):
    return [j for j, r in enumerate(rank_of_job) if r == rank]


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms, each stamped with the host's clock on
    arrival; the summary keeps the samples that arrived inside the `with` block (the timed region).
    The raw samples are also written to $BENCH_CLOCKS_DIR when that is set."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.rows = []          # (host time, line)
        self.t0 = self.t1 = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.monotonic(), line.strip()))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.monotonic() + 3.0      # the sampler is live before the region starts
            while not self.rows and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.t0 = time.monotonic()
        return self

    def __exit__(self, *a):
        self.t1 = time.monotonic()
        if self.proc:
            time.sleep(0.06)                       # let the last in-region sample arrive
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except Exception:
                self.proc.kill()
            self.thread.join(5)
            out = os.environ.get("BENCH_CLOCKS_DIR")
            if out:
                os.makedirs(out, exist_ok=True)
                with open(os.path.join(out, f"clocks_bench_{os.getpid()}.csv"), "w") as f:
                    for t, line in self.rows:
                        f.write(f"{t - self.t0:.3f},{line}\n")

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        parsed = []
        for t, line in self.rows:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                parsed.append((t, float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        inside = [r for r in parsed if self.t0 <= r[0] <= self.t1 + 0.06]
        rows = inside or parsed
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4][1:]) if v.lower().startswith("active")})
        out = {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
               "power_w_max": max(r[3] for r in rows), "samples": len(rows), "reasons": reasons}
        if not inside:
            out["note"] = "no sample arrived inside the timed region; these are the samples around it"
        return out


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of a per-rank float over all ranks (the rank itself when not distributed)."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def pack_rate(units: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed together (the whole pack, split across
    the ranks) over the slowest rank's time."""
    return units * steps / (max_ms / 1e3)


def link_probe(x_h, x_d, y_h, y_d, s_in, s_out, reps=3):
    """Host link bandwidth with pinned buffers: H2D alone, D2H alone, both at once (GB/s per
    direction), timed with events bracketing the copies' streams."""
    import torch

    def run(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        s = torch.cuda.current_stream()
        s.wait_stream(s_in)
        s.wait_stream(s_out)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    def h2d():
        s_in.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_in):
            x_d.copy_(x_h, non_blocking=True)

    def d2h():
        s_out.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_out):
            y_h.copy_(y_d, non_blocking=True)

    def both():
        h2d()
        d2h()

    bx, by = x_h.numel() * x_h.element_size(), y_h.numel() * y_h.element_size()
    t_both = run(both)
    return {"h2d_gbs": bx / run(h2d) / 1e9, "d2h_gbs": by / run(d2h) / 1e9,
            "concurrent_gbs_per_direction": max(bx, by) / t_both / 1e9}


def oracle_sample(wl, per_job):
    """A bounded sample of one projection for the CPU oracle: the first `per_job` tokens of every
    job (only those rows are drawn).  Returns (sub-workload, X, W, dY, per-projection job lists,
    tokens)."""
    import numpy as np
    from adapter_gemm_packed_gb300 import workloads as W
    from oracle import lora_oracle as orc
    sub, T = W.materialise_jobs(wl, None, per_job)
    X = W.rows_as_f64(T.X, wl.dtype)
    dY = W.rows_as_f64(T.dY, wl.dtype)
    if wl.dtype == "bf16_w4":
        Wm = orc.dequantize_w4(T.Wq, T.Wscale)
    else:
        Wm = W.rows_as_f64(T.Wt, wl.dtype).T.copy()
    # per projection of a shared-input pack (one otherwise): its jobs' adapters
    G = sub.n_groups
    segs = []
    for g in range(G):
        sg = []
        for j, (o, n) in enumerate(zip(sub.offsets, sub.n_tokens)):
            i = j * G + g
            sg.append(orc.Seg(o, n, T.At[i].astype(np.float64).T.copy(), T.Bt[i].astype(np.float64).T.copy(),
                              sub.alphas[i]))
        segs.append(sg)
    return sub, X, Wm, dY, segs, sub.N


def oracle_step(wl, X, Wm, dY, segs, state, t):
    """One oracle step of one projection: each output group's column slice with its adapters
    (Y side by side, dX summed), then AdamW on every adapter."""
    import numpy as np
    from oracle import lora_oracle as orc
    Y = np.zeros((X.shape[0], Wm.shape[1]))
    dX = np.zeros_like(X)
    for g, (o, w) in enumerate(zip(wl.group_offsets, wl.widths)):
        Y[:, o:o + w], H = orc.forward(X, Wm[:, o:o + w], segs[g])
        dXg, dA, dB, dH = orc.backward(X, Wm[:, o:o + w], dY[:, o:o + w], segs[g])
        dX += dXg
        for i, sg in enumerate(segs[g]):
            for name, p, gr in (("A", sg.A, dA[i]), ("B", sg.B, dB[i])):
                m, v = state.get((name, g, i), (0.0, 0.0))
                p2, m, v = orc.adamw(p, gr, m, v, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, t)
                state[(name, g, i)] = (m, v)
    return Y, dX


class OracleLayer:
    """The oracle's step over every projection of the workload, on a token sample."""

    def __init__(self, wl, per_job):
        self.samples = [oracle_sample(p, per_job) for p in parts_of(wl)]
        self.tokens = self.samples[0][-1]
        self.states = [{} for _ in self.samples]

    def step(self, t):
        for (sub, X, Wm, dY, segs, _), st in zip(self.samples, self.states):
            oracle_step(sub, X, Wm, dY, segs, st, t)


def cores_used():
    return os.cpu_count() or 1


def run_reference(args, wl, rank):
    """The reference arm of this metric: the fp64 CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return
    # size each step's sample so the whole run stays near --ref-budget-s seconds
    probe = OracleLayer(wl, 8)
    t0 = time.perf_counter()
    probe.step(1)
    per_tok = (time.perf_counter() - t0) / probe.tokens
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    per_job = int(max(1, min(args.ref_tokens_per_job, budget / per_tok / len(wl.n_tokens))))
    orl = OracleLayer(wl, per_job)
    for t in range(1, args.warmup + 1):
        orl.step(t)
    t0 = time.perf_counter()
    for t in range(args.warmup + 1, args.warmup + args.steps + 1):
        orl.step(t)
    dt = time.perf_counter() - t0
    value = orl.tokens * args.steps / dt
    sample = (f"first {per_job} tokens of each of the {len(wl.n_tokens)} jobs ({orl.tokens} tokens) through every "
              f"projection, full d_in x d_out")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Philox)", "config": config_of(wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(wl, ngpus):
    """The workload as both arms report it (identical dicts)."""
    parts = parts_of(wl)
    p0 = parts[0]
    c = {"workload": wl.name}
    if hasattr(wl, "parts"):
        c["projections"] = [{"name": n, "d_in": p.d_in, "d_out": p.d_out} for n, p in zip(labels_of(wl), parts)]
        c["jobs"] = len(p0.n_tokens)
        c["adapters"] = sum(p.n_adapters for p in parts)
    else:
        c["d_in"], c["d_out"] = p0.d_in, p0.d_out
        c["adapters"] = p0.n_adapters
    c.update({"ranks": p0.ranks, "tokens_per_step": wl.N, "dtype_io": p0.dtype,
              "parallelism": "one GPU" if ngpus == 1 else
              f"jobs sharded over {ngpus} GPUs (whole jobs, longest first; no collective)",
              "l2": "inputs larger than L2 (X and dY are N x d bf16, each above the 129 MB L2)"
              if p0.N * min(p0.d_in, p0.d_out) * 2 > 129e6 else "inputs smaller than L2"})
    return c


def options_of(wl, args):
    opts = []
    if not args.no_reuse:
        opts.append("MLORA_REUSE_STAGING (backward reuses the forward's bf16 shadows and staged H)")
    if args.window != "auto":
        opts.append({"pairs": "MLORA_WINDOW_PAIRS", "single": "MLORA_WINDOW_SINGLE"}[args.window])
    if args.no_overlap:
        opts.append("MLORA_NO_OVERLAP (each kernel launched after the previous one ends)")
    if args.overlap:
        opts.append("MLORA_OVERLAP (programmatic overlap whatever the plan's size)")
    if parts_of(wl)[0].dtype == "bf16_w4":
        opts.append("MLORA_W4_FUSED (codes expanded inside the base GEMMs)" if args.w4_fused else
                    "4-bit base expanded to bf16 once per call, then the bf16 GEMMs")
    return "; ".join(opts) or None


def traffic_record(wl_name, kernel):
    """DRAM bytes of one step's launches of `kernel` on workload `wl_name` from a committed ncu
    summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    r = rec.get(f"{wl_name}:{kernel}")
    if not r:
        return None
    for src, sha in r["sources"].items():
        data = open(os.path.join(ROOT, src), "rb").read()
        if hashlib.sha256(data).hexdigest()[:16] != sha:
            return None
    return r.get("bytes_per_step")


class PartRun:
    """One projection on this GPU: its plan and buffers (PackedLoRA), device-resident inputs and
    the pinned host copies the end-to-end pass streams in."""

    def __init__(self, wl, T, flags, label):
        import numpy as np
        import torch
        from adapter_gemm_packed_gb300.layer import PackedLoRA
        self.wl, self.label = wl, label
        scales = [np.float32(a) / np.float32(r) for a, r in zip(wl.alphas, wl.ranks)]
        if wl.groups is None:
            self.layer = PackedLoRA(wl.d_in, wl.d_out, wl.ranks, wl.n_tokens, scales, dtype=wl.dtype, At=T.At,
                                    Bt=T.Bt, flags=flags)
        else:
            # shared-input pack: one adapter per job and projection, the projections stacked in W
            self.layer = PackedLoRA(wl.d_in, wl.d_out, wl.nest(wl.ranks), wl.n_tokens, wl.nest(scales),
                                    dtype=wl.dtype, At=wl.nest(T.At), Bt=wl.nest(T.Bt), flags=flags,
                                    groups=wl.groups)
        tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16

        def host(a):
            t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if wl.dtype != "f32" else torch.from_numpy(a)
            return t.pin_memory()

        self.X_h, self.dY_h = host(T.X), host(T.dY)
        self.X, self.dY = self.X_h.cuda(), self.dY_h.cuda()
        if wl.dtype == "bf16_w4":
            self.Wt = (torch.from_numpy(T.Wq).cuda(), torch.from_numpy(T.Wscale).cuda())
        else:
            self.Wt = host(T.Wt).cuda()
        self.Y = torch.empty((wl.N, wl.d_out), dtype=tdt, device="cuda")
        self.dX = torch.empty((wl.N, wl.d_in), dtype=tdt, device="cuda")

    def in_bytes(self):
        return self.X.numel() * self.X.element_size() + self.dY.numel() * self.dY.element_size()

    def out_bytes(self):
        return self.Y.numel() * self.Y.element_size() + self.dX.numel() * self.dX.element_size()


def layer_step(runs, t, bufs=None, stream=None):
    """One training step of the layer: every projection's forward (first to last), every
    backward (last to first), then every AdamW step.  `bufs[i]` = (X, dY, Y, dX) of run i."""
    wl = runs[0].wl
    io = bufs or [(r.X, r.dY, r.Y, r.dX) for r in runs]
    for r, (X, dY, Y, dX) in zip(runs, io):
        r.layer.forward(X, r.Wt, Y, stream=stream)
    for r, (X, dY, Y, dX) in reversed(list(zip(runs, io))):
        r.layer.backward(X, r.Wt, dY, dX, stream=stream)
    for r in runs:
        r.layer.adamw(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, t, stream=stream)


def aggregate_kernels(runs, profs, steps, prof_step_ms, layered):
    """Per kernel over all projections: time per step, launches, share, and the achieved rate of
    its algorithmic FLOPs or bytes (their sum over the launches over the launches' summed time)."""
    agg = {}
    for r, prof in zip(runs, profs):
        for k, (ms_k, n_k) in prof.items():
            if n_k == 0:
                continue
            e = agg.setdefault(k, {"ms": 0.0, "launches": 0, "flops": 0.0, "bytes": 0.0, "by_projection": {}})
            e["ms"] += ms_k
            e["launches"] += n_k
            f, b = kernel_flops(r.wl, k), kernel_bytes(r.wl, k)
            pp = {"ms_per_launch": ms_k / n_k}
            if f:
                e["flops"] += f * n_k
                pp["tflops"] = f / (ms_k / n_k * 1e-3) / 1e12
            if b:
                e["bytes"] += b * n_k
                pp["gbs"] = b / (ms_k / n_k * 1e-3) / 1e9
            e["by_projection"][r.label] = pp
    out = {}
    for k, e in agg.items():
        v = {"ms_per_launch": e["ms"] / e["launches"], "launches": e["launches"],
             "launches_per_step": e["launches"] / steps, "ms_per_step": e["ms"] / steps,
             "share_of_step": e["ms"] / steps / prof_step_ms}
        if e["flops"]:
            v["tflops"] = e["flops"] / (e["ms"] * 1e-3) / 1e12
        if e["bytes"]:
            v["gbs"] = e["bytes"] / (e["ms"] * 1e-3) / 1e9
        if layered:
            v["by_projection"] = e["by_projection"]
        out[k] = v
    return out


def run_ours(args, wl, rank, world, local_rank):
    import torch
    from adapter_gemm_packed_gb300 import _mlora as M
    from adapter_gemm_packed_gb300 import workloads as W

    dist = world > 1
    torch.cuda.set_device(local_rank)
    parts, labels = parts_of(wl), labels_of(wl)
    layered = hasattr(wl, "parts")
    flags = (0 if args.no_reuse else M.MLORA_REUSE_STAGING) | (M.MLORA_W4_FUSED if args.w4_fused else 0)
    flags |= {"auto": 0, "pairs": M.MLORA_WINDOW_PAIRS, "single": M.MLORA_WINDOW_SINGLE}[args.window]
    flags |= M.MLORA_NO_OVERLAP if args.no_overlap else 0
    flags |= M.MLORA_OVERLAP if args.overlap else 0
    # this rank's jobs (all of them on one GPU)
    rank_of_job, load = shard(wl, world)
    mine = jobs_of_rank(rank_of_job, rank)
    runs = []
    for p, lab in zip(parts, labels):
        if not mine:
            break
        if world == 1:
            T = W.materialise(p)
            sub = p
        else:
            sub, T = W.materialise_jobs(p, mine)
        runs.append(PartRun(sub, T, flags, lab))
        del T
    stream = torch.cuda.current_stream()
    t_no = [0]

    def step():
        t_no[0] += 1
        if runs:
            layer_step(runs, t_no[0])

    def barrier():
        if dist:
            torch.distributed.barrier()

    def check(where):
        for r in runs:
            if r.layer.sync_status() != M.MLORA_OK:
                raise SystemExit(f"device status error {where} ({r.label})")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    check("during warm-up")

    # ---- timed region (device): K steps back to back on one stream
    launches0 = M.mlora_launch_count()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    launches = M.mlora_launch_count() - launches0
    check("in the timed region")
    ms_rank = ms
    ms = max_over_ranks(ms, device="cuda")

    # ---- per-kernel times: the same K steps again with the library recording a CUDA event pair
    # around every launch on the launching stream (events between launches serialise them, so
    # this pass is kept out of the headline number)
    for r in runs:
        M.mlora_profile_enable(r.layer.plan, True)
        M.mlora_profile_read(r.layer.plan)
    torch.cuda.synchronize()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    torch.cuda.synchronize()
    prof_ms = p0.elapsed_time(p1)
    profs = [M.mlora_profile_read(r.layer.plan) for r in runs]
    for r in runs:
        M.mlora_profile_enable(r.layer.plan, False)

    # ---- end to end through the public API: every step copies every projection's inputs X, dY
    # from pinned host memory to the device and its results Y, dX back.  The copies of step
    # i+1 / i-1 run on their own streams while step i computes (double-buffered device buffers,
    # ordered by events), as an input pipeline of a training loop would.
    e2e = None
    if not args.no_e2e and runs:
        Y_h = [torch.empty_like(r.Y, device="cpu").pin_memory() for r in runs]
        dX_h = [torch.empty_like(r.dX, device="cpu").pin_memory() for r in runs]
        dev = [[(r.X, r.dY, r.Y, r.dX),
                (torch.empty_like(r.X), torch.empty_like(r.dY), torch.empty_like(r.Y), torch.empty_like(r.dX))]
               for r in runs]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        h2d_done = [ev(), ev()]
        comp_done = [ev(), ev()]
        d2h_done = [ev(), ev()]
        started = [False, False]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if started[b]:
                    s_in.wait_event(comp_done[b])        # step i-2 has finished reading these inputs
                for r, d in zip(runs, dev):
                    d[b][0].copy_(r.X_h, non_blocking=True)
                    d[b][1].copy_(r.dY_h, non_blocking=True)
                h2d_done[b].record(s_in)
            stream.wait_event(h2d_done[b])
            if started[b]:
                stream.wait_event(d2h_done[b])           # step i-2's results have left these outputs
            t_no[0] += 1
            layer_step(runs, t_no[0], [d[b] for d in dev], stream=stream)
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for j, d in enumerate(dev):
                    Y_h[j].copy_(d[b][2], non_blocking=True)
                    dX_h[j].copy_(d[b][3], non_blocking=True)
                d2h_done[b].record(s_out)
            started[b] = True

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1), device="cuda")
        b_in = sum(r.in_bytes() for r in runs)
        b_out = sum(r.out_bytes() for r in runs)
        e2e = {"value": pack_rate(wl.N, args.steps, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": b_in, "d2h_bytes_per_step": b_out, "ms_per_step": ems / args.steps,
               "pipelined": "H2D and D2H copies on their own streams, double-buffered device buffers"}
        if dist:
            e2e["bytes_note"] = "h2d / d2h bytes are rank 0's share of the pack"
        # The host link bounds this number: measure it here (one direction at a time, then both at
        # once, on equal-sized pinned copies: the largest run's X and Y cut to the smaller of the
        # two) and report the per-direction rate the pipeline reached.
        big = max(runs, key=lambda r: min(r.X.numel(), r.Y.numel()))
        n = min(big.X.numel(), big.Y.numel())
        j = runs.index(big)
        link = link_probe(big.X_h.view(-1)[:n], big.X.view(-1)[:n], Y_h[j].view(-1)[:n], big.Y.view(-1)[:n],
                          s_in, s_out)
        step_s = ems / args.steps / 1e3
        e2e["link"] = dict(link, achieved_h2d_gbs=b_in / step_s / 1e9, achieved_d2h_gbs=b_out / step_s / 1e9,
                           frac_of_concurrent=max(b_in, b_out) / step_s / 1e9 / link["concurrent_gbs_per_direction"])
        check("in the end-to-end region")

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    step_ms = ms / args.steps
    prof_step_ms = prof_ms / args.steps
    kernels = aggregate_kernels(runs, profs, args.steps, prof_step_ms, layered)
    sustained = ms_rank >= SUSTAINED_AFTER_MS
    if parts[0].dtype != "f32":
        dom = max(("fwd_gemm", "bwd_gemm"), key=lambda k: kernels.get(k, {}).get("ms_per_step", 0))
        dk = kernels[dom]
        burst, sust = peaks.get("bf16_tflops"), peaks.get("bf16_tflops_sustained")
        peak = sust if (sustained and sust) else burst
        roof = {"kernel": dom, "bound": "tensor", "achieved": dk["tflops"], "peak": peak, "unit": "TFLOP/s",
                "frac": dk["tflops"] / peak,
                "peak_source": f"{peak_src} bf16_tflops_sustained (long power-capped loop; this timed region is "
                               f"{ms_rank / 1e3:.1f} s)" if peak == sust else
                               f"{peak_src} bf16_tflops (burst cuBLAS GEMM; this timed region is {ms_rank:.0f} ms)",
                "frac_of_burst": dk["tflops"] / burst if burst else None,
                "frac_of_sustained": dk["tflops"] / sust if sust else None,
                "launches_per_step": dk["launches_per_step"],
                "traffic": traffic_record(wl.name, dom)}
        if layered:
            roof["achieved_is"] = (f"algorithmic FLOPs of one step's {dom} launches (one per projection) over "
                                   f"their summed CUDA-event time; traffic is those launches' DRAM bytes")
    else:
        # fp32 path: plain FFMA.  Peak = SMs x 128 FFMA lanes x 2 FLOP x max SM clock.
        p0 = parts[0]
        dom = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
        nr = sum(n * r for n, r in zip(p0.n_tokens, p0.ranks))
        f = {"f32_forward": 2.0 * p0.N * p0.d_in * p0.d_out + 2.0 * nr * (p0.d_in + p0.d_out),     # XW, XA, HB
             "f32_backward": 2.0 * p0.N * p0.d_in * p0.d_out + 4.0 * nr * (p0.d_in + p0.d_out)}    # dYW^T, dH, dX_lora, dA, dB
        sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
        peak = sms * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        ach = f.get(dom, 0.0) / (kernels[dom]["ms_per_launch"] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "peak_source": "derived: SMs x 128 FP32 lanes x 2 FLOP x max SM clock", "traffic": None}
    hbm = peaks.get("hbm_gbs")
    for k in ("shrink", "dH", "dA", "dB", "adamw", "w4_expand"):
        if k in kernels and "gbs" in kernels[k]:
            kernels[k]["frac_of_hbm"] = kernels[k]["gbs"] / hbm
    line = {"metric": METRIC, "value": pack_rate(wl.N, args.steps, ms), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "f32": "f32", "bf16_w4": "bf16 (4-bit base)"}[parts[0].dtype],
            "data": "synthetic (seeded Philox; shapes of the named workload, random-init adapters)",
            "config": config_of(wl, world), "options": options_of(wl, args),
            "tflops": flops_per_step(wl) * args.steps / (ms / 1e3) / 1e12,
            "roofline": roof, "kernels": kernels, "kernel_timing_ms_per_step": prof_step_ms,
            "gpu_launches": launches, "e2e": e2e, "clocks": clk.summary()}
    if dist:
        toks = [sum(parts[0].n_tokens[j] for j in jobs_of_rank(rank_of_job, q)) for q in range(world)]
        line["shard"] = {"jobs_per_rank": [len(jobs_of_rank(rank_of_job, q)) for q in range(world)],
                         "tokens_per_rank": toks, "cost_balance_max_over_mean": max(load) / (sum(load) / world),
                         "note": "kernels, gpu_launches and e2e bytes are rank 0's"}
    if not args.no_cpu_baseline and world == 1:
        orl = OracleLayer(wl, args.ref_tokens_per_job)
        t, reps = 0, 0
        t0 = time.perf_counter()
        while reps < 1 or (time.perf_counter() - t0 < args.cpu_seconds and reps < 50):
            t += 1
            orl.step(t)
            reps += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": orl.tokens * reps / dt, "unit": "tokens/s", "cores": cores_used(),
                                "kind": "oracle",
                                "sample": f"first {args.ref_tokens_per_job} tokens of each job ({orl.tokens} tokens) "
                                          f"through every projection x {reps} steps, fp64 numpy "
                                          f"(BLAS threads = cores)"}
    print(json.dumps(line), flush=True)
    for r in runs:
        r.layer.close()


SWEEP_LAYERS = [("qwen2.5_3b_attn_2048x2048", 2048, 2048), ("qwen2.5_3b_mlp_up_2048x11008", 2048, 11008),
                ("qwen2.5_7b_attn_3584x3584", 3584, 3584), ("qwen2.5_7b_mlp_up_3584x18944", 3584, 18944)]
SWEEP_JOBS = [1, 2, 4, 8, 16, 32]


def run_sweep(args):
    """One JSON line per (layer, job count): a step of the whole pack (forward, backward, AdamW) as
    one plan, the same jobs one plan at a time back to back, and a PyTorch / cuBLAS comparator that
    batches the base GEMMs over all tokens but runs the LoRA products adapter by adapter (then one
    fused torch AdamW over all adapters).  Inputs are seeded device draws; the L2 is flushed before
    every timed step, outside the CUDA events."""
    import torch
    from adapter_gemm_packed_gb300 import _mlora as M
    from adapter_gemm_packed_gb300.layer import PackedLoRA

    torch.cuda.set_device(0)
    r, n_tok, s = 64, 1024, 2.0                 # s = alpha / r with alpha = 2 r
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    bf = torch.bfloat16
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")    # twice the 129 MB L2

    def timed(step):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        total = 0.0
        for _ in range(args.sweep_steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
        return total / args.sweep_steps

    def rel(a, b):
        return float((a.float() - b.float()).norm() / b.float().norm())

    gen = torch.Generator(device="cuda")
    layers = [x for x in SWEEP_LAYERS if not args.sweep_layers or x[0] in args.sweep_layers.split(",")]
    jobs = [int(j) for j in args.sweep_jobs.split(",")] if args.sweep_jobs else SWEEP_JOBS
    if not layers:
        raise SystemExit(f"--sweep-layers: none of {[x[0] for x in SWEEP_LAYERS]}")
    for name, d_in, d_out in layers:
        li = [x[0] for x in SWEEP_LAYERS].index(name)
        for n_jobs in jobs:
            gen.manual_seed(7000 + 100 * li + n_jobs)
            N = n_jobs * n_tok
            randn = lambda *shape: torch.randn(*shape, generator=gen, device="cuda")
            Wt = (randn(d_out, d_in) * 0.02).to(bf)
            At = [randn(r, d_in) * d_in ** -0.5 for _ in range(n_jobs)]
            Bt = [randn(d_out, r) * 0.02 for _ in range(n_jobs)]
            X = randn(N, d_in).to(bf)
            dY = (randn(N, d_out) * 0.01).to(bf)
            rows = [slice(j * n_tok, (j + 1) * n_tok) for j in range(n_jobs)]

            # the pack as one plan (its own copies of the masters, as every arm below)
            layer = PackedLoRA(d_in, d_out, [r] * n_jobs, [n_tok] * n_jobs, [s] * n_jobs, At=[a.clone() for a in At],
                               Bt=[b.clone() for b in Bt],
                               flags=M.MLORA_REUSE_STAGING)
            Y, dX = torch.empty(N, d_out, dtype=bf, device="cuda"), torch.empty(N, d_in, dtype=bf, device="cuda")
            layer.forward(X, Wt, Y)
            layer.backward(X, Wt, dY, dX)
            Y0, dX0 = Y.clone(), dX.clone()
            t = [0]

            def packed():
                t[0] += 1
                layer.forward(X, Wt, Y)
                layer.backward(X, Wt, dY, dX)
                layer.adamw(lr, b1, b2, eps, wd, t[0])

            # the same jobs, one plan each, run one after another
            singles = [PackedLoRA(d_in, d_out, [r], [n_tok], [s], At=[At[j].clone()], Bt=[Bt[j].clone()],
                                  flags=M.MLORA_REUSE_STAGING)
                       for j in range(n_jobs)]
            t1 = [0]

            def one_at_a_time():
                t1[0] += 1
                for j, L in enumerate(singles):
                    L.forward(X[rows[j]], Wt, Y[rows[j]])
                    L.backward(X[rows[j]], Wt, dY[rows[j]], dX[rows[j]])
                    L.adamw(lr, b1, b2, eps, wd, t1[0])

            # PyTorch comparator: batched base GEMMs, per-adapter LoRA products, fused AdamW
            A = [a.clone() for a in At]
            B = [b.clone() for b in Bt]
            opt = torch.optim.AdamW(A + B, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, fused=True)

            def torch_naive(update=True):
                Yt = torch.nn.functional.linear(X, Wt)
                Ab, Bb = [a.to(bf) for a in A], [b.to(bf) for b in B]
                Hs = []
                for j, sl in enumerate(rows):
                    H = X[sl] @ Ab[j].t()
                    Yt[sl] += s * (H @ Bb[j].t())
                    Hs.append(H)
                dXt = dY @ Wt
                for j, sl in enumerate(rows):
                    B[j].grad = (s * (dY[sl].t() @ Hs[j])).float()
                    dH = s * (dY[sl] @ Bb[j])
                    A[j].grad = (dH.t() @ X[sl]).float()
                    dXt[sl] += dH @ Ab[j]
                if update:
                    opt.step()
                return Yt, dXt

            Yt, dXt = torch_naive(update=False)
            agree = {"Y": rel(Y0, Yt), "dX": rel(dX0, dXt)}
            ms_packed = timed(packed)
            ms_single = timed(one_at_a_time)
            ms_torch = timed(torch_naive)
            if layer.sync_status() != M.MLORA_OK or any(L.sync_status() != M.MLORA_OK for L in singles):
                raise SystemExit("device status error in the sweep")
            flops = 4.0 * N * d_in * d_out + 6.0 * N * r * (d_in + d_out)
            print(json.dumps({"sweep": "packed_vs_sequential", "layer": name, "d_in": d_in, "d_out": d_out, "rank": r,
                              "jobs": n_jobs, "tokens": N, "packed_ms": ms_packed, "one_plan_per_job_ms": ms_single,
                              "torch_per_adapter_ms": ms_torch, "speedup_vs_one_plan_per_job": ms_single / ms_packed,
                              "speedup_vs_torch_per_adapter": ms_torch / ms_packed,
                              "packed_tflops": flops / (ms_packed * 1e-3) / 1e12,
                              "agreement_rel_frobenius": agree, "l2": "flushed before every timed step",
                              "steps": args.sweep_steps, "warmup": 3}), flush=True)
            layer.close()
            for L in singles:
                L.close()
            del layer, singles, opt, A, B, X, dY, Y, dX, Wt, At, Bt
            torch.cuda.empty_cache()


# Cost-table calibration: the seven Llama-3-8B projections, the Qwen-2.5 shapes of the sweep and the
# many-small-jobs down projection, each at several pack sizes of 1024-token jobs.
CALIBRATE_SHAPES = [(4096, 4096), (4096, 1024), (4096, 14336), (14336, 4096), (2048, 2048), (2048, 11008),
                    (3584, 3584), (3584, 18944), (28672, 8192)]
CALIBRATE_TOKENS = [1024, 4096, 16384, 65536, 143360]
CALIBRATE_RANKS = [8, 16, 32, 64, 128]


def run_calibrate(args):
    """Measure the step time (forward + backward + AdamW, back-to-back steps, inputs in device memory)
    of packs of 1024-token jobs with ranks cycling through 8..128, for every shape and size above,
    and write the cost table mlora_cost_estimate interpolates (adapter_gemm_packed_gb300/
    cost_table_gb300.json, or --calibrate-out)."""
    import torch
    from adapter_gemm_packed_gb300 import _mlora as M
    from adapter_gemm_packed_gb300 import cost
    from adapter_gemm_packed_gb300.layer import PackedLoRA

    torch.cuda.set_device(0)
    gen = torch.Generator(device="cuda")
    bf = torch.bfloat16
    points = []
    for d_in, d_out in CALIBRATE_SHAPES:
        for N in CALIBRATE_TOKENS:
            if N * (d_in + d_out) * 2 * 4 > 120e9:
                continue
            gen.manual_seed(11 * d_in + d_out + N)
            J = max(1, N // 1024)
            toks = [N // J] * J
            toks[-1] += N - sum(toks)
            ranks = [CALIBRATE_RANKS[j % len(CALIBRATE_RANKS)] for j in range(J)]
            At = [torch.randn(r, d_in, device="cuda", generator=gen) * d_in ** -0.5 for r in ranks]
            Bt = [torch.randn(d_out, r, device="cuda", generator=gen) * 0.02 for r in ranks]
            layer = PackedLoRA(d_in, d_out, ranks, toks, [2.0] * J, At=At, Bt=Bt, flags=M.MLORA_REUSE_STAGING)
            X = torch.randn(N, d_in, device="cuda", generator=gen).to(bf)
            dY = torch.randn(N, d_out, device="cuda", generator=gen).to(bf)
            Wt = (torch.randn(d_out, d_in, device="cuda", generator=gen) * 0.02).to(bf)
            Y = torch.empty(N, d_out, dtype=bf, device="cuda")
            dX = torch.empty(N, d_in, dtype=bf, device="cuda")
            t = [0]

            def step():
                t[0] += 1
                layer.forward(X, Wt, Y)
                layer.backward(X, Wt, dY, dX)
                layer.adamw(1e-3, 0.9, 0.999, 1e-8, 0.01, t[0])

            for _ in range(3):
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.calibrate_steps):
                step()
            e1.record()
            torch.cuda.synchronize()
            if layer.sync_status() != M.MLORA_OK:
                raise SystemExit("device status error in calibration")
            ms = e0.elapsed_time(e1) / args.calibrate_steps
            work = float(sum(n * r * (d_in + d_out) for n, r in zip(toks, ranks)))
            points.append({"d_in": d_in, "d_out": d_out, "n_tokens": N, "jobs": J, "lora_work": work, "step_ms": ms})
            print(json.dumps(points[-1]), flush=True)
            layer.close()
            del layer, X, dY, Wt, Y, dX, At, Bt
            torch.cuda.empty_cache()
    out = args.calibrate_out or cost.TABLE_PATH
    with open(out, "w") as f:
        json.dump({"what": "step time (forward + backward + AdamW) of packs of 1024-token jobs, ranks cycling "
                           "8..128, bf16, back-to-back steps with inputs in device memory; one GB300",
                   "command": "python bench.py --calibrate", "steps": args.calibrate_steps,
                   "gpu": torch.cuda.get_device_name(0), "points": points}, f, indent=1)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="layer (default: the 7 projections of a Llama-3-8B decoder layer), qproj, mlp_up, many_small, ...")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-reuse", action="store_true", help="rebuild the backward's staging (no MLORA_REUSE_STAGING)")
    ap.add_argument("--w4-fused", action="store_true", help="4-bit base: expand inside the GEMMs (MLORA_W4_FUSED)")
    ap.add_argument("--window", choices=["auto", "pairs", "single"], default="auto",
                    help="engine of the shrink / dH products (default: the planner's choice)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch every kernel after the previous one ends (MLORA_NO_OVERLAP)")
    ap.add_argument("--overlap", action="store_true",
                    help="keep the programmatic overlap whatever the plan's size (MLORA_OVERLAP)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens-per-job", type=int, default=64)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    ap.add_argument("--sweep", action="store_true",
                    help="packed vs sequential over Qwen-2.5 layer shapes (one JSON line per point, one GPU)")
    ap.add_argument("--sweep-steps", type=int, default=10)
    ap.add_argument("--sweep-layers", default="", help="comma-separated subset of the sweep's layer names")
    ap.add_argument("--sweep-jobs", default="", help="comma-separated job counts (default 1,2,4,8,16,32)")
    ap.add_argument("--calibrate", action="store_true",
                    help="measure the cost table of mlora_cost_estimate (one GPU) and write it")
    ap.add_argument("--calibrate-steps", type=int, default=10)
    ap.add_argument("--calibrate-out", default="")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.sweep or args.calibrate:
        if world > 1:
            raise SystemExit("--sweep and --calibrate run on one GPU")
        import __graft_entry__
        __graft_entry__.build()
        run_sweep(args) if args.sweep else run_calibrate(args)
        return
    wl = workload(args.workload)
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    run_ours(args, wl, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
