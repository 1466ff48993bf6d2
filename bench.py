#!/usr/bin/env python3
"""FlashAttention-2 forward benchmark on GB300: TFLOP/s and fraction of the
tensor-core roofline, one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one forward pass (one launch of the library's kernel) over the
workload's synthetic inputs, resident in HBM.  Default workload: B=4, H=32,
N_q=N_k=8192, d=128, bf16, non-causal, scale 1/sqrt(128).  FLOPs per step =
4*B*H*N_q*N_k*d (halved when causal).  With N GPUs (torchrun) every rank runs
its own copy of the workload (independent problems, no collective on the data
path): weak scaling, value = FLOPs of all ranks / slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (the correctness reference) on
the host cores, on a bounded sample of rows of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402
import torch  # noqa: E402

NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25   # dense tf32 / bf16 nominal tensor rates
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="large_nc")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--api", choices=["fa", "sdpa"], default="fa",
                    help="forward through fa.fwd (default) or through torch.nn.functional."
                         "scaled_dot_product_attention routed to this library")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and whitespace: what the compiler
    sees of the kernels (string literals are left alone; none holds '//')."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments and whitespace ignored), the
    key under which the committed DRAM-traffic records were taken."""
    h = hashlib.sha256()
    for f in sorted((ROOT / "attention_fa2_fwd_02_gb300" / "csrc").glob("*")):
        h.update(f.name.encode())
        h.update(_code_only(f.read_text(errors="replace")).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = ROOT / "profiles" / "dram_traffic.json"
    if not p.exists():
        return None
    try:
        d = json.loads(p.read_text())
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    ent = d.get("workloads", {}).get(workload)
    return None if ent is None else float(ent["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        target = str(self.dev)
        try:
            bus = torch.cuda.get_device_properties(self.dev).pci_bus_id  # type: ignore[attr-defined]
            if bus:
                target = bus
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", target],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(backend: str | None = None):
    """(world, rank, local_rank, torch.distributed or None) from the torchrun
    environment.  One process per GPU over NCCL; gloo when no GPU is present
    (the multi-rank logic is tested that way on CPU)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
        return world, rank, local, dist
    return 1, 0, 0, None


def max_over_ranks(x: float, dist) -> float:
    """The slowest rank's time (timing only: no collective touches the data)."""
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_step: float, world: int, slowest_ms_per_step: float) -> float:
    """Weak scaling: every rank runs its own copy of the workload, so the job
    processes world x flops per step in the slowest rank's step time (TFLOP/s)."""
    return flops_per_step * world / (slowest_ms_per_step * 1e-3) / 1e12


def workload_desc(w) -> dict:
    from attention_fa2_fwd_02_gb300.inputs import AxialBlockWorkload, AxialWorkload, VarlenWorkload
    if isinstance(w, VarlenWorkload):
        lens = w.lens
        kind = "causal (top-left, per sequence)" if w.causal else "non-causal"
        return {"workload": f"{w.name}: packed batch of {w.n_seq} sequences, lengths uniform in [{w.lo}, {w.hi}] "
                            f"(seed {w.seed}; total {sum(lens)} tokens, max {max(lens)}), H={w.H} d={w.d} bf16 "
                            f"{kind}, scale={w.scale:.6g}",
                "lengths": lens, "H": w.H, "H_kv": w.kv_heads, "d": w.d, "dtype": "bf16", "causal": w.causal,
                "scale": w.scale}
    if isinstance(w, AxialBlockWorkload):
        return {"workload": f"axial attention block x[{w.B},{w.H},{w.W},{w.D}] fp32, {w.heads} heads: LayerNorm + "
                            f"QKV + attention + out-projection + residual, row pass then column pass, "
                            f"random weights",
                "shape": list(w.shape), "heads": w.heads}
    if isinstance(w, AxialWorkload):
        return {"workload": f"axial attention core x[{w.B},{w.Hg},{w.Wg},{w.heads},{w.hd}] fp32, "
                            f"row + column, scale {w.scale}",
                "shape": list(w.shape), "scale": w.scale, "causal": False}
    kind = "causal" if w.causal else "non-causal"
    dt = "bf16" if w.dtype == torch.bfloat16 else "fp32"
    gqa = f" H_kv={w.kv_heads}" if w.kv_heads != w.H else ""
    dv = f" Dv={w.v_dim}" if w.v_dim != w.d else ""
    return {"workload": f"{w.name}: B={w.B} H={w.H}{gqa} N_q={w.N_q} N_k={w.N_k} d={w.d}{dv} {dt} {kind}, "
                        f"scale={w.scale:.6g}",
            "B": w.B, "H": w.H, "H_kv": w.kv_heads, "N_q": w.N_q, "N_k": w.N_k, "d": w.d, "Dv": w.v_dim,
            "dtype": dt, "causal": w.causal, "scale": w.scale}


def get_workload(name):
    """The workload; names ending in ``_bwd`` time the backward pass of the
    named forward workload (bf16, head dims up to 128)."""
    from attention_fa2_fwd_02_gb300.inputs import AXIAL, AXIAL_BLOCK, VARLEN, WORKLOADS
    if name in VARLEN:
        return VARLEN[name]
    if name == "axial":
        return AXIAL
    if name == "axial_block":
        return AXIAL_BLOCK
    base = name[:-4] if name.endswith("_bwd") else name
    if base not in WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(WORKLOADS)}, {sorted(VARLEN)}, "
                         f"axial, axial_block, or <bf16 workload>_bwd")
    w = WORKLOADS[base]
    if name.endswith("_bwd") and (w.dtype != torch.bfloat16 or max(w.d, w.v_dim) > 128):
        raise SystemExit(f"{name}: the backward runs on bf16 workloads with head dims up to 128")
    return w


def bwd_flops(w) -> float:
    """Backward FLOPs: five products per (b, h), 2*N_q*N_k times d for S, dK and
    dQ and times Dv for dP and dV (2.5x the forward's two when Dv = d); halved
    when causal."""
    f = 2.0 * w.B * w.H * w.N_q * w.N_k * (3 * w.d + 2 * w.v_dim)
    return f / 2 if w.causal else f


def bwd_oracle_sample(w, Q, K, V, G, budget_s: float):
    """The backward oracle (as it stands) on the leading n x n block of random
    (b, h) slices, n grown until one call takes ~budget_s / 4; returns
    (algorithmic flops, seconds, description)."""
    import oracle
    oracle.build()
    g = np.random.default_rng(0)
    n = 128
    flops, calls, t0 = 0.0, 0, time.perf_counter()
    while True:
        b, h = int(g.integers(w.B)), int(g.integers(w.H))
        nq, nk = min(n, w.N_q), min(n, w.N_k)
        t1 = time.perf_counter()
        hk = h // (w.H // w.kv_heads)
        oracle.attention_bwd(Q[b, h, :nq], K[b, hk, :nk], V[b, hk, :nk], G[b, h, :nq], w.scale, w.causal)
        one = time.perf_counter() - t1
        flops += 2.0 * nq * nk * (3 * w.d + 2 * w.v_dim) * (0.5 if w.causal else 1.0)
        calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
        if one < budget_s / 8 and n < min(w.N_q, w.N_k):
            n *= 2
    dt = time.perf_counter() - t0
    return flops, dt, (f"{calls} backward calls on leading blocks (up to {n}x{n}) of random (b,h) slices "
                       f"of the same inputs; flops counted as 10*n_q*n_k*d (halved causal)")


# ------------------------------------------------------------ CPU oracle leg
def oracle_sample(w, Q, K, V, budget_s: float, rows_per_call: int = 512):
    """Run the oracle (as it stands) on rows of the workload until ~budget_s
    seconds of CPU work; return (flops, seconds, description)."""
    import oracle
    oracle.build()
    from attention_fa2_fwd_02_gb300.inputs import AxialWorkload
    if isinstance(w, AxialWorkload):
        qr = Q.permute(0, 1, 3, 2, 4).reshape(-1, w.Wg, w.hd)
        kr = K.permute(0, 1, 3, 2, 4).reshape(-1, w.Wg, w.hd)
        vr = V.permute(0, 1, 3, 2, 4).reshape(-1, w.Wg, w.hd)
        qc = Q.permute(0, 2, 3, 1, 4).reshape(-1, w.Hg, w.hd)
        kc = K.permute(0, 2, 3, 1, 4).reshape(-1, w.Hg, w.hd)
        vc = V.permute(0, 2, 3, 1, 4).reshape(-1, w.Hg, w.hd)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.attention(qr, kr, vr, w.scale)
            oracle.attention(qc, kc, vc, w.scale)
            reps += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return w.flops * reps, dt, f"{reps} full row+column passes of the axial workload"
    g = np.random.default_rng(0)
    flops = 0.0
    n_rows = 0
    t0 = time.perf_counter()
    while True:
        b, h = int(g.integers(w.B)), int(g.integers(w.H))
        r0 = int(g.integers(0, max(1, w.N_q - rows_per_call + 1)))
        rows = np.arange(r0, min(w.N_q, r0 + rows_per_call))
        hk = h // (w.H // w.kv_heads)  # the K/V head of query head h
        oracle.attention(Q[b, h], K[b, hk], V[b, hk], w.scale, w.causal, rows=rows)
        nvis = np.minimum(rows + 1, w.N_k) if w.causal else np.full(rows.size, w.N_k)
        flops += float(2.0 * (w.d + w.v_dim) * nvis.sum())
        n_rows += rows.size
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return flops, dt, f"{n_rows} query rows ({rows_per_call}-row blocks of random (b,h) slices)"


def varlen_oracle_sample(w, q, k, v, cu, budget_s: float, rows_per_call: int = 512):
    """The oracle (as it stands) on blocks of query rows of random (sequence,
    head) pairs of the packed batch until ~budget_s seconds of CPU work;
    returns (flops, seconds, description)."""
    import oracle
    oracle.build()
    g = np.random.default_rng(0)
    G = w.H // w.kv_heads
    flops, n_rows = 0.0, 0
    t0 = time.perf_counter()
    while True:
        b, h = int(g.integers(w.n_seq)), int(g.integers(w.H))
        s0, s1 = int(cu[b]), int(cu[b + 1])
        n = s1 - s0
        r0 = int(g.integers(0, max(1, n - rows_per_call + 1)))
        rows = np.arange(r0, min(n, r0 + rows_per_call))
        oracle.attention(q[s0:s1, h], k[s0:s1, h // G], v[s0:s1, h // G], w.scale, w.causal, rows=rows)
        nvis = np.minimum(rows + 1, n) if w.causal else np.full(rows.size, n)
        flops += float(4.0 * w.d * nvis.sum())
        n_rows += rows.size
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return flops, dt, f"{n_rows} query rows ({rows_per_call}-row blocks of random (sequence, head) pairs)"


def axial_block_oracle_step(w, x, row, col):
    import oracle
    return oracle.axial_block(x, row, col, w.heads)


def run_reference(args, w):
    """--impl reference: the oracle on the host cores, each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    from attention_fa2_fwd_02_gb300.inputs import AxialBlockWorkload
    if isinstance(w, AxialBlockWorkload):  # the whole block per step (it is small)
        x, row, col = w.make()
        xn, rn, cn = x.numpy(), {k: v.numpy() for k, v in row.items()}, {k: v.numpy() for k, v in col.items()}
        steps, warm = args.steps, max(3, args.warmup)
        for _ in range(warm):
            axial_block_oracle_step(w, xn, rn, cn)
        t0 = time.perf_counter()
        for _ in range(steps):
            axial_block_oracle_step(w, xn, rn, cn)
        el = time.perf_counter() - t0
        val = w.flops * steps / el / 1e12
        print(json.dumps({
            "impl": "reference", "metric": "axial block TFLOP/s", "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(w),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": "the full block (row + column pass) per step, numpy fp64"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    from attention_fa2_fwd_02_gb300.inputs import VarlenWorkload
    if isinstance(w, VarlenWorkload):  # bounded row samples of the packed batch per step
        q, k, v, cu, _ = w.make()
        steps, warm = args.steps, max(3, args.warmup)
        budget = max(0.05, 120.0 / (steps + warm))
        for _ in range(warm):
            varlen_oracle_sample(w, q, k, v, cu, budget)
        tot_f, tot_t, desc = 0.0, 0.0, ""
        for _ in range(steps):
            f, dt, desc = varlen_oracle_sample(w, q, k, v, cu, budget)
            tot_f += f
            tot_t += dt
        val = tot_f / tot_t / 1e12
        print(json.dumps({
            "impl": "reference", "metric": "attention fwd TFLOP/s", "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": tot_t / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(w),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    Q, K, V = w.make()
    steps, warm = args.steps, max(3, args.warmup)
    if args.workload.endswith("_bwd"):
        from attention_fa2_fwd_02_gb300.inputs import normal
        G = normal(Q.shape[:-1] + V.shape[-1:], 4242, torch.bfloat16)  # dO: O's shape
        budget = max(0.05, 120.0 / (steps + warm))
        for _ in range(warm):
            bwd_oracle_sample(w, Q, K, V, G, budget)
        tot_f, tot_t, desc = 0.0, 0.0, ""
        for _ in range(steps):
            f, dt, desc = bwd_oracle_sample(w, Q, K, V, G, budget)
            tot_f += f
            tot_t += dt
        val = tot_f / tot_t / 1e12
        cfg = workload_desc(w)
        cfg["pass"] = "backward"
        line = {
            "impl": "reference", "metric": "attention bwd TFLOP/s", "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": tot_t / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    # size one step so that the whole run takes about two minutes
    f, dt, _ = oracle_sample(w, Q, K, V, budget_s=0.5)
    rate = f / dt
    per_step_s = max(0.02, 120.0 / (steps + warm))
    from attention_fa2_fwd_02_gb300.inputs import AxialWorkload
    if isinstance(w, AxialWorkload):
        sample_desc = "full axial workload (row + column) per step"
        def step():
            oracle_sample(w, Q, K, V, budget_s=0.0)
        step_flops = w.flops
    else:
        rows = max(1, min(w.N_q, int(rate * per_step_s / (2.0 * (w.d + w.v_dim) * w.N_k))))
        g = np.random.default_rng(1)
        sample_desc = f"{rows} query rows of one random (b,h) slice per step"
        def step():
            b, h = int(g.integers(w.B)), int(g.integers(w.H))
            hk = h // (w.H // w.kv_heads)
            oracle.attention(Q[b, h], K[b, hk], V[b, hk], w.scale, w.causal, rows=np.arange(rows))
        nvis = np.minimum(np.arange(rows) + 1, w.N_k) if w.causal else np.full(rows, w.N_k)
        step_flops = float(2.0 * (w.d + w.v_dim) * nvis.sum())
    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    val = step_flops * steps / el / 1e12
    line = {
        "impl": "reference", "metric": "attention fwd TFLOP/s", "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_desc(w),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg
def run_axial_block(args, w):
    """The fused axial block: two launches per step (row pass, column pass),
    HBM roofline, end to end with the grid copied in and out every step."""
    import attention_fa2_fwd_02_gb300 as fa
    world, rank, local, dist = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    warm, steps = max(3, args.warmup), max(1, args.steps)
    xh, row, col = w.make()
    xd = xh.to(dev)
    rowd, cold = ({k: v.to(dev) for k, v in p.items()} for p in (row, col))
    outd = torch.empty_like(xd)
    stream = torch.cuda.current_stream(dev)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20
    flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev)  # the grid fits in L2: flush

    def step():
        return fa.axial_block(xd, rowd, cold, heads=w.heads, out=outd)
    for _ in range(warm):
        flush.zero_()
        step()
    fa.check()
    graph = torch.cuda.CUDAGraph()  # microsecond launches: timed from a graph replay
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    for k in range(steps):
        flush.zero_()
        ev[k][0].record(stream)
        graph.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    fa.check()
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    step_ms = max_over_ranks(kernel_ms, dist)
    value = whole_job_value(w.flops, world, step_ms)
    peaks, peak_src = load_peaks()
    achieved = w.algorithmic_bytes / (kernel_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
            "frac": achieved / float(peaks["hbm_gbs"]), "traffic": recorded_traffic(args.workload),
            "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
            "timed": "row-pass + column-pass launches of fa_axial_pass_kernel"}
    e2e = None
    if not args.no_e2e:
        xp, op = xh.pin_memory(), torch.empty_like(xh).pin_memory()

        def e2e_step():
            xd.copy_(xp, non_blocking=True)
            step()
            op.copy_(outd, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(3, min(steps, 50))
        a.record(stream)
        for _ in range(n):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b) / n, dist)
        nb = xh.numel() * 4
        e2e = {"value": whole_job_value(w.flops, world, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": nb, "d2h_bytes_per_step": nb}
        fa.check()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xn, rn, cn = xh.numpy(), {k: v.numpy() for k, v in row.items()}, {k: v.numpy() for k, v in col.items()}
        t0, reps = time.perf_counter(), 0
        while True:
            axial_block_oracle_step(w, xn, rn, cn)
            reps += 1
            if time.perf_counter() - t0 >= min(args.cpu_seconds, 5.0):
                break
        dt = time.perf_counter() - t0
        cpu = {"value": w.flops * reps / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps} full blocks (row + column pass), numpy fp64; {dt:.1f} s"}
    if rank == 0:
        cfg = workload_desc(w)
        cfg["l2"] = "L2 flushed (%.0f MB write) between steps" % (flush.numel() * 4 / 2**20)
        cfg["parallelism"] = f"replicas x{world} (independent problems per GPU)"
        cfg["cuda_graph"] = True
        print(json.dumps({
            "metric": "axial block TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded i.i.d. N(0,1) grid and weights)",
            "config": cfg, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": 2 * steps, "kernel_ms": kernel_ms}), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_varlen(args, w):
    """A packed variable-length batch: one fa_fwd_varlen launch per step,
    tensor-core roofline, end to end with q, k, v and the offsets copied in
    and O, LSE copied out every step."""
    import attention_fa2_fwd_02_gb300 as fa
    world, rank, local, dist = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    warm, steps = max(3, args.warmup), max(1, args.steps)
    qh, kh, vh, cuh, _ = w.make()
    max_len = max(w.lens)
    qd, kd, vd, cud = qh.to(dev), kh.to(dev), vh.to(dev), cuh.to(dev)
    od = torch.empty_like(qd)
    ld = torch.empty((w.H, qh.shape[0]), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20
    in_bytes = sum(x.numel() * x.element_size() for x in (qd, kd, vd, cud))
    flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev) if in_bytes <= l2_bytes else None

    def step():
        return fa.fwd_varlen(qd, kd, vd, cud, cud, max_len, scale=w.scale, is_causal=w.causal, out=od, lse=ld)
    for _ in range(warm):
        step()
    fa.check()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    for k in range(steps):
        if flush is not None:
            flush.zero_()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    fa.check()
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    step_ms = max_over_ranks(kernel_ms, dist)
    value = whole_job_value(w.flops, world, step_ms)
    peaks, peak_src = load_peaks()
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": recorded_traffic(args.workload), "peak_source": f"bf16_tflops burst (of {peak_src})"}
    e2e = None
    if not args.no_e2e:
        hp = [x.pin_memory() for x in (qh, kh, vh, cuh)]
        op, lp = torch.empty(qh.shape, dtype=qh.dtype).pin_memory(), torch.empty(ld.shape).pin_memory()

        def e2e_step():
            for dst, src in zip((qd, kd, vd, cud), hp):
                dst.copy_(src, non_blocking=True)
            step()
            op.copy_(od, non_blocking=True)
            lp.copy_(ld, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(3, min(steps, 20))
        a.record(stream)
        for _ in range(n):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b) / n, dist)
        e2e = {"value": whole_job_value(w.flops, world, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": int(in_bytes), "d2h_bytes_per_step": int(od.numel() * 2 + ld.numel() * 4)}
        fa.check()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        f, dt, desc = varlen_oracle_sample(w, qh, kh, vh, cuh, budget_s=args.cpu_seconds)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{desc}; {dt:.1f} s of fp64 CPU work"}
    if rank == 0:
        cfg = workload_desc(w)
        cfg["l2"] = ("inputs larger than L2: %.0f MB vs %.0f MB" % (in_bytes / 2**20, l2_bytes / 2**20)
                     if flush is None else "L2 flushed between steps")
        cfg["parallelism"] = f"replicas x{world} (independent problems per GPU)"
        print(json.dumps({
            "metric": "attention fwd TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded i.i.d. N(0,1), seeded lengths)",
            "config": cfg, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": steps, "kernel_ms": kernel_ms}), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse_args()
    w = get_workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
        return
    from attention_fa2_fwd_02_gb300.inputs import AxialBlockWorkload, VarlenWorkload
    if isinstance(w, AxialBlockWorkload):
        run_axial_block(args, w)
        return
    if isinstance(w, VarlenWorkload):
        run_varlen(args, w)
        return
    import attention_fa2_fwd_02_gb300 as fa
    from attention_fa2_fwd_02_gb300.inputs import AxialWorkload

    world, rank, local, dist = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    warm = max(3, args.warmup)
    steps = max(1, args.steps)
    axial = isinstance(w, AxialWorkload)
    bwd = args.workload.endswith("_bwd")
    Qh, Kh, Vh = w.make()
    Qd, Kd, Vd = Qh.to(dev), Kh.to(dev), Vh.to(dev)
    if bwd:
        from attention_fa2_fwd_02_gb300.inputs import normal
        Gh = normal(Qh.shape[:-1] + Vh.shape[-1:], 4242, torch.bfloat16)  # dO: O's shape
        Gd = Gh.to(dev)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = getattr(props, "L2_cache_size", 0) or 129 * 2**20
    in_bytes = sum(x.numel() * x.element_size() for x in (Qd, Kd, Vd))
    if bwd:  # the backward also reads O, LSE and dO
        in_bytes = 2 * in_bytes + Gd.numel() * 2
    flush = None
    if in_bytes <= l2_bytes:
        flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev)

    n_split = 1  # key-range splits the library picks for this problem
    vt_bytes = 0  # fp32: bytes of the V^T workspace (the step is then the V^T pass + the attention kernel)
    if bwd:
        # forward outputs (not timed), then the backward as the step
        Od, Ld = fa.fwd(Qd, Kd, Vd, scale=w.scale, is_causal=w.causal, split_kv=1)
        dQd, dKd, dVd = torch.empty_like(Qd), torch.empty_like(Kd), torch.empty_like(Vd)
        ws = torch.empty(fa.lib().fa_bwd_workspace_bytes(w.B, w.H, w.N_q, max(w.d, w.v_dim)), dtype=torch.uint8,
                         device=dev)

        def step():
            return fa.bwd(Qd, Kd, Vd, Od, Ld, Gd, scale=w.scale, is_causal=w.causal, dQ=dQd, dK=dKd, dV=dVd,
                          workspace=ws)
        make_step = None
    elif axial:
        def make_step(Qx, Kx, Vx):
            def f():
                return fa.axial(Qx, Kx, Vx, scale=w.scale, with_lse=True)
            return f
        step = make_step(Qd, Kd, Vd)
    else:
        Od = torch.empty((*Qd.shape[:-1], Vd.shape[-1]), dtype=Qd.dtype, device=dev)
        Ld = torch.empty(Qd.shape[:-1], dtype=torch.float32, device=dev)
        code = fa.FA_BF16 if w.dtype == torch.bfloat16 else fa.FA_FP32
        if w.d in (64, 128) and w.kv_heads == w.H and w.v_dim == w.d:  # (split-KV: K/V with the query heads, Dv = d)
            n_split = fa.lib().fa_fwd_splitkv_choose(code, w.B, w.H, w.N_q, w.N_k, w.d, int(w.causal))
        ws = None
        if n_split > 1:  # the split path's scratch, allocated once outside the timed region
            ws = torch.empty(fa.lib().fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.N_q, w.d, n_split),
                             dtype=torch.uint8, device=dev)
        vt_bytes = 0
        if n_split == 1 and w.v_dim == w.d:  # fp32: V^T written once per call into this scratch
            vt_bytes = fa.lib().fa_fwd_ws_bytes(code, w.B, w.H, w.kv_heads, w.N_q, w.N_k, w.d)
            if vt_bytes > 0:
                ws = torch.empty(vt_bytes, dtype=torch.uint8, device=dev)

        def make_step(Qx, Kx, Vx, Ox=None, Lx=None):
            Ox = torch.empty((*Qx.shape[:-1], Vx.shape[-1]), dtype=Qx.dtype, device=dev) if Ox is None else Ox
            Lx = torch.empty(Qx.shape[:-1], dtype=torch.float32, device=dev) if Lx is None else Lx

            def f():
                return fa.fwd(Qx, Kx, Vx, scale=w.scale, is_causal=w.causal, out=Ox, lse=Lx,
                              split_kv=n_split, workspace=ws)
            return f
        step = make_step(Qd, Kd, Vd, Od, Ld)

        if args.api == "sdpa":  # the same forward, reached through PyTorch's SDPA entry point
            import torch.nn.functional as F
            from attention_fa2_fwd_02_gb300 import sdpa
            n_split = fa.lib().fa_fwd_splitkv_choose(code, w.B, w.H, w.N_q, w.N_k, w.d, int(w.causal)) \
                if (w.d in (64, 128) and w.kv_heads == w.H and w.v_dim == w.d) else 1

            def step():
                with sdpa.routed():
                    return F.scaled_dot_product_attention(Qd, Kd, Vd, is_causal=w.causal, scale=w.scale,
                                                          enable_gqa=w.kv_heads != w.H)

    for _ in range(warm):
        if flush is not None:
            flush.zero_()
        step()
    fa.check()
    # Inputs that fit in L2 (the tiny, tutorial and axial shapes): the steps
    # run on copies of the inputs that rotate over more than twice the L2
    # size, so no step finds its inputs in L2, and back to back: one CUDA
    # graph replays a launch on every copy, and a step's time is the replay
    # time over the number of launches (no flush and no timing event between
    # launches, whose own overhead, a few microseconds, would otherwise sit in
    # the time of a microsecond-scale kernel).
    rotating = flush is not None and not bwd and args.api == "fa" and make_step is not None
    n_copies = 1
    if rotating:
        per_copy = in_bytes + (2 if axial else 1) * (Qd.numel() * Qd.element_size() // Qd.shape[-1] *
                                                      (Vd.shape[-1] + 1))
        n_copies = int(min(8192, max(2, math.ceil(2 * l2_bytes / per_copy) + 1)))
        launches = [step] + [make_step(Qd.clone(), Kd.clone(), Vd.clone()) for _ in range(n_copies - 1)]
        for f in launches[1:]:
            f()
        torch.cuda.synchronize(dev)
        fa.check()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for f in launches:
                f()
        torch.cuda.synchronize(dev)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)
        fa.check()
        replays = max(1, math.ceil(steps / n_copies))
        rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
        sampler = ClockSampler(local)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler.start()
        time.sleep(0.3)
        for a, b in rev:
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop()
        fa.check()
        kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in rev) / n_copies
        steps = replays * n_copies
        step_ms = max_over_ranks(kernel_ms, dist)
        use_graph = True
        flops = bwd_flops(w) if bwd else w.flops
        value = whole_job_value(flops, world, step_ms)
    # Sub-millisecond launches are timed from a CUDA graph replay: the step is
    # the same single kernel launch, without the Python/ctypes host overhead
    # that would otherwise sit between the timing events.
    if not rotating:
        probe0, probe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        probe0.record(stream)
        step()
        probe1.record(stream)
        torch.cuda.synchronize(dev)
        use_graph = probe0.elapsed_time(probe1) < 1.0
        timed_step = step
    if not rotating and use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize(dev)
        timed_step = graph.replay
        for _ in range(3):
            timed_step()
        torch.cuda.synchronize(dev)
        fa.check()
    if not rotating:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(local)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sampler.start()
        time.sleep(0.3)  # let the sampler take its first reading before the load starts
        t_start.record(stream)
        for k in range(steps):
            if flush is not None:
                flush.zero_()
            ev[k][0].record(stream)
            timed_step()
            ev[k][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop()
        fa.check()
        launch_ms = [a.elapsed_time(b) for a, b in ev]
        kernel_ms = statistics.mean(launch_ms)
        wall_ms = t_start.elapsed_time(t_end)
        # with an L2 flush between steps the step time is the kernel time only
        step_ms = kernel_ms if flush is not None else wall_ms / steps
        step_ms = max_over_ranks(step_ms, dist)
        flops = bwd_flops(w) if bwd else w.flops
        value = whole_job_value(flops, world, step_ms)

    # --------------------------------------------------------- roofline
    peaks, peak_src = load_peaks()
    traffic = recorded_traffic(args.workload)
    if axial:
        bytes_per_launch = w.algorithmic_bytes
        achieved = bytes_per_launch / (kernel_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} hbm_gbs (of {peak_src})"}
    else:
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        base = float(peaks["bf16_tflops"])
        if w.dtype == torch.bfloat16:
            peak, note = base, f"bf16_tflops burst (of {peak_src})"
        else:
            peak = base * NOMINAL_TF32_OVER_BF16
            note = f"bf16_tflops burst x nominal tf32/bf16 ratio 1.1/2.25 (of {peak_src})"
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": note}
        if n_split > 1:  # the events bracket both launches of a split step
            roof["timed"] = f"split-KV attention kernel (n_split={n_split}) + merge kernel"
        if vt_bytes > 0:  # ... and both launches of an fp32 step with the V^T pass
            roof["timed"] = "V^T pass (fa_vt_kernel) + tf32 attention kernel"
        tile = 256 if max(w.d, w.v_dim) > 128 else (128 if max(w.d, w.v_dim) > 64 else 64)
        if not axial and not bwd and (w.d != tile or w.v_dim != tile) and w.d not in (16, 32):
            roof["tile_columns"] = (f"d={w.d}, Dv={w.v_dim} run on {tile}-column tiles: the tensor work is "
                                    f"{2 * tile / (w.d + w.v_dim):.3f}x the FLOPs counted")
        if bwd:  # the events bracket the three launches of a backward step
            roof["timed"] = "backward preprocess + tensor-core backward kernel + dQ conversion"


    # ------------------------------------------------------ end to end
    e2e = None
    if not args.no_e2e and bwd:
        # through the public API from host buffers: Q, K, V, O, LSE, dO in,
        # dQ, dK, dV out, every step
        hp = [x.pin_memory() for x in (Qh, Kh, Vh)]
        Op, Lp, Gp = Od.cpu().pin_memory(), Ld.cpu().pin_memory(), Gh.pin_memory()
        outs = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (Qh, Kh, Vh)]

        def e2e_step():
            for dst, src in zip((Qd, Kd, Vd, Od, Ld, Gd), (*hp, Op, Lp, Gp)):
                dst.copy_(src, non_blocking=True)
            step()
            for dst, src in zip(outs, (dQd, dKd, dVd)):
                dst.copy_(src, non_blocking=True)

        e_steps = max(3, min(steps, 20))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b) / e_steps, dist)
        h2d = sum(x.numel() * x.element_size() for x in (*hp, Op, Lp, Gp))
        d2h = sum(x.numel() * x.element_size() for x in outs)
        e2e = {"value": whole_job_value(flops, world, e_ms), "unit": "TFLOP/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
        fa.check()
    elif not args.no_e2e:
        Qp, Kp, Vp = (x.pin_memory() for x in (Qh, Kh, Vh))
        Op = torch.empty((*Qh.shape[:-1], Vh.shape[-1]), dtype=Qh.dtype).pin_memory()
        Lp = torch.empty(Qh.shape[:-1], dtype=torch.float32).pin_memory()
        if axial:
            Op2 = torch.empty_like(Op)
            Lp2 = torch.empty_like(Lp)

        def e2e_step():
            Qd.copy_(Qp, non_blocking=True)
            Kd.copy_(Kp, non_blocking=True)
            Vd.copy_(Vp, non_blocking=True)
            if axial:
                (o1, l1), (o2, l2) = step()
                Op.copy_(o1, non_blocking=True)
                Op2.copy_(o2, non_blocking=True)
                Lp.copy_(l1, non_blocking=True)
                Lp2.copy_(l2, non_blocking=True)
            elif args.api == "sdpa":  # the routed SDPA returns O only
                Op.copy_(step(), non_blocking=True)
            else:
                step()
                Op.copy_(Od, non_blocking=True)
                Lp.copy_(Ld, non_blocking=True)

        e_steps = max(3, min(steps, 20))
        pipelined = not axial and args.api == "fa"
        if pipelined:
            # The plain forward overlaps step k's upload, step k-1's kernel and
            # step k-2's download: two device buffer sets, one stream each
            # for uploads, kernels and downloads, ordered by events (uploads
            # split over three streams measured 7 % slower).  Every step
            # still copies its own inputs in and its outputs out inside the
            # timed region.
            sets = [(Qd, Kd, Vd, Od, Ld)]
            sets.append(tuple(torch.empty_like(x) for x in sets[0]))
            steps_b = [step, make_step(*sets[1])]
            outs_h = [(Op, Lp), (torch.empty_like(Op).pin_memory(), torch.empty_like(Lp).pin_memory())]
            s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
            in_done = [torch.cuda.Event() for _ in range(2)]
            comp_done = [torch.cuda.Event() for _ in range(2)]
            out_done = [torch.cuda.Event() for _ in range(2)]
            for e in comp_done:
                e.record(s_comp)
            for e in out_done:
                e.record(s_out)

            def e2e_pipe(k):
                b = k & 1
                q, kk, v, o, l = sets[b]
                with torch.cuda.stream(s_in):
                    s_in.wait_event(comp_done[b])  # step k-2's kernel is done with set b's inputs
                    q.copy_(Qp, non_blocking=True)
                    kk.copy_(Kp, non_blocking=True)
                    v.copy_(Vp, non_blocking=True)
                    in_done[b].record(s_in)
                with torch.cuda.stream(s_comp):
                    s_comp.wait_event(in_done[b])
                    s_comp.wait_event(out_done[b])  # step k-2's download has read set b's outputs
                    steps_b[b]()
                    comp_done[b].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[b])
                    outs_h[b][0].copy_(o, non_blocking=True)
                    outs_h[b][1].copy_(l, non_blocking=True)
                    out_done[b].record(s_out)

            for k in range(2):
                e2e_pipe(k)
            torch.cuda.synchronize(dev)
            if dist is not None:
                dist.barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s_in)
            for k in range(e_steps):
                e2e_pipe(k)
            s_out.wait_event(comp_done[(e_steps - 1) & 1])
            b.record(s_out)
            torch.cuda.synchronize(dev)
        else:
            for _ in range(2):
                e2e_step()
            torch.cuda.synchronize(dev)
            if dist is not None:
                dist.barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(e_steps):
                e2e_step()
            b.record(stream)
            torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(a.elapsed_time(b) / e_steps, dist)
        h2d = in_bytes
        d2h = Op.numel() * Op.element_size() + (0 if args.api == "sdpa" else Lp.numel() * 4)
        if axial:
            d2h *= 2
        e2e = {"value": whole_job_value(flops, world, e_ms), "unit": "TFLOP/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "overlap": ("uploads, kernels and downloads of consecutive steps overlap (two buffer sets, "
                           "three streams)") if pipelined else "none (one stream)"}
        fa.check()

    # ---------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        if bwd:
            f, dt, desc = bwd_oracle_sample(w, Qh, Kh, Vh, Gh, budget_s=args.cpu_seconds)
        else:
            f, dt, desc = oracle_sample(w, Qh, Kh, Vh, budget_s=args.cpu_seconds)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": f"{desc}; {dt:.1f} s of fp64 CPU work"}

    if rank == 0:
        cfg = workload_desc(w)
        if rotating:
            cfg["l2"] = ("inputs rotate over %d copies (%.0f MB > 2 x L2 %.0f MB); %d launches back to back per "
                         "graph replay, time per launch = replay time / %d" %
                         (n_copies, n_copies * per_copy / 2**20, l2_bytes / 2**20, n_copies, n_copies))
        else:
            cfg["l2"] = ("inputs larger than L2: %.0f MB vs %.0f MB" % (in_bytes / 2**20, l2_bytes / 2**20)
                         if flush is None else "L2 flushed (%.0f MB write) between steps" % (flush.numel() * 4 / 2**20))
        cfg["parallelism"] = f"replicas x{world} (independent problems per GPU)"
        cfg["cuda_graph"] = use_graph
        cfg["split_kv"] = n_split
        if vt_bytes > 0:
            cfg["v_transpose"] = f"V^T pass into a {vt_bytes / 2**20:.1f} MB workspace, then K-major V^T tiles"
        if args.api == "sdpa":
            cfg["api"] = "torch.nn.functional.scaled_dot_product_attention routed to this library"
        if bwd:
            cfg["pass"] = "backward (dQ, dK, dV from Q, K, V, O, LSE, dO); FLOPs = 2.5x the forward's"
        line = {
            "metric": "attention bwd TFLOP/s" if bwd else "attention fwd TFLOP/s", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if (not axial and w.dtype == torch.bfloat16) else ("f32" if axial else "tf32"),
            "data": "synthetic (seeded i.i.d. N(0,1))", "config": cfg,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            # one kernel per step, plus the merge kernel when the keys are split
            # or the V^T pass before it (fp32)
            # (a backward step is three launches: preprocess, kernel, dQ conversion)
            "gpu_launches": steps * (3 if bwd else (2 if (n_split > 1 or vt_bytes > 0) else 1)),
            "kernel_ms": kernel_ms,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
