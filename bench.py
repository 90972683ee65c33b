"""Benchmark of the DCP hot path on GB300: reshard -> per-rank partial attention -> LSE merge.

One step = one pass of the whole path over one batch: the page-level reshard from the CP
layer-split source layout into the DCP page-interleaved pools, partial MLA decode attention
on every DCP rank, and the exact LSE merge.  Default workload: 32 requests x 8192 tokens,
64 heads, q_len 1, BF16 KV, page 64, DCP=8, resharded from one CP source shard (1 layer).

Prints one JSON line.  --impl reference times the float64 CPU oracle instead (bounded
sample of the same workload, on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dcp_inputs as di  # noqa: E402

METRIC = "DCP decode attn KV GB/s + TFLOP/s and reshard GB/s, % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM bytes per launch measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum) for the
# kernels below on the default workload, with the hash of the kernel source they were taken
# on; a changed source reports traffic null until it is re-measured.
NCU_TRAFFIC = {
    # (kernel, workload): (source hash, bytes per launch); profiles/attn_kernel__batch-32x8192-h64-bf16-dcp8.md
    ("reshard_kernel", "batch-32x8192-h64-q1-bf16-dcp8"): ("37f38495550d4afc", 551839000),
    ("attn_kernel", "batch-32x8192-h64-q1-bf16-dcp8"): ("49a82f8ae989d93b", 331932928),
}


def _src_hash(name: str) -> str:
    p = os.path.join(ROOT, "decode_context_paged_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------ workload
class Workload:
    """The default batch workload, resident in HBM, plus its per-step algorithmic sizes."""

    def __init__(self, device, seed: int = 1):
        self.B, self.T, self.H, self.N = 32, 1, 64, 8
        self.n_tokens = 8192
        self.dtype = "bf16"
        lens = [self.n_tokens] * self.B
        self.rc = di.reshard_case(lens, n_layers=1, layer_counts=[1], n_dcp=self.N, dtype=self.dtype,
                                  contiguous_src=True, seed=seed, device=device, dst_slots=512)
        self.q = di.random_q(self.B, self.T, self.H, di._gen(seed + 7, device), device)
        self.seq_lens = torch.tensor(lens, dtype=torch.int32, device=device)
        self.pools = [p[0] for p in self.rc.dst_pools]
        self.kv_scale = 1.0
        self.scale = di.SOFTMAX_SCALE
        R = self.B * self.T * self.H
        self.o_part = torch.empty((self.N, self.B, self.T, self.H, 512), dtype=torch.float32, device=device)
        self.lse_part = torch.empty((self.N, self.B, self.T, self.H), dtype=torch.float32, device=device)
        self.o = torch.empty((self.B, self.T, self.H, 512), dtype=torch.float32, device=device)
        self.lse = torch.empty((self.B, self.T, self.H), dtype=torch.float32, device=device)
        import decode_context_paged_gb300 as dcp
        self.ws = dcp.alloc_workspace(self.B, self.T, self.H, self.N, self.rc.dst_vpages.numel(), device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        pages = self.rc.dst_vpages.numel()
        elem = 2 if self.dtype == "bf16" else 1
        page_bytes = 64 * 576 * elem
        tokens = sum(lens)
        self.bytes = {
            "reshard": 2 * pages * page_bytes,                       # read + write every page
            "attn": tokens * 576 * elem + self.q.numel() * 2 + self.N * R * (512 + 1) * 4,
            "merge": self.N * R * (512 + 1) * 4 + R * (512 + 1) * 4,
        }
        self.flops_attn = 2 * tokens * self.T * self.H * (576 + 512)
        self.name = f"batch-{self.B}x{self.n_tokens}-h{self.H}-q{self.T}-{self.dtype}-dcp{self.N}"

    def step(self, dcp, events=None):
        rc = self.rc
        if events:
            events[0].record()
        dcp.reshard_pages(rc.req_page_ptr, rc.src_pages, rc.dst_vpages, 1, rc.src_pools, rc.src_pool_pages,
                          rc.dst_pools, rc.dst_slots, dev_error=self.err)
        if events:
            events[1].record()
        dcp.partial_decode_attn(self.q, self.seq_lens, rc.req_page_ptr, rc.dst_vpages, self.pools, self.scale,
                                self.kv_scale, o_part=self.o_part, lse_part=self.lse_part, workspace=self.ws,
                                dev_error=self.err)
        if events:
            events[2].record()
        dcp.lse_merge(self.o_part, self.lse_part, self.o, self.lse)
        if events:
            events[3].record()


LAUNCHES_PER_STEP = 6  # reshard, plan pages, plan units, attention, chunk combine, merge


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        return dist, rank, ws, local
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(wl, max_seconds: float = 20.0):
    """Times the float64 oracle on a bounded sample of the workload: whole requests (their
    reshard, per-rank partial attention and merge), adding requests until ~max_seconds."""
    import numpy as np

    import oracle
    oracle.build()
    rc = wl.rc
    ptr = rc.req_page_ptr.cpu().numpy()
    src_pages = rc.src_pages.cpu().numpy()
    vp = rc.dst_vpages.cpu().numpy()
    src = [p.cpu().view(torch.uint8).numpy().reshape(-1) for p in rc.src_pools]
    qb = wl.q.cpu().view(torch.int16).numpy().view(np.uint16)
    per_req_bytes = sum(wl.bytes.values()) / wl.B
    done, t_total = 0, 0.0
    while done < wl.B and t_total < max_seconds:
        b = done
        p0, p1 = int(ptr[b]), int(ptr[b + 1])
        sub_ptr = np.array([0, p1 - p0], np.int64)
        dst = [np.zeros(rc.dst_slots * rc.page_bytes, np.uint8) for _ in range(wl.N)]
        t0 = time.perf_counter()
        oracle.reshard(sub_ptr, src_pages[p0:p1], vp[p0:p1], rc.page_bytes, 1, src, rc.src_pool_pages, wl.N,
                       dst, rc.dst_slots)
        pools = [d.view(np.uint16).reshape(rc.dst_slots, 64, 576) for d in dst]
        parts = [oracle.attention(qb[b:b + 1], np.array([wl.n_tokens], np.int32), sub_ptr, vp[p0:p1], pools,
                                  oracle.BF16, 1.0, wl.scale, wl.N, rank=d, q_len=wl.T, num_heads=wl.H)
                 for d in range(wl.N)]
        oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        t_total += time.perf_counter() - t0
        done += 1
    gbs = done * per_req_bytes / t_total / 1e9
    return gbs, done, t_total, oracle.num_threads()


# ------------------------------------------------------------------------------- main
def run_reference(args):
    dist, rank, world, local = dist_setup()
    if rank != 0:
        return
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = Workload(dev)
    for _ in range(args.warmup):
        pass  # the oracle has no warm state; warm-up steps are not needed for a CPU program
    vals = []
    samples = []
    for _ in range(args.steps):
        gbs, done, secs, threads = oracle_sample(wl, max_seconds=args.ref_seconds)
        vals.append(gbs)
        samples.append((done, secs))
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(s for _, s in samples) / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "l2": "inputs larger than L2"},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{samples[0][0]} of {wl.B} requests per step (reshard + {wl.N} partials + merge)"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import decode_context_paged_gb300 as dcp
    dist, rank, world, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = Workload(dev, seed=1 + rank)
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 3)):
        wl.step(dcp)
    torch.cuda.synchronize()
    if int(wl.err.item()) != 0:
        raise RuntimeError(f"device error word {int(wl.err.item())}")

    # ---- timed region: K steps, per-stage events on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for k in range(args.steps):
            wl.step(dcp, ev[k])
        end.record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    ms = start.elapsed_time(end)
    ms = max_over_ranks(dist, ms)
    stage_ms = {
        "reshard": sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps,
        "attn": sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps,
        "merge": sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps,
    }
    step_bytes = sum(wl.bytes.values())
    ms_step = ms / args.steps
    value = world * step_bytes / (ms_step * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers
    host_src = [p.cpu().pin_memory() for p in wl.rc.src_pools]
    host_q = wl.q.cpu().pin_memory()
    host_o = torch.empty(wl.o.shape, dtype=torch.float32).pin_memory()
    host_l = torch.empty(wl.lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_src) + host_q.numel() * 2
    d2h = host_o.numel() * 4 + host_l.numel() * 4

    def e2e_step():
        for hs, ds in zip(host_src, wl.rc.src_pools):
            ds.copy_(hs, non_blocking=True)
        wl.q.copy_(host_q, non_blocking=True)
        wl.step(dcp)
        host_o.copy_(wl.o, non_blocking=True)
        host_l.copy_(wl.lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / args.steps
    e2e_value = world * step_bytes / (e2e_ms * 1e-3) / 1e9

    if rank != 0:
        return
    hbm, bf16, bf16_sus, peak_kind = peaks()
    stage_gbs = {k: wl.bytes[k] / (stage_ms[k] * 1e-3) / 1e9 for k in stage_ms}
    attn_tflops = wl.flops_attn / (stage_ms["attn"] * 1e-3) / 1e12
    dom = max(stage_ms, key=stage_ms.get)
    kernel_of = {"reshard": "reshard_kernel", "attn": "attn_kernel", "merge": "lse_merge_kernel"}
    src_of = {"reshard": "dcp_reshard.cu", "attn": "dcp_attn.cu", "merge": "dcp_merge.cu"}
    tr = NCU_TRAFFIC.get((kernel_of[dom], wl.name))
    traffic = tr[1] if tr and tr[0] == _src_hash(src_of[dom]) else None
    roof = {"kernel": kernel_of[dom], "bound": "hbm", "achieved": stage_gbs[dom], "peak": hbm, "unit": "GB/s",
            "frac": stage_gbs[dom] / hbm, "peak_kind": peak_kind, "traffic": traffic,
            "algorithmic_bytes": wl.bytes[dom]}
    cpu = None
    if not args.no_cpu_baseline:
        gbs, done, secs, threads = oracle_sample(wl, max_seconds=args.ref_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{done} of {wl.B} requests (reshard + {wl.N} partials + merge), {secs:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "l2": "inputs larger than L2 (302 MB pools)",
                   "bytes_per_step": step_bytes, "parallelism": f"replicas x{world}"},
        "stages": {
            "reshard": {"ms": stage_ms["reshard"], "GB/s": stage_gbs["reshard"], "frac_hbm": stage_gbs["reshard"] / hbm},
            "attn": {"ms": stage_ms["attn"], "GB/s": stage_gbs["attn"], "TFLOP/s": attn_tflops,
                     "frac_hbm": stage_gbs["attn"] / hbm, "frac_bf16": attn_tflops / bf16},
            "merge": {"ms": stage_ms["merge"], "GB/s": stage_gbs["merge"], "frac_hbm": stage_gbs["merge"] / hbm},
        },
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
