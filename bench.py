"""Benchmark of the DCP hot path on GB300: reshard -> per-rank partial attention -> LSE merge.

One step = one pass of the whole path over one batch: the page-level reshard from the CP
layer-split source layout into the DCP page-interleaved pools, partial MLA decode attention
on every DCP rank, and the exact LSE merge.  Default workload (the largest): 64 requests of
2K-500K tokens (log-uniform, multiples of 64), 8 layers, FP8-E4M3 KV, page 64, resharded from a
CP4 layer split into DCP=8, then per layer the attention of 64 heads (q_len 1) on every rank and
the merge.  The attention's plan is made once per step (it depends only on the page table) on a
side stream while the reshard runs; the attention and the merge run as one library call per
layer (dcp_decode_attn_merged_run); --unfused times dcp_partial_decode_attn and dcp_lse_merge
as separate calls.

Timing: after the warm-up and a half-second soak of the same step (under which nvidia-smi
samples the clocks), K steps between two CUDA events give the value; a second pass of K steps
with events around every stage gives the stage times and the roofline's kernel duration.  The
end-to-end number runs the step through the same calls with the inputs uploaded from pinned
host memory every step (double-buffered, the next step's upload on a copy stream) and the
merged output read back.

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
L2_BYTES = 129 << 20  # GB300 L2

# DRAM bytes per launch measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum) for the
# kernels below on the default workload, with the hash of the kernel source they were taken
# on (for the reshard: dcp_reshard.cu and the copy ring header); a changed source reports
# traffic null until it is re-measured.
NCU_TRAFFIC = {
    # (kernel, workload): (source hash, DRAM bytes per launch).  The agent attention and the
    # batch kernels are captured on their own workload; the others on smaller cases of the same
    # kernel (the long1 config, and agent8's reshard on the long-copy grid), scaled by the units
    # processed: pages for the reshard, requests for the attention.
    ("reshard_kernel", "batch-32x8192-h64-q1-bf16-dcp8"): ("26b6b9b40d4d64dd", 552448000),
    ("reshard_kernel", "agent-48x100000-h64-q1-e4m3-dcp8"): ("26b6b9b40d4d64dd", 5236858368),
    ("reshard_kernel", "e2e-64x463936-h64-q1-e4m3-dcp8-L8-cp4"): ("26b6b9b40d4d64dd", 44745598653),
    ("attn_kernel", "batch-32x8192-h64-q1-bf16-dcp8"): ("b5795b2a10f59e5a", 325355776),
    ("attn_kernel", "agent-48x100000-h64-q1-e4m3-dcp8"): ("b5795b2a10f59e5a", 2790926848),
    ("attn_kernel", "long-4x1048576-h64-q4-e4m3-dcp8"): ("b5795b2a10f59e5a", 2528633856),
}


def _src_hash(names) -> str:
    """sha256/16 of one kernel source file, or of several concatenated in order."""
    h = hashlib.sha256()
    for name in ([names] if isinstance(names, str) else names):
        with open(os.path.join(ROOT, "decode_context_paged_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


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
WORKLOADS = {
    # name: (lengths, heads, q_len, DCP ranks, KV dtype, layers, CP source ranks, slots per rank)
    "tiny": (lambda: [1024], 16, 1, 4, "bf16", 1, 1, 4),
    "batch": (lambda: [8192] * 32, 64, 1, 8, "bf16", 1, 1, 512),
    "agent": (lambda: [100_000] * 48, 64, 1, 8, "e4m3", 1, 1, 9408),
    "long": (lambda: [1 << 20] * 4, 64, 4, 8, "e4m3", 1, 1, 8192),
    "e2e": (lambda: di.e2e_lengths(), 64, 1, 8, "e4m3", di.E2E_LAYERS, di.E2E_NCP, None),
    # smaller cases of the same kernels, for profiler captures (not bench lines): 8 of the agent
    # workload's requests, 1 of the long workload's
    "agent8": (lambda: [100_000] * 8, 64, 1, 8, "e4m3", 1, 1, 1568),
    "long1": (lambda: [1 << 20], 64, 4, 8, "e4m3", 1, 1, 2048),
    # a small multi-layer case (CP2 -> DCP4, 4 layers) for the tests of the layer pipeline
    "layers4": (lambda: [3000, 700, 64 * 40 + 5], 64, 1, 4, "e4m3", 4, 2, None),
}


class Workload:
    """One workload resident in HBM (source pools, destination pools, Q, outputs) plus its
    per-step algorithmic bytes.  A step = reshard all layers, then per layer partial attention
    on every DCP rank and the LSE merge."""

    def __init__(self, name: str, device, seed: int = 1, fused: bool = True, staging_mb: int = 0,
                 naive: bool = False, layout: str = "page", overlap_plan: bool = True, oracle_only: bool = False,
                 overlap_layers: bool = True):
        """oracle_only: inputs for the oracle arm -- the layer split from the oracle, no library
        call, no workspace (that arm loads nothing but the oracle)."""
        if oracle_only:
            import oracle
            split = oracle.layer_range
            dcp = None
        else:
            import decode_context_paged_gb300 as dcp
            split = dcp.layer_range
        self.layout = layout  # "token": token-interleaved DCP (row-gather reshard, token-layout attention)
        self.fused = fused
        # the attention's plan depends only on the page table: made once per step on a side stream
        # while the reshard runs, then run for every layer
        self.overlap_plan = overlap_plan and fused and layout == "page" and device.type == "cuda" and not oracle_only
        self.side = torch.cuda.Stream(device) if self.overlap_plan else None
        self.naive = naive  # reshard stage as the pages' initial design: full transfer, then in-place shard
        self.pack = staging_mb > 0  # reshard stage in bounded pack mode (per path: filter, pack, unpack)
        lens_fn, self.H, self.T, self.N, self.dtype, self.L, self.n_cp, slots = WORKLOADS[name]
        lens = lens_fn()
        self.lens = lens
        self.B = len(lens)
        counts = [e - s for s, e in (split(self.L, self.n_cp, r) for r in range(self.n_cp))]
        # layer pipeline (several layers): the reshard runs layer by layer on a stream of higher
        # priority (one call per layer, on the source rank's pool view of that layer), and each
        # layer's attention starts as soon as its layer has arrived, so the attention of the
        # first layers overlaps the transfer of the rest
        self.layer_rank = [r for r in range(self.n_cp) for _ in range(counts[r])]
        self.layer_in_rank = [l - sum(counts[:self.layer_rank[l]]) for l in range(self.L)]
        self.layer_pipe = (overlap_layers and self.overlap_plan and not naive and staging_mb == 0
                           and layout == "page" and self.L > 1)
        if self.layer_pipe:
            self.rs = torch.cuda.Stream(device, priority=-1)
            self.layer_done = [torch.cuda.Event() for _ in range(self.L)]
        self.rc = di.reshard_case(lens, n_layers=self.L, layer_counts=counts, n_dcp=self.N, dtype=self.dtype,
                                  contiguous_src=True, seed=seed, device=device, dst_slots=slots)
        self.q = di.random_q(self.B, self.T, self.H, di._gen(seed + 7, device), device)
        self.seq_lens = torch.tensor(lens, dtype=torch.int32, device=device)
        if layout == "token":
            # destination: the token-interleaved table and per-rank pools (same pages per rank)
            g = torch.Generator().manual_seed(seed + 11)
            tslots = sum(-(-(-(-n // self.N)) // 64) for n in lens) + 1
            tptr, tv = di.token_page_table(lens, self.N, tslots, g)
            self.tok_ptr, self.tok_vp, self.tok_slots = tptr.to(device), tv.to(device), tslots
            self.tok_pools = [torch.empty((self.L, tslots, 64, 576), dtype=self.rc.src_pools[0].dtype, device=device)
                              for _ in range(self.N)]
            for t in self.tok_pools:
                t.view(torch.uint8).zero_()
            self.layer_pools = [[p[l] for p in self.tok_pools] for l in range(self.L)]
        else:
            self.layer_pools = [[p[l] for p in self.rc.dst_pools] for l in range(self.L)]
        self.kv_scale = di.FP8_KV_SCALE if self.dtype == "e4m3" else 1.0
        self.scale = di.SOFTMAX_SCALE
        R = self.B * self.T * self.H
        self.R = R
        self.o_part = torch.empty((self.N, self.B, self.T, self.H, 512), dtype=torch.float32, device=device)
        self.lse_part = torch.empty((self.N, self.B, self.T, self.H), dtype=torch.float32, device=device)
        self.o = torch.empty((self.L, self.B, self.T, self.H, 512), dtype=torch.float32, device=device)
        self.lse = torch.empty((self.L, self.B, self.T, self.H), dtype=torch.float32, device=device)
        n_entries = self.tok_vp.numel() if layout == "token" else self.rc.dst_vpages.numel()
        # (the workspace is sized for the device's SM count; the oracle arm has none)
        self.ws = (dcp.alloc_workspace(self.B, self.T, self.H, self.N, n_entries, device)
                   if device.type == "cuda" and not oracle_only else None)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        pages = self.rc.dst_vpages.numel()
        elem = 2 if self.dtype == "bf16" else 1
        page_bytes = 64 * 576 * elem
        tokens = sum(lens)
        self.bytes = {
            "reshard": 2 * pages * page_bytes * self.L,              # read + write every page of every layer
            "attn": self.L * (tokens * 576 * elem + self.q.numel() * 2 + self.N * R * (512 + 1) * 4),
            "merge": self.L * (self.N * R * (512 + 1) * 4 + R * (512 + 1) * 4),
        }
        keys = sum(sum(n - self.T + t + 1 for t in range(self.T)) for n in lens)  # visible (row, key) per head
        self.flops_attn = 2 * keys * self.H * (576 + 512) * self.L
        self.name = (f"{name}-{self.B}x{max(lens)}-h{self.H}-q{self.T}-{self.dtype}-dcp{self.N}"
                     + (f"-L{self.L}-cp{self.n_cp}" if self.L > 1 else ""))
        # reshard + per layer: plan count (+ FP8 Q split), plan build, attention, chunk combine, merge;
        # with the plan made once per step: 2 plan launches + per layer (FP8 Q split), attention, 2 merge
        self.launches_per_step = (1 + self.L * 5 if not self.overlap_plan else
                                  3 + self.L * (4 if self.dtype == "e4m3" else 3))
        if self.layer_pipe:
            self.launches_per_step += self.L - 1  # one reshard launch per layer
        if self.naive:
            n_pages = self.rc.dst_vpages.numel()
            need = self.N * self.L * n_pages * self.rc.page_bytes
            if need > (96 << 30):
                raise SystemExit(f"--naive needs {need / 2**30:.0f} GiB of receive buffers for this workload")
            self.recv = [torch.empty((self.L, n_pages, 64, 576), dtype=self.rc.src_pools[0].dtype, device=device)
                         for _ in range(self.N)]
            self.launches_per_step += 1
            # full transfer: N x (read + write) of the KV; in-place shard: read + write once
            self.naive_moved_bytes = (self.N + 1) * self.bytes["reshard"]
        if self.pack:
            # per path (r, d): its filtered page count (fixed by the page table, known to the host as in
            # the pages' sender) and the chunk item ranges through the bounded staging buffer
            self.staging = torch.empty(staging_mb << 20, dtype=torch.uint8, device=device)
            vp = self.rc.dst_vpages.cpu()
            owner = vp % self.N if self.N > 1 else torch.zeros_like(vp)
            self.pack_paths = []
            start = 0
            for r, cnt in enumerate(counts):
                for d in range(self.N):
                    n_idx = int((owner == d).sum())
                    self.pack_paths.append((r, d, start, cnt, n_idx,
                                            dcp.pack_chunks(cnt * n_idx, self.rc.page_bytes, self.staging.numel())))
                start += cnt
            n_chunks = sum(len(p[5]) for p in self.pack_paths)
            self.launches_per_step += len(self.pack_paths) + 2 * n_chunks - 1
            self.pack_moved_bytes = 2 * self.bytes["reshard"]  # every page in and out of the staging buffer
        self.l2_note = ("inputs larger than L2" if self.bytes["reshard"] // 2 > L2_BYTES
                        else "inputs smaller than L2 (not a bench line: no flush between steps)")
        # CUDA-event stages: the fused attention call moves the merge's bytes into its stage
        self.stage_bytes = ({"reshard": self.bytes["reshard"], "attn": self.bytes["attn"] + self.bytes["merge"]}
                            if fused else dict(self.bytes))

    def step(self, dcp, events=None, inputs=None):
        """events: dict stage -> list of (start, end) event pairs, appended per call (the stages
        then run one after the other, so that each one's time can be attributed).
        inputs: (source pools, q) to use instead of the resident ones."""
        rc = self.rc
        src_pools, q = inputs if inputs is not None else (rc.src_pools, self.q)
        if self.layer_pipe and events is None:
            self._pipelined_step(dcp, src_pools, q)
            return

        def rec(stage, fn):
            if events is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            events.setdefault(stage, []).append((a, b))

        def pack_reshard():
            for r, d, start, cnt, n_idx, chunks in self.pack_paths:
                slot, src, _ = dcp.filter_page_indices(rc.dst_vpages, self.N, d, rc.src_pages)
                for begin, n in chunks:
                    dcp.pack_pages(src, n_idx, cnt, begin, n, src_pools[r], self.staging, dev_error=self.err)
                    dcp.unpack_pages(slot, n_idx, cnt, start, begin, n, self.staging, rc.dst_pools[d],
                                     dev_error=self.err)

        def naive_reshard():
            dcp.naive_full_transfer(rc.src_pages, self.L, src_pools, rc.src_pool_pages, self.recv,
                                    dev_error=self.err)
            dcp.naive_inplace_shard(rc.dst_vpages, self.L, self.recv, rc.dst_pools, rc.dst_slots, dev_error=self.err)

        def token_reshard():
            dcp.token_reshard(self.seq_lens, rc.req_page_ptr, rc.src_pages, self.tok_ptr, self.tok_vp, self.L,
                              src_pools, rc.src_pool_pages, self.tok_pools, self.tok_slots, dev_error=self.err)

        if self.overlap_plan:
            main = torch.cuda.current_stream()
            self.side.wait_stream(main)  # the previous step's runs are done with the workspace
            with torch.cuda.stream(self.side):
                rec("plan", lambda: dcp.attn_plan((self.B, self.T, self.H), rc.req_page_ptr, rc.dst_vpages,
                                                  self.layer_pools[0], self.ws, dev_error=self.err))
        if self.layout == "token":
            rec("reshard", token_reshard)
        elif self.naive:
            rec("reshard", naive_reshard)
        elif self.pack:
            rec("reshard", pack_reshard)
        else:
            rec("reshard", lambda: dcp.reshard_pages(rc.req_page_ptr, rc.src_pages, rc.dst_vpages, self.L,
                                                     src_pools, rc.src_pool_pages, rc.dst_pools, rc.dst_slots,
                                                     dev_error=self.err))
        if self.overlap_plan:
            torch.cuda.current_stream().wait_stream(self.side)
        for l in range(self.L):
            if self.fused:
                tbl = (self.tok_ptr, self.tok_vp) if self.layout == "token" else (rc.req_page_ptr, rc.dst_vpages)
                rec("attn", lambda: dcp.decode_attn_merged(q, self.seq_lens, tbl[0], tbl[1],
                                                           self.layer_pools[l], self.scale, self.kv_scale,
                                                           o_part=self.o_part, lse_part=self.lse_part, o_out=self.o[l],
                                                           lse_out=self.lse[l], workspace=self.ws, dev_error=self.err,
                                                           planned=self.overlap_plan, layout=self.layout))
                continue
            tbl = (self.tok_ptr, self.tok_vp) if self.layout == "token" else (rc.req_page_ptr, rc.dst_vpages)
            rec("attn", lambda: dcp.partial_decode_attn(q, self.seq_lens, tbl[0], tbl[1],
                                                        self.layer_pools[l], self.scale, self.kv_scale,
                                                        o_part=self.o_part, lse_part=self.lse_part, workspace=self.ws,
                                                        dev_error=self.err, layout=self.layout))
            rec("merge", lambda: dcp.lse_merge(self.o_part, self.lse_part, self.o[l], self.lse[l]))




    def _pipelined_step(self, dcp, src_pools, q):
        rc = self.rc
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)  # the previous step's runs are done with the workspace
        with torch.cuda.stream(self.side):
            dcp.attn_plan((self.B, self.T, self.H), rc.req_page_ptr, rc.dst_vpages, self.layer_pools[0], self.ws,
                          dev_error=self.err)
        self.rs.wait_stream(main)  # the previous step's attention is done with the destination pools
        with torch.cuda.stream(self.rs):
            for l in range(self.L):
                r = self.layer_rank[l]
                dcp.reshard_pages(rc.req_page_ptr, rc.src_pages, rc.dst_vpages, 1, [src_pools[r][self.layer_in_rank[l]]],
                                  rc.src_pool_pages, [p[l] for p in rc.dst_pools], rc.dst_slots, n_dcp=self.N,
                                  dev_error=self.err)
                self.layer_done[l].record(self.rs)
        main.wait_stream(self.side)
        for l in range(self.L):
            main.wait_event(self.layer_done[l])
            dcp.decode_attn_merged(q, self.seq_lens, rc.req_page_ptr, rc.dst_vpages, self.layer_pools[l], self.scale,
                                   self.kv_scale, o_part=self.o_part, lse_part=self.lse_part, o_out=self.o[l],
                                   lse_out=self.lse[l], workspace=self.ws, dev_error=self.err, planned=True)
        main.wait_stream(self.rs)


def dist_setup():
    """One process per GPU under torchrun (NCCL); gloo on a host without CUDA (the oracle arm,
    and the CPU tests of this logic)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
        return dist, rank, ws, local
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(wl, max_seconds: float = 20.0):
    """Times the float64 oracle on a bounded sample of the workload: request by request, the
    reshard of the request's pages (every layer), then for layer 0 the per-rank partial
    attention and merge of a subset of the request's query rows, until ~max_seconds.
    Returns (GB/s over the sample's share of the step's algorithmic bytes, a description, seconds,
    threads, seconds per stage)."""
    import numpy as np

    import oracle
    oracle.build()
    rc = wl.rc
    ptr = rc.req_page_ptr.cpu().numpy()
    src_pages = rc.src_pages.cpu().numpy()
    vp = rc.dst_vpages.cpu().numpy()
    src = [p.cpu().view(torch.uint8).numpy().reshape(-1) for p in rc.src_pools]
    qb = wl.q.cpu().view(torch.int16).numpy().view(np.uint16)
    dt = oracle.BF16 if wl.dtype == "bf16" else oracle.E4M3
    pages_total = len(vp)
    rows_per_req = wl.T * wl.H
    step_rows = wl.B * rows_per_req * wl.L
    attn_merge = wl.bytes["attn"] + wl.bytes["merge"]
    done_bytes, t_total, n_req, n_rows = 0.0, 0.0, 0, 0
    t_stage = {"reshard": 0.0, "attention": 0.0, "merge": 0.0}
    # request by request, cycling through the workload's requests until the time budget is spent
    while t_total < max_seconds and n_req < 64 * wl.B:
        b = n_req % wl.B
        p0, p1 = int(ptr[b]), int(ptr[b + 1])
        sub_ptr = np.array([0, p1 - p0], np.int64)
        # rows: all of them when the request is short, fewer for long contexts
        keys = wl.lens[b]
        n_sel = max(1, min(rows_per_req, int(4e9 / (keys * 2176 * 2))))
        rows = np.arange(n_sel, dtype=np.int64) * max(1, rows_per_req // n_sel)
        dst = [np.zeros(wl.L * rc.dst_slots * rc.page_bytes, np.uint8) for _ in range(wl.N)]
        t0 = time.perf_counter()
        oracle.reshard(sub_ptr, src_pages[p0:p1], vp[p0:p1], rc.page_bytes, wl.L, src, rc.src_pool_pages, wl.N,
                       dst, rc.dst_slots)
        t1 = time.perf_counter()
        esz = 2 if wl.dtype == "bf16" else 1
        pools = [d.reshape(wl.L, rc.dst_slots * 64 * 576 * esz)[0].view(np.uint16 if esz == 2 else np.uint8)
                 .reshape(rc.dst_slots, 64, 576) for d in dst]
        parts = [oracle.attention(qb[b:b + 1], np.array([wl.lens[b]], np.int32), sub_ptr, vp[p0:p1], pools,
                                  dt, wl.kv_scale, wl.scale, wl.N, rank=d, rows=rows, q_len=wl.T, num_heads=wl.H)
                 for d in range(wl.N)]
        t2 = time.perf_counter()
        oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        t3 = time.perf_counter()
        t_stage["reshard"] += t1 - t0
        t_stage["attention"] += t2 - t1  # (the pools' views between the two are free)
        t_stage["merge"] += t3 - t2
        t_total += t3 - t0
        done_bytes += wl.bytes["reshard"] * (p1 - p0) / pages_total + attn_merge * len(rows) / step_rows
        n_req += 1
        n_rows += len(rows)
    gbs = done_bytes / t_total / 1e9
    passes = (f"{n_req // wl.B} passes over all {wl.B} requests" + (f" + {n_req % wl.B} requests" if n_req % wl.B else "")
              if n_req >= wl.B else f"{n_req} of {wl.B} requests")
    desc = (f"{passes}: each request's reshard ({wl.L} layers) + layer-0 partial attention over {wl.N} ranks and "
            f"merge for {n_rows} of {n_req * rows_per_req} query rows; {t_total:.1f} s")
    return gbs, desc, t_total, oracle.num_threads(), t_stage


# ------------------------------------------------------------------------------- main
def run_reference(args):
    dist, rank, world, local = dist_setup()
    if rank != 0:
        return
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = Workload(args.config, dev, oracle_only=True)
    vals, secs, desc, threads, stages = [], [], "", 1, {}
    # the oracle has no warm state: warm-up steps are not run; the whole run stays near two
    # minutes of host time however many steps are asked for
    per_step = min(args.ref_seconds, max(2.0, 120.0 / max(args.steps, 1)))
    for _ in range(args.steps):
        gbs, desc, t, threads, stages = oracle_sample(wl, max_seconds=per_step)
        vals.append(gbs)
        secs.append(t)
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, world),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
                         "stage_seconds": stages},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, world: int) -> dict:
    """The `config` object of both arms' JSON lines."""
    return {"workload": wl.name, "l2": wl.l2_note, "bytes_per_step": sum(wl.bytes.values()),
            "parallelism": f"replicas x{world}"}


def fp8_dense_peak_tflops(dev, n: int = 8192, reps: int = 10):
    """Dense E4M3 x E4M3 -> BF16 GEMM throughput of this GPU (cuBLASLt through torch._scaled_mm,
    n^3, best of `reps`, CUDA events): the tensor roofline of the FP8 contraction.  None if the
    call is unavailable."""
    try:
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev, dtype=torch.float32)
        for _ in range(3):
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:  # noqa: BLE001 -- the bench falls back to the nominal ratio
        return None


def _stage_ms(events, steps):
    return {k: sum(a.elapsed_time(b) for a, b in v) / steps for k, v in events.items()}


def run_ours(args):
    import decode_context_paged_gb300 as dcp
    dist, rank, world, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # all work on a stream of our own: the legacy default stream would serialise against the
    # side stream (plan) and the copy stream (end-to-end uploads)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    wl = Workload(args.config, dev, seed=1 + rank, fused=not args.unfused, staging_mb=args.staging_mb,
                  naive=args.naive, layout=args.layout, overlap_plan=not args.no_plan_overlap,
                  overlap_layers=not args.no_layer_overlap)

    for _ in range(max(args.warmup, 3)):
        wl.step(dcp)
    torch.cuda.synchronize()
    if int(wl.err.item()) != 0:
        raise RuntimeError(f"device error word {int(wl.err.item())}")
    if args.profile_steps:
        # for a profiler: the warm-up and K plain steps, nothing else (no soak, no timing, no
        # host-buffer run, no oracle); prints no bench line
        for _ in range(args.steps):
            wl.step(dcp)
        torch.cuda.synchronize()
        if int(wl.err.item()) != 0:
            raise RuntimeError(f"device error word {int(wl.err.item())}")
        print(f"profile run: {wl.name}, {max(args.warmup, 3)} + {args.steps} steps", flush=True)
        return

    # ---- timed region: K steps between two CUDA events on the launching stream.  Then a second
    # timed pass of K steps with events around every stage (stage times, the roofline's kernel
    # duration); an event between two launches stops the second one from starting early
    # (programmatic dependent launch), so that pass's step is a little slower.
    events = {}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_start, s_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # nvidia-smi samples every 100 ms: keep the same step running for about half a second
        # (untimed) so that the samples see the GPU under this load, then time
        t_soak, soak_steps = time.perf_counter(), 0
        while time.perf_counter() - t_soak < 0.5:
            for _ in range(8):
                wl.step(dcp)
            soak_steps += 8
            torch.cuda.synchronize()
        barrier(dist)
        start.record(stream)
        for _ in range(args.steps):
            wl.step(dcp)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        s_start.record(stream)
        for _ in range(args.steps):
            wl.step(dcp, events)
        s_end.record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, start.elapsed_time(end))
    staged_ms_step = max_over_ranks(dist, s_start.elapsed_time(s_end)) / args.steps
    stage_ms = _stage_ms(events, args.steps)
    step_bytes = sum(wl.bytes.values())
    ms_step = ms / args.steps
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    if int(wl.err.item()) != 0:
        raise RuntimeError(f"device error word {int(wl.err.item())}")

    # ---- end to end through the public API with host buffers (pinned)
    host_src = [p.cpu().pin_memory() for p in wl.rc.src_pools]
    host_q = wl.q.cpu().pin_memory()
    host_o = torch.empty(wl.o.shape, dtype=torch.float32).pin_memory()
    host_l = torch.empty(wl.lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_src) + host_q.numel() * 2
    d2h = host_o.numel() * 4 + host_l.numel() * 4

    # Every step uploads its inputs (the prefill-side pools and Q) from pinned host memory and
    # reads its result back.  The inputs are double-buffered on the device and uploaded on a copy
    # stream, so that step i + 1's upload overlaps step i's kernels; the host link then bounds the
    # step (about 210 GB/s host to device on GB300, by the copy engines and by SM loads alike).
    dev_in = [(wl.rc.src_pools, wl.q), ([torch.empty_like(p) for p in wl.rc.src_pools], torch.empty_like(wl.q))]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def upload(b):
        copy_stream.wait_event(consumed[b])  # the step that last read buffer b is done
        with torch.cuda.stream(copy_stream):
            for hs, ds in zip(host_src, dev_in[b][0]):
                ds.copy_(hs, non_blocking=True)
            dev_in[b][1].copy_(host_q, non_blocking=True)
        copied[b].record(copy_stream)

    def e2e_run(n):
        upload(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                upload(b ^ 1)
            stream.wait_event(copied[b])
            wl.step(dcp, inputs=dev_in[b])
            consumed[b].record(stream)
            host_o.copy_(wl.o, non_blocking=True)
            host_l.copy_(wl.lse, non_blocking=True)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 10))
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / e2e_steps
    # the host link on its own: one pinned upload of the largest input, best of 3
    bi = max(range(len(host_src)), key=lambda i: host_src[i].numel())
    big = host_src[bi]
    link_ms = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dev_in[0][0][bi].copy_(big, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        link_ms.append(a.elapsed_time(b))
    link_gbs = big.numel() * big.element_size() / (min(link_ms) * 1e-3) / 1e9
    e2e_value = world * step_bytes / (e2e_ms * 1e-3) / 1e9

    if rank != 0:
        return
    hbm, bf16, bf16_sus, peak_kind = peaks()
    plan_ms = stage_ms.pop("plan", None)  # on the side stream, overlapped with the reshard
    plan_info = None
    if plan_ms is not None and wl.layout != "token":  # the plan's queue, read back after the timed passes
        torch.cuda.synchronize()
        plan_info = dcp.attn_plan_info((wl.B, wl.T, wl.H), wl.rc.dst_vpages.numel(), wl.layer_pools[0], wl.ws)
    stage_gbs = {k: wl.stage_bytes[k] / (stage_ms[k] * 1e-3) / 1e9 for k in stage_ms}
    attn_tflops = wl.flops_attn / (stage_ms["attn"] * 1e-3) / 1e12
    dom = max(stage_ms, key=stage_ms.get)
    kernel_of = {"reshard": "reshard_kernel", "attn": "attn_kernel", "merge": "lse_merge_kernel"}
    src_of = {"reshard": ("dcp_reshard.cu", "dcp_copy_ring.cuh"), "attn": "dcp_attn.cu", "merge": "dcp_merge.cu"}
    tr = NCU_TRAFFIC.get((kernel_of[dom], wl.name))
    traffic = tr[1] if tr and tr[0] == _src_hash(src_of[dom]) else None
    # the tensor roofline uses the peak of the MMA kind executed: E4M3 measured on this GPU (a
    # cuBLASLt FP8 GEMM), else twice the BF16 peak (the nominal ratio)
    if wl.dtype == "e4m3":
        fp8 = fp8_dense_peak_tflops(dev)
        tc_peak, tc_kind = (fp8, "measured here: cuBLASLt e4m3 8192^3 GEMM, best of 10") if fp8 else (
            2.0 * bf16, peak_kind + " bf16 x2 (nominal e4m3 ratio)")
    else:
        tc_peak, tc_kind = bf16, peak_kind + " bf16"
    attn_bound = "tensor" if wl.flops_attn / tc_peak / 1e12 > wl.stage_bytes["attn"] / hbm / 1e9 else "hbm"
    if dom == "attn" and attn_bound == "tensor":
        roof = {"kernel": "attn_kernel", "bound": "tensor", "achieved": attn_tflops, "peak": tc_peak,
                "unit": "TFLOP/s", "frac": attn_tflops / tc_peak, "peak_kind": tc_kind,
                "traffic": traffic, "algorithmic_flops": wl.flops_attn}
    else:
        roof = {"kernel": kernel_of[dom], "bound": "hbm", "achieved": stage_gbs[dom], "peak": hbm, "unit": "GB/s",
                "frac": stage_gbs[dom] / hbm, "peak_kind": peak_kind, "traffic": traffic,
                "algorithmic_bytes": wl.stage_bytes[dom]}
    cpu = None
    if not args.no_cpu_baseline:
        gbs, desc, secs, threads, t_stage = oracle_sample(wl, max_seconds=args.ref_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc,
               "stage_seconds": t_stage}
        if wl.name.startswith(("tiny", "batch")):  # the small workloads: one core as well
            import oracle
            oracle.set_num_threads(1)
            try:
                g1, d1, _, _, _ = oracle_sample(wl, max_seconds=min(5.0, args.ref_seconds))
            finally:
                oracle.set_num_threads(threads)
            cpu["single_core"] = {"value": g1, "unit": "GB/s", "cores": 1, "sample": d1}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "e4m3 (fp32 accumulate)",
        "data": "synthetic",
        "config": workload_config(wl, world),
        "schedule": ("layer pipeline: the reshard layer by layer on a high-priority stream, each layer's "
                     "attention as soon as its layer has arrived (the stage pass below runs the stages one "
                     "after the other)" if wl.layer_pipe else "stages in order"),
        "stages": {
            "reshard": {"ms": stage_ms["reshard"], "GB/s": stage_gbs["reshard"], "frac_hbm": stage_gbs["reshard"] / hbm,
                        **({"mode": f"bounded pack, {args.staging_mb} MB staging buffer",
                            "moved_GB/s": wl.pack_moved_bytes / (stage_ms["reshard"] * 1e-3) / 1e9,
                            "moved_frac_hbm": wl.pack_moved_bytes / (stage_ms["reshard"] * 1e-3) / 1e9 / hbm}
                           if wl.pack else
                           {"mode": "naive: full transfer to every DCP rank + in-place shard",
                            "moved_GB/s": wl.naive_moved_bytes / (stage_ms["reshard"] * 1e-3) / 1e9,
                            "moved_frac_hbm": wl.naive_moved_bytes / (stage_ms["reshard"] * 1e-3) / 1e9 / hbm}
                           if wl.naive else {"mode": "token-interleaved row gather"} if wl.layout == "token"
                           else {"mode": "direct"})},
            "attn": {"ms": stage_ms["attn"], "GB/s": stage_gbs["attn"], "TFLOP/s": attn_tflops,
                     "frac_hbm": stage_gbs["attn"] / hbm, "frac_tensor": attn_tflops / tc_peak,
                     "tensor_peak_TFLOP/s": tc_peak, "tensor_peak_kind": tc_kind, "bound": attn_bound,
                     "includes_merge": wl.fused},
            **({} if wl.fused else {"merge": {"ms": stage_ms["merge"], "GB/s": stage_gbs["merge"],
                                              "frac_hbm": stage_gbs["merge"] / hbm}}),
            **({"plan": {"ms": plan_ms, "stream": "side, overlapped with the reshard; once per step",
                         **({"units": plan_info["units"], "split_pairs": plan_info["split_pairs"],
                             "tiles_per_chunk": plan_info["tiles_per_chunk"]} if plan_info else {})}}
               if plan_ms is not None else {}),
            "pass": {"steps": args.steps, "ms_per_step": staged_ms_step,
                     "note": "second timed pass with CUDA events around each stage"},
            "attn_plus_merge_frac_of_roofline": (
                max((wl.bytes["attn"] + wl.bytes["merge"]) / hbm / 1e9, wl.flops_attn / tc_peak / 1e12)
                / ((stage_ms["attn"] + stage_ms.get("merge", 0.0)) * 1e-3)),
        },
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "h2d_GB/s": h2d / (e2e_ms * 1e-3) / 1e9, "link_h2d_GB/s": link_gbs,
                "frac_of_link": h2d / (e2e_ms * 1e-3) / 1e9 / link_gbs,
                "note": "inputs double-buffered on the device, next step's upload on a copy stream"},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": {**clk.summary(), "window": f"{soak_steps} untimed steps of the same work, then both timed passes"},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="e2e",
                    help="e2e (default, the largest workload): 64 requests of 2K-500K, 8 layers, CP4 -> DCP8, "
                         "E4M3; batch: 32 x 8192 BF16; agent: 48 x 100K E4M3; long: 4 x 1M, q_len 4, E4M3; "
                         "tiny: 1 x 1024 (a check, not a bench)")
    ap.add_argument("--ref-seconds", type=float, default=15.0,
                    help="host-time budget of one oracle sample (cpu_baseline; per step of --impl reference at most)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle sample in the CUDA arm")
    ap.add_argument("--layout", choices=["page", "token"], default="page",
                    help="token: token-interleaved DCP (rank i holds tokens i, i + N, ...) instead of pages")
    ap.add_argument("--naive", action="store_true",
                    help="reshard as the pages' initial design: full KV to every DCP rank, then an in-place shard")
    ap.add_argument("--staging-mb", type=int, default=0,
                    help="reshard in bounded pack mode through a staging buffer of this many MB (0: direct)")
    ap.add_argument("--no-plan-overlap", action="store_true",
                    help="make the attention plan inside every attention call instead of once per step on a "
                         "side stream overlapped with the reshard")
    ap.add_argument("--profile-steps", action="store_true",
                    help="run only the warm-up and --steps plain steps (for ncu captures; no bench line)")
    ap.add_argument("--no-layer-overlap", action="store_true",
                    help="several layers: reshard all layers before the first attention instead of starting "
                         "each layer's attention as soon as its layer has arrived")
    ap.add_argument("--unfused", action="store_true",
                    help="partial attention and the LSE merge as separate calls (default: one call)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
