"""Rank bodies for the multi-rank control tests (gloo on CPU, spawned processes)."""
from __future__ import annotations

import datetime
import os
import sys
import time
import traceback

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _init(rank, world, port):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=20))
    return dist


def run(rank, world, port, scenario, out_q):
    """Runs ``scenario`` on this rank and puts (rank, result or exception text) on out_q."""
    try:
        dist = _init(rank, world, port)
        res = SCENARIOS[scenario](rank, world, dist)
        out_q.put((rank, "ok", res))
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent test
        out_q.put((rank, type(e).__name__, f"{e}\n{traceback.format_exc()}"))


def _size_broadcast_divergent(rank, world, dist):
    import torch
    from decode_context_paged_gb300 import control
    gate = control.StepGate(dist.distributed_c10d._get_default_store(), world, timeout_s=10)
    owner = 0
    # the owner matched 5 slots; rank 1 matched 5 as well, rank 2 only 3 (prefix divergence)
    local = {0: 5, 1: 5, 2: 3}[rank]
    kv = torch.arange(5 * 4, dtype=torch.float32).reshape(5, 4) if rank == owner else torch.empty((0, 4))
    calls = []
    committed, data = control.size_broadcast(torch.arange(local), kv, owner, gate=gate, step="layer0")
    calls.append("layer0")
    # second step: the owner has no prefix at all -> every rank skips, consistently
    local2 = {0: 0, 1: 4, 2: 0}[rank]
    c2, d2 = control.size_broadcast(torch.arange(local2), torch.empty((0, 4)), owner, gate=gate, step="layer1")
    calls.append("layer1")
    return {"committed": committed, "data": None if data is None else data.tolist(), "skip2": (c2, d2),
            "calls": calls}


def _gate_catches_a_skipping_rank(rank, world, dist):
    import torch
    from decode_context_paged_gb300 import control
    gate = control.StepGate(dist.distributed_c10d._get_default_store(), world, timeout_s=3)
    prefix = torch.arange(0 if rank == 1 else 6)
    t0 = time.monotonic()
    if rank == 1 and prefix.numel() == 0:
        # the early return the size broadcast replaced: this rank leaves the protocol
        return {"skipped": True}
    try:
        control.size_broadcast(prefix, torch.zeros((6, 2)), 0, gate=gate, step="buggy")
    except control.GateTimeout as e:
        return {"gate_timeout": str(e), "seconds": time.monotonic() - t0}
    return {"completed": True}


def _consensus_and_padded(rank, world, dist):
    import torch
    from decode_context_paged_gb300 import control
    n = control.consensus_prefix_len({0: 7, 1: 5, 2: 9}[rank])
    vals = torch.arange({0: 3, 1: 5, 2: 0}[rank], dtype=torch.float64) + 10 * rank
    s = control.padded_all_reduce(vals, op=dist.ReduceOp.SUM)
    m = control.padded_all_reduce(vals, op=dist.ReduceOp.MAX)
    # integers past 2^53 stay exact (a float64 reduction would round them)
    big = torch.tensor([(1 << 60) + 1 + rank] * (rank + 1), dtype=torch.int64)
    bs = control.padded_all_reduce(big, op=dist.ReduceOp.SUM)
    bm = control.padded_all_reduce(big, op=dist.ReduceOp.MIN)
    return {"prefix": n, "sum": s.tolist(), "max": m.tolist(), "big_sum": bs.tolist(), "big_min": bm.tolist(),
            "big_dtype": str(bs.dtype)}


def _gather_and_merge(rank, world, dist):
    import numpy as np
    import torch
    import dcp_inputs as di
    import oracle
    from decode_context_paged_gb300 import control
    case = di.attention_case([700, 130, 64 * 5 + 3], H=4, T=2, n_dcp=world, dtype="bf16", slots_per_rank=None,
                             seed=13, device="cpu")
    qb = case.q.view(torch.int16).numpy().view(np.uint16)
    pools = [p.view(torch.int16).numpy().view(np.uint16) for p in case.pools]
    args = (qb, case.seq_lens.numpy(), case.req_page_ptr.numpy(), case.dst_vpages.numpy(), pools, oracle.BF16, 1.0,
            case.softmax_scale, world)
    o_d, l_d = oracle.attention(*args, rank=rank, q_len=case.T, num_heads=case.H)  # this rank's shard only

    def merge(o, l):
        mo, ml = oracle.lse_merge(o.numpy(), l.numpy())
        return torch.from_numpy(mo), torch.from_numpy(ml)

    o, l = control.gather_and_merge(torch.from_numpy(o_d), torch.from_numpy(l_d), merge=merge)
    ro, rl = oracle.attention(*args, rank=-1, q_len=case.T, num_heads=case.H)
    return {"o_err": float(np.abs(o.numpy() - ro).max()), "lse_err": float(np.abs(l.numpy() - rl).max())}


SCENARIOS = {
    "size_broadcast_divergent": _size_broadcast_divergent,
    "gate_catches_a_skipping_rank": _gate_catches_a_skipping_rank,
    "consensus_and_padded": _consensus_and_padded,
    "gather_and_merge": _gather_and_merge,
}
