"""Multi-rank control of the DCP transfer path (host side).

"Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding":
  * 6.7 "Bootstrap": the decode side's DCP rank is d = attn_tp_rank mod N_dcp, and (N_dcp, d)
    travel with every request to the prefill side, which filters each transfer by the metadata
    of the request it serves (heterogeneous decode groups, DCP size changes between requests).
  * 4.2 "Prefix KV Broadcast: Size-Broadcast Protocol": every rank joins a one-element broadcast
    of the owner's element count n first; then either every rank skips (n = 0) or every rank
    joins the same n-element broadcast, and a non-owner commits the received data only when its
    own count equals n.
  * Conclusion: consensus prefix lengths and padded all-reduces keep every rank in the same
    collectives; "SGLang's path": one exchange per layer gathers the ranks' partial (O, LSE) and
    merges them exactly.

A rank that leaves the protocol (the early return the size broadcast replaced) would leave the
others blocked in a collective.  StepGate lets every rank check, before a protocol step, that
all ranks reached it: a missing rank shows up as a GateTimeout on the others after a bounded
wait, never as a hang.
"""
from __future__ import annotations

import time
from dataclasses import dataclass

import torch
import torch.distributed as dist


# ------------------------------------------------------------------------------ bootstrap
@dataclass(frozen=True)
class DstKVInfo:
    """Per-request destination metadata: the decode side's DCP size and this rank's DCP rank."""
    dcp_size: int
    dcp_rank: int


def decode_dst_info(attn_tp_rank: int, dcp_size: int) -> DstKVInfo:
    """Decode side: d = attn_tp_rank mod N_dcp (6.7); a single rank when N_dcp <= 1."""
    if dcp_size < 1 or attn_tp_rank < 0:
        raise ValueError("dcp_size >= 1 and attn_tp_rank >= 0 required")
    return DstKVInfo(dcp_size, attn_tp_rank % dcp_size if dcp_size > 1 else 0)


def transfer_filter_params(info: DstKVInfo | None, local_dcp_size: int, local_tp_rank: int) -> tuple[int, int]:
    """Prefill side: the (N_dcp, d) to filter one request's transfer with.  The request's own
    metadata is authoritative; the local values are only the fallback (6.7)."""
    if info is not None:
        return info.dcp_size, info.dcp_rank
    fb = decode_dst_info(local_tp_rank, local_dcp_size)
    return fb.dcp_size, fb.dcp_rank


# ------------------------------------------------------------------------------- step gate
class GateTimeout(RuntimeError):
    """Raised on the ranks that reached a protocol step when another rank did not."""


class StepGate:
    """Before a protocol step, every rank announces itself in the process group's store and
    waits (bounded) until all ranks did; the step name must be unique per step and rank-invariant."""

    def __init__(self, store, world_size: int, timeout_s: float = 5.0, poll_s: float = 0.005):
        self.store = store
        self.world = world_size
        self.timeout_s = timeout_s
        self.poll_s = poll_s

    def arrive(self, step: str) -> None:
        key = f"dcp_gate/{step}"
        self.store.add(key, 1)
        t0 = time.monotonic()
        while True:
            n = self.store.add(key, 0)
            if n >= self.world:
                return
            if time.monotonic() - t0 > self.timeout_s:
                raise GateTimeout(f"step {step!r}: {n} of {self.world} ranks arrived within {self.timeout_s:.1f} s")
            time.sleep(self.poll_s)


# ------------------------------------------------------------------------- size broadcast
def size_broadcast(local_slots: torch.Tensor, kv: torch.Tensor, owner: int, group=None,
                   gate: StepGate | None = None, step: str = "") -> tuple[bool, torch.Tensor | None]:
    """4.2's protocol.  ``local_slots``: this rank's matched prefix slots; ``kv``: on the owner,
    the KV elements of its slots ([n][...]); elsewhere a tensor whose trailing shape and dtype
    the received elements take.  Returns (committed, data): the owner and every non-owner whose
    own count equals n commit the n elements; the others consume the broadcast without
    committing; with n = 0 every rank skips and returns (False, None)."""
    rank = dist.get_rank(group)
    if gate is not None:
        gate.arrive(f"{step}/count")
    n_t = torch.tensor([local_slots.numel() if rank == owner else 0], dtype=torch.int64)
    dist.broadcast(n_t, src=owner, group=group)  # every rank joins: the count decides for all
    n = int(n_t.item())
    if n == 0:
        return False, None
    buf = kv.contiguous().clone() if rank == owner else torch.empty((n, *kv.shape[1:]), dtype=kv.dtype)
    if rank == owner and buf.shape[0] != n:
        raise ValueError("owner's KV rows and slot count differ")
    if gate is not None:
        gate.arrive(f"{step}/data")
    dist.broadcast(buf, src=owner, group=group)  # every rank joins the same n-element broadcast
    commit = rank == owner or local_slots.numel() == n
    return commit, (buf if commit else None)


# ------------------------------------------------------------------ consensus / all-reduce
def consensus_prefix_len(local_len: int, group=None) -> int:
    """Every rank uses the prefix length all ranks matched: the minimum over ranks."""
    t = torch.tensor([int(local_len)], dtype=torch.int64)
    dist.all_reduce(t, op=dist.ReduceOp.MIN, group=group)
    return int(t.item())


def _pad_value(op, dtype: torch.dtype):
    """The identity of `op` in `dtype` (integers: 0, or the type's extreme for MAX / MIN)."""
    if op == dist.ReduceOp.SUM:
        return 0
    info = torch.finfo(dtype) if dtype.is_floating_point else torch.iinfo(dtype)
    if op == dist.ReduceOp.MAX:
        return float("-inf") if dtype.is_floating_point else info.min
    if op == dist.ReduceOp.MIN:
        return float("inf") if dtype.is_floating_point else info.max
    raise ValueError(f"padded_all_reduce: unsupported op {op}")


def padded_all_reduce(values: torch.Tensor, op=dist.ReduceOp.SUM, group=None) -> torch.Tensor:
    """All-reduce of 1-D tensors whose length differs per rank: the ranks agree on the longest
    length (an all-reduce MAX every rank joins), pad with op's identity and reduce; every rank
    joins both collectives whatever its own length (even 0).  The reduction runs in the values'
    own dtype, so integers stay exact (every rank must pass the same dtype)."""
    n = torch.tensor([values.numel()], dtype=torch.int64)
    dist.all_reduce(n, op=dist.ReduceOp.MAX, group=group)
    width = int(n.item())
    buf = torch.full((width,), _pad_value(op, values.dtype), dtype=values.dtype)
    buf[:values.numel()] = values
    dist.all_reduce(buf, op=op, group=group)
    return buf


# ------------------------------------------------------------------------------ exchange
def gather_and_merge(o_local: torch.Tensor, lse_local: torch.Tensor, merge=None, group=None):
    """The per-layer exchange: all-gather every DCP rank's partial (O_d [rows][512], LSE_d
    [rows]) in rank order, then the exact LSE merge (default: the library's dcp_lse_merge on the
    gathered device tensors).  Returns (O, LSE)."""
    world = dist.get_world_size(group)
    os_ = [torch.empty_like(o_local) for _ in range(world)]
    ls_ = [torch.empty_like(lse_local) for _ in range(world)]
    dist.all_gather(os_, o_local.contiguous(), group=group)
    dist.all_gather(ls_, lse_local.contiguous(), group=group)
    o, lse = torch.stack(os_), torch.stack(ls_)
    if merge is None:
        from . import lse_merge as merge
    return merge(o, lse)
