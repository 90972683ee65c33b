"""Helpers shared by the GPU parity tests: host copies for the oracle and comparisons."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances for floating-point attention outputs (max-abs): 2e-2 on O and 1e-3 on LSE.
O_TOL = 2e-2
LSE_TOL = 1e-3


def q_bits(case) -> np.ndarray:
    return case.q.cpu().view(torch.int16).numpy().view(np.uint16)


def pool_bytes(case) -> list:
    if case.dtype == "bf16":
        return [p.cpu().view(torch.int16).numpy().view(np.uint16) for p in case.pools]
    return [p.cpu().view(torch.uint8).numpy() for p in case.pools]


def oracle_attention(case, rank=-1, rows=None, qb=None, pools=None, layout=None):
    qb = q_bits(case) if qb is None else qb
    pools = pool_bytes(case) if pools is None else pools
    return oracle.attention(qb, case.seq_lens.cpu().numpy(), case.req_page_ptr.cpu().numpy(),
                            case.dst_vpages.cpu().numpy(), pools,
                            oracle.BF16 if case.dtype == "bf16" else oracle.E4M3, case.kv_scale,
                            case.softmax_scale, case.n_dcp, rank=rank, rows=rows, q_len=case.T,
                            num_heads=case.H, layout=layout or getattr(case, "layout", "page"))


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what: str, o_tol=O_TOL, lse_tol=LSE_TOL):
    """Element-wise comparison; -inf LSE must match exactly (empty shards)."""
    o_gpu = np.asarray(o_gpu, np.float64).reshape(o_ref.shape)
    lse_gpu = np.asarray(lse_gpu, np.float64).reshape(lse_ref.shape)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    ninf_ref = np.isneginf(lse_ref)
    ninf_gpu = np.isneginf(lse_gpu)
    assert np.array_equal(ninf_ref, ninf_gpu), f"{what}: empty-shard rows differ"
    do = float(np.abs(o_gpu - o_ref).max()) if o_ref.size else 0.0
    fin = ~ninf_ref
    dl = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert do <= o_tol, f"{what}: O max-abs error {do:.3e} > {o_tol}"
    assert dl <= lse_tol, f"{what}: LSE max-abs error {dl:.3e} > {lse_tol}"
    return do, dl
