"""Seeded random shapes through the fused entry point (every rank's partial plus the merge).

Each case draws the batch size, the sequence lengths (at least q_len), the head count (including
counts that leave a partial query group of fewer than 64 rows), q_len, the DCP size and the KV
type, then compares every rank's partial and the merged output with the oracle row by row.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    T = int(rng.integers(1, 4))
    B = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(T, 3000, size=B)]
    if rng.random() < 0.3:  # a request shorter than one page
        lens[int(rng.integers(0, B))] = int(rng.integers(T, 64))
    H = int(rng.choice([16, 32, 48, 64, 80, 112, 128]))
    N = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    dtype = "e4m3" if rng.random() < 0.5 else "bf16"
    return f"r{i}-b{B}-t{T}-h{H}-n{N}-{dtype}", lens, H, T, N, dtype


CASES = [_draw(i) for i in range(16)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,lens,H,T,N,dtype", CASES, ids=[c[0] for c in CASES])
def test_random_shapes_fused(cuda_device, name, lens, H, T, N, dtype):
    case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=len(name) + 77,
                             device=cuda_device, name=name)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o_part = torch.full((N, case.B, T, H, 512), float("nan"), device=cuda_device)
    lse_part = torch.full((N, case.B, T, H), float("nan"), device=cuda_device)
    o, lse, _, _ = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                          case.softmax_scale, case.kv_scale, o_part=o_part, lse_part=lse_part,
                                          dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = case.rows
    qb, pools = q_bits(case), pool_bytes(case)
    for d in range(N):
        ro, rl = oracle_attention(case, rank=d, qb=qb, pools=pools)
        compare(o_part[d].cpu().numpy().reshape(R, 512), lse_part[d].cpu().numpy().reshape(R), ro, rl,
                f"{name} rank {d}")
    ro, rl = oracle_attention(case, qb=qb, pools=pools)
    compare(o.cpu().numpy().reshape(R, 512), lse.cpu().numpy().reshape(R), ro, rl, f"{name} merged")
