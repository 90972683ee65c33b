"""GPU parity of the fused partial-attention + LSE-merge entry point (dcp_decode_attn_merged).

The merged output must match the float64 oracle's unsharded attention (the merge of the
ranks' partials is exact, "SGLang's path") within the attention tolerances; the partials it leaves in
o_part / lse_part must equal those of dcp_partial_decode_attn bit for bit (same kernels), and
its merged rows must equal dcp_lse_merge of those partials (same arithmetic, ascending rank
order).  Cases cover requests whose ranks are all single-chunk, requests with a rank in
several chunks, both in one call, empty ranks, q_len 4 and 96 heads.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits

pytestmark = pytest.mark.gpu

CASES = [
    # name, lens, H, T, N, dtype
    ("ragged", [1000, 130, 64 * 9 + 5], 64, 1, 4, "bf16"),
    ("empty-ranks", [64, 200, 1], 64, 1, 8, "bf16"),
    ("causal-q4", [64 * 7 + 3, 66, 260], 64, 4, 2, "bf16"),
    ("heads-96", [700, 333], 96, 1, 3, "bf16"),
    ("dcp1", [1500], 64, 1, 1, "bf16"),
    ("ragged-fp8", [1000, 130, 64 * 9 + 5], 64, 1, 4, "e4m3"),
    ("causal-q4-fp8", [64 * 7 + 3, 66, 260], 64, 4, 2, "e4m3"),
    ("mixed-len-fp8", [70_000, 9_000], 64, 1, 8, "e4m3"),
    # one request whose ranks run in several chunks next to single-chunk requests
    ("chunked-and-single", [64 * 1024 + 17, 3000, 200], 64, 1, 2, "bf16"),
    ("chunked-and-single-fp8", [64 * 1024 + 17, 3000, 200], 64, 1, 2, "e4m3"),
]


def _run(case, ws=None):
    err = torch.zeros(1, dtype=torch.int32, device=case.q.device)
    o, l, op, lp = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                          case.softmax_scale, case.kv_scale, workspace=ws, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o, l, op, lp


@pytest.mark.parametrize("name,lens,H,T,N,dtype", CASES, ids=[c[0] for c in CASES])
def test_merged_matches_oracle_and_unfused(cuda_device, name, lens, H, T, N, dtype):
    case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=3 + len(name),
                             device=cuda_device, name=name)
    o, l, op, lp = _run(case)
    # partials: identical to the partial-attention entry point
    op_ref, lp_ref = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                             case.softmax_scale, case.kv_scale)
    om_ref, lm_ref = dcp.lse_merge(op_ref, lp_ref)
    torch.cuda.synchronize()
    assert torch.equal(op, op_ref) and torch.equal(lp, lp_ref)
    # merged rows: the separate merge of the same partials, up to fp32 rounding
    assert torch.equal(torch.isneginf(l), torch.isneginf(lm_ref))
    fin = ~torch.isneginf(lm_ref)
    assert float((l[fin] - lm_ref[fin]).abs().max()) <= 1e-6 if fin.any() else True
    assert float((o - om_ref).abs().max()) <= 1e-6
    # merged rows against the unsharded float64 oracle (sampled for the long case)
    R = case.rows
    rows = None if sum(lens) < 50_000 else np.arange(0, R, 5)
    ro, rl = oracle_attention(case, rows=rows, qb=q_bits(case), pools=pool_bytes(case))
    on, ln = o.cpu().numpy().reshape(R, 512), l.cpu().numpy().reshape(R)
    if rows is not None:
        on, ln = on[rows], ln[rows]
    compare(on, ln, ro, rl, f"{name} merged")


def test_merged_consecutive_calls_reuse_workspace(cuda_device):
    """Repeated calls on one workspace give identical results (nothing carries over)."""
    case = di.attention_case([3000, 900, 64 * 40], H=64, T=1, n_dcp=4, dtype="bf16", slots_per_rank=None, seed=9,
                             device=cuda_device, name="reuse")
    ws = dcp.alloc_workspace(case.B, case.T, case.H, case.n_dcp, case.dst_vpages.numel(), cuda_device)
    first = [t.clone() for t in _run(case, ws)[:2]]
    for _ in range(3):
        again = _run(case, ws)[:2]
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])


@pytest.mark.gpu
def test_control_gather_and_merge_on_a_one_rank_nccl_group(cuda_device, monkeypatch):
    """The per-layer exchange of the multi-GPU deployment (all-gather of the partials, then the
    library's merge) through a real NCCL group; one GPU per box here, so one rank holding every
    DCP partial as its own rows' stack is gathered and merged."""
    import socket

    import torch.distributed as dist

    from decode_context_paged_gb300 import control
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    monkeypatch.setenv("MASTER_ADDR", "127.0.0.1")
    monkeypatch.setenv("MASTER_PORT", str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=cuda_device)
    try:
        case = di.attention_case([900, 70], H=16, T=1, n_dcp=1, dtype="bf16", slots_per_rank=None, seed=12,
                                 device=cuda_device, name="nccl-1")
        o, lse = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                         case.softmax_scale)
        R = case.rows
        om, lm = control.gather_and_merge(o[0].reshape(R, 512), lse[0].reshape(R))
        torch.cuda.synchronize()
        ro, rl = oracle_attention(case, qb=q_bits(case), pools=pool_bytes(case))
        compare(om.cpu().numpy().reshape(R, 512), lm.cpu().numpy().reshape(R), ro, rl, "nccl gather + merge")
    finally:
        dist.destroy_process_group()
