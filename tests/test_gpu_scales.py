"""Non-default scales through every attention entry point.

The FP8 KV scale multiplies both the scores and V, and the softmax scale only the scores; each
entry point (per-rank partials, fused with the merge, plan once then run, the static-scratch
variant) carries them on its own path to the kernels, so each is compared with the oracle at
scales other than the ones every other test uses.
"""
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,kv_scale,softmax_scale", [("e4m3", 0.011, 0.05), ("e4m3", 0.04, 0.11),
                                                          ("bf16", 1.0, 0.031)])
def test_every_entry_point_carries_the_scales(cuda_device, dtype, kv_scale, softmax_scale):
    case = di.attention_case([1500, 333, 64 * 20], H=64, T=2, n_dcp=4, dtype=dtype, slots_per_rank=None, seed=31,
                             device=cuda_device, name="scales")
    case.kv_scale, case.softmax_scale = kv_scale, softmax_scale
    R, N = case.rows, case.n_dcp
    qb, pools = q_bits(case), pool_bytes(case)
    ref = [oracle_attention(case, rank=d, qb=qb, pools=pools) for d in range(N)]
    ref_m = oracle_attention(case, qb=qb, pools=pools)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools, softmax_scale, kv_scale)

    def check_parts(o, lse, what):
        torch.cuda.synchronize()
        assert int(err.item()) == 0, what
        for d in range(N):
            compare(o[d].cpu().numpy().reshape(R, 512), lse[d].cpu().numpy().reshape(R), *ref[d], f"{what} rank {d}")

    o, lse = dcp.partial_decode_attn(*args, dev_error=err)
    check_parts(o, lse, "partial")
    mo, ml, o, lse = dcp.decode_attn_merged(*args, dev_error=err)
    check_parts(o, lse, "fused")
    compare(mo.cpu().numpy().reshape(R, 512), ml.cpu().numpy().reshape(R), *ref_m, "fused merged")
    ws = dcp.alloc_workspace(case.B, case.T, case.H, N, case.dst_vpages.numel(), cuda_device)
    dcp.attn_plan((case.B, case.T, case.H), case.req_page_ptr, case.dst_vpages, case.pools, ws, dev_error=err)
    o, lse = dcp.partial_decode_attn(*args, workspace=ws, dev_error=err, planned=True)
    check_parts(o, lse, "planned run")
    mo, ml, o, lse = dcp.decode_attn_merged(*args, workspace=ws, dev_error=err, planned=True)
    check_parts(o, lse, "planned fused")
    compare(mo.cpu().numpy().reshape(R, 512), ml.cpu().numpy().reshape(R), *ref_m, "planned fused merged")
    o, lse = dcp.partial_decode_attn_static(*args, dev_error=err)
    check_parts(o, lse, "static")
