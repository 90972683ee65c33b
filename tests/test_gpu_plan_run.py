"""GPU: a plan made once (dcp_attn_plan) and run for several layers (dcp_partial_decode_attn_run,
dcp_decode_attn_merged_run) gives, run after run, exactly the one-call results for each layer's
Q and pools (same kernels; the work counter is reset by every run).  Chunked segments included."""
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp

pytestmark = pytest.mark.gpu

CASES = [
    ("ragged", [1000, 130, 64 * 9 + 5], 64, 1, 4, "bf16"),
    ("causal-q4-fp8", [64 * 7 + 3, 66, 260], 64, 4, 2, "e4m3"),
    ("mixed-len-fp8", [70_000, 9_000], 64, 1, 8, "e4m3"),
    ("chunked", [64 * 1024 + 17, 3000], 64, 1, 2, "bf16"),
]


@pytest.mark.parametrize("name,lens,H,T,N,dtype", CASES, ids=[c[0] for c in CASES])
def test_plan_once_run_per_layer_equals_one_call(cuda_device, name, lens, H, T, N, dtype):
    layers = [di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=s, device=cuda_device,
                                name=name) for s in (1, 2, 3)]
    base = layers[0]
    for c in layers[1:]:  # one page table for the step: same table, new Q and pools per layer
        c.req_page_ptr, c.dst_vpages = base.req_page_ptr, base.dst_vpages
    ws = dcp.alloc_workspace(base.B, T, H, N, base.dst_vpages.numel(), cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dcp.attn_plan((base.B, T, H), base.req_page_ptr, base.dst_vpages, base.pools, ws, dev_error=err)
    for c in layers:
        args = (c.q, c.seq_lens, c.req_page_ptr, c.dst_vpages, c.pools, c.softmax_scale, c.kv_scale)
        o_r, l_r = dcp.partial_decode_attn(*args, workspace=ws, dev_error=err, planned=True)
        o_1, l_1 = dcp.partial_decode_attn(*args, dev_error=err)
        m_r = dcp.decode_attn_merged(*args, workspace=ws, dev_error=err, planned=True)
        m_1 = dcp.decode_attn_merged(*args, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(o_r, o_1) and torch.equal(l_r, l_1)
        for a, b in zip(m_r, m_1):
            assert torch.equal(a, b)


MISMATCH = [
    # what differs between the plan and the run
    ("fewer-requests", dict(B=2)),
    ("other-dtype", dict(dtype="e4m3")),
    ("other-heads", dict(H=32)),
    ("other-ranks", dict(N=2)),
    ("no-plan", dict(no_plan=True)),
]


@pytest.mark.parametrize("what,change", MISMATCH, ids=[m[0] for m in MISMATCH])
def test_planned_run_refuses_a_mismatched_plan(cuda_device, what, change):
    """A planned run whose arguments do not match the plan in the workspace (or a workspace that
    holds no plan) sets DEVERR_PLAN_MISMATCH and computes nothing: outputs keep their sentinel."""
    lens, H, N = [1000, 130, 64 * 9 + 5], 64, 4
    base = di.attention_case(lens, H=H, T=1, n_dcp=N, dtype="bf16", slots_per_rank=None, seed=4, device=cuda_device)
    run = di.attention_case(lens[:change.get("B", 3)], H=change.get("H", H), T=1, n_dcp=change.get("N", N),
                            dtype=change.get("dtype", "bf16"), slots_per_rank=None, seed=5, device=cuda_device)
    ws = dcp.alloc_workspace(3, 1, H, N, base.dst_vpages.numel(), cuda_device)
    ws.fill_(0)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    if not change.get("no_plan"):
        dcp.attn_plan((base.B, 1, H), base.req_page_ptr, base.dst_vpages, base.pools, ws, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    need = dcp.workspace_size(run.B, 1, run.H, run.n_dcp, run.dst_vpages.numel())
    wsr = ws if need <= ws.numel() else torch.cat([ws, torch.zeros(need - ws.numel(), dtype=torch.uint8,
                                                                   device=cuda_device)])
    o = torch.full((run.n_dcp, run.B, 1, run.H, 512), 7.0, device=cuda_device)
    l = torch.full((run.n_dcp, run.B, 1, run.H), 7.0, device=cuda_device)
    oo = torch.full((run.B, 1, run.H, 512), 7.0, device=cuda_device)
    lo = torch.full((run.B, 1, run.H), 7.0, device=cuda_device)
    dcp.decode_attn_merged(run.q, run.seq_lens, run.req_page_ptr, run.dst_vpages, run.pools, run.softmax_scale,
                           run.kv_scale, o_part=o, lse_part=l, o_out=oo, lse_out=lo, workspace=wsr, dev_error=err,
                           planned=True)
    torch.cuda.synchronize()
    assert int(err.item()) & dcp.DEVERR_PLAN_MISMATCH
    assert dcp.device_error_status(int(err.item())) == -4  # DCP_ERR_WORKSPACE
    for t in (o, l, oo, lo):
        assert bool((t == 7.0).all())
    # the matching run afterwards is fine
    if not change.get("no_plan") and wsr is ws:
        err.zero_()
        dcp.decode_attn_merged(base.q, base.seq_lens, base.req_page_ptr, base.dst_vpages, base.pools,
                               base.softmax_scale, base.kv_scale, workspace=ws, dev_error=err, planned=True)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
