"""The allocation-free partial-attention entry point (dcp_partial_decode_attn_static).

It serves callers that cannot call cudaMalloc — a host whose pool allocator owns all device
memory, or a decode loop where allocating is not allowed — by using the library's fixed
device scratch array instead of a caller workspace.  Its outputs must match the regular
entry point's on the same inputs, on consecutive calls (the array keeps the previous call's
contents, which must not leak into the next result).  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu


def _compare(case):
    err = torch.zeros(1, dtype=torch.int32, device=case.q.device)
    ref_o, ref_l = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages,
                                           case.pools, case.softmax_scale, case.kv_scale, dev_error=err)
    o = torch.full_like(ref_o, float("nan"))
    l = torch.full_like(ref_l, float("nan"))
    dcp.partial_decode_attn_static(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                   case.softmax_scale, case.kv_scale, o_part=o, lse_part=l, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ro, rl, go, gl = (t.cpu().numpy() for t in (ref_o, ref_l, o, l))
    assert np.isfinite(go).all()
    assert np.array_equal(np.isneginf(rl), np.isneginf(gl))
    fin = np.isfinite(rl)
    assert np.abs(go - ro).max() <= O_TOL
    assert np.abs(gl[fin] - rl[fin]).max() <= LSE_TOL


def test_static_scratch_matches_workspace_entry_point_twice(cuda_device):
    long_case = di.attention_case([64 * 1024 + 17], H=64, T=1, n_dcp=2, dtype="bf16", slots_per_rank=None,
                                  seed=21, device=cuda_device, name="chunked")
    ragged = di.attention_case([1000, 130, 64 * 9 + 5], H=64, T=1, n_dcp=4, dtype="bf16",
                               slots_per_rank=None, seed=3, device=cuda_device, name="ragged")
    _compare(long_case)   # first call: sets up the scratch address, uses chunk partials
    _compare(ragged)      # second call in a row: different sizes over the stale scratch
    _compare(long_case)


def test_static_scratch_rejects_sizes_over_the_limit(cuda_device):
    case = di.attention_case([64], H=64, T=1, n_dcp=1, dtype="bf16", slots_per_rank=None, seed=1,
                             device=cuda_device)
    big_pages = torch.zeros(4_000_000, dtype=torch.int32, device=cuda_device)  # needs > 64 MiB of scratch
    ptr = torch.tensor([0, 64], dtype=torch.int64, device=cuda_device)
    with pytest.raises(dcp.DcpError) as e:
        dcp.partial_decode_attn_static(case.q, case.seq_lens, ptr, big_pages, case.pools, case.softmax_scale)
    assert e.value.status == -4
