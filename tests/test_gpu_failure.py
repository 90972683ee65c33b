"""The device-side failure path: a pipeline wait runs out, the host reads the status, and the
context keeps working (no fault, trap or hang is involved)."""
import time

import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits


def test_selftest_rejects_bad_limits():
    # argument checks happen on the host, before any launch (no GPU needed)
    lib = dcp.library()
    assert lib.dcp_selftest_wait_timeout(0, 1, 1, None) == -1
    assert lib.dcp_selftest_wait_timeout(2_000_000_000, 1, 1, None) == -1
    assert lib.dcp_selftest_wait_timeout(1000, None, 1, None) == -1


@pytest.mark.gpu
def test_wait_times_out_and_the_context_stays_usable(cuda_device):
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ok = torch.full((1,), 7, dtype=torch.int32, device=cuda_device)
    t0 = time.monotonic()
    dcp.selftest_wait_timeout(2_000_000, err, ok)  # 2 ms
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(ok.item()) == 0
    assert int(err.item()) & dcp.DEVERR_TIMEOUT
    assert dcp.device_error_status(int(err.item())) == -6  # DCP_ERR_TIMEOUT
    assert elapsed < 5.0
    # the next call on the same context computes correctly
    case = di.attention_case([700, 64], H=16, T=1, n_dcp=2, dtype="bf16", slots_per_rank=None, seed=4,
                             device=cuda_device, name="after-timeout")
    err2 = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o, lse, _, _ = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                          case.softmax_scale, dev_error=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    ro, rl = oracle_attention(case, qb=q_bits(case), pools=pool_bytes(case))
    compare(o.cpu().numpy().reshape(case.rows, 512), lse.cpu().numpy().reshape(case.rows), ro, rl, "after timeout")
