"""A skewed batch: many short requests next to two long ones, with more (rank, request)
segments than SMs, so that the plan sizes its chunks from the per-SM share of all tiles and cuts
only the long segments into chunks.  Every rank's partial and the merged output are checked
against the oracle on sampled rows of every request."""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,n_short", [("e4m3", 22), ("bf16", 22), ("e4m3", 38)])
def test_skewed_batch_with_more_segments_than_sms(cuda_device, dtype, n_short):
    # 24 requests: 192 segments, chunks of the average segment; 40 requests: 320 segments, chunks
    # grown to 0.6 of the per-SM share of all tiles (larger than the average segment)
    rng = np.random.default_rng(7)
    lens = [60_000, 61_111] + [int(x) for x in rng.integers(1, 3000, size=n_short)]
    H, T, N = 64, 1, 8
    case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=17,
                             device=cuda_device, name="skew")
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o, lse, o_part, lse_part = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages,
                                                      case.pools, case.softmax_scale, case.kv_scale, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # rows 0, 21, 42, 63 of every request (q_len 1: row = b * H + h)
    rows = np.array([b * H + h for b in range(len(lens)) for h in (0, 21, 42, 63)], np.int64)
    qb, pools = q_bits(case), pool_bytes(case)
    R = case.rows
    for d in range(N):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o_part[d].cpu().numpy().reshape(R, 512)[rows], lse_part[d].cpu().numpy().reshape(R)[rows], ro, rl,
                f"skew rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(o.cpu().numpy().reshape(R, 512)[rows], lse.cpu().numpy().reshape(R)[rows], ro, rl, "skew merged")
