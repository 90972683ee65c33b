"""GPU parity of the token-interleaved DCP layout ("SGLang's path": rank i holds tokens i,
i + N, ...): the row-gather reshard bit for bit, and the per-rank partial attention over the
token-interleaved table (plus the exact merge) within 2e-2 max-abs on O and 1e-3 on LSE."""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
import oracle
from _parity import compare, pool_bytes, q_bits

pytestmark = pytest.mark.gpu

CASES = [
    # name, lens, H, T, N, dtype
    ("ragged", [1000, 130, 64 * 9 + 5], 64, 1, 4, "bf16"),
    ("causal-q4", [64 * 7 + 3, 66, 260], 64, 4, 2, "bf16"),
    ("heads-96", [700, 333], 96, 1, 3, "bf16"),
    ("dcp1", [1500], 64, 1, 1, "bf16"),
    ("ragged-fp8", [1000, 130, 64 * 9 + 5], 64, 1, 4, "e4m3"),
    ("long-mixed-fp8", [40_000, 3_000], 64, 1, 8, "e4m3"),
]


def _oracle(case, rank=-1, rows=None):
    return oracle.attention(q_bits(case), case.seq_lens.cpu().numpy(), case.req_page_ptr.cpu().numpy(),
                            case.dst_vpages.cpu().numpy(), pool_bytes(case),
                            oracle.BF16 if case.dtype == "bf16" else oracle.E4M3, case.kv_scale, case.softmax_scale,
                            case.n_dcp, rank=rank, rows=rows, q_len=case.T, num_heads=case.H, layout="token")


@pytest.mark.parametrize("name,lens,H,T,N,dtype", CASES, ids=[c[0] for c in CASES])
def test_token_layout_attention_matches_oracle(cuda_device, name, lens, H, T, N, dtype):
    case = di.token_attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, seed=11 + len(name), device=cuda_device,
                                   name=name)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o, l = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                   case.softmax_scale, case.kv_scale, dev_error=err, layout="token")
    om, lm = dcp.lse_merge(o, l)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = case.rows
    rows = None if sum(lens) < 20_000 else np.arange(0, R, 3)
    o, l, om, lm = (x.cpu().numpy() for x in (o, l, om, lm))
    for d in range(N) if N <= 4 else (0, N - 1):
        ro, rl = _oracle(case, rank=d, rows=rows)
        og, lg = o[d].reshape(R, 512), l[d].reshape(R)
        if rows is not None:
            og, lg = og[rows], lg[rows]
        compare(og, lg, ro, rl, f"{name} rank {d}")
    ro, rl = _oracle(case, rows=rows)
    og, lg = om.reshape(R, 512), lm.reshape(R)
    if rows is not None:
        og, lg = og[rows], lg[rows]
    compare(og, lg, ro, rl, f"{name} merged")


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_token_reshard_matches_oracle_bit_exact(cuda_device, dtype):
    lens, n_layers, counts, N = [64 * 12 + 7, 300, 65], 3, [2, 1], 3
    rc = di.reshard_case(lens, n_layers=n_layers, layer_counts=counts, n_dcp=N, dtype=dtype, contiguous_src=False,
                         seed=41, device=cuda_device)
    slots = sum(-(-(-(-n // N)) // 64) for n in lens) + 2
    tptr, tv = di.token_page_table(lens, N, slots, torch.Generator().manual_seed(5))
    dst = [torch.empty((n_layers, slots, 64, 576), dtype=rc.src_pools[0].dtype, device=cuda_device)
           for _ in range(N)]
    for t in dst:
        t.view(torch.uint8).fill_(di.SENTINEL_BYTE)
    seq = torch.tensor(lens, dtype=torch.int32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dcp.token_reshard(seq, rc.req_page_ptr, rc.src_pages, tptr.to(cuda_device), tv.to(cuda_device), n_layers,
                      rc.src_pools, rc.src_pool_pages, dst, slots, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = [np.full(t.numel() * t.element_size(), di.SENTINEL_BYTE, np.uint8) for t in dst]
    row_bytes = 576 * (2 if dtype == "bf16" else 1)
    assert oracle.token_reshard(lens, rc.req_page_ptr.cpu().numpy(), rc.src_pages.cpu().numpy(), tptr.numpy(),
                                tv.numpy(), row_bytes, n_layers,
                                [p.cpu().view(torch.uint8).numpy().reshape(-1) for p in rc.src_pools],
                                rc.src_pool_pages, N, ref, slots) == 0
    for a, b in zip(dst, ref):
        assert np.array_equal(a.cpu().view(torch.uint8).numpy().reshape(-1), b)


@pytest.mark.parametrize("name,lens,H,T,N,dtype", [CASES[0], CASES[1], CASES[4]], ids=["ragged", "causal-q4", "ragged-fp8"])
def test_token_layout_fused_call_matches_oracle(cuda_device, name, lens, H, T, N, dtype):
    """dcp_decode_attn_merged_tokens: every rank's partial over the token-interleaved table and
    the merge in one call."""
    case = di.token_attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, seed=11 + len(name), device=cuda_device,
                                   name=name)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    om, lm, o, l = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                          case.softmax_scale, case.kv_scale, dev_error=err, layout="token")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = case.rows
    for d in range(N):
        ro, rl = _oracle(case, rank=d)
        compare(o[d].cpu().numpy().reshape(R, 512), l[d].cpu().numpy().reshape(R), ro, rl, f"{name} fused rank {d}")
    ro, rl = _oracle(case)
    compare(om.cpu().numpy().reshape(R, 512), lm.cpu().numpy().reshape(R), ro, rl, f"{name} fused merged")
