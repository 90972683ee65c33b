"""Pools larger than 4 GiB per rank: pages at the highest slots, past every 32-bit byte offset.

The reshard writes a request's pages into the last slots of two destination pools of more than
4.4 GB each; the attention (fused with the merge) then reads them there.  The oracle sees the
same pages through compact copies (only the used slots, renumbered), which leaves the attention
unchanged because it depends only on each request's pages in order.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
import oracle

PAGE = 64


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,slots", [("bf16", 60_000), ("e4m3", 120_000)])
def test_reshard_and_attention_past_4gib(cuda_device, dtype, slots):
    N, n_tok, H = 2, 2000, 16
    n_pages = (n_tok + PAGE - 1) // PAGE
    page_bytes = PAGE * 576 * (2 if dtype == "bf16" else 1)
    assert slots * page_bytes > (1 << 32)
    g = di._gen(5, cuda_device)
    # source: one CP rank, one layer, the request's pages in a small pool
    src_pool = di.random_pool(n_pages, dtype, g, cuda_device, layers=1)
    src_pages = torch.arange(n_pages, dtype=torch.int32)
    # destination: page j -> owner j mod N at one of the top slots of its rank
    slot = np.array([slots - 1 - 3 * (j // N) for j in range(n_pages)], np.int64)
    owner = np.arange(n_pages) % N
    vpages = torch.tensor(slot * N + owner, dtype=torch.int32)
    ptr = torch.tensor([0, n_pages], dtype=torch.int64)
    dst = [torch.empty((1, slots, PAGE, 576), dtype=src_pool.dtype, device=cuda_device) for _ in range(N)]
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dcp.reshard_pages(ptr.to(cuda_device), src_pages.to(cuda_device), vpages.to(cuda_device), 1, [src_pool], n_pages,
                      dst, slots, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for j in range(n_pages):  # bit-exact at the far end of the pools
        a = dst[owner[j]][0, slot[j]].view(torch.uint8)
        b = src_pool[0, j].view(torch.uint8)
        assert torch.equal(a, b), f"page {j}"

    q = di.random_q(1, 1, H, g, cuda_device)
    seq = torch.tensor([n_tok], dtype=torch.int32, device=cuda_device)
    kv_scale = di.FP8_KV_SCALE if dtype == "e4m3" else 1.0
    o, lse, o_part, lse_part = dcp.decode_attn_merged(q, seq, ptr.to(cuda_device), vpages.to(cuda_device),
                                                      [d[0] for d in dst], di.SOFTMAX_SCALE, kv_scale,
                                                      dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # oracle on compact pools: rank d's used slots renumbered 0, 1, ... in page order
    compact_slot = np.zeros(n_pages, np.int64)
    pools = []
    for d in range(N):
        js = [j for j in range(n_pages) if owner[j] == d]
        for k, j in enumerate(js):
            compact_slot[j] = k
        rows = torch.stack([src_pool[0, j] for j in js]).cpu()
        pools.append(rows.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16"
                     else rows.view(torch.uint8).numpy())
    vp_c = (compact_slot * N + owner).astype(np.int32)
    qb = q.cpu().view(torch.int16).numpy().view(np.uint16)
    dt = oracle.BF16 if dtype == "bf16" else oracle.E4M3
    ro, rl = oracle.attention(qb, np.array([n_tok], np.int32), ptr.numpy(), vp_c, pools, dt, kv_scale,
                              di.SOFTMAX_SCALE, N, q_len=1, num_heads=H)
    assert np.abs(o.cpu().numpy().reshape(H, 512) - ro).max() <= 2e-2
    assert np.abs(lse.cpu().numpy().reshape(H) - rl).max() <= 1e-3
    for d in range(N):
        rpo, rpl = oracle.attention(qb, np.array([n_tok], np.int32), ptr.numpy(), vp_c, pools, dt, kv_scale,
                                    di.SOFTMAX_SCALE, N, rank=d, q_len=1, num_heads=H)
        assert np.abs(o_part[d].cpu().numpy().reshape(H, 512) - rpo).max() <= 2e-2
        assert np.abs(lse_part[d].cpu().numpy().reshape(H) - rpl).max() <= 1e-3
