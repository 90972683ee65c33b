"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Reshard and index filtering must match bit for bit; attention and merge outputs within
2e-2 max-abs on O and 1e-3 on LSE.  Sizes span several 128-token tiles and ragged tails;
the full-size workloads are checked on sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
import oracle
from _parity import compare, oracle_attention, pool_bytes, q_bits

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------------------- merge
@pytest.mark.parametrize("n,rows", [(1, 7), (4, 300), (8, 1024), (3, 1)])
def test_lse_merge_matches_oracle(cuda_device, n, rows):
    g = torch.Generator().manual_seed(n * 1000 + rows)
    o = torch.randn((n, rows, 512), generator=g, dtype=torch.float32)
    lse = 4 * torch.randn((n, rows), generator=g, dtype=torch.float32)
    if n > 1:
        lse[0, ::5] = -float("inf")           # empty shards
    lse[:, rows // 2] = -float("inf")         # an all-empty row
    o_gpu, l_gpu = dcp.lse_merge(o.to(cuda_device), lse.to(cuda_device))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.lse_merge(o.double().numpy(), lse.double().numpy())
    compare(o_gpu.cpu().numpy(), l_gpu.cpu().numpy(), o_ref, l_ref, "merge", o_tol=1e-5, lse_tol=1e-5)


# ---------------------------------------------------------------------------- filter
@pytest.mark.parametrize("n_dcp,n", [(1, 100), (4, 256), (8, 20000), (3, 1), (8, 0)])
def test_filter_matches_oracle_bit_exact(cuda_device, n_dcp, n):
    g = torch.Generator().manual_seed(n + n_dcp)
    vals = torch.randperm(max(4 * n, 1), generator=g)[:n].to(torch.int32)
    src = torch.randperm(max(4 * n, 1), generator=g)[:n].to(torch.int32)
    for d in range(n_dcp):
        slot, s, cnt = dcp.filter_page_indices(vals.to(cuda_device), n_dcp, d, src.to(cuda_device))
        torch.cuda.synchronize()
        k = int(cnt.item())
        ref_src, ref_dst = oracle.transfer_filter(src.numpy(), vals.numpy(), n_dcp, d)
        assert k == ref_dst.size
        assert np.array_equal(slot[:k].cpu().numpy(), ref_dst)
        assert np.array_equal(s[:k].cpu().numpy(), ref_src)


def test_filter_256_pages_to_64(cuda_device):
    """The 6.3 log line: 256 pages -> 64 per rank at DCP=4."""
    vals = torch.arange(256, dtype=torch.int32, device=cuda_device)
    for d in range(4):
        _, _, cnt = dcp.filter_page_indices(vals, 4, d)
        assert int(cnt.item()) == 64


# --------------------------------------------------------------------------- reshard
def _reshard_both(case, only_src=-1, only_dst=-1, expect_status=0):
    err = torch.zeros(1, dtype=torch.int32, device=case.src_pools[0].device)
    before = [p.cpu().view(torch.uint8).numpy().reshape(-1).copy() for p in case.dst_pools]
    dcp.reshard_pages(case.req_page_ptr, case.src_pages, case.dst_vpages, case.n_layers, case.src_pools,
                      case.src_pool_pages, case.dst_pools, case.dst_slots, n_dcp=case.n_dcp,
                      only_src_rank=only_src, only_dst_rank=only_dst, dev_error=err)
    torch.cuda.synchronize()
    gpu = [p.cpu().view(torch.uint8).numpy().reshape(-1) for p in case.dst_pools]
    src = [p.cpu().view(torch.uint8).numpy().reshape(-1).copy() for p in case.src_pools]
    ref = before
    st = oracle.reshard(case.req_page_ptr.cpu().numpy(), case.src_pages.cpu().numpy(),
                        case.dst_vpages.cpu().numpy(), case.page_bytes, case.n_layers, src,
                        case.src_pool_pages, case.n_dcp, ref, case.dst_slots, only_src, only_dst)
    assert st == expect_status
    return gpu, ref, int(err.item())


def _counts(n_layers, n_cp):
    return [e - s for s, e in (oracle.layer_range(n_layers, n_cp, r) for r in range(n_cp))]


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("lens,n_layers,n_cp,n_dcp,contig", [
    ([1024], 1, 1, 4, False),                      # tiny: 16 pages, 1 source shard, DCP=4
    ([3000, 64, 700, 129, 5000], 8, 4, 8, True),   # CP4 layer-split -> DCP8, ragged lengths
    ([640, 200], 5, 3, 3, False),                  # uneven layer split, odd N
    ([300], 2, 2, 1, True),                        # DCP=1: identity filter
])
def test_reshard_bit_exact(cuda_device, dtype, lens, n_layers, n_cp, n_dcp, contig):
    case = di.reshard_case(lens, n_layers, _counts(n_layers, n_cp), n_dcp, dtype, contig, seed=len(lens),
                           device=cuda_device, dst_slots=None)
    gpu, ref, err = _reshard_both(case)
    assert err == 0
    for a, b in zip(gpu, ref):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("ctas", [1, 7, 76, 151, 1000])
def test_reshard_on_forced_grids_bit_exact(cuda_device, monkeypatch, ctas):
    """The copy kernel's CTA count forced (DCP_RING_CTAS): one CTA, odd counts, the half grid
    used for long copies, and more CTAs than chunks; the chunk ranges must still tile the work."""
    monkeypatch.setenv("DCP_RING_CTAS", str(ctas))
    case = di.reshard_case([3000, 64, 700, 129, 5000], 8, _counts(8, 4), 8, "e4m3", True, seed=ctas,
                           device=cuda_device)
    gpu, ref, err = _reshard_both(case)
    assert err == 0
    for a, b in zip(gpu, ref):
        assert np.array_equal(a, b)


def test_reshard_single_paths_compose(cuda_device):
    case = di.reshard_case([2000, 900], 6, _counts(6, 3), 4, "e4m3", True, seed=5, device=cuda_device)
    for r in range(3):
        for d in range(4):
            gpu, ref, err = _reshard_both(case, only_src=r, only_dst=d)
            assert err == 0
            for a, b in zip(gpu, ref):
                assert np.array_equal(a, b)
    full = [p.clone() for p in case.dst_pools]
    fresh = di.reshard_case([2000, 900], 6, _counts(6, 3), 4, "e4m3", True, seed=5, device=cuda_device)
    _reshard_both(fresh)
    for a, b in zip(full, fresh.dst_pools):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_reshard_out_of_range_sets_device_error(cuda_device):
    case = di.reshard_case([256], 1, [1], 4, "bf16", True, seed=3, device=cuda_device)
    case.dst_vpages[1] = case.dst_slots * 4 + 1   # slot past the pool
    gpu, ref, err = _reshard_both(case, expect_status=-2)
    assert err & dcp.DEVERR_OUT_OF_RANGE
    for a, b in zip(gpu, ref):
        assert np.array_equal(a, b)


# ------------------------------------------------------------------------- attention
def _run_attention(case):
    err = torch.zeros(1, dtype=torch.int32, device=case.q.device)
    o, l = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                   case.softmax_scale, case.kv_scale, dev_error=err)
    om, lm = dcp.lse_merge(o, l)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o.cpu().numpy(), l.cpu().numpy(), om.cpu().numpy(), lm.cpu().numpy()


def _check_all(case, o, l, om, lm):
    qb, pools = q_bits(case), pool_bytes(case)
    R = case.rows
    for d in range(case.n_dcp):
        ro, rl = oracle_attention(case, rank=d, qb=qb, pools=pools)
        compare(o[d].reshape(R, 512), l[d].reshape(R), ro, rl, f"{case.name} rank {d}")
    ro, rl = oracle_attention(case, qb=qb, pools=pools)
    return compare(om.reshape(R, 512), lm.reshape(R), ro, rl, f"{case.name} merged")


ATTN_CASES = [
    # name, lens, H, T, N, dtype
    ("tiny", [1024], 16, 1, 4, "bf16"),
    ("ragged", [1000, 130, 64 * 9 + 5], 64, 1, 4, "bf16"),
    ("empty-ranks", [64, 200, 1], 64, 1, 8, "bf16"),
    ("causal-q4", [64 * 7 + 3, 66, 260], 64, 4, 2, "bf16"),
    ("heads-96", [700, 333], 96, 1, 3, "bf16"),
    ("dcp1", [1500], 64, 1, 1, "bf16"),
    ("tiny-fp8", [1024], 16, 1, 4, "e4m3"),
    ("ragged-fp8", [1000, 130, 64 * 9 + 5], 64, 1, 4, "e4m3"),
    ("empty-ranks-fp8", [64, 200, 1], 64, 1, 8, "e4m3"),
    ("causal-q4-fp8", [64 * 7 + 3, 66, 260], 64, 4, 2, "e4m3"),
    ("heads-96-fp8", [700, 333], 96, 1, 3, "e4m3"),
    # long segments per rank (chunked) next to short ones
    ("mixed-len-fp8", [70_000, 9_000], 64, 1, 8, "e4m3"),
    # the largest DCP size, 32 heads (half a query group), 128 heads (two groups) with q_len 2
    ("dcp16", [5000, 700, 1], 64, 1, 16, "bf16"),
    ("dcp16-fp8", [5000, 70], 64, 1, 16, "e4m3"),
    ("heads-32", [900, 64], 32, 1, 4, "bf16"),
    ("heads-128-q2-fp8", [1200, 300], 128, 2, 4, "e4m3"),
]


@pytest.mark.parametrize("name,lens,H,T,N,dtype", ATTN_CASES, ids=[c[0] for c in ATTN_CASES])
def test_attention_matches_oracle(cuda_device, name, lens, H, T, N, dtype):
    case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=len(name),
                             device=cuda_device, name=name)
    _check_all(case, *_run_attention(case))


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_attention_multi_chunk_combine(cuda_device, dtype):
    """A long single request splits into many chunks per rank (in-call chunk merge)."""
    case = di.attention_case([64 * 1024 + 17], H=64, T=1, n_dcp=2, dtype=dtype, slots_per_rank=None,
                             seed=21, device=cuda_device, name="long-chunked")
    o, l, om, lm = _run_attention(case)
    rows = np.arange(0, 64, 7)
    qb, pools = q_bits(case), pool_bytes(case)
    for d in range(2):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(64, 512)[rows], l[d].reshape(64)[rows], ro, rl, f"chunked rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(64, 512)[rows], lm.reshape(64)[rows], ro, rl, "chunked merged")


def test_attention_batch_full_size_sampled(cuda_device):
    """32 x 8192 tokens, 64 heads, BF16, DCP=8 at full size; sampled rows vs the oracle."""
    case = di.batch_case(cuda_device)
    o, l, om, lm = _run_attention(case)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(case.rows, 48, replace=False))
    qb, pools = q_bits(case), pool_bytes(case)
    for d in (0, 5):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(-1, 512)[rows], l[d].reshape(-1)[rows], ro, rl, f"batch rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(-1, 512)[rows], lm.reshape(-1)[rows], ro, rl, "batch merged")


def _sampled(case, o, l, om, lm, n_rows, ranks, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(case.rows, n_rows, replace=False))
    qb, pools = q_bits(case), pool_bytes(case)
    for d in ranks:
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(-1, 512)[rows], l[d].reshape(-1)[rows], ro, rl, f"{case.name} rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(-1, 512)[rows], lm.reshape(-1)[rows], ro, rl, f"{case.name} merged")


def test_attention_agent_full_size_sampled(cuda_device):
    """48 x 100,000 tokens, 64 heads, FP8-E4M3, DCP=8 over a ~2.8 GB pool; 64 sampled rows on
    every rank's partials and the merged output."""
    case = di.agent_case(cuda_device)
    _sampled(case, *_run_attention(case), n_rows=64, ranks=range(8))


def test_attention_agent_dcp1_check(cuda_device):
    """The 1/8 check of the agent workload: 6 requests run at DCP=1 over one pool holding all
    their pages equal their DCP=8 partials merged."""
    case = di.agent_case(cuda_device)
    sub = di.AttnCase(B=6, T=1, H=64, n_dcp=8, dtype="e4m3", seq_lens=case.seq_lens[:6],
                      req_page_ptr=case.req_page_ptr[:7].clone(),
                      dst_vpages=case.dst_vpages[:int(case.req_page_ptr[6])].clone(), q=case.q[:6].contiguous(),
                      pools=case.pools, slots_per_rank=case.slots_per_rank, kv_scale=case.kv_scale, name="agent-6")
    o8, l8, om, lm = _run_attention(sub)
    one = torch.cat(sub.pools, 0)
    vp = (sub.dst_vpages % 8) * sub.slots_per_rank + sub.dst_vpages // 8
    single = di.AttnCase(B=6, T=1, H=64, n_dcp=1, dtype="e4m3", seq_lens=sub.seq_lens, req_page_ptr=sub.req_page_ptr,
                         dst_vpages=vp.to(torch.int32), q=sub.q, pools=[one], slots_per_rank=8 * sub.slots_per_rank,
                         kv_scale=sub.kv_scale, name="agent-6-dcp1")
    o1, l1, _, _ = _run_attention(single)
    compare(om.reshape(-1, 512), lm.reshape(-1), o1[0].reshape(-1, 512).astype(np.float64),
            l1[0].reshape(-1).astype(np.float64), "DCP=1 vs DCP=8 merged")
    # and the DCP=1 run itself against the oracle (unsharded attention over the one pool)
    rows = np.sort(np.random.default_rng(1).choice(single.rows, 48, replace=False))
    ro, rl = oracle_attention(single, rows=rows)
    compare(o1[0].reshape(-1, 512)[rows], l1[0].reshape(-1)[rows], ro, rl, "agent 6 requests at DCP=1")


def test_attention_long_eagle_full_size_sampled(cuda_device):
    """4 x 1,048,576 tokens, q_len 4 causal, FP8, DCP=8: for every request and every one of the
    4 new tokens, 4 heads, on every rank's partials and the merged output."""
    case = di.long_eagle_case(cuda_device)
    o, l, om, lm = _run_attention(case)
    rows = np.array([(b * case.T + t) * case.H + h for b in range(case.B) for t in range(case.T)
                     for h in (0, 21, 42, 63)], np.int64)
    qb, pools = q_bits(case), pool_bytes(case)
    for d in range(case.n_dcp):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(-1, 512)[rows], l[d].reshape(-1)[rows], ro, rl, f"long rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(-1, 512)[rows], lm.reshape(-1)[rows], ro, rl, "long merged")


def test_attention_and_merge_with_no_requests(cuda_device):
    """An empty batch is a no-op (no launch, no error)."""
    case = di.attention_case([64], H=64, T=1, n_dcp=2, dtype="bf16", slots_per_rank=None, seed=1,
                             device=cuda_device)
    q = case.q[:0]
    seq = case.seq_lens[:0]
    ptr = case.req_page_ptr[:1]
    o, l = dcp.partial_decode_attn(q, seq, ptr, case.dst_vpages[:0], case.pools, case.softmax_scale)
    om, lm, _, _ = dcp.decode_attn_merged(q, seq, ptr, case.dst_vpages[:0], case.pools, case.softmax_scale)
    torch.cuda.synchronize()
    assert o.numel() == 0 and om.numel() == 0 and lm.numel() == 0
