"""Full-size parity of the workloads the benchmark times.

* Reshard, bit-exact, every page of every layer: the batch workload (32 x 8192, BF16, one layer),
  the agent workload (48 x 100,000, FP8, one layer) and the end-to-end workload (64 requests of
  2K-500K tokens, 8 layers, CP4 layer split -> DCP8, FP8).  The last two are long copies (several
  GB), which the copy kernel runs on one CTA per pair of SMs ("Serving Macaron-V1 at Scale", 2:
  every path (r, d) moves L_r x P_d; 6.3: transfer with source-side filtering; 6.4: the physical
  page is the copy unit).
* The end-to-end workload's attention: one plan for the page table, then the fused attention +
  merge on each of the 8 layers, sampled rows of the shortest, the longest and two middle
  requests against the oracle on every rank's partials and on the merged output.

The oracle runs request by request on a relabelled sub-problem: the request's source pages
numbered from 0 and, per destination rank, its pages at consecutive local slots (the page table
of the sub-problem keeps each page's owner); the GPU's pages are gathered from the slots the
generator chose.  Slots no request names must keep the sentinel byte.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
import oracle
from _parity import compare

pytestmark = pytest.mark.gpu


def half_grid_threshold(device) -> int:
    """Bytes moved (read + write) from which the copy kernels run one CTA per pair of SMs."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return max(sms // 2, 1) * (16 << 20)


def run_reshard(rc):
    err = torch.zeros(1, dtype=torch.int32, device=rc.src_pools[0].device)
    dcp.reshard_pages(rc.req_page_ptr, rc.src_pages, rc.dst_vpages, rc.n_layers, rc.src_pools, rc.src_pool_pages,
                      rc.dst_pools, rc.dst_slots, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def check_reshard_by_request(rc):
    """Every request's pages of every layer against the oracle; untouched slots keep the sentinel."""
    ptr = rc.req_page_ptr.cpu().numpy()
    src_pages = rc.src_pages.cpu()
    owner, slot = rc.page_owner, rc.page_slot
    N = max(rc.n_dcp, 1)
    pb = rc.page_bytes
    checked = 0
    for b in range(len(rc.seq_lens)):
        p0, p1 = int(ptr[b]), int(ptr[b + 1])
        n = p1 - p0
        if n == 0:
            continue
        # sub-problem: source pages 0..n-1; rank d's pages of the request at local slots 0, 1, ...
        own = owner[p0:p1]
        local = torch.empty(n, dtype=torch.int64)
        k = [0] * N
        for d in range(N):
            sel = own == d
            k[d] = int(sel.sum())
            local[sel] = torch.arange(k[d])
        vsub = (local * N + own if rc.n_dcp > 1 else local).to(torch.int32).numpy()
        idx = src_pages[p0:p1].to(torch.int64).to(rc.src_pools[0].device)
        src = [np.ascontiguousarray(p.index_select(1, idx).cpu().view(torch.uint8).numpy().reshape(-1))
               for p in rc.src_pools]
        kmax = max(max(k), 1)
        ref = [np.full(rc.n_layers * kmax * pb, di.SENTINEL_BYTE, np.uint8) for _ in range(N)]
        st = oracle.reshard(np.array([0, n], np.int64), np.arange(n, dtype=np.int32), vsub, pb, rc.n_layers, src, n,
                            rc.n_dcp, ref, kmax)
        assert st == 0
        for d in range(N):
            if k[d] == 0:
                continue
            sl = slot[p0:p1][own == d].to(rc.dst_pools[d].device)
            gpu = rc.dst_pools[d].index_select(1, sl).cpu().view(torch.uint8).numpy().reshape(rc.n_layers, k[d], pb)
            want = ref[d].reshape(rc.n_layers, kmax, pb)[:, :k[d]]
            if not np.array_equal(gpu, want):
                bad = np.argwhere((gpu != want).any(axis=2))[0]
                raise AssertionError(f"{rc.name}: request {b}, rank {d}, layer {bad[0]}, page {bad[1]} differs")
            checked += rc.n_layers * k[d]
        del src, ref
    for d in range(N):
        used = torch.zeros(rc.dst_slots, dtype=torch.bool)
        used[slot[owner == d]] = True
        free = torch.nonzero(~used).flatten().to(rc.dst_pools[d].device)
        if free.numel():
            rest = rc.dst_pools[d].index_select(1, free).view(torch.uint8)
            assert bool((rest == di.SENTINEL_BYTE).all()), f"{rc.name}: a slot no request names was written"
    return checked


def test_batch_reshard_full_size_bit_exact(cuda_device):
    rc = di.reshard_case([8192] * 32, n_layers=1, layer_counts=[1], n_dcp=8, dtype="bf16", contiguous_src=True,
                         seed=1, device=cuda_device, dst_slots=512, name="batch-32x8192-bf16-dcp8")
    run_reshard(rc)
    assert check_reshard_by_request(rc) == rc.dst_vpages.numel()


def test_agent_reshard_full_size_bit_exact(cuda_device):
    rc = di.reshard_case([100_000] * 48, n_layers=1, layer_counts=[1], n_dcp=8, dtype="e4m3", contiguous_src=True,
                         seed=1, device=cuda_device, dst_slots=9408, name="agent-48x100000-fp8-dcp8")
    moved = 2 * rc.dst_vpages.numel() * rc.page_bytes
    assert moved >= half_grid_threshold(cuda_device)  # the long-copy grid (one CTA per SM pair)
    run_reshard(rc)
    assert check_reshard_by_request(rc) == rc.dst_vpages.numel()


@pytest.fixture(scope="module")
def e2e(cuda_device):
    counts = di.e2e_layer_counts(oracle.layer_range)
    assert counts == [2, 2, 2, 2]
    rc = di.e2e_reshard_case(cuda_device, counts)
    run_reshard(rc)
    yield rc
    del rc
    torch.cuda.empty_cache()


def test_e2e_reshard_full_size_bit_exact(cuda_device, e2e):
    rc = e2e
    moved = 2 * rc.n_layers * rc.dst_vpages.numel() * rc.page_bytes
    assert moved >= half_grid_threshold(cuda_device)
    assert len(rc.seq_lens) == 64 and min(rc.seq_lens) >= 2048 and max(rc.seq_lens) <= 500_032
    assert check_reshard_by_request(rc) == rc.n_layers * rc.dst_vpages.numel()


def test_e2e_attention_every_layer_sampled(cuda_device, e2e):
    rc = e2e
    B, T, H, N, L = len(rc.seq_lens), 1, 64, 8, rc.n_layers
    q = di.random_q(B, T, H, di._gen(8, cuda_device), cuda_device)
    seq = torch.tensor(rc.seq_lens, dtype=torch.int32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ws = dcp.alloc_workspace(B, T, H, N, rc.dst_vpages.numel(), cuda_device)
    layer_pools = [[p[l] for p in rc.dst_pools] for l in range(L)]
    dcp.attn_plan((B, T, H), rc.req_page_ptr, rc.dst_vpages, layer_pools[0], ws, dev_error=err)
    o_part = torch.empty((L, N, B, T, H, 512), dtype=torch.float32, device=cuda_device)
    lse_part = torch.empty((L, N, B, T, H), dtype=torch.float32, device=cuda_device)
    o = torch.empty((L, B, T, H, 512), dtype=torch.float32, device=cuda_device)
    lse = torch.empty((L, B, T, H), dtype=torch.float32, device=cuda_device)
    for l in range(L):
        dcp.decode_attn_merged(q, seq, rc.req_page_ptr, rc.dst_vpages, layer_pools[l], di.SOFTMAX_SCALE,
                               di.FP8_KV_SCALE, o_part=o_part[l], lse_part=lse_part[l], o_out=o[l], lse_out=lse[l],
                               workspace=ws, dev_error=err, planned=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    order = np.argsort(np.array(rc.seq_lens), kind="stable")
    picks = [int(order[0]), int(order[len(order) // 3]), int(order[2 * len(order) // 3]), int(order[-1])]
    heads = np.arange(0, H, 9)
    rows = np.sort(np.concatenate([b * H + heads for b in picks])).astype(np.int64)
    qb = q.cpu().view(torch.int16).numpy().view(np.uint16)
    sl, ptr, vp = seq.cpu().numpy(), rc.req_page_ptr.cpu().numpy(), rc.dst_vpages.cpu().numpy()
    for l in range(L):
        pools = [p.cpu().view(torch.uint8).numpy() for p in layer_pools[l]]
        op = o_part[l].reshape(N, -1, 512).cpu().numpy()
        lp = lse_part[l].reshape(N, -1).cpu().numpy()
        for d in range(N):
            ro, rlse = oracle.attention(qb, sl, ptr, vp, pools, oracle.E4M3, di.FP8_KV_SCALE, di.SOFTMAX_SCALE, N,
                                        rank=d, rows=rows, q_len=T, num_heads=H)
            compare(op[d][rows], lp[d][rows], ro, rlse, f"e2e layer {l} rank {d}")
        ro, rlse = oracle.attention(qb, sl, ptr, vp, pools, oracle.E4M3, di.FP8_KV_SCALE, di.SOFTMAX_SCALE, N,
                                    rows=rows, q_len=T, num_heads=H)
        compare(o[l].reshape(-1, 512).cpu().numpy()[rows], lse[l].reshape(-1).cpu().numpy()[rows], ro, rlse,
                f"e2e layer {l} merged")
        del pools
