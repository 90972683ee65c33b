"""GPU parity of the reshard's other modes, bit for bit: the bounded pack mode
(dcp_pack_pages / dcp_unpack_pages) and the naive full-transfer + in-place-shard baseline.

For every path (source rank r, destination rank d) of a multi-layer CP2 -> DCP4 reshard, the
path's filtered page list comes from dcp_filter_page_indices on the GPU; packing its items chunk
by chunk through a bounded staging buffer and unpacking each chunk must give the staging bytes
of the float64 oracle's pack, chunk for chunk, and the destination pool of the oracle's reshard
of that path (and of the GPU reshard of that path).  Item ranges come from pack_chunks.
"""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
import oracle

pytestmark = pytest.mark.gpu


def _u8(t):
    return t.cpu().view(torch.uint8).numpy().reshape(-1)


def _sentinel_like(t):
    return torch.empty_like(t).view(torch.uint8).fill_(di.SENTINEL_BYTE).view(t.dtype)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("cap_pages", [5, 64, 100000])
def test_pack_unpack_matches_oracle_and_reshard(cuda_device, dtype, cap_pages):
    lens = [64 * 40 + 3, 900, 64 * 9]
    counts = [2, 1]  # 3 layers over 2 CP ranks
    case = di.reshard_case(lens, n_layers=3, layer_counts=counts, n_dcp=4, dtype=dtype, contiguous_src=False,
                           seed=17, device=cuda_device)
    pb = case.page_bytes
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    starts = [0, counts[0]]
    src_u8 = [_u8(p) for p in case.src_pools]
    for r in range(2):
        for d in range(4):
            slot, src, cnt = dcp.filter_page_indices(case.dst_vpages, 4, d, case.src_pages)
            n_idx = int(cnt.item())
            n_items = counts[r] * n_idx
            staging = torch.empty(cap_pages * pb, dtype=torch.uint8, device=cuda_device)
            got = _sentinel_like(case.dst_pools[d])
            ref_pool = np.full(got.numel() * got.element_size(), di.SENTINEL_BYTE, np.uint8)
            src_idx_h, slot_h = src[:n_idx].cpu().numpy(), slot[:n_idx].cpu().numpy()
            for begin, n in dcp.pack_chunks(n_items, pb, staging.numel()):
                dcp.pack_pages(src, n_idx, counts[r], begin, n, case.src_pools[r], staging, dev_error=err)
                ref = np.zeros(n * pb, np.uint8)
                assert oracle.pack(src_idx_h, counts[r], begin, n, pb, src_u8[r], case.src_pool_pages, ref) == 0
                assert np.array_equal(_u8(staging)[:n * pb], ref)
                dcp.unpack_pages(slot, n_idx, counts[r], starts[r], begin, n, staging, got, dev_error=err)
                assert oracle.unpack(slot_h, counts[r], starts[r], begin, n, pb, ref, ref_pool, 3,
                                     case.dst_slots) == 0
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert np.array_equal(_u8(got), ref_pool)
            # the GPU reshard of the same path into a fresh sentinel pool
            fresh = [_sentinel_like(p) for p in case.dst_pools]
            dcp.reshard_pages(case.req_page_ptr, case.src_pages, case.dst_vpages, 3, case.src_pools,
                              case.src_pool_pages, fresh, case.dst_slots, only_src_rank=r, only_dst_rank=d,
                              dev_error=err)
            torch.cuda.synchronize()
            assert torch.equal(fresh[d].view(torch.uint8), got.view(torch.uint8))


def test_pack_out_of_range_sets_device_error(cuda_device):
    case = di.reshard_case([64 * 8], n_layers=1, layer_counts=[1], n_dcp=1, dtype="bf16", contiguous_src=True,
                           seed=2, device=cuda_device)
    idx = torch.tensor([0, case.src_pool_pages + 5, 1], dtype=torch.int32, device=cuda_device)
    staging = torch.full((3 * case.page_bytes,), 7, dtype=torch.uint8, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dcp.pack_pages(idx, 3, 1, 0, 3, case.src_pools[0], staging, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dcp.DEVERR_OUT_OF_RANGE
    pb = case.page_bytes
    s = _u8(staging)
    src = _u8(case.src_pools[0]).reshape(-1, pb)
    assert np.array_equal(s[:pb], src[0]) and np.array_equal(s[2 * pb:], src[1])
    assert (s[pb:2 * pb] == 7).all()


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_naive_transfer_and_inplace_shard_match_oracle_and_reshard(cuda_device, dtype):
    """The 6.1 baseline: the receive buffers equal the oracle's full transfer bit for bit, and
    the in-place shard leaves the DCP pools exactly as the 2D reshard does."""
    lens = [64 * 30 + 5, 700, 64 * 3]
    counts = [2, 2]  # 4 layers over 2 CP ranks
    case = di.reshard_case(lens, n_layers=4, layer_counts=counts, n_dcp=4, dtype=dtype, contiguous_src=False,
                           seed=31, device=cuda_device)
    pb = case.page_bytes
    n_pages = case.dst_vpages.numel()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    recv = [torch.empty((4, n_pages, 64, 576), dtype=case.src_pools[0].dtype, device=cuda_device) for _ in range(4)]
    dcp.naive_full_transfer(case.src_pages, 4, case.src_pools, case.src_pool_pages, recv, dev_error=err)
    got = [_sentinel_like(p) for p in case.dst_pools]
    dcp.naive_inplace_shard(case.dst_vpages, 4, recv, got, case.dst_slots, dev_error=err)
    ref = [_sentinel_like(p) for p in case.dst_pools]
    dcp.reshard_pages(case.req_page_ptr, case.src_pages, case.dst_vpages, 4, case.src_pools, case.src_pool_pages,
                      ref, case.dst_slots, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_recv = [np.zeros(4 * n_pages * pb, np.uint8) for _ in range(4)]
    assert oracle.full_transfer(case.src_pages.cpu().numpy(), pb, 4, [_u8(p) for p in case.src_pools],
                                case.src_pool_pages, 4, ref_recv) == 0
    for a, b in zip(recv, ref_recv):
        assert np.array_equal(_u8(a), b)
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
