"""Pins for the float64 oracle (CPU only).

Each test ties an oracle function to something other than itself: a worked example printed
on the pages (tests/golden/), a closed form, an invariant the pages state, a special case
that reduces to a library routine (torch dtype casts, scipy softmax / logsumexp), or brute
force on tiny inputs.  Together they are chosen so that a dropped term, a wrong sign or
index, a transposed operand, an off-by-one mask or a wrong log base fails at least one.

Citations: [P1] "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding" (Mind Lab), by
section; [P2] "SGLang's path" (serving-k3, module 05), its paragraph on decode context
parallelism.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import dcp_inputs as di
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ----------------------------------------------------------------------------- layer split
def test_layer_split_worked_example():
    """Layer assignment, worked example 78 layers / 8 CP ranks (4.1; restated in 6.5)."""
    for row in _golden_rows("layer_split_78_8.txt"):
        r, s, e = map(int, row.split())
        assert oracle.layer_range(78, 8, r) == (s, e)


@pytest.mark.parametrize("n_layers,n_cp", [(8, 4), (1, 1), (7, 3), (78, 8), (5, 8), (61, 7)])
def test_layer_split_is_balanced_contiguous_partition(n_layers, n_cp):
    """Ranges tile [0, L) in rank order; sizes differ by at most one, larger ones first."""
    ranges = [oracle.layer_range(n_layers, n_cp, r) for r in range(n_cp)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n_layers
    for (s0, e0), (s1, e1) in zip(ranges, ranges[1:]):
        assert e0 == s1
    sizes = [e - s for s, e in ranges]
    assert max(sizes) - min(sizes) <= 1
    assert sizes == sorted(sizes, reverse=True)
    assert sum(sizes) == n_layers


# ---------------------------------------------------------------------------- page filter
def test_filter_round_robin_16_pages_4_ranks():
    """Animation 3 of 5.1: 16 pages to 4 ranks by page_idx % 4, local slot p // 4."""
    for row in _golden_rows("dcp_pages_16_4.txt"):
        left, right = row.split("|")
        d, *pages = map(int, left.split())
        slots = list(map(int, right.split()))
        out = oracle.filter_indices(np.arange(16), 4, d)
        assert out.tolist() == slots
        # the kept global pages are exactly the owned ones
        assert [s * 4 + d for s in out.tolist()] == pages


def test_filter_256_pages_to_64_per_rank():
    """6.3 log line: 256 pages -> 64 (1/4 of the full sequence) at DCP=4."""
    idx = np.arange(256)
    for d in range(4):
        assert oracle.filter_indices(idx, 4, d).size == 64


@pytest.mark.parametrize("n_dcp", [0, 1])
def test_filter_identity_without_dcp(n_dcp):
    """6.2: with N_dcp <= 1 the indices come back unchanged."""
    idx = np.array([5, 3, 99, 0, 7], np.int32)
    assert oracle.filter_indices(idx, n_dcp, 0).tolist() == idx.tolist()


@pytest.mark.parametrize("n_dcp", [2, 3, 4, 8])
def test_filter_outputs_partition_the_input(n_dcp):
    """Guarantees 1-4 of 6.2: the ranks' kept pages partition the input, each rank keeps
    its pages in input order, and slot * N + d rebuilds the global page."""
    rng = np.random.default_rng(n_dcp)
    idx = rng.permutation(500)[:301].astype(np.int32)
    rebuilt = {}
    for d in range(n_dcp):
        out = oracle.filter_indices(idx, n_dcp, d)
        owned = [int(p) for p in idx if int(p) % n_dcp == d]
        assert out.size == len(owned)
        for pos, s in enumerate(out.tolist()):
            g = s * n_dcp + d
            assert g == owned[pos]
            rebuilt[g] = d
    assert sorted(rebuilt) == sorted(idx.tolist())


@pytest.mark.parametrize("n_dcp", [1, 4, 8])
def test_transfer_filter_masks_on_decode_value(n_dcp):
    """6.3: the mask comes from the decode-side value; the prefill-side indices pass through."""
    rng = np.random.default_rng(7)
    n = 200
    src = rng.permutation(1000)[:n].astype(np.int32)
    dst = rng.permutation(4000)[:n].astype(np.int32)
    seen = []
    for d in range(max(n_dcp, 1)):
        s, t = oracle.transfer_filter(src, dst, n_dcp, d)
        back = {int(a): int(b) for a, b in zip(src, dst)}
        for a, b in zip(s.tolist(), t.tolist()):
            full = b * n_dcp + d if n_dcp > 1 else b
            assert back[a] == full
            seen.append(a)
        # order preserved
        pos = [int(np.nonzero(src == a)[0][0]) for a in s.tolist()]
        assert pos == sorted(pos)
    assert sorted(seen) == sorted(src.tolist())


# -------------------------------------------------------------------------------- reshard
def _tagged_source(case_pages, layer_counts, page_bytes, src_pool_pages, rng):
    """Source pools whose every page starts with a unique 8-byte tag (rank, layer, page)."""
    pools = []
    for r, lc in enumerate(layer_counts):
        p = rng.integers(0, 256, size=lc * src_pool_pages * page_bytes, dtype=np.uint8)
        v = p.reshape(lc, src_pool_pages, page_bytes)
        for l in range(lc):
            for s in range(src_pool_pages):
                v[l, s, :8] = np.frombuffer(np.array([r, l, s, 0x51], np.int16).tobytes(), np.uint8)
        pools.append(p)
    return pools


@pytest.mark.parametrize("n_layers,n_cp,n_dcp,lens", [
    (8, 4, 8, [3000, 700, 64, 129]),
    (5, 2, 3, [64 * 7, 1, 190]),
    (1, 1, 4, [1024]),
    (3, 3, 1, [200, 64]),
])
def test_reshard_is_a_lossless_permutation(n_layers, n_cp, n_dcp, lens):
    """2 / 6.3 / 6.4: every (layer, page) of every request lands exactly once, in the rank
    and slot the decode-side page value names, byte for byte; untouched slots keep the
    sentinel; total bytes written equal the full KV (6.1: no N-fold duplication)."""
    rng = np.random.default_rng(11)
    page_bytes = 64 * 576  # FP8 page; the copy is byte-exact so the element type is moot
    pages = [(n + 63) // 64 for n in lens]
    total = sum(pages)
    ranges = [oracle.layer_range(n_layers, n_cp, r) for r in range(n_cp)]
    counts = [e - s for s, e in ranges]
    ptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int64)
    n_ranks = max(n_dcp, 1)
    slots = total // n_ranks + 3
    g = torch.Generator().manual_seed(3)
    _, vp = di.page_table(lens, n_dcp, slots, g)
    vp = vp.numpy()
    src_pool_pages = total + 5
    src_pages = rng.permutation(src_pool_pages)[:total].astype(np.int32)
    src = _tagged_source(pages, counts, page_bytes, src_pool_pages, rng)
    dst = [np.full(n_layers * slots * page_bytes, di.SENTINEL_BYTE, np.uint8) for _ in range(n_ranks)]
    assert oracle.reshard(ptr, src_pages, vp, page_bytes, n_layers, src, src_pool_pages, n_dcp,
                          dst, slots) == 0
    written = set()
    for l in range(n_layers):
        r = next(i for i, (s, e) in enumerate(ranges) if s <= l < e)
        for i in range(total):
            v = int(vp[i])
            d, s = (v % n_dcp, v // n_dcp) if n_dcp > 1 else (0, v)
            got = dst[d].reshape(n_layers, slots, page_bytes)[l, s]
            want = src[r].reshape(counts[r], src_pool_pages, page_bytes)[l - ranges[r][0], src_pages[i]]
            assert np.array_equal(got, want)
            assert (d, l, s) not in written
            written.add((d, l, s))
    n_sentinel = 0
    for d in range(n_ranks):
        v = dst[d].reshape(n_layers, slots, page_bytes)
        for l in range(n_layers):
            for s in range(slots):
                if (d, l, s) not in written:
                    assert (v[l, s] == di.SENTINEL_BYTE).all()
                    n_sentinel += 1
    assert len(written) == n_layers * total
    assert len(written) + n_sentinel == n_ranks * n_layers * slots


def test_reshard_paths_compose_and_each_carries_one_nth():
    """2 (2D reshard target, all (r, d) paths) and 5.3 (each path carries 1/N_dcp of the
    sequence): running the paths one at a time gives the full result, and each path writes
    its layers x 1/N of the pages."""
    rng = np.random.default_rng(5)
    n_layers, n_cp, n_dcp = 6, 3, 4
    lens = [64 * 64, 64 * 32]
    pages = [(n + 63) // 64 for n in lens]
    total = sum(pages)
    ranges = [oracle.layer_range(n_layers, n_cp, r) for r in range(n_cp)]
    counts = [e - s for s, e in ranges]
    ptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int64)
    slots = total // n_dcp
    g = torch.Generator().manual_seed(9)
    _, vp = di.page_table(lens, n_dcp, slots, g)
    src_pages = np.arange(total, dtype=np.int32)
    page_bytes = 128
    src = _tagged_source(pages, counts, page_bytes, total, rng)
    full = [np.zeros(n_layers * slots * page_bytes, np.uint8) for _ in range(n_dcp)]
    oracle.reshard(ptr, src_pages, vp.numpy(), page_bytes, n_layers, src, total, n_dcp, full, slots)
    parts = [np.zeros(n_layers * slots * page_bytes, np.uint8) for _ in range(n_dcp)]
    for r, d in itertools.product(range(n_cp), range(n_dcp)):
        before = [p.copy() for p in parts]
        oracle.reshard(ptr, src_pages, vp.numpy(), page_bytes, n_layers, src, total, n_dcp, parts,
                       slots, only_src=r, only_dst=d)
        changed_pages = sum(int((a != b).reshape(-1, page_bytes).any(axis=1).sum())
                            for a, b in zip(before, parts))
        assert changed_pages == counts[r] * total // n_dcp
    for a, b in zip(full, parts):
        assert np.array_equal(a, b)


def test_reshard_rejects_out_of_range_slot():
    page_bytes = 64
    src = [np.zeros(4 * page_bytes, np.uint8)]
    dst = [np.zeros(2 * page_bytes, np.uint8) for _ in range(2)]
    ptr = np.array([0, 2], np.int64)
    st = oracle.reshard(ptr, np.array([0, 1], np.int32), np.array([0, 9], np.int32), page_bytes, 1,
                        src, 4, 2, dst, 2)
    assert st == -2


def _path_case(seed=7):
    """5 layers split over 2 CP ranks, 3 DCP ranks, ragged requests; tagged source pages."""
    rng = np.random.default_rng(seed)
    n_layers, n_cp, n_dcp = 5, 2, 3
    lens = [64 * 7, 1, 190, 2000]
    pages = [(n + 63) // 64 for n in lens]
    total = sum(pages)
    ranges = [oracle.layer_range(n_layers, n_cp, r) for r in range(n_cp)]
    counts = [e - s for s, e in ranges]
    ptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int64)
    slots = total // n_dcp + 4
    g = torch.Generator().manual_seed(seed)
    _, vp = di.page_table(lens, n_dcp, slots, g)
    src_pool_pages = total + 3
    src_pages = rng.permutation(src_pool_pages)[:total].astype(np.int32)
    page_bytes = 96
    src = _tagged_source(pages, counts, page_bytes, src_pool_pages, rng)
    return dict(n_layers=n_layers, n_cp=n_cp, n_dcp=n_dcp, ranges=ranges, counts=counts, ptr=ptr, slots=slots,
                vp=vp.numpy(), src_pages=src_pages, src_pool_pages=src_pool_pages, page_bytes=page_bytes, src=src)


@pytest.mark.parametrize("cap", [1, 7, "layer", "all", "all+3"])
def test_pack_unpack_chunks_compose_to_path_reshard(cap):
    """Bounded pack ([P3]): packing a path's pages chunk by chunk into a fixed staging buffer and
    unpacking each chunk gives exactly the path's reshard ([P1] 2, 6.3); every staging page holds
    the source page of its item (layer-major order, checked by the source tags); the bytes moved
    equal items x page bytes whatever the buffer size, and one chunk suffices exactly when the
    items fit (the pack trigger: pages x item bytes > buffer bytes)."""
    c = _path_case()
    pb = c["page_bytes"]
    for r, d in itertools.product(range(c["n_cp"]), range(c["n_dcp"])):
        src_idx, dst_slot = oracle.transfer_filter(c["src_pages"], c["vp"], c["n_dcp"], d)
        n_idx = src_idx.size
        n_items = c["counts"][r] * n_idx
        per = {"layer": n_idx, "all": n_items, "all+3": n_items + 3}.get(cap, cap)
        per = max(per, 1)
        staging = np.zeros(per * pb, np.uint8)
        got = [np.full(c["n_layers"] * c["slots"] * pb, di.SENTINEL_BYTE, np.uint8) for _ in range(c["n_dcp"])]
        moved, n_chunks = 0, 0
        for begin in range(0, n_items, per):
            n = min(per, n_items - begin)
            staging[:] = 0
            assert oracle.pack(src_idx, c["counts"][r], begin, n, pb, c["src"][r], c["src_pool_pages"], staging) == 0
            for m in range(n):
                k = begin + m
                j, i = divmod(k, n_idx)
                tag = np.frombuffer(staging[m * pb:m * pb + 8].tobytes(), np.int16)
                assert list(tag) == [r, j, src_idx[i], 0x51]
            assert oracle.unpack(dst_slot, c["counts"][r], c["ranges"][r][0], begin, n, pb, staging, got[d],
                                 c["n_layers"], c["slots"]) == 0
            moved += n * pb
            n_chunks += 1
        assert moved == n_items * pb
        assert n_chunks == -(-n_items // per)
        assert (n_chunks == 1) == (n_items * pb <= per * pb)
        ref = [np.full(c["n_layers"] * c["slots"] * pb, di.SENTINEL_BYTE, np.uint8) for _ in range(c["n_dcp"])]
        assert oracle.reshard(c["ptr"], c["src_pages"], c["vp"], pb, c["n_layers"], c["src"], c["src_pool_pages"],
                              c["n_dcp"], ref, c["slots"], only_src=r, only_dst=d) == 0
        for a, b in zip(got, ref):
            assert np.array_equal(a, b)


def test_pack_rejects_out_of_range_index_and_copies_the_rest():
    pb = 32
    src = np.arange(3 * 4 * pb, dtype=np.uint8) % 251  # 3 layers x 4 pages
    src_idx = np.array([2, 9, 0], np.int32)             # entry 1 is past the pool
    staging = np.full(4 * pb, 7, np.uint8)
    assert oracle.pack(src_idx, 3, 2, 4, pb, src, 4, staging) == -2   # items 2..5
    v = src.reshape(3, 4, pb)
    assert np.array_equal(staging[0:pb], v[0, 0])       # item 2: layer 0, entry 2
    assert np.array_equal(staging[pb:2 * pb], v[1, 2])  # item 3: layer 1, entry 0
    assert (staging[2 * pb:3 * pb] == 7).all()          # item 4: layer 1, entry 1 (skipped)
    assert np.array_equal(staging[3 * pb:], v[1, 0])    # item 5: layer 1, entry 2


@pytest.mark.parametrize("n_dcp", [1, 3, 4])
def test_naive_transfer_then_inplace_shard_equals_2d_reshard(n_dcp):
    """6.1: the initial design (full unsharded KV to every DCP rank, then an in-place shard)
    ends in the same DCP layout as the 2D reshard, after N_dcp times the transfer: every rank's
    receive buffer holds the whole sequence, and the shard discards (N_dcp - 1) / N_dcp of it."""
    c = _path_case(seed=4)
    pb, L = c["page_bytes"], c["n_layers"]
    total = c["src_pages"].size
    vp = c["vp"] if n_dcp == 3 else _table_for(c, n_dcp)
    n_ranks = max(n_dcp, 1)
    slots = total // n_ranks + 4
    recv = [np.zeros(L * total * pb, np.uint8) for _ in range(n_ranks)]
    assert oracle.full_transfer(c["src_pages"], pb, L, c["src"], c["src_pool_pages"], n_dcp, recv) == 0
    for d in range(n_ranks):  # the whole sequence, page-table order, at every rank
        for l in range(L):
            r = next(i for i, (s0, e0) in enumerate(c["ranges"]) if s0 <= l < e0)
            for i in range(total):
                tag = np.frombuffer(recv[d][(l * total + i) * pb:(l * total + i) * pb + 8].tobytes(), np.int16)
                assert list(tag) == [r, l - c["ranges"][r][0], c["src_pages"][i], 0x51]
    got = [np.full(L * slots * pb, di.SENTINEL_BYTE, np.uint8) for _ in range(n_ranks)]
    assert oracle.inplace_shard(vp, pb, L, n_dcp, recv, got, slots) == 0
    ref = [np.full(L * slots * pb, di.SENTINEL_BYTE, np.uint8) for _ in range(n_ranks)]
    assert oracle.reshard(c["ptr"], c["src_pages"], vp, pb, L, c["src"], c["src_pool_pages"], n_dcp, ref, slots) == 0
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    transferred = sum(x.size for x in recv)
    assert transferred == n_ranks * L * total * pb  # N_dcp x the KV; the 2D reshard moves 1 x


def _table_for(c, n_dcp):
    pages = [int(c["ptr"][b + 1] - c["ptr"][b]) for b in range(len(c["ptr"]) - 1)]
    total = sum(pages)
    g = torch.Generator().manual_seed(23)
    _, vp = di.page_table([64 * n for n in pages], n_dcp, total // max(n_dcp, 1) + 4, g)
    return vp.numpy()


# ------------------------------------------------------------------- token-interleaved layout
def _dense_layouts(lens, n_dcp, H=3, T=2, seed=3):
    """One dense BF16 token sequence per request, laid out page-interleaved ([P1] 5.1: token t
    at row t mod 64 of entry t div 64) and token-interleaved ([P2]: rank t mod N, local token
    t div N), with the same queries."""
    page = di.attention_case(lens, H=H, T=T, n_dcp=n_dcp, dtype="bf16", slots_per_rank=None, seed=seed,
                             device="cpu")
    tok = di.token_attention_case(lens, H=H, T=T, n_dcp=n_dcp, dtype="bf16", seed=seed + 1, device="cpu")
    tok.q = page.q.clone()
    n_r = max(n_dcp, 1)
    g = torch.Generator().manual_seed(seed + 7)
    for b, n in enumerate(lens):
        dense = torch.randn((n, 576), generator=g).to(torch.bfloat16)
        pp, pv = page.req_page_ptr.numpy(), page.dst_vpages.numpy()
        tp, tv = tok.req_page_ptr.numpy(), tok.dst_vpages.numpy()
        for t in range(n):
            v = int(pv[pp[b] + t // 64])
            page.pools[v % n_r if n_dcp > 1 else 0][v // n_r if n_dcp > 1 else v, t % 64] = dense[t]
            d, qd = t % n_r, t // n_r
            w = int(tv[tp[b] + (qd // 64) * n_r + d])
            tok.pools[d][w // n_r if n_dcp > 1 else w, qd % 64] = dense[t]
    return page, tok


def _call_layout(case, rank=-1):
    q_bits, raw, _ = _np_case(case)
    return oracle.attention(q_bits, case.seq_lens.numpy(), case.req_page_ptr.numpy(), case.dst_vpages.numpy(), raw,
                            oracle.BF16, 1.0, case.softmax_scale, case.n_dcp, rank=rank, q_len=case.T,
                            num_heads=case.H, layout=case.layout)


@pytest.mark.parametrize("lens,n_dcp", [([130, 70, 5], 3), ([64 * 9 + 1], 4), ([200], 1)])
def test_token_layout_attention_equals_page_layout_and_merges_exactly(lens, n_dcp):
    """[P2]: with rank i holding tokens i, i + N, ..., the unsharded attention equals the
    page-interleaved layout's over the same token sequence (both are the dense attention), and
    the merge of the per-rank partials is exact (the LSE recombination)."""
    page, tok = _dense_layouts(lens, n_dcp)
    o_p, l_p = _call_layout(page)
    o_t, l_t = _call_layout(tok)
    np.testing.assert_allclose(o_t, o_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_t, l_p, rtol=0, atol=1e-12)
    parts = [_call_layout(tok, rank=d) for d in range(max(n_dcp, 1))]
    o_m, l_m = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o_m, o_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_m, l_p, rtol=0, atol=1e-12)


def test_token_layout_rank_partial_brute_force():
    """Rank d's partial covers exactly the tokens t = d mod N with t <= n - T + q (scipy)."""
    lens, n_dcp, H, T = [150, 67], 3, 2, 2
    page, tok = _dense_layouts(lens, n_dcp, H=H, T=T, seed=5)
    q_bits, raw, dec = _np_case(page)
    for d in range(n_dcp):
        o, l = _call_layout(tok, rank=d)
        for b, n in enumerate(lens):
            pp, pv = page.req_page_ptr.numpy(), page.dst_vpages.numpy()
            keys = []
            for tt in range(n):
                v = int(pv[pp[b] + tt // 64])
                keys.append(dec[v % n_dcp][v // n_dcp, tt % 64])
            keys = np.stack(keys)
            for t in range(T):
                for h in range(H):
                    row = (b * T + t) * H + h
                    vis = [tt for tt in range(n) if tt % n_dcp == d and tt <= n - T + t]
                    qv = torch.from_numpy(q_bits[b, t, h].view(np.int16)).view(torch.bfloat16).double().numpy()
                    if not vis:
                        assert np.isneginf(l[row]) and not o[row].any()
                        continue
                    sc = page.softmax_scale * (keys[vis] @ qv)
                    assert l[row] == pytest.approx(logsumexp(sc), abs=1e-10)
                    np.testing.assert_allclose(o[row], softmax(sc) @ keys[vis][:, :512], rtol=0, atol=1e-10)


def test_token_reshard_puts_token_t_at_rank_t_mod_n():
    """[P2] layout from the prefill pages: token t of layer l lands at rank t mod N, local token
    t div N (row (t div N) mod 64 of the page named by entry ((t div N) div 64) N + t mod N); rows
    past the sequence keep the sentinel; layers come from their owning CP rank ([P1] 4.1)."""
    rng = np.random.default_rng(2)
    lens, n_dcp, n_layers, n_cp = [130, 64, 3], 3, 3, 2
    ranges = [oracle.layer_range(n_layers, n_cp, r) for r in range(n_cp)]
    pages = [(n + 63) // 64 for n in lens]
    sptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int64)
    src_pool_pages = sum(pages) + 2
    src_pages = rng.permutation(src_pool_pages)[:sum(pages)].astype(np.int32)
    row_bytes = 16
    pb = 64 * row_bytes
    src = []
    for r, (l0, l1) in enumerate(ranges):
        p = np.zeros(((l1 - l0), src_pool_pages, 64, row_bytes), np.uint8)
        for l in range(l1 - l0):
            for s in range(src_pool_pages):
                for i in range(64):
                    p[l, s, i, :8] = np.frombuffer(np.array([r, l, s, i], np.int16).tobytes(), np.uint8)
        src.append(p.reshape(-1))
    slots = 8
    tptr, tv = di.token_page_table(lens, n_dcp, slots, torch.Generator().manual_seed(1))
    tptr, tv = tptr.numpy(), tv.numpy()
    dst = [np.full(n_layers * slots * pb, di.SENTINEL_BYTE, np.uint8) for _ in range(n_dcp)]
    assert oracle.token_reshard(lens, sptr, src_pages, tptr, tv, row_bytes, n_layers, src, src_pool_pages, n_dcp,
                                dst, slots) == 0
    hit = set()
    for l in range(n_layers):
        r = next(i for i, (s0, e0) in enumerate(ranges) if s0 <= l < e0)
        for b, n in enumerate(lens):
            for t in range(n):
                d, qd = t % n_dcp, t // n_dcp
                w = int(tv[tptr[b] + (qd // 64) * n_dcp + d])
                assert w % n_dcp == d
                off = ((l * slots + w // n_dcp) * 64 + qd % 64) * row_bytes
                tag = list(np.frombuffer(dst[d][off:off + 8].tobytes(), np.int16))
                assert tag == [r, l - ranges[r][0], src_pages[sptr[b] + t // 64], t % 64]
                hit.add((d, off))
    for d in range(n_dcp):
        rows = dst[d].reshape(-1, row_bytes)
        for k in range(rows.shape[0]):
            if (d, k * row_bytes) not in hit:
                assert (rows[k] == di.SENTINEL_BYTE).all()


# ------------------------------------------------------------------------------- decoders
def test_bf16_decode_matches_format_and_torch():
    """BF16 = upper half of binary32: known encodings, and all 65536 codes vs torch's cast."""
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC000) == -2.0
    assert oracle.bf16_value(0x7F80) == math.inf
    assert oracle.bf16_value(0x0001) == 2.0 ** -133
    codes = np.arange(65536, dtype=np.uint16)
    mine = oracle.decode_bf16(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_decode_matches_format_and_torch():
    """E4M3 (OCP FP8): known encodings, and all 256 codes vs torch.float8_e4m3fn."""
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    assert oracle.e4m3_value(0x80) == 0.0 and math.copysign(1, oracle.e4m3_value(0x80)) < 0
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# ----------------------------------------------------------------------------- attention
def _np_case(case):
    """Host copies of an AttnCase: q bits, pool bytes, decoded pools (torch casts)."""
    q_bits = case.q.cpu().view(torch.int16).numpy().view(np.uint16)
    pools = [p.cpu() for p in case.pools]
    raw = [(p.view(torch.int16).numpy().view(np.uint16) if case.dtype == "bf16"
            else p.view(torch.uint8).numpy()) for p in pools]
    dec = [p.double().numpy() * case.kv_scale for p in pools]
    return q_bits, raw, dec


def _call(case, raw, q_bits, rank=-1, rows=None, n_dcp=None):
    return oracle.attention(q_bits, case.seq_lens.cpu().numpy(), case.req_page_ptr.cpu().numpy(),
                            case.dst_vpages.cpu().numpy(), raw,
                            oracle.BF16 if case.dtype == "bf16" else oracle.E4M3, case.kv_scale,
                            case.softmax_scale, case.n_dcp if n_dcp is None else n_dcp, rank=rank,
                            rows=rows, q_len=case.T, num_heads=case.H)


def _brute(case, q_bits, dec, b, t, h, rank=-1):
    """Gather the visible keys with explicit loops, then scipy softmax / logsumexp."""
    n = int(case.seq_lens[b])
    ptr = case.req_page_ptr.cpu().numpy()
    vp = case.dst_vpages.cpu().numpy()
    keys = []
    for j in range(ptr[b + 1] - ptr[b]):
        v = int(vp[ptr[b] + j])
        d, s = divmod(v, case.n_dcp)[::-1] if case.n_dcp > 1 else (0, v)
        if rank >= 0 and d != rank:
            continue
        for i in range(64):
            if 64 * j + i <= n - case.T + t:
                keys.append(dec[d][s, i])
    q = torch.from_numpy(q_bits[b, t, h].view(np.int16)).view(torch.bfloat16).double().numpy()
    if not keys:
        return np.zeros(512), -math.inf
    K = np.stack(keys)
    s = case.softmax_scale * (K @ q)
    return softmax(s) @ K[:, :512], logsumexp(s)


def _small(lens, H=4, T=1, n_dcp=3, dtype="bf16", seed=0, slots=None):
    return di.attention_case(lens, H=H, T=T, n_dcp=n_dcp, dtype=dtype, slots_per_rank=slots,
                             seed=seed, device="cpu")


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_attention_single_key_closed_form(dtype):
    """One visible key: O = its first 512 dims, LSE = its scaled score."""
    case = _small([1], H=3, n_dcp=1, dtype=dtype)
    q_bits, raw, dec = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    v = int(case.dst_vpages[0])
    k = dec[0][v, 0]
    for h in range(3):
        q = torch.from_numpy(q_bits[0, 0, h].view(np.int16)).view(torch.bfloat16).double().numpy()
        assert lse[h] == pytest.approx(case.softmax_scale * float(k @ q), abs=1e-12)
        np.testing.assert_allclose(o[h], k[:512], rtol=0, atol=1e-12)


def test_attention_identical_keys_closed_form():
    """n identical keys: O = that key's V, LSE = s + ln n (natural log, every key counted)."""
    case = _small([64 * 3 - 5], H=2, n_dcp=1)
    q_bits, raw, dec = _np_case(case)
    row = case.pools[0][0, 0].clone()
    case.pools[0][:] = row
    q_bits, raw, dec = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    n = 64 * 3 - 5
    k = dec[0][0, 0]
    for h in range(2):
        q = torch.from_numpy(q_bits[0, 0, h].view(np.int16)).view(torch.bfloat16).double().numpy()
        s = case.softmax_scale * float(k @ q)
        assert lse[h] == pytest.approx(s + math.log(n), abs=1e-12)
        np.testing.assert_allclose(o[h], k[:512], rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype,T,n_dcp,lens", [
    ("bf16", 1, 3, [130, 64, 1, 257]),
    ("e4m3", 2, 4, [200, 65, 127]),
    ("bf16", 4, 2, [64 * 5 + 3, 66]),
])
def test_attention_brute_force(dtype, T, n_dcp, lens):
    """Unsharded and per-rank rows vs explicit gathering + scipy softmax / logsumexp."""
    case = _small(lens, H=3, T=T, n_dcp=n_dcp, dtype=dtype, seed=len(lens))
    q_bits, raw, dec = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    parts = [_call(case, raw, q_bits, rank=d) for d in range(n_dcp)]
    for b, t, h in itertools.product(range(case.B), range(T), range(3)):
        r = (b * T + t) * 3 + h
        bo, bl = _brute(case, q_bits, dec, b, t, h)
        np.testing.assert_allclose(o[r], bo, rtol=0, atol=1e-11)
        assert lse[r] == pytest.approx(bl, abs=1e-11)
        for d in range(n_dcp):
            bo, bl = _brute(case, q_bits, dec, b, t, h, rank=d)
            np.testing.assert_allclose(parts[d][0][r], bo, rtol=0, atol=1e-11)
            if bl == -math.inf:
                assert parts[d][1][r] == -math.inf
            else:
                assert parts[d][1][r] == pytest.approx(bl, abs=1e-11)


def test_attention_causal_equals_shorter_sequence():
    """Multi-token verify: query t of T sees exactly the first n - T + t + 1 tokens, i.e.
    the same row of a q_len=1 call on a sequence shortened by T - 1 - t tokens."""
    T = 4
    case = _small([64 * 3 + 2], H=2, T=T, n_dcp=2, seed=4)
    q_bits, raw, _ = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    n = int(case.seq_lens[0])
    for t in range(T):
        short = di.AttnCase(B=1, T=1, H=2, n_dcp=2, dtype="bf16",
                            seq_lens=torch.tensor([n - (T - 1 - t)], dtype=torch.int32),
                            req_page_ptr=case.req_page_ptr, dst_vpages=case.dst_vpages,
                            q=case.q[:, t:t + 1], pools=case.pools,
                            slots_per_rank=case.slots_per_rank, kv_scale=1.0)
        qs = np.ascontiguousarray(q_bits[:, t:t + 1])
        o1, l1 = _call(short, raw, qs)
        for h in range(2):
            np.testing.assert_array_equal(o[t * 2 + h], o1[h])
            assert lse[t * 2 + h] == l1[h]


def test_attention_page_relocation_invariance():
    """Moving pages to other slots (table updated) leaves every result bit-identical."""
    case = _small([300, 520], H=2, n_dcp=3, seed=8, slots=12)
    q_bits, raw, _ = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(1))
    vp = case.dst_vpages.clone()
    pools = [torch.empty_like(p) for p in case.pools]
    for d in range(3):
        pools[d][perm] = case.pools[d]
    for i in range(vp.numel()):
        v = int(vp[i])
        vp[i] = int(perm[v // 3]) * 3 + v % 3
    moved = di.AttnCase(B=2, T=1, H=2, n_dcp=3, dtype="bf16", seq_lens=case.seq_lens,
                        req_page_ptr=case.req_page_ptr, dst_vpages=vp, q=case.q, pools=pools,
                        slots_per_rank=12, kv_scale=1.0)
    q2, raw2, _ = _np_case(moved)
    o2, l2 = _call(moved, raw2, q2)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, l2)


def test_attention_fp8_scale_placement():
    """E4M3 pool with kv_scale = 2^-3 equals a BF16 pool holding the same values times 2^-3
    (exactly representable): the scale multiplies both K (scores) and V (output)."""
    case = _small([190, 64], H=2, n_dcp=2, dtype="e4m3", seed=6)
    case.kv_scale = 0.125
    q_bits, raw, dec = _np_case(case)
    o8, l8 = _call(case, raw, q_bits)
    bf = [(p.double() * 0.125).to(torch.bfloat16) for p in case.pools]
    assert all(torch.equal(b.double(), p.double() * 0.125) for b, p in zip(bf, case.pools))
    case16 = di.AttnCase(B=2, T=1, H=2, n_dcp=2, dtype="bf16", seq_lens=case.seq_lens,
                         req_page_ptr=case.req_page_ptr, dst_vpages=case.dst_vpages, q=case.q,
                         pools=bf, slots_per_rank=case.slots_per_rank, kv_scale=1.0)
    q2, raw2, _ = _np_case(case16)
    o16, l16 = _call(case16, raw2, q2)
    np.testing.assert_allclose(o8, o16, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l8, l16, rtol=0, atol=1e-13)


def test_dcp1_equals_unsharded():
    """A DCP=1 run over one pool holding every page equals the unsharded multi-rank run."""
    case = _small([400, 64 * 4, 3], H=2, n_dcp=4, seed=12)
    q_bits, raw, _ = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    slots = case.slots_per_rank
    one = torch.cat(case.pools, 0)  # rank d's slot s -> slot d * slots + s
    vp = case.dst_vpages.clone()
    vp = (vp % 4) * slots + vp // 4
    single = di.AttnCase(B=3, T=1, H=2, n_dcp=1, dtype="bf16", seq_lens=case.seq_lens,
                         req_page_ptr=case.req_page_ptr, dst_vpages=vp.to(torch.int32), q=case.q,
                         pools=[one], slots_per_rank=4 * slots, kv_scale=1.0)
    q1, raw1, _ = _np_case(single)
    o1, l1 = _call(single, raw1, q1)
    np.testing.assert_array_equal(o, o1)
    np.testing.assert_array_equal(lse, l1)


@pytest.mark.parametrize("T,lens", [(1, [900, 64, 2, 64 * 9 + 1]), (4, [65, 64 * 6 + 2])])
def test_merged_shards_equal_unsharded(T, lens):
    """5.2 and the exactness claim of the second page: merging the N partials (O_d, LSE_d)
    reproduces full softmax attention to float64 rounding, including empty shards."""
    n_dcp = 4
    case = _small(lens, H=3, T=T, n_dcp=n_dcp, seed=13)
    q_bits, raw, _ = _np_case(case)
    o, lse = _call(case, raw, q_bits)
    parts = [_call(case, raw, q_bits, rank=d) for d in range(n_dcp)]
    assert any(np.isneginf(p[1]).any() for p in parts)  # an empty shard is exercised
    om, lm = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------------- merge
def test_merge_closed_forms():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((1, 5, 8))
    l = rng.standard_normal((1, 5))
    om, lm = oracle.lse_merge(o, l)                      # one part: identity
    np.testing.assert_array_equal(om, o[0])
    np.testing.assert_array_equal(lm, l[0])
    o2 = rng.standard_normal((2, 5, 8))
    l2 = np.repeat(l, 2, axis=0)                         # equal LSEs: mean and + ln 2
    om, lm = oracle.lse_merge(o2, l2)
    np.testing.assert_allclose(om, o2.mean(0), atol=1e-15)
    np.testing.assert_allclose(lm, l[0] + math.log(2), atol=1e-15)
    l3 = np.stack([l[0], np.full(5, -np.inf)])           # an empty part weighs nothing
    om, lm = oracle.lse_merge(o2, l3)
    np.testing.assert_array_equal(om, o2[0])
    np.testing.assert_array_equal(lm, l[0])
    om, lm = oracle.lse_merge(o2, np.full((2, 5), -np.inf))  # all empty
    assert (om == 0).all() and np.isneginf(lm).all()


def test_merge_matches_logsumexp_and_is_order_invariant():
    """LSE = scipy logsumexp over parts; O = softmax(LSE_d)-weighted sum; rank order free."""
    rng = np.random.default_rng(1)
    n, rows, v = 8, 37, 16
    o = rng.standard_normal((n, rows, v))
    l = 5 * rng.standard_normal((n, rows))
    l[3, 4] = -np.inf
    om, lm = oracle.lse_merge(o, l)
    np.testing.assert_allclose(lm, logsumexp(l, axis=0), rtol=0, atol=1e-12)
    w = softmax(l, axis=0)
    np.testing.assert_allclose(om, np.einsum("nr,nrv->rv", w, o), rtol=0, atol=1e-12)
    perm = rng.permutation(n)
    op, lp = oracle.lse_merge(o[perm], l[perm])
    np.testing.assert_allclose(op, om, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lp, lm, rtol=0, atol=1e-13)
