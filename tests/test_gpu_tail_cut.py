"""GPU: the plan's tail cut.  Persistent CTAs take units largest first; when the last round of
the queue is only partly filled, the plan cuts the chunks of that round into pieces of about
(their work / number of SMs) tiles, merged like chunks.  The unit counts the device plan reports
(dcp_attn_plan_info) must equal a host restatement of that rule, and the results must match the
oracle on every rank whether or not a segment was cut."""
import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits

pytestmark = pytest.mark.gpu


def _pair_tiles(case):
    """128-token tiles of every (rank, request) pair, rank-major (pair = d * B + b)."""
    ptr = case.req_page_ptr.cpu().numpy()
    own = (case.dst_vpages.cpu().numpy() % case.n_dcp) if case.n_dcp > 1 else np.zeros(int(ptr[-1]), np.int64)
    tiles = []
    for d in range(case.n_dcp):
        for b in range(case.B):
            pages = int((own[ptr[b]:ptr[b + 1]] == d).sum())
            tiles.append((pages + 1) // 2)
    return tiles


def _expected(case, tpc, sms):
    """(units, pairs with several pieces, whether the tail is cut) by the rule the plan applies (host restatement): chunks
    of tpc tiles; the queue in (size descending, request, rank, chunk) order; if its last round
    is partly filled, the chunks from that round's first position on laid end to end and cut at
    the multiples of q = their tiles x G / SMs, when that pays and fits the workspace."""
    G = case.T * ((case.H + 63) // 64)
    B, N = case.B, case.n_dcp
    tiles = _pair_tiles(case)
    chunks, items = {}, []
    for d in range(N):
        for b in range(B):
            pr = d * B + b
            t = tiles[pr]
            chunks[pr] = 1 if t == 0 else -(-t // tpc)
            items += [(max(0, min(tpc, t - c * tpc)), (b * N + d, c), pr) for c in range(chunks[pr])]
    split = {pr for pr, ch in chunks.items() if ch > 1}
    part_before = sum(ch * G for ch in chunks.values() if ch > 1)
    n_pages = int(case.req_page_ptr[-1])
    max_partials = (G * (n_pages + N * B)) // tpc + G
    max_units = N * B * G + max_partials
    u_c = len(items)
    total = u_c * G
    full = total // sms
    if full < 1 or total % sms == 0:
        return total, len(split), False
    ts = -(-(full * sms) // G)
    tail = sorted(items, key=lambda x: (-x[0], x[1]))[ts:]
    s_tail, smax = sum(x[0] for x in tail), (tail[0][0] if tail else -1)
    q = -(-(s_tail * G) // sms)
    cuts = s_tail // q if q else 0
    pays = q >= 8 and 4 * smax > 5 * q + 16
    fits = (u_c - ts <= 512 and total + cuts * G <= max_units and part_before + (cuts + u_c - ts) * G <= max_partials)
    if not (pays and fits):
        return total, len(split), False
    extra, o = 0, 0
    for sz, _, pr in tail:
        k = (o + sz - 1) // q - o // q + 1 if sz > 0 else 1
        if k > 1:
            split.add(pr)
        extra += k - 1
        o += sz
    return (u_c + extra) * G, len(split), True


def _plan(case):
    ws = dcp.alloc_workspace(case.B, case.T, case.H, case.n_dcp, case.dst_vpages.numel(), case.q.device)
    err = torch.zeros(1, dtype=torch.int32, device=case.q.device)
    dcp.attn_plan((case.B, case.T, case.H), case.req_page_ptr, case.dst_vpages, case.pools, ws, dev_error=err)
    info = dcp.attn_plan_info((case.B, case.T, case.H), case.dst_vpages.numel(), case.pools, ws)
    assert int(err.item()) == 0 and info["valid"]
    return ws, info


def _cut_case(device, sms, T=1):
    """(ceil(SMs / 4.8) + 8) / q_len requests x 81,920 tokens at DCP=8: 80-tile segments, enough
    units (at least SMs / 0.6) that the plan keeps each segment whole, and a partly filled last
    round (16 of 320 units past it on 152 SMs) that the rule cuts.  With q_len 2 every chunk is
    two units (the query groups of the two new tokens), cut alike."""
    B = -(-sms * 10 // (48 * T)) + 8 // T
    return di.attention_case([81_920] * B, H=64, T=T, n_dcp=8, dtype="e4m3", slots_per_rank=None, seed=41 + T,
                             device=device, name=f"tail-cut-{B}x81920-q{T}-fp8-dcp8")


def test_plan_info_on_a_workspace_without_a_plan(cuda_device):
    case = di.attention_case([1000, 300], H=64, T=1, n_dcp=4, dtype="bf16", slots_per_rank=None, seed=2,
                             device=cuda_device)
    ws = dcp.alloc_workspace(case.B, case.T, case.H, case.n_dcp, case.dst_vpages.numel(), cuda_device)
    ws.zero_()
    info = dcp.attn_plan_info((case.B, case.T, case.H), case.dst_vpages.numel(), case.pools, ws)
    assert info["valid"] is False and info["units"] == 0 and info["split_pairs"] == 0


@pytest.mark.parametrize("T", [1, 2])
def test_tail_cut_counts_and_parity(cuda_device, T):
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    case = _cut_case(cuda_device, sms, T)
    ws, info = _plan(case)
    units, split, cut = _expected(case, info["tiles_per_chunk"], sms)
    assert cut and split > 0, "the case is built so that the rule cuts"
    assert (info["units"], info["split_pairs"]) == (units, split)
    # planned run and one-call run: partials of every rank and the merged output vs the oracle
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools, case.softmax_scale, case.kv_scale)
    om, lm, o, l = dcp.decode_attn_merged(*args, workspace=ws, dev_error=err, planned=True)
    o1, l1 = dcp.partial_decode_attn(*args, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o, o1) and torch.equal(l, l1)
    o, l, om, lm = (t.cpu().numpy() for t in (o, l, om, lm))
    # two heads of every request and new token: every (rank, request, query group) is checked,
    # cut or not
    rows = np.array([(b * case.T + t) * case.H + h for b in range(case.B) for t in range(case.T)
                     for h in (b % 64, 63 - b % 64)], np.int64)
    qb, pools = q_bits(case), pool_bytes(case)
    for d in range(case.n_dcp):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(-1, 512)[rows], l[d].reshape(-1)[rows], ro, rl, f"{case.name} rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(-1, 512)[rows], lm.reshape(-1)[rows], ro, rl, f"{case.name} merged")


@pytest.mark.parametrize("name", ["agent", "batch"])
def test_tail_cut_rule_on_the_workloads(cuda_device, name):
    """The agent workload (384 equal segments) is cut on a 152-SM GB300; the batch workload's
    8-tile segments are not (a cut would cost more than it saves)."""
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    case = di.agent_case(cuda_device) if name == "agent" else di.batch_case(cuda_device)
    _, info = _plan(case)
    assert (info["units"], info["split_pairs"]) == _expected(case, info["tiles_per_chunk"], sms)[:2]
    if sms == 152:
        assert (info["split_pairs"] > 0) == (name == "agent")


# Seeded mixed lengths (multiples of 64 tokens), chosen so that on a 152-SM GB300 some segments
# are already chunked and the last round is cut: the boundary size's chunks are then taken by
# their (request, rank, chunk) rank and pieces join pairs that already hold several chunks.
MIXED = [(1, 24, (300, 1700), 2, "e4m3"), (25, 40, (300, 1700), 1, "e4m3"), (25, 40, (300, 1700), 1, "bf16")]


@pytest.mark.parametrize("seed,B,pages,T,dtype", MIXED, ids=[f"seed{m[0]}-q{m[3]}-{m[4]}" for m in MIXED])
def test_tail_cut_with_mixed_lengths_and_chunked_segments(cuda_device, seed, B, pages, T, dtype):
    import random
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    rng = random.Random(seed)
    lens = [64 * rng.randint(*pages) for _ in range(B)]
    case = di.attention_case(lens, H=64, T=T, n_dcp=8, dtype=dtype, slots_per_rank=None, seed=seed,
                             device=cuda_device, name=f"mixed-{seed}-{dtype}")
    ws, info = _plan(case)
    units, split, cut = _expected(case, info["tiles_per_chunk"], sms)
    assert (info["units"], info["split_pairs"]) == (units, split)
    if sms == 152:  # the premise of the case: segments already chunked, and a cut tail
        tiles = _pair_tiles(case)
        assert cut and max(tiles) > info["tiles_per_chunk"]
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools, case.softmax_scale, case.kv_scale)
    om, lm, o, l = dcp.decode_attn_merged(*args, workspace=ws, dev_error=err, planned=True)
    o1, l1 = dcp.partial_decode_attn(*args, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o, o1) and torch.equal(l, l1)
    o, l, om, lm = (t.cpu().numpy() for t in (o, l, om, lm))
    rows = np.array([(b * case.T + t) * case.H + h for b in range(case.B) for t in range(case.T)
                     for h in ((7 * b) % 64, 63 - (5 * b) % 64)], np.int64)
    qb, pools = q_bits(case), pool_bytes(case)
    for d in range(case.n_dcp):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(-1, 512)[rows], l[d].reshape(-1)[rows], ro, rl, f"{case.name} rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(-1, 512)[rows], lm.reshape(-1)[rows], ro, rl, f"{case.name} merged")


def test_tail_cut_on_the_token_interleaved_layout(cuda_device):
    """The token-interleaved layout's one-call attention makes the same plan (its table holds
    rank d's local page jj at entry jj N + d): the cut applies alike, and the partials of every
    rank and their merge match the oracle over that layout."""
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    B = -(-sms * 10 // 48) + 8
    case = di.token_attention_case([81_920] * B, H=64, T=1, n_dcp=8, dtype="e4m3", seed=47, device=cuda_device,
                                   name=f"tail-cut-tokens-{B}x81920")
    ws = dcp.alloc_workspace(case.B, case.T, case.H, case.n_dcp, case.dst_vpages.numel(), cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o, l = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                   case.softmax_scale, case.kv_scale, workspace=ws, dev_error=err, layout="token")
    info = dcp.attn_plan_info((case.B, case.T, case.H), case.dst_vpages.numel(), case.pools, ws)
    om, lm = dcp.lse_merge(o, l)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and info["valid"]
    units, split, cut = _expected(case, info["tiles_per_chunk"], sms)
    assert (info["units"], info["split_pairs"]) == (units, split) and cut
    o, l, om, lm = (t.cpu().numpy() for t in (o, l, om, lm))
    rows = np.array([b * case.H + h for b in range(case.B) for h in ((3 * b) % 64, 63 - b % 64)], np.int64)
    qb, pools = q_bits(case), pool_bytes(case)
    for d in range(case.n_dcp):
        ro, rl = oracle_attention(case, rank=d, rows=rows, qb=qb, pools=pools)
        compare(o[d].reshape(-1, 512)[rows], l[d].reshape(-1)[rows], ro, rl, f"{case.name} rank {d}")
    ro, rl = oracle_attention(case, rows=rows, qb=qb, pools=pools)
    compare(om.reshape(-1, 512)[rows], lm.reshape(-1)[rows], ro, rl, f"{case.name} merged")
