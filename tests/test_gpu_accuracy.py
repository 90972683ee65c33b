"""GPU parity on the inputs that stress the attention's arithmetic.

* Peaked softmax: a few planted keys per request take most of the weight, so a rounding
  error on one weight goes straight into O instead of averaging out over many keys.  Run on
  long (rank, request) segments (at least 128 pages per rank) and short ones, for both KV
  types, with q_len 1 and 4.
* A raised softmax scale: scores spread by tens of units, so a handful of keys dominate.
* Non-finite tail rows: the rows of a request's last page past its length are not part of the
  sequence ("Serving Macaron-V1 at Scale", 5.1: pages of 64 tokens; a ragged length leaves the
  last page partly filled).  They are filled with NaN here (BF16 0x7FC0, E4M3 0xFF / 0x7F) and
  must not reach the output.

Comparison: element-wise against the float64 oracle, 2e-2 max-abs on O and 1e-3 on LSE.
"""
import math

import numpy as np
import pytest
import torch

import dcp_inputs as di
import decode_context_paged_gb300 as dcp
from _parity import compare, oracle_attention, pool_bytes, q_bits

pytestmark = pytest.mark.gpu


def _kv_float(case, d, slot, rows):
    """float64 values of pool d's page `slot`, rows `rows` (the FP8 scale applied)."""
    x = case.pools[d][slot][rows].float().double().cpu().numpy()
    return x * (case.kv_scale if case.dtype == "e4m3" else 1.0)


def plant_peaks(case, margins, seed):
    """Per request: give every head's Q one shared rope direction w and plant len(margins)
    keys at random visible positions whose rope part is w scaled so that the key's score sits
    `margin` above the expected log-sum-exp of the background keys.  Returns the planted
    (request, position) pairs."""
    g = torch.Generator().manual_seed(seed)
    ptr = case.req_page_ptr.cpu()
    sl = case.seq_lens.cpu()
    var = 576.0 * case.softmax_scale ** 2          # score variance of N(0,1) rows
    planted = []
    for b in range(case.B):
        n = int(sl[b])
        w = torch.randn(64, generator=g)
        case.q[b, :, :, 512:] = w.to(case.q.device, torch.bfloat16)
        wq = case.q[b, 0, 0, 512:].double().cpu()
        bg = math.log(max(n - case.T + 1, 1)) + var / 2
        pos = torch.randperm(n - case.T + 1, generator=g)[:len(margins)]
        for p, m in zip(pos.tolist(), margins):
            beta = (bg + m) / (float(wq @ wq) * case.softmax_scale)
            e = int(ptr[b]) + p // 64
            d, slot = int(case.page_owner[e]), int(case.page_slot[e])
            rope = beta * wq
            if case.dtype == "e4m3":
                rope = (rope / case.kv_scale).clamp(-448.0, 448.0)
            case.pools[d][slot, p % 64, 512:] = rope.to(case.pools[d].device, case.pools[d].dtype)
            planted.append((b, p))
    return planted


def top_weight(case, lse_ref, b):
    """Largest single-key softmax weight of request b's rows (new token 0), from float64 scores
    of every key: checks that a test's input really is peaked."""
    sl = int(case.seq_lens[b])
    ptr = case.req_page_ptr.cpu()
    limit = sl - case.T  # visible keys of new token 0
    q = case.q[b, 0].double().cpu().numpy()  # [H][576]
    best = np.full(case.H, -np.inf)
    for e in range(int(ptr[b]), int(ptr[b + 1])):
        j = e - int(ptr[b])
        rows = np.arange(64)
        pos = 64 * j + rows
        keep = pos <= limit
        if not keep.any():
            continue
        k = _kv_float(case, int(case.page_owner[e]), int(case.page_slot[e]), slice(0, 64))[keep]
        s = case.softmax_scale * (k @ q.T)  # [keys][H]
        best = np.maximum(best, s.max(axis=0))
    r0 = (b * case.T) * case.H
    return np.exp(best - lse_ref[r0:r0 + case.H])


def _run_both(case):
    err = torch.zeros(1, dtype=torch.int32, device=case.q.device)
    o, l = dcp.partial_decode_attn(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                   case.softmax_scale, case.kv_scale, dev_error=err, layout=case.layout)
    om, lm, _, _ = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                          case.softmax_scale, case.kv_scale, dev_error=err, layout=case.layout)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o.cpu().numpy(), l.cpu().numpy(), om.cpu().numpy(), lm.cpu().numpy()


def _check(case, o, l, om, lm):
    qb, pools = q_bits(case), pool_bytes(case)
    R = case.rows
    lay = case.layout
    for d in range(case.n_dcp):
        ro, rl = oracle_attention(case, rank=d, qb=qb, pools=pools, layout=lay)
        compare(o[d].reshape(R, 512), l[d].reshape(R), ro, rl, f"{case.name} rank {d}")
    ro, rl = oracle_attention(case, qb=qb, pools=pools, layout=lay)
    compare(om.reshape(R, 512), lm.reshape(R), ro, rl, f"{case.name} merged")
    return rl


PEAK_CASES = [
    # name, lens, H, T, N, dtype: long segments (>= 128 pages per rank) and short ones
    ("long-fp8", [70_000, 70_016], 64, 1, 8, "e4m3"),
    ("short-fp8", [3000, 5000, 200], 64, 1, 4, "e4m3"),
    ("long-q4-fp8", [70_000], 64, 4, 8, "e4m3"),
    ("long-bf16", [70_000], 64, 1, 8, "bf16"),
    ("short-bf16", [3000, 640], 64, 1, 4, "bf16"),
]


@pytest.mark.parametrize("name,lens,H,T,N,dtype", PEAK_CASES, ids=[c[0] for c in PEAK_CASES])
def test_peaked_softmax_matches_oracle(cuda_device, name, lens, H, T, N, dtype):
    case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=40 + len(name),
                             device=cuda_device, name="peaked-" + name)
    plant_peaks(case, margins=(0.5, 1.0, 2.0), seed=7)
    rl = _check(case, *_run_both(case))
    w = np.concatenate([top_weight(case, rl, b) for b in range(case.B)])
    assert np.median(w) > 0.4 and w.max() > 0.5, f"input not peaked: median top weight {np.median(w):.2f}"


SCALE_CASES = [
    ("long-fp8", [70_000, 66_000], 64, 1, 8, "e4m3"),
    ("short-fp8", [2000, 900], 64, 1, 4, "e4m3"),
    ("long-bf16", [70_000], 64, 1, 8, "bf16"),
]


@pytest.mark.parametrize("name,lens,H,T,N,dtype", SCALE_CASES, ids=[c[0] for c in SCALE_CASES])
def test_raised_softmax_scale_matches_oracle(cuda_device, name, lens, H, T, N, dtype):
    """Softmax scale 8/sqrt(192): scores spread by ~14 units, a few keys carry the weight."""
    case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=60 + len(name),
                             device=cuda_device, name="scale8-" + name)
    case.softmax_scale = 8.0 / math.sqrt(192.0)
    rl = _check(case, *_run_both(case))
    w = top_weight(case, rl, 0)
    assert np.median(w) > 0.2, f"input not peaked: median top weight {np.median(w):.2f}"


def fill_tail_rows(case):
    """Rows past each request's length in the pages its table names get NaN bits.  Page
    layout: entry j holds positions 64 j + i; token layout: entry jj N + d holds (64 jj + i) N + d."""
    ptr = case.req_page_ptr.cpu()
    sl = case.seq_lens.cpu()
    n = max(case.n_dcp, 1)
    filled = 0
    for b in range(case.B):
        seq = int(sl[b])
        for e in range(int(ptr[b]), int(ptr[b + 1])):
            j = e - int(ptr[b])
            if case.layout == "token":
                jj, d = j // n, j % n
                nv = max(0, min(64, -(-(seq - d) // n) - 64 * jj)) if seq > d else 0
            else:
                nv = max(0, min(64, seq - 64 * j))
            if nv == 64:
                continue
            pool = case.pools[int(case.page_owner[e])]
            rows = pool[int(case.page_slot[e]), nv:]
            if case.dtype == "bf16":
                rows.view(torch.int16).fill_(0x7FC0)
            else:
                u8 = rows.view(torch.uint8)
                u8.fill_(0xFF)
                u8[:, 1::2] = 0x7F
            filled += 64 - nv
    return filled


TAIL_CASES = [
    # name, lens, H, T, N, dtype, layout
    ("ragged-bf16", [1000, 130, 64 * 9 + 5], 64, 1, 4, "bf16", "page"),
    ("ragged-fp8", [1000, 130, 64 * 9 + 5], 64, 1, 4, "e4m3", "page"),
    ("long-fp8", [70_000 + 17, 3000 + 1], 64, 1, 8, "e4m3", "page"),
    ("causal-q4-bf16", [64 * 7 + 3, 260], 64, 4, 2, "bf16", "page"),
    ("causal-q4-fp8", [64 * 7 + 3, 260], 64, 4, 2, "e4m3", "page"),
    ("token-bf16", [1000, 333], 64, 1, 4, "bf16", "token"),
    ("token-fp8", [1000, 333], 64, 1, 4, "e4m3", "token"),
    ("heads-96-fp8", [700, 333], 96, 1, 3, "e4m3", "page"),
]


@pytest.mark.parametrize("name,lens,H,T,N,dtype,layout", TAIL_CASES, ids=[c[0] for c in TAIL_CASES])
def test_nan_tail_rows_do_not_reach_the_output(cuda_device, name, lens, H, T, N, dtype, layout):
    if layout == "token":
        case = di.token_attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, seed=80 + len(name),
                                       device=cuda_device, name="nan-tail-" + name)
    else:
        case = di.attention_case(lens, H=H, T=T, n_dcp=N, dtype=dtype, slots_per_rank=None, seed=80 + len(name),
                                 device=cuda_device, name="nan-tail-" + name)
    assert fill_tail_rows(case) > 0
    _check(case, *_run_both(case))


def test_nan_tail_rows_static_and_planned(cuda_device):
    """The same through the planned run and the allocation-free entry point."""
    case = di.attention_case([1000, 130, 64 * 9 + 5], H=64, T=1, n_dcp=4, dtype="e4m3", slots_per_rank=None,
                             seed=91, device=cuda_device, name="nan-tail-planned")
    assert fill_tail_rows(case) > 0
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ws = dcp.alloc_workspace(case.B, case.T, case.H, case.n_dcp, case.dst_vpages.numel(), cuda_device)
    dcp.attn_plan((case.B, case.T, case.H), case.req_page_ptr, case.dst_vpages, case.pools, ws, dev_error=err)
    om, lm, o, l = dcp.decode_attn_merged(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                          case.softmax_scale, case.kv_scale, workspace=ws, dev_error=err,
                                          planned=True)
    so, sl = dcp.partial_decode_attn_static(case.q, case.seq_lens, case.req_page_ptr, case.dst_vpages, case.pools,
                                            case.softmax_scale, case.kv_scale, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _check(case, so.cpu().numpy(), sl.cpu().numpy(), om.cpu().numpy(), lm.cpu().numpy())
    _check(case, o.cpu().numpy(), l.cpu().numpy(), om.cpu().numpy(), lm.cpu().numpy())
