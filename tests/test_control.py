"""Multi-rank control of the transfer path on CPU ranks (gloo, 127.0.0.1): per-request
bootstrap ("Serving Macaron-V1 at Scale", 6.7), the size-broadcast protocol (4.2) under prefix
divergence, a rank that leaves the protocol (caught by the step gate as a bounded-time error,
never a hang), consensus prefix length and padded all-reduce, and the all-gather + exact LSE
merge exchange ("SGLang's path") against the float64 oracle."""
import multiprocessing as mp
import socket

import numpy as np
import pytest
import torch

import oracle
from decode_context_paged_gb300 import control


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(scenario, world, timeout=90):
    import _control_workers as w
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=w.run, args=(r, world, port, scenario, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, status, res = q.get(timeout=timeout)
        out[rank] = (status, res)
    for p in procs:
        p.join(timeout=30)
        if p.is_alive():
            p.kill()
    return out


def test_bootstrap_per_request_metadata():
    """6.7: d = attn_tp_rank mod N_dcp on the decode side; the request's own (N_dcp, d) decides
    the prefill filter, so decode groups of different DCP sizes coexist and a request after a
    DCP change is filtered with its new size; local values are only the fallback."""
    vp = np.arange(16, dtype=np.int32)            # Animation 3: 16 pages
    src = np.arange(100, 116, dtype=np.int32)
    group_a = [control.decode_dst_info(r, 4) for r in range(4)]   # DCP=4 group
    group_b = [control.decode_dst_info(r, 1) for r in range(2)]   # DCP=1 group
    assert [i.dcp_rank for i in group_a] == [0, 1, 2, 3] and [i.dcp_rank for i in group_b] == [0, 0]
    assert control.decode_dst_info(6, 4).dcp_rank == 2
    for info in group_a:
        n, d = control.transfer_filter_params(info, local_dcp_size=2, local_tp_rank=1)
        s, dst = oracle.transfer_filter(src, vp, n, d)
        assert list(s) == list(src[d::4]) and list(dst) == list(range(4))
    n, d = control.transfer_filter_params(group_b[1], local_dcp_size=4, local_tp_rank=3)
    s, dst = oracle.transfer_filter(src, vp, n, d)
    assert (n, d) == (1, 0) and list(s) == list(src) and list(dst) == list(vp)
    # no per-request metadata: local fallback attn_tp_rank mod dcp_size
    assert control.transfer_filter_params(None, local_dcp_size=4, local_tp_rank=7) == (4, 3)
    # the DCP size changes between requests (2 -> 4) without any global renegotiation
    assert control.transfer_filter_params(control.decode_dst_info(3, 2), 4, 3) == (2, 1)
    assert control.transfer_filter_params(control.decode_dst_info(3, 4), 2, 3) == (4, 3)


def test_size_broadcast_consistent_under_prefix_divergence():
    out = _run("size_broadcast_divergent", 3)
    assert all(s == "ok" for s, _ in out.values()), out
    r = {k: v[1] for k, v in out.items()}
    want = np.arange(20, dtype=np.float32).reshape(5, 4).tolist()
    assert r[0]["committed"] and r[0]["data"] == want            # the owner
    assert r[1]["committed"] and r[1]["data"] == want            # same count: commits
    assert not r[2]["committed"] and r[2]["data"] is None        # diverged: consumes, no commit
    assert all(v["skip2"] == (False, None) for v in r.values())  # owner empty: all skip
    assert all(v["calls"] == ["layer0", "layer1"] for v in r.values())


def test_a_rank_leaving_the_protocol_is_caught_not_hung():
    out = _run("gate_catches_a_skipping_rank", 3, timeout=60)
    assert out[1] == ("ok", {"skipped": True})
    for rank in (0, 2):
        status, res = out[rank]
        assert status == "ok" and "gate_timeout" in res, out
        assert res["seconds"] < 10


def test_consensus_prefix_and_padded_all_reduce():
    out = _run("consensus_and_padded", 3)
    assert all(s == "ok" for s, _ in out.values()), out
    for _, res in out.values():
        assert res["prefix"] == 5
        assert res["sum"] == [0 + 10 + 0, 1 + 11, 2 + 12, 13, 14]
        assert res["max"] == [10, 11, 12, 13, 14]
        # ranks pass 1, 2, 3 copies of 2^60 + 1 + rank: exact int64 sums and minima
        b = (1 << 60) + 1
        assert res["big_dtype"] == "torch.int64"
        assert res["big_sum"] == [3 * b + 3, 2 * b + 3, b + 2]
        assert res["big_min"] == [b, b + 1, b + 2]


@pytest.mark.parametrize("world", [2, 4])
def test_all_gather_and_merge_equals_unsharded_attention(world):
    out = _run("gather_and_merge", world)
    assert all(s == "ok" for s, _ in out.values()), out
    for _, res in out.values():
        assert res["o_err"] < 1e-12 and res["lse_err"] < 1e-12
