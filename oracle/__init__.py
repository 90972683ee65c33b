"""Float64 CPU oracle for the DCP hot path (test infrastructure).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` leg may import this package.  The product library
(``decode_context_paged_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``dcp_oracle.c`` (plain C, float64, OpenMP over independent rows);
this module only builds it with gcc and marshals numpy arrays through ctypes.  Every C
function cites the passage of the pages it restates:

* "Serving Macaron-V1 at Scale: Page-Level 2D KV Resharding": 4.1 layer assignment,
  5.1 page ownership, 5.2 LSE merge, 6.2 page index filter, 6.3 transfer filtering,
  6.4 page-granular transfer.
* "SGLang's path" (serving-k3 module 05): partial attention with an exact log-sum-exp
  recombination.

Pins: tests/test_oracle_pins.py.  No function is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdcp_oracle.so")
_lock = threading.Lock()
_lib = None

PAGE_TOKENS = 64
K_DIM = 576
V_DIM = 512
BF16 = 0
E4M3 = 1


def build(force: bool = False) -> str:
    """Compile dcp_oracle.c into libdcp_oracle.so next to it (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.dcpo_num_threads.restype = i32
            lib.dcpo_set_num_threads.argtypes = [i32]
            lib.dcpo_layer_range.argtypes = [i32, i32, i32, vp, vp]
            lib.dcpo_filter_indices.argtypes = [vp, i64, i32, i32, vp]
            lib.dcpo_filter_indices.restype = i64
            lib.dcpo_transfer_filter.argtypes = [vp, vp, i64, i32, i32, vp, vp]
            lib.dcpo_transfer_filter.restype = i64
            lib.dcpo_reshard.argtypes = [i32, vp, vp, vp, i64, i32, i32, vp, i64, i32, vp, i64,
                                         i32, i32]
            lib.dcpo_reshard.restype = i32
            lib.dcpo_bf16_value.argtypes = [ctypes.c_uint16]
            lib.dcpo_bf16_value.restype = dbl
            lib.dcpo_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.dcpo_e4m3_value.restype = dbl
            lib.dcpo_decode_bf16.argtypes = [vp, vp, i64]
            lib.dcpo_decode_e4m3.argtypes = [vp, vp, i64]
            lib.dcpo_attention.argtypes = [i32, i32, i32, vp, vp, vp, vp, i32, dbl, dbl, i32, vp,
                                           i64, i32, vp, i64, vp, vp]
            lib.dcpo_attention.restype = i32
            lib.dcpo_lse_merge.argtypes = [i32, i64, i32, vp, vp, vp, vp]
            lib.dcpo_attention_tokens.argtypes = lib.dcpo_attention.argtypes
            lib.dcpo_attention_tokens.restype = i32
            lib.dcpo_token_reshard.argtypes = [i32, vp, vp, vp, vp, vp, i64, i32, i32, vp, i64, i32, vp, i64]
            lib.dcpo_token_reshard.restype = i32
            lib.dcpo_full_transfer.argtypes = [i64, vp, i64, i32, i32, vp, i64, i32, vp]
            lib.dcpo_full_transfer.restype = i32
            lib.dcpo_inplace_shard.argtypes = [i64, vp, i64, i32, i32, vp, vp, i64]
            lib.dcpo_inplace_shard.restype = i32
            lib.dcpo_pack.argtypes = [i64, vp, i32, i64, i64, i64, vp, i64, vp]
            lib.dcpo_pack.restype = i32
            lib.dcpo_unpack.argtypes = [i64, vp, i32, i32, i64, i64, i64, vp, vp, i32, i64]
            lib.dcpo_unpack.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().dcpo_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's parallel loops from now on (n < 1: one per processor)."""
    _load().dcpo_set_num_threads(int(n))


def layer_range(n_layers: int, n_cp: int, r: int) -> tuple[int, int]:
    s = np.zeros(1, np.int32)
    e = np.zeros(1, np.int32)
    _load().dcpo_layer_range(n_layers, n_cp, r, _ptr(s), _ptr(e))
    return int(s[0]), int(e[0])


def filter_indices(kv_indices, n_dcp: int, d: int) -> np.ndarray:
    idx = _c(kv_indices, np.int32)
    out = np.zeros(max(idx.size, 1), np.int32)
    k = _load().dcpo_filter_indices(_ptr(idx), idx.size, n_dcp, d, _ptr(out))
    return out[:k].copy()


def transfer_filter(transfer_idx, dst_idx, n_dcp: int, d: int) -> tuple[np.ndarray, np.ndarray]:
    s = _c(transfer_idx, np.int32)
    t = _c(dst_idx, np.int32)
    assert s.size == t.size
    os_ = np.zeros(max(s.size, 1), np.int32)
    od = np.zeros(max(s.size, 1), np.int32)
    k = _load().dcpo_transfer_filter(_ptr(s), _ptr(t), s.size, n_dcp, d, _ptr(os_), _ptr(od))
    return os_[:k].copy(), od[:k].copy()


def reshard(req_page_ptr, src_pages, dst_vpages, page_bytes: int, n_layers: int,
            src_pools: list[np.ndarray], src_pool_pages: int, n_dcp: int,
            dst_pools: list[np.ndarray], dst_slots: int, only_src: int = -1,
            only_dst: int = -1) -> int:
    """Byte-exact reshard into ``dst_pools`` (modified in place).  Pools are uint8 arrays."""
    rpp = _c(req_page_ptr, np.int64)
    sp = _c(src_pages, np.int32)
    dv = _c(dst_vpages, np.int32)
    for p in list(src_pools) + list(dst_pools):
        assert p.dtype == np.uint8 and p.flags["C_CONTIGUOUS"]
    sarr = (ctypes.c_void_p * len(src_pools))(*[_ptr(p) for p in src_pools])
    darr = (ctypes.c_void_p * len(dst_pools))(*[_ptr(p) for p in dst_pools])
    return int(_load().dcpo_reshard(rpp.size - 1, _ptr(rpp), _ptr(sp), _ptr(dv), page_bytes,
                                    n_layers, len(src_pools), ctypes.addressof(sarr),
                                    src_pool_pages, n_dcp, ctypes.addressof(darr), dst_slots,
                                    only_src, only_dst))


def token_reshard(seq_lens, src_page_ptr, src_pages, tok_page_ptr, tok_vpages, row_bytes: int, n_layers: int,
                  src_pools: list, src_pool_pages: int, n_dcp: int, dst_pools: list, dst_slots: int) -> int:
    """Token-interleaved reshard (row gather) into ``dst_pools`` (modified in place)."""
    sl = _c(seq_lens, np.int32)
    spp = _c(src_page_ptr, np.int64)
    sp = _c(src_pages, np.int32)
    tpp = _c(tok_page_ptr, np.int64)
    tv = _c(tok_vpages, np.int32)
    for p in list(src_pools) + list(dst_pools):
        assert p.dtype == np.uint8 and p.flags["C_CONTIGUOUS"]
    sarr = (ctypes.c_void_p * len(src_pools))(*[_ptr(p) for p in src_pools])
    darr = (ctypes.c_void_p * len(dst_pools))(*[_ptr(p) for p in dst_pools])
    return int(_load().dcpo_token_reshard(sl.size, _ptr(sl), _ptr(spp), _ptr(sp), _ptr(tpp), _ptr(tv), row_bytes,
                                          n_layers, len(src_pools), ctypes.addressof(sarr), src_pool_pages, n_dcp,
                                          ctypes.addressof(darr), dst_slots))


def full_transfer(src_pages, page_bytes: int, n_layers: int, src_pools: list, src_pool_pages: int, n_dcp: int,
                  recv: list) -> int:
    """Naive transfer: every page of every layer to every DCP rank's receive buffer [L][pages]."""
    sp = _c(src_pages, np.int32)
    for p in list(src_pools) + list(recv):
        assert p.dtype == np.uint8 and p.flags["C_CONTIGUOUS"]
    sarr = (ctypes.c_void_p * len(src_pools))(*[_ptr(p) for p in src_pools])
    rarr = (ctypes.c_void_p * len(recv))(*[_ptr(p) for p in recv])
    return int(_load().dcpo_full_transfer(sp.size, _ptr(sp), page_bytes, n_layers, len(src_pools),
                                          ctypes.addressof(sarr), src_pool_pages, n_dcp, ctypes.addressof(rarr)))


def inplace_shard(dst_vpages, page_bytes: int, n_layers: int, n_dcp: int, recv: list, dst_pools: list,
                  dst_slots: int) -> int:
    """Each rank keeps the pages it owns from its full copy, at their DCP slots."""
    dv = _c(dst_vpages, np.int32)
    for p in list(recv) + list(dst_pools):
        assert p.dtype == np.uint8 and p.flags["C_CONTIGUOUS"]
    rarr = (ctypes.c_void_p * len(recv))(*[_ptr(p) for p in recv])
    darr = (ctypes.c_void_p * len(dst_pools))(*[_ptr(p) for p in dst_pools])
    return int(_load().dcpo_inplace_shard(dv.size, _ptr(dv), page_bytes, n_layers, n_dcp, ctypes.addressof(rarr),
                                          ctypes.addressof(darr), dst_slots))


def pack(src_idx, n_layers: int, item_begin: int, n_items: int, page_bytes: int, src_pool: np.ndarray,
         src_pool_pages: int, staging: np.ndarray) -> int:
    """Bounded-pack send side: items [item_begin, item_begin + n_items) of one path into staging."""
    si = _c(src_idx, np.int32)
    assert src_pool.dtype == np.uint8 and staging.dtype == np.uint8
    assert staging.size >= n_items * page_bytes and src_pool.flags["C_CONTIGUOUS"] and staging.flags["C_CONTIGUOUS"]
    return int(_load().dcpo_pack(si.size, _ptr(si), n_layers, item_begin, n_items, page_bytes, _ptr(src_pool),
                                 src_pool_pages, _ptr(staging)))


def unpack(dst_slot, n_layers: int, layer_offset: int, item_begin: int, n_items: int, page_bytes: int,
           staging: np.ndarray, dst_pool: np.ndarray, num_layers: int, dst_slots: int) -> int:
    """Bounded-pack receive side: the same item range from staging into the destination pool."""
    ds = _c(dst_slot, np.int32)
    assert dst_pool.dtype == np.uint8 and dst_pool.flags["C_CONTIGUOUS"]
    return int(_load().dcpo_unpack(ds.size, _ptr(ds), n_layers, layer_offset, item_begin, n_items, page_bytes,
                                   _ptr(staging), _ptr(dst_pool), num_layers, dst_slots))


def bf16_value(bits: int) -> float:
    return float(_load().dcpo_bf16_value(bits))


def e4m3_value(bits: int) -> float:
    return float(_load().dcpo_e4m3_value(bits))


def decode_bf16(bits) -> np.ndarray:
    a = _c(bits, np.uint16)
    out = np.empty(a.shape, np.float64)
    _load().dcpo_decode_bf16(_ptr(a), _ptr(out), a.size)
    return out


def decode_e4m3(bits) -> np.ndarray:
    a = _c(bits, np.uint8)
    out = np.empty(a.shape, np.float64)
    _load().dcpo_decode_e4m3(_ptr(a), _ptr(out), a.size)
    return out


def attention(q_bits, seq_lens, req_page_ptr, dst_vpages, kv_pools: list[np.ndarray],
              dtype: int, kv_scale: float, softmax_scale: float, n_dcp: int, rank: int = -1,
              rows=None, q_len: int = 1, num_heads: int | None = None, layout: str = "page"):
    """Partial (rank >= 0) or unsharded (rank = -1) attention in float64.  layout "page": entry j
    of a request's table holds positions 64 j + i; "token": entry jj * N + d is rank d's local page
    jj, holding positions (64 jj + i) * N + d.

    q_bits: uint16 BF16 bits [B][T][H][576]; kv_pools: per-rank arrays whose raw bytes are
    [slots][64][576] BF16 (uint16) or E4M3 (uint8).  Returns (o [rows][512], lse [rows]).
    """
    q = _c(q_bits, np.uint16)
    b_count = q.shape[0]
    if num_heads is None:
        num_heads = q.shape[2]
    sl = _c(seq_lens, np.int32)
    rpp = _c(req_page_ptr, np.int64)
    dv = _c(dst_vpages, np.int32)
    pools = [np.ascontiguousarray(p) for p in kv_pools]
    elem = 2 if dtype == BF16 else 1
    slots = pools[0].nbytes // (PAGE_TOKENS * K_DIM * elem)
    for p in pools:
        assert p.nbytes == slots * PAGE_TOKENS * K_DIM * elem
    parr = (ctypes.c_void_p * len(pools))(*[_ptr(p) for p in pools])
    if rows is None:
        n_rows = b_count * q_len * num_heads
        rws = None
    else:
        rws = _c(rows, np.int64)
        n_rows = rws.size
    o = np.zeros((n_rows, V_DIM), np.float64)
    lse = np.zeros(n_rows, np.float64)
    fn = _load().dcpo_attention_tokens if layout == "token" else _load().dcpo_attention
    st = fn(b_count, q_len, num_heads, _ptr(q), _ptr(sl), _ptr(rpp), _ptr(dv),
                                dtype, float(kv_scale), float(softmax_scale), n_dcp,
                                ctypes.addressof(parr), slots, rank,
                                _ptr(rws) if rws is not None else None, n_rows, _ptr(o), _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle attention: page slot out of range (status {st})")
    return o, lse


def lse_merge(o_part, lse_part):
    """Exact LSE merge in float64.  o_part [n][rows][v], lse_part [n][rows]."""
    op = _c(o_part, np.float64)
    lp = _c(lse_part, np.float64)
    n, rows, v = op.shape
    assert lp.shape == (n, rows)
    o = np.empty((rows, v), np.float64)
    lse = np.empty(rows, np.float64)
    _load().dcpo_lse_merge(n, rows, v, _ptr(op), _ptr(lp), _ptr(o), _ptr(lse))
    return o, lse
