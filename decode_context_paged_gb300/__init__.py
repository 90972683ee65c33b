"""GB300-native decode context parallelism (DCP) hot path: Python binding of libdcp.so.

The three stages of the method run in hand-written sm_103a CUDA kernels behind the C ABI in
``include/dcp.h``; this module only marshals torch tensors (device pointers, sizes, the
current stream) into those calls and turns status codes into exceptions.  There is no CPU
fallback: if ``libdcp.so`` is missing or the GPU is absent the calls raise.

Entry points (same names as the C ABI):
  layer_range              CP layer split ("Serving Macaron-V1 at Scale", 4.1)
  filter_page_indices      source-side page-index filter (6.2, 6.3)
  reshard_pages            CP layer-split -> DCP page reshard, all paths in one launch (2, 6.3, 6.4)
  partial_decode_attn      per-rank paged MLA decode attention -> partial O + LSE (5.2)
  lse_merge                exact LSE merge of the partials (5.2)
  decode_attn_merged       every rank's attention and the merge in one call
  attn_plan                the attention's plan, made once and run per layer (planned=True)
  token_reshard            reshard into the token-interleaved layout ("SGLang's path"); the
                           attention over it: partial_decode_attn / decode_attn_merged(layout="token")
  naive_full_transfer,     the initial design kept as a baseline (6.1): full KV to every DCP rank,
  naive_inplace_shard        then an in-place shard
  pack_pages, unpack_pages one path's pages through a bounded staging buffer (pack_chunks plans it)
  partial_decode_attn_static  the attention without a caller workspace
  selftest_wait_timeout    runs the bounded device wait to its limit (failure-path test)
The host-side multi-rank control (bootstrap, size broadcast, consensus prefix, exchange) is in
``decode_context_paged_gb300.control``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdcp.so")

DCP_OK = 0
DCP_KV_BF16 = 0
DCP_KV_FP8_E4M3 = 1
DEVERR_OUT_OF_RANGE = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_PLAN_MISMATCH = 0x4
DEVERR_LAYOUT = 0x8
PAGE = 64
K_DIM = 576
V_DIM = 512

_lib = None


class DcpError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "(nvcc, sm_103a); there is no fallback path")
        lib = ctypes.CDLL(LIB_PATH)
        i32, i64, f32, vp, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
        lib.dcp_version.restype = i32
        lib.dcp_status_string.argtypes = [i32]
        lib.dcp_status_string.restype = ctypes.c_char_p
        lib.dcp_device_error_status.argtypes = [ctypes.c_int32]
        lib.dcp_device_error_status.restype = i32
        lib.dcp_layer_range.argtypes = [i32, i32, i32, vp, vp]
        lib.dcp_layer_range.restype = i32
        lib.dcp_filter_page_indices.argtypes = [i64, vp, vp, i32, i32, vp, vp, vp, vp]
        lib.dcp_token_reshard.argtypes = [i32, vp, vp, vp, vp, i64, vp, i32, i32, i32, vp, i64, i32, vp, i64, vp, vp]
        lib.dcp_token_reshard.restype = i32
        lib.dcp_naive_full_transfer.argtypes = [i64, vp, i32, i32, i32, vp, i64, i32, vp, vp, vp]
        lib.dcp_naive_full_transfer.restype = i32
        lib.dcp_naive_inplace_shard.argtypes = [i64, vp, i32, i32, i32, vp, vp, i64, vp, vp]
        lib.dcp_naive_inplace_shard.restype = i32
        lib.dcp_pack_pages.argtypes = [i64, vp, i32, i64, i64, i32, vp, i64, vp, sz, vp, vp]
        lib.dcp_pack_pages.restype = i32
        lib.dcp_unpack_pages.argtypes = [i64, vp, i32, i32, i64, i64, i32, vp, sz, vp, i32, i64, vp, vp]
        lib.dcp_unpack_pages.restype = i32
        lib.dcp_filter_page_indices.restype = i32
        lib.dcp_reshard_pages.argtypes = [i32, vp, i64, vp, vp, i32, i32, i32, i32, i32, vp, i64, i32,
                                          vp, i64, i32, i32, vp, vp]
        lib.dcp_reshard_pages.restype = i32
        lib.dcp_partial_decode_attn_workspace_size.argtypes = [i32, i32, i32, i32, i64]
        lib.dcp_partial_decode_attn_workspace_size.restype = sz
        lib.dcp_partial_decode_attn.argtypes = [i32, i32, i32, vp, vp, vp, i64, vp, i32, i32, f32, f32, i32,
                                                vp, i64, i32, vp, vp, vp, sz, vp, vp]
        lib.dcp_partial_decode_attn.restype = i32
        lib.dcp_partial_decode_attn_tokens.argtypes = lib.dcp_partial_decode_attn.argtypes
        lib.dcp_partial_decode_attn_tokens.restype = i32
        lib.dcp_partial_decode_attn_run.argtypes = lib.dcp_partial_decode_attn.argtypes
        lib.dcp_partial_decode_attn_run.restype = i32
        lib.dcp_attn_plan.argtypes = [i32, i32, i32, vp, i64, vp, i32, i32, i64, i32, vp, sz, vp, vp]
        lib.dcp_attn_plan.restype = i32
        lib.dcp_attn_plan_info.argtypes = [i32, i32, i32, i64, i32, i32, vp, sz, vp, vp]
        lib.dcp_attn_plan_info.restype = i32
        lib.dcp_partial_decode_attn_static.argtypes = [i32, i32, i32, vp, vp, vp, i64, vp, i32, i32, f32, f32,
                                                       i32, vp, i64, i32, vp, vp, vp, vp]
        lib.dcp_partial_decode_attn_static.restype = i32
        lib.dcp_decode_attn_merged.argtypes = [i32, i32, i32, vp, vp, vp, i64, vp, i32, i32, f32, f32, i32, vp,
                                               i64, vp, vp, vp, vp, vp, sz, vp, vp]
        lib.dcp_decode_attn_merged.restype = i32
        lib.dcp_decode_attn_merged_run.argtypes = lib.dcp_decode_attn_merged.argtypes
        lib.dcp_decode_attn_merged_run.restype = i32
        lib.dcp_decode_attn_merged_tokens.argtypes = lib.dcp_decode_attn_merged.argtypes
        lib.dcp_decode_attn_merged_tokens.restype = i32
        lib.dcp_lse_merge.argtypes = [i32, i64, i32, vp, vp, vp, vp, vp]
        lib.dcp_lse_merge.restype = i32
        lib.dcp_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp, vp]
        lib.dcp_selftest_wait_timeout.restype = i32
        _lib = lib
    return _lib


def library():
    """The loaded ctypes handle of libdcp.so."""
    return _load()


def version() -> int:
    return int(_load().dcp_version())


def status_string(status: int) -> str:
    return _load().dcp_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != DCP_OK:
        raise DcpError(status, what)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _dptr(t: torch.Tensor | None, name: str, dtype=None, device=True) -> int | None:
    if t is None:
        return None
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _kv_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DCP_KV_BF16
    if t.dtype == torch.float8_e4m3fn:
        return DCP_KV_FP8_E4M3
    raise ValueError(f"KV pools must be bfloat16 or float8_e4m3fn, got {t.dtype}")


def _ptr_array(tensors, name) -> ctypes.Array:
    return (ctypes.c_void_p * len(tensors))(*[_dptr(t, f"{name}[{i}]") for i, t in enumerate(tensors)])


def _check_pools(kv_pools) -> tuple[int, int]:
    """Every pool [slots][64][576] of one dtype; returns (slots, dtype code)."""
    if not kv_pools:
        raise ValueError("kv_pools is empty")
    slots = kv_pools[0].shape[0]
    dtype = _kv_code(kv_pools[0])
    for p in kv_pools:
        if p.shape != (slots, PAGE, K_DIM) or p.dtype != kv_pools[0].dtype:
            raise ValueError("every kv pool must be [slots][64][576] of one dtype")
    return slots, dtype


def _check_out(t: torch.Tensor | None, shape: tuple, name: str) -> None:
    """A caller-supplied output must be fp32 of exactly this shape (the kernels write all of it)."""
    if t is not None and (tuple(t.shape) != tuple(shape) or t.dtype != torch.float32):
        raise ValueError(f"{name} must be float32 {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def _pool_pages(t: torch.Tensor, name: str) -> tuple[int, int]:
    """(layers, pages) of a pool [layers][pages][64][576] (or [pages][64][576] as one layer)."""
    if t.dim() == 4 and tuple(t.shape[2:]) == (PAGE, K_DIM):
        return t.shape[0], t.shape[1]
    if t.dim() == 3 and tuple(t.shape[1:]) == (PAGE, K_DIM):
        return 1, t.shape[0]
    raise ValueError(f"{name} must be [layers][pages][64][576]")


def device_error_status(word: int) -> int:
    return int(_load().dcp_device_error_status(int(word)))


def layer_range(n_layers: int, n_cp: int, r: int) -> tuple[int, int]:
    s, e = ctypes.c_int(0), ctypes.c_int(0)
    _check(_load().dcp_layer_range(n_layers, n_cp, r, ctypes.addressof(s), ctypes.addressof(e)),
           "dcp_layer_range")
    return s.value, e.value


def filter_page_indices(dst_vpages: torch.Tensor, n_dcp: int, d: int,
                        transfer_idx: torch.Tensor | None = None, stream=None):
    """Returns (slots, src or None, count tensor); the first ``count`` entries are valid."""
    n = dst_vpages.numel()
    out_slot = torch.empty(max(n, 1), dtype=torch.int32, device=dst_vpages.device)
    out_src = torch.empty_like(out_slot) if transfer_idx is not None else None
    count = torch.zeros(1, dtype=torch.int64, device=dst_vpages.device)
    _check(_load().dcp_filter_page_indices(n, _dptr(dst_vpages, "dst_vpages", torch.int32),
                                           _dptr(transfer_idx, "transfer_idx", torch.int32), n_dcp, d,
                                           _dptr(out_slot, "out_slot"), _dptr(out_src, "out_src"),
                                           _dptr(count, "count"), _stream(stream)),
           "dcp_filter_page_indices")
    return out_slot, out_src, count


def token_reshard(seq_lens: torch.Tensor, src_page_ptr: torch.Tensor, src_pages: torch.Tensor,
                  tok_page_ptr: torch.Tensor, tok_vpages: torch.Tensor, num_layers: int, src_pools: list,
                  src_pool_pages: int, dst_pools: list, dst_slots_per_rank: int, dev_error: torch.Tensor | None = None,
                  stream=None) -> None:
    """Row gather into the token-interleaved layout (rank d holds tokens d, d + N, ...)."""
    dtype = _kv_code(src_pools[0])
    sp = _ptr_array(src_pools, "src_pools")
    dp = _ptr_array(dst_pools, "dst_pools")
    _check(_load().dcp_token_reshard(seq_lens.numel(), _dptr(seq_lens, "seq_lens", torch.int32),
                                     _dptr(src_page_ptr, "src_page_ptr", torch.int64),
                                     _dptr(src_pages, "src_pages", torch.int32),
                                     _dptr(tok_page_ptr, "tok_page_ptr", torch.int64), tok_vpages.numel(),
                                     _dptr(tok_vpages, "tok_vpages", torch.int32), dtype, num_layers, len(src_pools),
                                     ctypes.addressof(sp), src_pool_pages, len(dst_pools), ctypes.addressof(dp),
                                     dst_slots_per_rank, _dptr(dev_error, "dev_error", torch.int32), _stream(stream)),
           "dcp_token_reshard")


def naive_full_transfer(src_pages: torch.Tensor, num_layers: int, src_pools: list, src_pool_pages: int,
                        recv_bufs: list, dev_error: torch.Tensor | None = None, stream=None) -> None:
    """Baseline: every page of every layer to every DCP rank's receive buffer [L][pages][64][576]."""
    dtype = _kv_code(src_pools[0])
    sp = _ptr_array(src_pools, "src_pools")
    rp = _ptr_array(recv_bufs, "recv_bufs")
    _check(_load().dcp_naive_full_transfer(src_pages.numel(), _dptr(src_pages, "src_pages", torch.int32), dtype,
                                           num_layers, len(src_pools), ctypes.addressof(sp), src_pool_pages,
                                           len(recv_bufs), ctypes.addressof(rp),
                                           _dptr(dev_error, "dev_error", torch.int32), _stream(stream)),
           "dcp_naive_full_transfer")


def naive_inplace_shard(dst_vpages: torch.Tensor, num_layers: int, recv_bufs: list, dst_pools: list,
                        dst_slots_per_rank: int, dev_error: torch.Tensor | None = None, stream=None) -> None:
    """Baseline: each rank keeps the pages it owns from its full copy, at their DCP slots."""
    dtype = _kv_code(dst_pools[0])
    rp = _ptr_array(recv_bufs, "recv_bufs")
    dp = _ptr_array(dst_pools, "dst_pools")
    _check(_load().dcp_naive_inplace_shard(dst_vpages.numel(), _dptr(dst_vpages, "dst_vpages", torch.int32), dtype,
                                           num_layers, len(dst_pools), ctypes.addressof(rp), ctypes.addressof(dp),
                                           dst_slots_per_rank, _dptr(dev_error, "dev_error", torch.int32),
                                           _stream(stream)),
           "dcp_naive_inplace_shard")


def pack_chunks(n_items: int, page_bytes: int, staging_bytes: int) -> list:
    """Item ranges (begin, count) of a path's bounded pack: as many whole pages per chunk as the
    staging buffer holds; one chunk when everything fits."""
    per = staging_bytes // page_bytes
    if per < 1:
        raise ValueError("the staging buffer holds no page")
    return [(b, min(per, n_items - b)) for b in range(0, n_items, per)]


def pack_pages(src_idx: torch.Tensor, n_idx: int, n_layers: int, item_begin: int, n_items: int,
               src_pool: torch.Tensor, staging: torch.Tensor, dev_error: torch.Tensor | None = None,
               stream=None) -> None:
    """Bounded-pack send side of one path: items [item_begin, item_begin + n_items) (layer-major
    over the first n_idx entries of src_idx) from src_pool [n_layers][pages][64][576] into staging."""
    dtype = _kv_code(src_pool)
    _check(_load().dcp_pack_pages(n_idx, _dptr(src_idx, "src_idx", torch.int32), n_layers, item_begin, n_items,
                                  dtype, _dptr(src_pool, "src_pool"), src_pool.shape[1], _dptr(staging, "staging"),
                                  staging.numel() * staging.element_size(), _dptr(dev_error, "dev_error", torch.int32),
                                  _stream(stream)),
           "dcp_pack_pages")


def unpack_pages(dst_slot: torch.Tensor, n_idx: int, n_layers: int, layer_offset: int, item_begin: int,
                 n_items: int, staging: torch.Tensor, dst_pool: torch.Tensor, dev_error: torch.Tensor | None = None,
                 stream=None) -> None:
    """Bounded-pack receive side: the same items from staging into dst_pool
    [num_layers][slots][64][576] at layer layer_offset + j, slot dst_slot[i]."""
    dtype = _kv_code(dst_pool)
    _check(_load().dcp_unpack_pages(n_idx, _dptr(dst_slot, "dst_slot", torch.int32), n_layers, layer_offset,
                                    item_begin, n_items, dtype, _dptr(staging, "staging"),
                                    staging.numel() * staging.element_size(), _dptr(dst_pool, "dst_pool"),
                                    dst_pool.shape[0], dst_pool.shape[1], _dptr(dev_error, "dev_error", torch.int32),
                                    _stream(stream)),
           "dcp_unpack_pages")


def reshard_pages(req_page_ptr: torch.Tensor, src_pages: torch.Tensor, dst_vpages: torch.Tensor,
                  num_layers: int, src_pools: list, src_pool_pages: int, dst_pools: list,
                  dst_slots_per_rank: int, n_dcp: int | None = None, only_src_rank: int = -1,
                  only_dst_rank: int = -1, dev_error: torch.Tensor | None = None, stream=None) -> None:
    """Page-level reshard (all (r, d) paths in one launch); dst_pools are written in place."""
    dtype = _kv_code(src_pools[0])
    n_dcp = len(dst_pools) if n_dcp is None else n_dcp
    if n_dcp > len(dst_pools):
        raise ValueError(f"n_dcp = {n_dcp} but only {len(dst_pools)} destination pools")
    n_cp = len(src_pools)
    for r, p in enumerate(src_pools):
        lay, pages = _pool_pages(p, f"src_pools[{r}]")
        s0 = (num_layers // n_cp) * r + min(r, num_layers % n_cp)  # rank r's share of the layers
        need = num_layers // n_cp + (1 if r < num_layers % n_cp else 0)
        # the library addresses layer l of the pool at l * src_pool_pages pages
        if (p.dtype != src_pools[0].dtype or lay < need or src_pool_pages > pages
                or (need > 1 and src_pool_pages != pages)):
            raise ValueError(f"src_pools[{r}] must be [{need}][src_pool_pages = {src_pool_pages}][64][576] "
                             f"(layers from {s0}), got {tuple(p.shape)} {p.dtype}")
    for d, p in enumerate(dst_pools[:n_dcp]):
        lay, pages = _pool_pages(p, f"dst_pools[{d}]")
        if (p.dtype != src_pools[0].dtype or lay < num_layers or dst_slots_per_rank > pages
                or (num_layers > 1 and dst_slots_per_rank != pages)):
            raise ValueError(f"dst_pools[{d}] must be [{num_layers}][dst_slots_per_rank = {dst_slots_per_rank}]"
                             f"[64][576], got {tuple(p.shape)} {p.dtype}")
    sp = _ptr_array(src_pools, "src_pools")
    dp = _ptr_array(dst_pools, "dst_pools")
    _check(_load().dcp_reshard_pages(req_page_ptr.numel() - 1, _dptr(req_page_ptr, "req_page_ptr", torch.int64),
                                     dst_vpages.numel(), _dptr(src_pages, "src_pages", torch.int32),
                                     _dptr(dst_vpages, "dst_vpages", torch.int32), PAGE, K_DIM, dtype,
                                     num_layers, len(src_pools), ctypes.addressof(sp), src_pool_pages,
                                     n_dcp, ctypes.addressof(dp), dst_slots_per_rank, only_src_rank,
                                     only_dst_rank, _dptr(dev_error, "dev_error", torch.int32),
                                     _stream(stream)),
           "dcp_reshard_pages")


def workspace_size(num_requests: int, q_len: int, num_heads: int, n_dcp: int, num_pages: int) -> int:
    return int(_load().dcp_partial_decode_attn_workspace_size(num_requests, q_len, num_heads, n_dcp,
                                                              num_pages))


def alloc_workspace(num_requests: int, q_len: int, num_heads: int, n_dcp: int, num_pages: int,
                    device) -> torch.Tensor:
    n = workspace_size(num_requests, q_len, num_heads, n_dcp, num_pages)
    if n == 0:
        raise DcpError(-1, "dcp_partial_decode_attn_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def partial_decode_attn(q: torch.Tensor, seq_lens: torch.Tensor, req_page_ptr: torch.Tensor,
                        dst_vpages: torch.Tensor, kv_pools: list, softmax_scale: float,
                        kv_scale: float = 1.0, only_rank: int = -1, o_part: torch.Tensor | None = None,
                        lse_part: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        dev_error: torch.Tensor | None = None, stream=None, layout: str = "page",
                        planned: bool = False):
    """Per-rank partial attention.  q: bf16 [B][T][H][576]; kv_pools: per-rank [slots][64][576].
    layout "token": the page table is token-interleaved (dcp_partial_decode_attn_tokens).
    planned: run the plan attn_plan stored in ``workspace`` (dcp_partial_decode_attn_run).
    Returns (o_part [N][B][T][H][512] fp32, lse_part [N][B][T][H] fp32)."""
    B, T, H, kd = q.shape
    if kd != K_DIM:
        raise ValueError("q must be [B][T][H][576]")
    N = len(kv_pools)
    slots, dtype = _check_pools(kv_pools)
    _check_out(o_part, (N, B, T, H, V_DIM), "o_part")
    _check_out(lse_part, (N, B, T, H), "lse_part")
    dev = q.device
    if o_part is None:
        o_part = torch.empty((N, B, T, H, V_DIM), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((N, B, T, H), dtype=torch.float32, device=dev)
    num_pages = dst_vpages.numel()
    if workspace is None:
        workspace = alloc_workspace(B, T, H, N, num_pages, dev)
    kp = _ptr_array(kv_pools, "kv_pools")
    if planned and (workspace is None or layout == "token"):
        raise ValueError("a planned run needs the workspace holding the plan (page layout)")
    fn = (_load().dcp_partial_decode_attn_run if planned else
          _load().dcp_partial_decode_attn_tokens if layout == "token" else _load().dcp_partial_decode_attn)
    _check(fn(B, T, H, _dptr(q, "q", torch.bfloat16),
                                           _dptr(seq_lens, "seq_lens", torch.int32),
                                           _dptr(req_page_ptr, "req_page_ptr", torch.int64), num_pages,
                                           _dptr(dst_vpages, "dst_vpages", torch.int32), PAGE, dtype,
                                           float(kv_scale), float(softmax_scale), N, ctypes.addressof(kp),
                                           slots, only_rank, _dptr(o_part, "o_part", torch.float32),
                                           _dptr(lse_part, "lse_part", torch.float32),
                                           _dptr(workspace, "workspace"), workspace.numel(),
                                           _dptr(dev_error, "dev_error", torch.int32), _stream(stream)),
           "dcp_partial_decode_attn")
    return o_part, lse_part


def attn_plan(q_shape: tuple, req_page_ptr: torch.Tensor, dst_vpages: torch.Tensor, kv_pools: list,
              workspace: torch.Tensor, only_rank: int = -1, dev_error: torch.Tensor | None = None, stream=None) -> None:
    """The attention's plan for this page table into ``workspace`` (dcp_attn_plan); q_shape =
    (B, T, H); kv_pools give the DCP size, slots per rank and dtype."""
    B, T, H = q_shape[:3]
    _check_pools(kv_pools)
    _check(_load().dcp_attn_plan(B, T, H, _dptr(req_page_ptr, "req_page_ptr", torch.int64), dst_vpages.numel(),
                                 _dptr(dst_vpages, "dst_vpages", torch.int32), _kv_code(kv_pools[0]), len(kv_pools),
                                 kv_pools[0].shape[0], only_rank, _dptr(workspace, "workspace"), workspace.numel(),
                                 _dptr(dev_error, "dev_error", torch.int32), _stream(stream)),
           "dcp_attn_plan")


def attn_plan_info(q_shape: tuple, num_pages: int, kv_pools: list, workspace: torch.Tensor, stream=None) -> dict:
    """The header of the plan in ``workspace`` (dcp_attn_plan_info, synchronous): work units in
    the queue, (rank, request) pairs split into several pieces, tiles per chunk, and whether the
    workspace holds a plan at all."""
    B, T, H = q_shape[:3]
    _check_pools(kv_pools)
    info = (ctypes.c_int32 * 4)()
    _check(_load().dcp_attn_plan_info(B, T, H, int(num_pages), _kv_code(kv_pools[0]), len(kv_pools),
                                      _dptr(workspace, "workspace"), workspace.numel(), ctypes.addressof(info),
                                      _stream(stream)),
           "dcp_attn_plan_info")
    return {"units": info[0], "split_pairs": info[1], "tiles_per_chunk": info[2], "valid": bool(info[3])}


def decode_attn_merged(q: torch.Tensor, seq_lens: torch.Tensor, req_page_ptr: torch.Tensor,
                       dst_vpages: torch.Tensor, kv_pools: list, softmax_scale: float, kv_scale: float = 1.0,
                       o_part: torch.Tensor | None = None, lse_part: torch.Tensor | None = None,
                       o_out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, dev_error: torch.Tensor | None = None, stream=None,
                       planned: bool = False, layout: str = "page"):
    """Every rank's partial attention plus their exact LSE merge in one call (planned: run the
    plan attn_plan stored in ``workspace``, dcp_decode_attn_merged_run; layout "token": the page
    table is token-interleaved, dcp_decode_attn_merged_tokens).
    Returns (o_out [B][T][H][512], lse_out [B][T][H], o_part, lse_part), all fp32."""
    if layout not in ("page", "token"):
        raise ValueError("layout must be 'page' or 'token'")
    if planned and (workspace is None or layout == "token"):
        raise ValueError("a planned run needs the workspace holding the plan (page layout)")
    B, T, H, kd = q.shape
    if kd != K_DIM:
        raise ValueError("q must be [B][T][H][576]")
    N = len(kv_pools)
    slots, dtype = _check_pools(kv_pools)
    _check_out(o_part, (N, B, T, H, V_DIM), "o_part")
    _check_out(lse_part, (N, B, T, H), "lse_part")
    dev = q.device
    if o_part is None:
        o_part = torch.empty((N, B, T, H, V_DIM), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((N, B, T, H), dtype=torch.float32, device=dev)
    _check_out(o_out, (B, T, H, V_DIM), "o_out")
    _check_out(lse_out, (B, T, H), "lse_out")
    if o_out is None:
        o_out = torch.empty((B, T, H, V_DIM), dtype=torch.float32, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    num_pages = dst_vpages.numel()
    if workspace is None:
        workspace = alloc_workspace(B, T, H, N, num_pages, dev)
    kp = _ptr_array(kv_pools, "kv_pools")
    fn = (_load().dcp_decode_attn_merged_run if planned else
          _load().dcp_decode_attn_merged_tokens if layout == "token" else _load().dcp_decode_attn_merged)
    _check(fn(B, T, H, _dptr(q, "q", torch.bfloat16),
                                          _dptr(seq_lens, "seq_lens", torch.int32),
                                          _dptr(req_page_ptr, "req_page_ptr", torch.int64), num_pages,
                                          _dptr(dst_vpages, "dst_vpages", torch.int32), PAGE, dtype,
                                          float(kv_scale), float(softmax_scale), N, ctypes.addressof(kp), slots,
                                          _dptr(o_part, "o_part", torch.float32),
                                          _dptr(lse_part, "lse_part", torch.float32),
                                          _dptr(o_out, "o_out", torch.float32),
                                          _dptr(lse_out, "lse_out", torch.float32),
                                          _dptr(workspace, "workspace"), workspace.numel(),
                                          _dptr(dev_error, "dev_error", torch.int32), _stream(stream)),
           "dcp_decode_attn_merged")
    return o_out, lse_out, o_part, lse_part


def partial_decode_attn_static(q: torch.Tensor, seq_lens: torch.Tensor, req_page_ptr: torch.Tensor,
                               dst_vpages: torch.Tensor, kv_pools: list, softmax_scale: float,
                               kv_scale: float = 1.0, only_rank: int = -1, o_part: torch.Tensor | None = None,
                               lse_part: torch.Tensor | None = None, dev_error: torch.Tensor | None = None,
                               stream=None):
    """Same as partial_decode_attn, for callers that cannot allocate device memory: the call
    uses the library's fixed device scratch array instead of a workspace.  The outputs must be
    passed in by such callers (they are only allocated here when omitted, for convenience)."""
    B, T, H, kd = q.shape
    if kd != K_DIM:
        raise ValueError("q must be [B][T][H][576]")
    N = len(kv_pools)
    slots, dtype = _check_pools(kv_pools)
    _check_out(o_part, (N, B, T, H, V_DIM), "o_part")
    _check_out(lse_part, (N, B, T, H), "lse_part")
    dev = q.device
    if o_part is None:
        o_part = torch.empty((N, B, T, H, V_DIM), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((N, B, T, H), dtype=torch.float32, device=dev)
    kp = _ptr_array(kv_pools, "kv_pools")
    _check(_load().dcp_partial_decode_attn_static(B, T, H, _dptr(q, "q", torch.bfloat16),
                                                  _dptr(seq_lens, "seq_lens", torch.int32),
                                                  _dptr(req_page_ptr, "req_page_ptr", torch.int64),
                                                  dst_vpages.numel(), _dptr(dst_vpages, "dst_vpages", torch.int32),
                                                  PAGE, dtype, float(kv_scale), float(softmax_scale), N,
                                                  ctypes.addressof(kp), slots, only_rank,
                                                  _dptr(o_part, "o_part", torch.float32),
                                                  _dptr(lse_part, "lse_part", torch.float32),
                                                  _dptr(dev_error, "dev_error", torch.int32), _stream(stream)),
           "dcp_partial_decode_attn_static")
    return o_part, lse_part


def lse_merge(o_part: torch.Tensor, lse_part: torch.Tensor, o_out: torch.Tensor | None = None,
              lse_out: torch.Tensor | None = None, stream=None):
    """Merge [N][rows...][v] partials into [rows...][v]; returns (o, lse)."""
    n = o_part.shape[0]
    v = o_part.shape[-1]
    rows = lse_part[0].numel()
    if o_part.numel() != n * rows * v:
        raise ValueError("o_part / lse_part shapes disagree")
    for t, want, name in ((o_out, rows * v, "o_out"), (lse_out, rows, "lse_out")):
        if t is not None and (t.numel() != want or t.dtype != torch.float32):
            raise ValueError(f"{name} must be float32 with {want} elements")
    if o_out is None:
        o_out = torch.empty(o_part.shape[1:], dtype=torch.float32, device=o_part.device)
    if lse_out is None:
        lse_out = torch.empty(lse_part.shape[1:], dtype=torch.float32, device=o_part.device)
    _check(_load().dcp_lse_merge(n, rows, v, _dptr(o_part, "o_part", torch.float32),
                                 _dptr(lse_part, "lse_part", torch.float32),
                                 _dptr(o_out, "o_out", torch.float32), _dptr(lse_out, "lse_out", torch.float32),
                                 _stream(stream)),
           "dcp_lse_merge")
    return o_out, lse_out


def selftest_wait_timeout(limit_ns: int, dev_error: torch.Tensor, out_ok: torch.Tensor, stream=None) -> None:
    """Run the library's bounded pipeline wait on a barrier nothing completes (see dcp.h):
    afterwards dev_error has DEVERR_TIMEOUT set and out_ok holds 0."""
    _check(_load().dcp_selftest_wait_timeout(int(limit_ns), _dptr(dev_error, "dev_error", torch.int32),
                                             _dptr(out_ok, "out_ok", torch.int32), _stream(stream)),
           "dcp_selftest_wait_timeout")
