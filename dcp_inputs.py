"""Seeded synthetic inputs shared by the tests, the smoke run and the benchmark.

This module only draws random data and lays it out in the formats the DCP entry points
take; it computes nothing the method computes.  Both the float64 oracle and the CUDA path
consume what it returns.

Recipe (shapes follow the pages' workloads; values are synthetic):

* Q: ``[B][T][H][576]`` BF16, N(0, 1) rounded to nearest-even.
* KV pools: one per DCP rank, ``[slots][64][576]``; BF16 N(0, 1), or FP8-E4M3 of N(0, 1)
  divided by a per-tensor scale ``kv_scale = 8 / 448`` (the E4M3 range then covers +-8
  sigma; values are clamped there before the round-to-nearest-even cast).
* Page table: logical page ``j`` of request ``b`` is owned by rank ``j mod N`` (round-robin
  ownership) and sits in a seeded uniformly random free slot of that rank's pool; the table
  stores the decode-side global page value ``slot * N + owner``.
* Sequence lengths: given per config; the last page of a request may be partly filled, and
  its tail rows hold finite random data like every other row.
* Source (prefill, CP layer-split) pools: ``[layers owned][pages][64][576]`` with random
  content; each request's source pages are contiguous or a seeded random permutation.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE = 64
K_DIM = 576
V_DIM = 512
FP8_KV_SCALE = 8.0 / 448.0
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_into(out: torch.Tensor, gen: torch.Generator, scale: float | None,
                chunk: int = 1 << 27) -> None:
    """Fill ``out`` (bf16 or float8_e4m3fn) with N(0,1) values (divided by ``scale`` for fp8)."""
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        x = torch.randn(n, generator=gen, device=out.device, dtype=torch.float32)
        if out.dtype == torch.float8_e4m3fn:
            x = (x / scale).clamp_(-448.0, 448.0)
        flat[s:s + n] = x.to(out.dtype)


def kv_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}[name]


def random_pool(n_slots: int, dtype: str, gen: torch.Generator, device, layers: int = 0) -> torch.Tensor:
    shape = (n_slots, PAGE, K_DIM) if layers == 0 else (layers, n_slots, PAGE, K_DIM)
    t = torch.empty(shape, dtype=kv_dtype(dtype), device=device)
    _randn_into(t, gen, FP8_KV_SCALE)
    return t


def random_q(b: int, t: int, h: int, gen: torch.Generator, device) -> torch.Tensor:
    q = torch.empty((b, t, h, K_DIM), dtype=torch.bfloat16, device=device)
    _randn_into(q, gen, None)
    return q


def check_page_table(req_page_ptr: torch.Tensor, dst_vpages: torch.Tensor) -> None:
    """Checks a destination page table against the contract the library leaves to its caller:
    CSR offsets non-decreasing from 0 to the table's length, and no page value twice (two
    entries with one value would write, and read, the same pool slot).  Values outside the pools
    are not checked here: the library flags those on the device.  Raises ValueError."""
    ptr = req_page_ptr.detach().to("cpu", torch.int64)
    vp = dst_vpages.detach().to("cpu", torch.int64)
    if ptr.numel() < 1 or int(ptr[0]) != 0 or int(ptr[-1]) != vp.numel():
        raise ValueError("req_page_ptr must run from 0 to the number of page entries")
    if ptr.numel() > 1 and bool((ptr[1:] < ptr[:-1]).any()):
        raise ValueError("req_page_ptr must be non-decreasing")
    if vp.numel() and torch.unique(vp).numel() != vp.numel():
        raise ValueError("a destination page value appears more than once in the table")


def page_table(seq_lens, n_dcp: int, slots_per_rank: int, gen: torch.Generator, with_slots: bool = False):
    """Round-robin ownership with seeded random slots.  Returns (req_page_ptr, dst_vpages), and
    with ``with_slots`` also the owner rank and pool slot the generator chose for every entry
    (int64 CPU tensors), so that tests can address a page's rows without decoding its value."""
    pages = [(int(n) + PAGE - 1) // PAGE for n in seq_lens]
    ptr = [0]
    for p in pages:
        ptr.append(ptr[-1] + p)
    n_ranks = max(n_dcp, 1)
    perms = [torch.randperm(slots_per_rank, generator=gen, device="cpu") for _ in range(n_ranks)]
    used = [0] * n_ranks
    vp = torch.empty(ptr[-1], dtype=torch.int64)
    owners = torch.empty(ptr[-1], dtype=torch.int64)
    slots_of = torch.empty(ptr[-1], dtype=torch.int64)
    k = 0
    for p in pages:
        j = torch.arange(p)
        owner = j % n_ranks
        for d in range(n_ranks):
            sel = owner == d
            cnt = int(sel.sum())
            if used[d] + cnt > slots_per_rank:
                raise ValueError("pool too small for the page table")
            slots = perms[d][used[d]:used[d] + cnt]
            used[d] += cnt
            vp[k:k + p][sel] = slots * n_ranks + d if n_dcp > 1 else slots
            owners[k:k + p][sel] = d
            slots_of[k:k + p][sel] = slots
        k += p
    out = (torch.tensor(ptr, dtype=torch.int64), vp.to(torch.int32))
    check_page_table(*out)
    return out + (owners, slots_of) if with_slots else out


def token_page_table(seq_lens, n_dcp: int, slots_per_rank: int, gen: torch.Generator, with_slots: bool = False):
    """Token-interleaved layout: rank d holds tokens d, d + N, ...; a request's table entry
    jj * N + d names rank d's local page jj at a seeded random free slot.  Every rank gets the
    same number of local pages, ceil(ceil(n / N) / 64).  Returns (req_page_ptr, dst_vpages), and
    with ``with_slots`` also every entry's owner rank and pool slot (int64 CPU tensors)."""
    n_ranks = max(n_dcp, 1)
    local = [-(-(-(-int(n) // n_ranks)) // PAGE) for n in seq_lens]
    perms = [torch.randperm(slots_per_rank, generator=gen, device="cpu") for _ in range(n_ranks)]
    used = [0] * n_ranks
    ptr, vp, owners, slots_of = [0], [], [], []
    for p in local:
        for jj in range(p):
            for d in range(n_ranks):
                if used[d] >= slots_per_rank:
                    raise ValueError("pool too small for the page table")
                slot = int(perms[d][used[d]])
                used[d] += 1
                vp.append(slot * n_ranks + d if n_dcp > 1 else slot)
                owners.append(d)
                slots_of.append(slot)
        ptr.append(ptr[-1] + p * n_ranks)
    out = (torch.tensor(ptr, dtype=torch.int64), torch.tensor(vp, dtype=torch.int32))
    check_page_table(*out)
    if with_slots:
        out += (torch.tensor(owners, dtype=torch.int64), torch.tensor(slots_of, dtype=torch.int64))
    return out


@dataclass
class AttnCase:
    """One partial-attention workload (all tensors on ``device``)."""
    B: int
    T: int
    H: int
    n_dcp: int
    dtype: str
    seq_lens: torch.Tensor          # int32 [B]
    req_page_ptr: torch.Tensor      # int64 [B+1]
    dst_vpages: torch.Tensor        # int32 [pages]
    q: torch.Tensor                 # bf16 [B][T][H][576]
    pools: list                     # per rank [slots][64][576]
    slots_per_rank: int
    kv_scale: float
    softmax_scale: float = SOFTMAX_SCALE
    name: str = ""
    layout: str = "page"            # "token": the table is token-interleaved (token_page_table)
    page_owner: torch.Tensor | None = None  # int64 CPU [pages]: rank whose pool holds each entry
    page_slot: torch.Tensor | None = None   # int64 CPU [pages]: that pool's slot

    @property
    def rows(self) -> int:
        return self.B * self.T * self.H

    @property
    def max_tokens(self) -> int:
        return int(self.seq_lens.max().item()) if self.B else 0


def attention_case(seq_lens, H: int, T: int, n_dcp: int, dtype: str, slots_per_rank: int | None,
                   seed: int, device, name: str = "") -> AttnCase:
    gen_cpu = _gen(seed, "cpu")
    gen_dev = _gen(seed + 1000003, device)
    seq_lens = [int(n) for n in seq_lens]
    n_ranks = max(n_dcp, 1)
    per_rank = [0] * n_ranks
    for n in seq_lens:
        p = (n + PAGE - 1) // PAGE
        for d in range(n_ranks):
            per_rank[d] += (p - d + n_ranks - 1) // n_ranks if p > d else 0
    need = max(per_rank) if per_rank else 0
    if slots_per_rank is None:
        slots_per_rank = max(need, 1)
    ptr, vp, owner, slot = page_table(seq_lens, n_dcp, slots_per_rank, gen_cpu, with_slots=True)
    q = random_q(len(seq_lens), T, H, gen_dev, device)
    pools = [random_pool(slots_per_rank, dtype, gen_dev, device) for _ in range(n_ranks)]
    return AttnCase(B=len(seq_lens), T=T, H=H, n_dcp=n_dcp, dtype=dtype,
                    seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                    req_page_ptr=ptr.to(device), dst_vpages=vp.to(device), q=q, pools=pools,
                    slots_per_rank=slots_per_rank,
                    kv_scale=FP8_KV_SCALE if dtype == "e4m3" else 1.0, name=name, page_owner=owner,
                    page_slot=slot)


@dataclass
class ReshardCase:
    """A CP layer-split -> DCP page-interleaved reshard workload."""
    n_layers: int
    n_cp: int
    n_dcp: int
    dtype: str
    seq_lens: list
    req_page_ptr: torch.Tensor      # int64 [B+1]
    src_pages: torch.Tensor         # int32 [pages]  prefill-side page index
    dst_vpages: torch.Tensor        # int32 [pages]  decode-side global page value
    src_pools: list                 # per CP rank [layers owned][src_pool_pages][64][576]
    src_pool_pages: int
    dst_pools: list                 # per DCP rank [n_layers][slots][64][576]
    dst_slots: int
    layer_counts: list = field(default_factory=list)
    name: str = ""
    page_owner: torch.Tensor | None = None  # int64 CPU [pages]: destination rank of each entry
    page_slot: torch.Tensor | None = None   # int64 CPU [pages]: its slot in that rank's pool

    @property
    def page_bytes(self) -> int:
        return PAGE * K_DIM * (2 if self.dtype == "bf16" else 1)


def token_attention_case(seq_lens, H: int, T: int, n_dcp: int, dtype: str, seed: int, device,
                         name: str = "") -> AttnCase:
    """An attention workload over the token-interleaved layout (token_page_table)."""
    gen_cpu = _gen(seed, "cpu")
    gen_dev = _gen(seed + 1000003, device)
    seq_lens = [int(n) for n in seq_lens]
    n_ranks = max(n_dcp, 1)
    slots = max(1, sum(-(-(-(-n // n_ranks)) // PAGE) for n in seq_lens))
    ptr, vp, owner, slot = token_page_table(seq_lens, n_dcp, slots, gen_cpu, with_slots=True)
    q = random_q(len(seq_lens), T, H, gen_dev, device)
    pools = [random_pool(slots, dtype, gen_dev, device) for _ in range(n_ranks)]
    return AttnCase(B=len(seq_lens), T=T, H=H, n_dcp=n_dcp, dtype=dtype,
                    seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                    req_page_ptr=ptr.to(device), dst_vpages=vp.to(device), q=q, pools=pools, slots_per_rank=slots,
                    kv_scale=FP8_KV_SCALE if dtype == "e4m3" else 1.0, name=name, layout="token",
                    page_owner=owner, page_slot=slot)


SENTINEL_BYTE = 0xA5


def reshard_case(seq_lens, n_layers: int, layer_counts: list, n_dcp: int, dtype: str,
                 contiguous_src: bool, seed: int, device, dst_slots: int | None = None,
                 src_pool_pages: int | None = None, name: str = "") -> ReshardCase:
    """``layer_counts[r]`` = layers held by source rank r (the layer split itself is the
    caller's; the generator only sizes the pools).  Destination pools are filled with the
    sentinel byte so stray or missing writes show."""
    gen_cpu = _gen(seed, "cpu")
    gen_dev = _gen(seed + 1000003, device)
    pages = [(int(n) + PAGE - 1) // PAGE for n in seq_lens]
    total = sum(pages)
    n_ranks = max(n_dcp, 1)
    per_rank = [0] * n_ranks
    for p in pages:
        for d in range(n_ranks):
            per_rank[d] += (p - d + n_ranks - 1) // n_ranks if p > d else 0
    if dst_slots is None:
        dst_slots = max(max(per_rank), 1)
    ptr, vp, owner, slot = page_table(seq_lens, n_dcp, dst_slots, gen_cpu, with_slots=True)
    if src_pool_pages is None:
        src_pool_pages = max(total, 1)
    if contiguous_src:
        src = torch.arange(total, dtype=torch.int32)
    else:
        src = torch.randperm(src_pool_pages, generator=gen_cpu)[:total].to(torch.int32)
    src_pools = [random_pool(src_pool_pages, dtype, gen_dev, device, layers=c) for c in layer_counts]
    dst_pools = []
    for _ in range(n_ranks):
        t = torch.empty((n_layers, dst_slots, PAGE, K_DIM), dtype=kv_dtype(dtype), device=device)
        t.view(torch.uint8).fill_(SENTINEL_BYTE)
        dst_pools.append(t)
    return ReshardCase(n_layers=n_layers, n_cp=len(layer_counts), n_dcp=n_dcp, dtype=dtype,
                       seq_lens=list(seq_lens), req_page_ptr=ptr.to(device),
                       src_pages=src.to(device), dst_vpages=vp.to(device), src_pools=src_pools,
                       src_pool_pages=src_pool_pages, dst_pools=dst_pools, dst_slots=dst_slots,
                       layer_counts=list(layer_counts), name=name, page_owner=owner, page_slot=slot)


def log_uniform_lengths(count: int, lo: int, hi: int, seed: int) -> list:
    """Lengths exp(U[ln lo, ln hi]) rounded to a multiple of 64 (at least 64)."""
    g = _gen(seed, "cpu")
    u = torch.rand(count, generator=g, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [max(PAGE, int(round(float(v) / PAGE)) * PAGE) for v in x]


# The five workloads, by what they are.
def tiny_case(device, seed: int = 0) -> AttnCase:
    """1 request x 1024 tokens (16 pages), 16 heads, q_len 1, BF16, DCP=4."""
    return attention_case([1024], H=16, T=1, n_dcp=4, dtype="bf16", slots_per_rank=4,
                          seed=seed, device=device, name="tiny-1x1024-h16-bf16-dcp4")


def batch_case(device, seed: int = 1) -> AttnCase:
    """32 requests x 8192 tokens, 64 heads, q_len 1, BF16, DCP=8, 512 slots per rank."""
    return attention_case([8192] * 32, H=64, T=1, n_dcp=8, dtype="bf16", slots_per_rank=512,
                          seed=seed, device=device, name="batch-32x8192-h64-bf16-dcp8")


def agent_case(device, seed: int = 2) -> AttnCase:
    """48 requests x 100,000 tokens, 64 heads, q_len 1, FP8, DCP=8 over a ~2.8 GB pool."""
    return attention_case([100_000] * 48, H=64, T=1, n_dcp=8, dtype="e4m3", slots_per_rank=9408,
                          seed=seed, device=device, name="agent-48x100000-h64-fp8-dcp8")


def long_eagle_case(device, seed: int = 3) -> AttnCase:
    """4 requests x 1,048,576 tokens, 64 heads, q_len 4 (causal), FP8, DCP=8."""
    return attention_case([1 << 20] * 4, H=64, T=4, n_dcp=8, dtype="e4m3", slots_per_rank=8192,
                          seed=seed, device=device, name="long-4x1048576-h64-q4-fp8-dcp8")


E2E_LAYERS = 8
E2E_NCP = 4


def e2e_lengths(seed: int = 4) -> list:
    return log_uniform_lengths(64, 2048, 500_000, seed)


def e2e_layer_counts(layer_range) -> list:
    """Layers held by each of the E2E_NCP source ranks under the caller's layer split."""
    return [e - s for s, e in (layer_range(E2E_LAYERS, E2E_NCP, r) for r in range(E2E_NCP))]


def e2e_reshard_case(device, layer_counts: list, seed: int = 1) -> ReshardCase:
    """64 requests of 2K-500K tokens (log-uniform, multiples of 64), 8 layers, CP4 layer-split
    source with each request's pages contiguous, DCP=8 destination, FP8-E4M3."""
    return reshard_case(e2e_lengths(), n_layers=E2E_LAYERS, layer_counts=layer_counts, n_dcp=8, dtype="e4m3",
                        contiguous_src=True, seed=seed, device=device, name="e2e-64x2K-500K-L8-cp4-dcp8-fp8")
