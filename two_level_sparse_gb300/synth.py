"""Seeded synthetic inputs for the two-level candidate indexer.

This module only draws random operands and lays them out in the library's
memory format; it holds none of the indexer's arithmetic.  Both the CUDA path
and the CPU oracle consume what it produces.

Operand formats (the ones the DeepSeek-V4.1 indexer pages describe):

* query: MXFP4 -- two e2m1 codes per byte (element ``2i`` in the low nibble)
  and one ue8m0 scale byte per 32 elements, ``q_fp4[rows, H, D/2]`` and
  ``q_sf[rows, H, D/32]`` (vLLM ``sparse_attn_indexer.py``, "MXFP4 layout"
  comment: 2 values per byte, ue8m0 scale per block of 32);
* head weights ``w[rows, H]`` fp32;
* index-K: FP8 e4m3 values plus one fp32 scale per position, stored in pages of
  64 positions.  One page is ``64*128`` value bytes followed by ``64`` little-
  endian fp32 scales (8448 bytes).  Pages sit in a pool in a random physical
  order behind an int32 page table ``page_table[num_req, max_pages]``
  (vLLM ``sparse_attn_indexer.py``, K-gather workspace: ``(T, head_dim)`` fp8
  values + ``(T, 4)`` bytes of fp32 scale per position);
* index-K, MXFP4 variant (the same file's ``use_fp4_cache`` path: ``head_dim
  / 2`` packed bytes and ``head_dim / 32`` ue8m0 scales per position): a page
  is ``64*64`` bytes of packed e2m1 codes followed by one 32-bit word per
  position whose byte ``j`` scales elements ``32j .. 32j + 31`` (4352 bytes).

Workloads (one source layer + four consumer layers, each with its own q, w and
K pool, one shared page table):

* decode: row ``t`` is request ``t``; its positions live in its own pages;
* prefill: every row belongs to one request; row ``t`` reaches ``L_t``
  positions of the shared pages (causal).
"""
from __future__ import annotations

import dataclasses
import math

import torch

H = 64
D = 128
BLOCK = 8
PAGE = 64
PAGE_VALUE_BYTES = PAGE * D
PAGE_BYTES = PAGE * D + PAGE * 4
KV_FP8, KV_MXFP4 = 0, 1
PAGE_VALUE_BYTES_MXFP4 = PAGE * D // 2
PAGE_BYTES_MXFP4 = PAGE_VALUE_BYTES_MXFP4 + PAGE * 4
LAYOUT_DECODE = 0
LAYOUT_PREFILL = 1
LAYOUT_VARLEN = 2  # a prefill chunk of several requests: rows req_start[r] .. req_start[r + 1] - 1 are request r
TOPK_POSITIONS = 512


@dataclasses.dataclass
class Layer:
    q_fp4: torch.Tensor  # uint8 [rows, H, D/2]
    q_sf: torch.Tensor  # uint8 [rows, H, D/32]
    w: torch.Tensor  # float32 [rows, H]
    k_pool: torch.Tensor  # uint8 [num_pages, PAGE_BYTES]


@dataclasses.dataclass
class Workload:
    name: str
    layout: int
    seq_len: torch.Tensor  # int32 [rows]
    page_table: torch.Tensor  # int32 [num_req, max_pages]
    layers: list  # [source, consumer_1, ..., consumer_4]
    topk_blocks: int
    topk: int = TOPK_POSITIONS
    req_start: torch.Tensor = None  # int32 [num_req + 1] (LAYOUT_VARLEN only)

    def row_req(self):
        """numpy int64 [rows]: the request of every row (LAYOUT_VARLEN), else None."""
        if self.layout != LAYOUT_VARLEN:
            return None
        import numpy as np

        starts = self.req_start.cpu().numpy().astype(np.int64)
        return np.repeat(np.arange(len(starts) - 1), np.diff(starts))

    @property
    def rows(self) -> int:
        return int(self.seq_len.shape[0])

    @property
    def max_len(self) -> int:
        return int(self.seq_len.max().item()) if self.rows else 0

    @property
    def num_pages(self) -> int:
        return int(self.layers[0].k_pool.shape[0])

    @property
    def kv(self) -> int:
        return KV_MXFP4 if int(self.layers[0].k_pool.shape[1]) == PAGE_BYTES_MXFP4 else KV_FP8

    def to(self, device) -> "Workload":
        mv = lambda t: t.to(device)
        return Workload(
            self.name,
            self.layout,
            mv(self.seq_len),
            mv(self.page_table),
            [Layer(mv(l.q_fp4), mv(l.q_sf), mv(l.w), mv(l.k_pool)) for l in self.layers],
            self.topk_blocks,
            self.topk,
            None if self.req_start is None else mv(self.req_start),
        )


def _k_pages(num_pages: int, gen: torch.Generator, device, chunk_pages: int = 2048) -> torch.Tensor:
    """FP8 e4m3 of N(0,1) values and U[0.5, 2) fp32 scales, page by page."""
    pool = torch.empty(num_pages, PAGE_BYTES, dtype=torch.uint8, device=device)
    for p0 in range(0, num_pages, chunk_pages):
        n = min(chunk_pages, num_pages - p0)
        vals = torch.randn(n * PAGE, D, generator=gen, device=device)
        pool[p0 : p0 + n, :PAGE_VALUE_BYTES] = (
            vals.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, PAGE_VALUE_BYTES)
        )
        scale = torch.rand(n, PAGE, generator=gen, device=device) * 1.5 + 0.5
        pool[p0 : p0 + n, PAGE_VALUE_BYTES:] = scale.view(torch.uint8).reshape(n, PAGE * 4)
    return pool


def _k_pages_mxfp4(num_pages: int, gen: torch.Generator, device, chunk_pages: int = 4096) -> torch.Tensor:
    """MXFP4 pages: uniformly random e2m1 codes (both nibbles of every byte)
    and ue8m0 scales with exponents uniform in [-4, 0] (codes 123..127), the
    same distribution as the queries."""
    pool = torch.empty(num_pages, PAGE_BYTES_MXFP4, dtype=torch.uint8, device=device)
    for p0 in range(0, num_pages, chunk_pages):
        n = min(chunk_pages, num_pages - p0)
        pool[p0 : p0 + n, :PAGE_VALUE_BYTES_MXFP4] = torch.randint(
            0, 256, (n, PAGE_VALUE_BYTES_MXFP4), generator=gen, device=device, dtype=torch.uint8)
        pool[p0 : p0 + n, PAGE_VALUE_BYTES_MXFP4:] = torch.randint(
            123, 128, (n, PAGE * 4), generator=gen, device=device, dtype=torch.uint8)
    return pool


def _layer(rows: int, num_pages: int, gen: torch.Generator, device, kv: int = KV_FP8) -> Layer:
    q_fp4 = torch.randint(0, 256, (rows, H, D // 2), generator=gen, device=device, dtype=torch.uint8)
    # ue8m0 exponent uniform in [-4, 0]: codes 123..127
    q_sf = torch.randint(123, 128, (rows, H, D // 32), generator=gen, device=device, dtype=torch.uint8)
    w = torch.randn(rows, H, generator=gen, device=device) * (1.0 / math.sqrt(H))
    pool = _k_pages_mxfp4(num_pages, gen, device) if kv == KV_MXFP4 else _k_pages(num_pages, gen, device)
    return Layer(q_fp4, q_sf, w.float(), pool)


def _duplicate_blocks(layer: Layer, page_table: torch.Tensor, seq_len: torch.Tensor, req_rows,
                      frac: float, gen: torch.Generator) -> None:
    """Overwrite ``frac`` of each request's full, non-newest blocks with a byte
    copy (values and scales) of another such block of the same request."""
    pool = layer.k_pool
    rb = D // 2 if int(pool.shape[1]) == PAGE_BYTES_MXFP4 else D  # value bytes per position
    pvb = PAGE * rb
    for r, L in req_rows:
        nb = (L + BLOCK - 1) // BLOCK
        nfull = nb - 1  # every block but the newest is full
        if nfull < 2:
            continue
        count = max(1, int(math.floor(frac * nfull)))
        dsts = torch.randperm(nfull, generator=gen)[:count].tolist()
        for dst in dsts:
            src = int(torch.randint(0, nfull - 1, (1,), generator=gen).item())
            if src >= dst:
                src += 1
            sp, so = int(page_table[r, src // 8]), (src % 8) * BLOCK
            dp, do = int(page_table[r, dst // 8]), (dst % 8) * BLOCK
            pool[dp, do * rb : (do + BLOCK) * rb] = pool[sp, so * rb : (so + BLOCK) * rb]
            pool[dp, pvb + do * 4 : pvb + (do + BLOCK) * 4] = pool[sp, pvb + so * 4 : pvb + (so + BLOCK) * 4]


def make_workload(name: str, layout: int, seq_len, topk_blocks: int, seed: int, layers: int = 5,
                  dup_frac: float = 0.0, device="cpu", topk: int = TOPK_POSITIONS, kv: int = KV_FP8) -> Workload:
    """Build one workload from explicit per-row lengths."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    seq_len = torch.as_tensor(seq_len, dtype=torch.int32).cpu()
    rows = int(seq_len.shape[0])
    if layout == LAYOUT_DECODE:
        pages_per = [(int(L) + PAGE - 1) // PAGE for L in seq_len.tolist()]
        num_pages = sum(pages_per)
        max_pages = max(pages_per) if pages_per else 0
        perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 7919))
        page_table = torch.full((rows, max(max_pages, 1)), -1, dtype=torch.int32)
        off = 0
        for r, n in enumerate(pages_per):
            page_table[r, :n] = perm[off : off + n].to(torch.int32)
            off += n
        req_rows = [(r, int(L)) for r, L in enumerate(seq_len.tolist())]
    else:
        max_len = int(seq_len.max().item()) if rows else 0
        num_pages = (max_len + PAGE - 1) // PAGE
        page_table = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 7919))
        page_table = page_table.to(torch.int32).reshape(1, max(num_pages, 0))
        if num_pages == 0:
            page_table = torch.full((1, 1), -1, dtype=torch.int32)
        req_rows = [(0, max_len)]
    num_pages = max(num_pages, 1)
    ls = [_layer(rows, num_pages, gen, device, kv) for _ in range(layers)]
    if dup_frac > 0:
        cpu_gen = torch.Generator().manual_seed(seed + 104729)
        for l in ls:
            pool_cpu = l.k_pool.cpu()
            _duplicate_blocks(Layer(l.q_fp4, l.q_sf, l.w, pool_cpu), page_table, seq_len, req_rows, dup_frac,
                              cpu_gen)
            l.k_pool.copy_(pool_cpu)
    return Workload(name, layout, seq_len.to(device), page_table.to(device), ls, topk_blocks, topk)


def make_varlen_workload(name: str, prefixes, rows_per_req, topk_blocks: int, seed: int, layers: int = 5,
                         device="cpu", topk: int = TOPK_POSITIONS, kv: int = KV_FP8) -> Workload:
    """A prefill chunk of several requests: request r contributes
    rows_per_req[r] causal rows after a prefix of prefixes[r] compressed
    positions (row i of the request reaches prefixes[r] + i + 1 positions).
    Every request has its own pages (random physical order) in one pool per
    layer; rows are grouped by request."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lens, starts = [], [0]
    for pre, n in zip(prefixes, rows_per_req):
        lens.extend(int(pre) + i + 1 for i in range(int(n)))
        starts.append(starts[-1] + int(n))
    seq_len = torch.as_tensor(lens, dtype=torch.int32)
    rows = int(seq_len.shape[0])
    pages_per = [(int(pre) + int(n) + PAGE - 1) // PAGE for pre, n in zip(prefixes, rows_per_req)]
    num_pages = max(sum(pages_per), 1)
    max_pages = max(max(pages_per) if pages_per else 0, 1)
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 7919))
    page_table = torch.full((len(pages_per), max_pages), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(pages_per):
        page_table[r, :n] = perm[off : off + n].to(torch.int32)
        off += n
    ls = [_layer(rows, num_pages, gen, device, kv) for _ in range(layers)]
    return Workload(name, LAYOUT_VARLEN, seq_len.to(device), page_table.to(device), ls, topk_blocks, topk,
                    torch.as_tensor(starts, dtype=torch.int32).to(device))


# A multi-request prefill chunk of 16384 rows: four requests of 4096 rows each
# after prefixes of 16 K, 64 K, 128 K and 240 K compressed positions.
VARLEN_CHUNK = dict(name="varlen_prefill_4x4096rows_prefix16k-240k_K2048",
                    prefixes=(16384, 65536, 131072, 245760), rows_per_req=(4096, 4096, 4096, 4096), topk_blocks=2048,
                    seed=5)


def varlen_chunk_workload(device="cpu", layers: int = 5) -> Workload:
    return make_varlen_workload(device=device, layers=layers, **VARLEN_CHUNK)


def _uniform_lengths(rows, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (rows,), generator=g, dtype=torch.int64).to(torch.int32)


def config_lengths(cid: int) -> torch.Tensor:
    """Per-row compressed lengths of the five standard workloads."""
    if cid == 0:
        return _uniform_lengths(4, 1024, 4096, 0)
    if cid == 1:
        return _uniform_lengths(64, 16384, 65536, 1)
    if cid == 2:
        rows = 128
        g = torch.Generator().manual_seed(2)
        n_short = int(math.floor(0.1 * rows + 0.5))
        short = torch.randperm(rows, generator=g)[:n_short]
        L = torch.randint(131072, 262144 + 1, (rows,), generator=g, dtype=torch.int64)
        L[short] = torch.randint(512, 16384 + 1, (n_short,), generator=g, dtype=torch.int64)
        return L.to(torch.int32)
    if cid == 3:
        i = torch.arange(4096, dtype=torch.int64)
        return ((61440 + i + 1) // 4).to(torch.int32)
    if cid == 4:
        i = torch.arange(16384, dtype=torch.int64)
        return (262144 - 16384 + i + 1).to(torch.int32)
    raise ValueError(cid)


CONFIG_NAMES = {
    0: "tiny_decode_4rows_L1k-4k_K128",
    1: "decode_64rows_L16k-64k_K2048",
    2: "long_decode_128rows_L512-256k_K2048",
    3: "prefill_4096rows_prefix61440_K2048",
    4: "prefill_16384rows_ctx262144_K2048",
}
CONFIG_LAYOUT = {0: LAYOUT_DECODE, 1: LAYOUT_DECODE, 2: LAYOUT_DECODE, 3: LAYOUT_PREFILL, 4: LAYOUT_PREFILL}
CONFIG_TOPK_BLOCKS = {0: 128, 1: 2048, 2: 2048, 3: 2048, 4: 2048}


def config_workload(cid: int, device="cpu", layers: int = 5, kv: int = KV_FP8) -> Workload:
    """Standard workload ``cid``; ``kv = KV_MXFP4`` draws MXFP4 pools instead
    of FP8 ones (same lengths, queries and weights; name suffixed)."""
    return make_workload(
        CONFIG_NAMES[cid] + ("_mxfp4" if kv == KV_MXFP4 else ""),
        CONFIG_LAYOUT[cid],
        config_lengths(cid),
        CONFIG_TOPK_BLOCKS[cid],
        seed=cid,
        layers=layers,
        dup_frac=0.05 if cid == 0 else 0.0,
        device=device,
        kv=kv,
    )


def _request_lengths(wl: Workload) -> list:
    """The number of positions each request's pages must hold."""
    L = wl.seq_len.cpu().tolist()
    if wl.layout == LAYOUT_DECODE:
        return L
    if wl.layout == LAYOUT_PREFILL:
        return [max(L) if L else 0]
    starts = wl.req_start.cpu().tolist()
    return [max(L[a:b]) if b > a else 0 for a, b in zip(starts[:-1], starts[1:])]


def shard_workload(wl: Workload, world: int) -> list:
    """The ``world`` context shards of an FP8 workload, interleave 1: global
    position s of a request lives on shard s % world at local position
    s // world (vLLM sparse_attn_indexer.py, two-level candidate filtering
    under DCP).  Each shard gets its own pools and page table holding its
    positions, and the local lengths; queries and weights are replicated.
    Pure data movement (the sharded cache layout), no arithmetic of the
    method."""
    assert wl.kv == KV_FP8
    dev = wl.seq_len.device
    L = wl.seq_len.to(torch.int64)
    req_len = _request_lengths(wl)
    pt = wl.page_table.to(torch.int64)
    shards = []
    for r in range(world):
        local_len = [max(0, (n - r + world - 1) // world) for n in req_len]
        pages = [(n + PAGE - 1) // PAGE for n in local_len]
        num_pages = max(sum(pages), 1)
        lpt = torch.full((len(pages), max(max(pages) if pages else 0, 1)), -1, dtype=torch.int32)
        src_page, src_slot, dst_page, dst_slot = [], [], [], []
        off = 0
        for q, (n, np_) in enumerate(zip(local_len, pages)):
            lpt[q, :np_] = torch.arange(off, off + np_, dtype=torch.int32)
            if n:
                j = torch.arange(n, device=dev)
                s = j * world + r
                src_page.append(pt[q].to(dev)[s // PAGE])
                src_slot.append(s % PAGE)
                dst_page.append(off + j // PAGE)
                dst_slot.append(j % PAGE)
            off += np_
        layers = []
        for l in wl.layers:
            pool = torch.zeros(num_pages, PAGE_BYTES, dtype=torch.uint8, device=dev)
            if src_page:
                sp, ss, dp, ds = (torch.cat(x) for x in (src_page, src_slot, dst_page, dst_slot))
                vals = l.k_pool[:, :PAGE_VALUE_BYTES].reshape(-1, PAGE, D)
                scl = l.k_pool[:, PAGE_VALUE_BYTES:].reshape(-1, PAGE, 4)
                pool[:, :PAGE_VALUE_BYTES].view(-1, PAGE, D)[dp, ds] = vals[sp, ss]
                pool[:, PAGE_VALUE_BYTES:].view(-1, PAGE, 4)[dp, ds] = scl[sp, ss]
            layers.append(Layer(l.q_fp4, l.q_sf, l.w, pool))
        local = torch.clamp(L - r + world - 1, min=0) // world
        shards.append(Workload(f"{wl.name}_shard{r}of{world}", wl.layout, local.to(torch.int32).to(dev),
                               lpt.to(dev), layers, wl.topk_blocks, wl.topk, wl.req_start))
    return shards
