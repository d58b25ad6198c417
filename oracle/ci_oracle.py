"""CPU oracle for the DeepSeek-V4.1 two-level candidate indexer.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library: it decodes the quantized operands exactly, scores in float64
with plain numpy, takes block maxima, and selects by full sorts.

What it computes follows these passages:

* score -- ``logit[t, s] = sum_h w[t, h] * ReLU(q[t, h] . k[s])`` over every
  reachable compressed position ``s < L_t`` (sglang PR #40352 "Score prefill
  consumer index layers on candidate blocks with DeepGEMM", Motivation and
  Design; vLLM ``sparse_attn_indexer.py``, the ``fp8_fp4_mqa_logits`` and
  ``fp8_fp4_paged_mqa_logits`` calls).  The per-position fp32 K scale
  multiplies the decoded e4m3 vector; the ue8m0 query scale multiplies each
  32-element block of the decoded e2m1 query (same file, "MXFP4 layout"
  comment and ``_gather_workspace_shapes``).  With the MXFP4 index-K cache
  (the same file's ``use_fp4_cache`` path: ``head_dim / 2`` packed bytes and
  ``head_dim / 32`` ue8m0 scales per position) K is decoded exactly like the
  query and there is no per-position scale (it is 1).
* level one -- one key per block of 8 positions, the maximum score inside the
  block; the row's newest block is forced to +inf so it is always kept; rows
  with at most ``K`` blocks keep every block (PR #40352, Design, "Level one";
  the ``block_amax.cuh`` listing in the review of the same PR states the
  contract: ``amax[b, i] = max(scores[b, 8i : 8i + 8])`` for
  ``i < ceil(L_b / 8)``, the last key +inf, rows with ``<= topk`` blocks
  skipped).  The kept block ids are returned ascending, padded with INT32_MAX.
* level two -- a consumer layer scores only positions inside the candidate
  blocks and below ``L_t`` and keeps its top-512, returned ascending, ``-1``
  past ``min(512, valid)`` (PR #40352, Design, "Level two").
* the source layer's own top-512 is the plain dense top-512 over all
  ``s < L_t`` (PR #40352, Design: the source "runs its own top-512").

Readings where the pages are silent: ties are broken toward the lower index,
for blocks and for positions; element ``2i`` of an MXFP4 byte pair is the low
nibble.
"""
from __future__ import annotations

import numpy as np

H = 64
D = 128
BLOCK = 8
PAGE = 64
PAGE_VALUE_BYTES = PAGE * D
PAGE_BYTES = PAGE_VALUE_BYTES + PAGE * 4
PAGE_VALUE_BYTES_MXFP4 = PAGE * D // 2
PAGE_BYTES_MXFP4 = PAGE_VALUE_BYTES_MXFP4 + PAGE * 4
INT32_MAX = 2**31 - 1

# Magnitudes of the eight e2m1 codes (sign in bit 3), as tabulated by the OCP
# Microscaling Formats (MX) v1.0 specification for FP4 E2M1.
_E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


# ----------------------------------------------------------------------------- decoding
def decode_e2m1(codes) -> np.ndarray:
    """4-bit e2m1 codes -> float64 values."""
    c = np.asarray(codes).astype(np.int64)
    mag = _E2M1_MAGNITUDE[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def unpack_fp4(packed) -> np.ndarray:
    """``[..., n]`` bytes -> ``[..., 2n]`` 4-bit codes, element 2i = low nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def decode_ue8m0(codes) -> np.ndarray:
    """ue8m0 scale byte ``c`` -> ``2**(c - 127)`` (code 255 is NaN)."""
    c = np.asarray(codes).astype(np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


def decode_e4m3(codes) -> np.ndarray:
    """FP8 e4m3 ("fn": bias 7, subnormals, no infinities, S.1111.111 = NaN)."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 7
    mag = np.where(exp == 0, man * 2.0**-9, (1.0 + man / 8.0) * np.ldexp(1.0, exp - 7))
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def decode_query(q_fp4_row, q_sf_row) -> np.ndarray:
    """MXFP4 vectors ``[..., D/2]`` + ``[..., D/32]`` -> float64 ``[..., D]``
    (one row's query, or MXFP4 K vectors)."""
    vals = decode_e2m1(unpack_fp4(q_fp4_row))
    scale = np.repeat(decode_ue8m0(q_sf_row), 32, axis=-1)
    return vals * scale


def page_values_and_scales(k_pool):
    """Views of a ``[num_pages, PAGE_BYTES]`` pool: e4m3 bytes ``[pages, 64, 128]``
    and fp32 scales ``[pages, 64]``."""
    pool = np.ascontiguousarray(np.asarray(k_pool, dtype=np.uint8))
    pages = pool.reshape(-1, PAGE_BYTES)
    vals = pages[:, :PAGE_VALUE_BYTES].reshape(-1, PAGE, D)
    scales = np.ascontiguousarray(pages[:, PAGE_VALUE_BYTES:]).view("<f4").reshape(-1, PAGE)
    return vals, scales


def page_values_and_scales_mxfp4(k_pool):
    """Views of a ``[num_pages, PAGE_BYTES_MXFP4]`` pool: packed e2m1 bytes
    ``[pages, 64, 64]`` and ue8m0 scale bytes ``[pages, 64, 4]`` (byte ``j`` of
    a position scales its elements ``32j .. 32j + 31``)."""
    pool = np.ascontiguousarray(np.asarray(k_pool, dtype=np.uint8))
    pages = pool.reshape(-1, PAGE_BYTES_MXFP4)
    vals = pages[:, :PAGE_VALUE_BYTES_MXFP4].reshape(-1, PAGE, D // 2)
    scales = pages[:, PAGE_VALUE_BYTES_MXFP4:].reshape(-1, PAGE, D // 32)
    return vals, scales


def is_mxfp4_pool(k_pool) -> bool:
    return np.asarray(k_pool).shape[-1] == PAGE_BYTES_MXFP4


def gather_keys(k_pool, page_row, positions):
    """Decoded K vectors ``[n, D]`` and per-position scales ``[n]`` at logical
    positions of one request, read through its page-table row.  An FP8 pool
    gives e4m3 vectors and their fp32 scales; an MXFP4 pool gives e2m1 vectors
    with their ue8m0 block scales applied, and scales of 1."""
    positions = np.asarray(positions, dtype=np.int64)
    page_row = np.asarray(page_row, dtype=np.int64)
    phys = page_row[positions // PAGE]
    off = positions % PAGE
    if is_mxfp4_pool(k_pool):
        vals, scales = page_values_and_scales_mxfp4(k_pool)
        k = decode_query(vals[phys, off], scales[phys, off])
        return k, np.ones(len(positions), dtype=np.float64)
    vals, scales = page_values_and_scales(k_pool)
    k = decode_e4m3(vals[phys, off])
    ks = scales[phys, off].astype(np.float64)
    return k, ks


# ----------------------------------------------------------------------------- scoring
def score_positions(q, w, k, kscale):
    """Scores of positions given decoded operands.

    ``q``: ``[H, D]``, ``w``: ``[H]``, ``k``: ``[n, D]``, ``kscale``: ``[n]``.
    Returns ``logit[n] = sum_h w_h * max(kscale * (q_h . k), 0)`` and
    ``tolmag[n] = sum_h |w_h * max(kscale * (q_h . k), 0)|``, both float64.
    """
    x = (q @ k.T) * kscale[None, :]
    r = np.maximum(x, 0.0)
    w64 = np.asarray(w, dtype=np.float64)
    return w64 @ r, np.abs(w64) @ r


def request_of(layout, t, row_req=None):
    """The request whose pages row ``t`` reads: itself for decode rows (layout
    0), request 0 for a one-request prefill chunk (layout 1), ``row_req[t]``
    for a chunk of several requests (layout 2; sglang PR #40352, Design: the
    chunk's rows carry their request starts and per-request rows)."""
    if layout == 0:
        return t
    if layout == 1:
        return 0
    return int(row_req[t])


def row_operands(layer, page_table, layout, t, row_req=None):
    """Decoded query, weights and page-table row of row ``t`` of one layer."""
    q = decode_query(np.asarray(layer.q_fp4[t]), np.asarray(layer.q_sf[t]))
    w = np.asarray(layer.w[t], dtype=np.float64)
    return q, w, np.asarray(page_table[request_of(layout, t, row_req)])


def dense_row_scores(layer, page_table, layout, t, L, row_req=None):
    """Scores and tolerance magnitudes of every position ``s < L`` of row ``t``."""
    q, w, prow = row_operands(layer, page_table, layout, t, row_req)
    pos = np.arange(L, dtype=np.int64)
    k, ks = gather_keys(layer.k_pool, prow, pos)
    return score_positions(q, w, k, ks)


# ----------------------------------------------------------------------------- level one
def num_blocks(L: int) -> int:
    return (int(L) + BLOCK - 1) // BLOCK


def block_keys(logit, L):
    """Block maxima of one row's scores, newest block forced to +inf.

    Returns ``(keys[nb], argmax_position[nb])``; the argmax of the newest block
    is reported as its maximum-score position although its key is +inf.
    """
    L = int(L)
    nb = num_blocks(L)
    padded = np.full(nb * BLOCK, -np.inf)
    padded[:L] = logit[:L]
    blocks = padded.reshape(nb, BLOCK)
    keys = blocks.max(axis=1)
    arg = blocks.argmax(axis=1) + np.arange(nb) * BLOCK
    if nb:
        keys[nb - 1] = np.inf
    return keys, arg


def select_blocks(keys, nb: int, K: int):
    """Top-``K`` block ids by (key descending, id ascending), returned ascending
    and INT32_MAX padded to ``K``; rows with ``nb <= K`` keep every block."""
    out = np.full(K, INT32_MAX, dtype=np.int64)
    if nb <= K:
        chosen = np.arange(nb)
    else:
        ids = np.arange(nb)
        order = np.lexsort((ids, -np.asarray(keys[:nb], dtype=np.float64)))
        chosen = np.sort(order[:K])
    out[: len(chosen)] = chosen
    return out, min(nb, K)


# ----------------------------------------------------------------------------- level two
def top_positions(scores, positions, P: int):
    """Top-``P`` of ``positions`` by (score descending, position ascending),
    returned ascending and ``-1`` padded to ``P``."""
    out = np.full(P, -1, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    if positions.size:
        order = np.lexsort((positions, -np.asarray(scores, dtype=np.float64)))
        take = np.sort(positions[order[:P]])
        out[: take.size] = take
    return out


def candidate_positions(blocks, nvalid: int, L: int):
    """Positions ``s < L`` inside the first ``nvalid`` candidate blocks."""
    b = np.asarray(blocks[:nvalid], dtype=np.int64)
    pos = (b[:, None] * BLOCK + np.arange(BLOCK)[None, :]).reshape(-1)
    return pos[pos < L]


def sparse_row_scores(layer, page_table, layout, t, positions, row_req=None):
    """Scores and tolerance magnitudes of row ``t`` at the given positions."""
    q, w, prow = row_operands(layer, page_table, layout, t, row_req)
    k, ks = gather_keys(layer.k_pool, prow, positions)
    return score_positions(q, w, k, ks)


def select_row(layer, page_table, layout, t, L, blocks, nvalid, P, row_req=None):
    """A layer's top-``P`` positions of row ``t`` inside its candidate blocks.

    Returns ``(positions[P], candidate_positions, scores, tolmag)`` where the
    last three describe every candidate position, for tolerance checks.
    """
    pos = candidate_positions(blocks, nvalid, L)
    logit, tolmag = sparse_row_scores(layer, page_table, layout, t, pos, row_req)
    return top_positions(logit, pos, P), pos, logit, tolmag


# ----------------------------------------------------------------------------- one row, both levels
def source_row(layer, page_table, layout, t, L, K, P, row_req=None):
    """The source layer's work for row ``t``: dense scores, block keys, the
    published top-``K`` blocks and its own dense top-``P`` positions."""
    logit, tolmag = dense_row_scores(layer, page_table, layout, t, L, row_req)
    keys, arg = block_keys(logit, L)
    nb = num_blocks(L)
    blocks, nvalid = select_blocks(keys, nb, K)
    own = top_positions(logit, np.arange(L), P)
    return dict(logit=logit, tolmag=tolmag, keys=keys, key_arg=arg, blocks=blocks, nvalid=nvalid, top=own)


def prefill_tail_rows(req_start, tail_lens):
    """The rows ``prefill_tail`` keeps, in order: the last ``tail_lens[r]``
    rows of each request ``r`` (fewer when the request has fewer rows)
    (sglang PR #40352, Design: prefill_tail restricts what was published to
    the last rows of each request, for the late layers that run on the tail
    only)."""
    rows = []
    for r in range(len(req_start) - 1):
        lo, hi = int(req_start[r]), int(req_start[r + 1])
        n = min(max(int(tail_lens[r]), 0), hi - lo)
        rows.extend(range(hi - n, hi))
    return np.asarray(rows, dtype=np.int64)

