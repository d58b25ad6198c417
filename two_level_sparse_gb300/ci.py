"""ctypes binding of libci.so (include/ci.h), same entry-point names.

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes the cudaStream_t, and a non-zero status becomes a
``CIError``.  Every step of the computation runs in the library's kernels.
Importing this module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libci.so")

CI_OK = 0
CI_ERR = {
    -1: "CI_ERR_NULL",
    -2: "CI_ERR_SHAPE",
    -3: "CI_ERR_ALIGN",
    -4: "CI_ERR_RANGE",
    -5: "CI_ERR_UNSUPPORTED",
    -6: "CI_ERR_CUDA",
}
LAYOUT_DECODE = 0
LAYOUT_PREFILL = 1
LAYOUT_VARLEN = 2
KV_FP8, KV_MXFP4 = 0, 1
PAGE_BYTES = {KV_FP8: 64 * 128 + 64 * 4, KV_MXFP4: 64 * 64 + 64 * 4}
DEVERR_LEN, DEVERR_PAGE, DEVERR_BLOCK, DEVERR_TIMEOUT, DEVERR_REQ, DEVERR_POS = 1, 2, 4, 8, 16, 32
Q_MXFP4, Q_FP8 = 0, 1

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64

SIGNATURES = {
    "ci_score_dense_amax8": [_P, _P, _P, _P, _I64, _I32, _P, _I32, _I32, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _I64,
                             _P, _P],
    "ci_publish_blocks": [_P, _I32, _I32, _P, _I64, _I32, _P, _I64, _P, _P, _P],
    "ci_publish_blocks2": [_P, _I32, _I32, _P, _I64, _I32, _P, _I64, _P, _I32, _P, _I64, _P, _P, _P],
    "ci_prefill_tail": [_P, _I32, _P, _I32, _P, _I64, _P, _I32, _P, _P, _I64, _P, _P, _I32, _P, _P],
    "ci_select_sparse": [_P, _P, _P, _P, _I64, _I32, _P, _I32, _I32, _I32, _P, _P, _I32, _I32, _P, _I64, _P, _I32, _I32,
                         _I32, _P, _P, _I64, _P, _P],
    "ci_select_sparse_layers": [_I32, _P, _P, _P, _P, _I64, _I32, _P, _I32, _I32, _I32, _P, _P, _I32, _I32, _P, _P,
                                _P, _P, _I32, _I32, _P, _P, _I64, _P, _P],
    "ci_dcp_merge_keys": [_P, _I32, _I64, _I64, _P, _I32, _I32, _I32, _P, _I64, _P, _P],
    "ci_dcp_merge_topk": [_P, _P, _I32, _I64, _I64, _I32, _I32, _P, _P, _I64, _P],
    "ci_q_rope_quant": [_P, _P, _P, _I32, _P, ctypes.c_float, ctypes.c_float, _I32, _I32, _I32, _P, _P, _P, _P, _P],
    "ci_strerror": [ctypes.c_int],
    "ci_version": [],
}


class CIError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({CI_ERR.get(status, '?')}: {strerror(status)})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, argtypes in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = ctypes.c_char_p if name == "ci_strerror" else ctypes.c_int
    return lib


lib = _load()


def strerror(status: int) -> str:
    return lib.ci_strerror(status).decode()


def version() -> int:
    return lib.ci_version()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != CI_OK:
        raise CIError(fn, status)


def _expect(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def kv_format(k_pool) -> int:
    """The page format of a pool, from its page size (8448 bytes: FP8, 4352: MXFP4)."""
    for fmt, nbytes in PAGE_BYTES.items():
        if k_pool.dim() == 2 and int(k_pool.shape[1]) == nbytes:
            return fmt
    raise ValueError(f"k_pool must be [num_pages, 8448] (FP8) or [num_pages, 4352] (MXFP4), got {tuple(k_pool.shape)}")


def _req_start(layout, req_start):
    if int(layout) == LAYOUT_VARLEN:
        _expect(req_start, torch.int32, "req_start")
    return _ptr(req_start)


def ci_score_dense_amax8(q_fp4, q_sf, w, k_pool, page_table, layout, seq_len, max_len, skip_le_blocks, keys,
                         dev_err=None, stream=None, req_start=None, block_positions=8):
    """Block keys of the source layer (see include/ci.h)."""
    for t, d, n in ((q_fp4, torch.uint8, "q_fp4"), (q_sf, torch.uint8, "q_sf"), (w, torch.float32, "w"),
                    (k_pool, torch.uint8, "k_pool"), (page_table, torch.int32, "page_table"),
                    (seq_len, torch.int32, "seq_len"), (keys, torch.float32, "keys")):
        _expect(t, d, n)
    rows = int(seq_len.shape[0])
    _check("ci_score_dense_amax8", lib.ci_score_dense_amax8(
        _ptr(q_fp4), _ptr(q_sf), _ptr(w), _ptr(k_pool), int(k_pool.shape[0]), kv_format(k_pool), _ptr(page_table),
        int(page_table.shape[0]), int(page_table.shape[1]), int(layout), _req_start(layout, req_start), _ptr(seq_len),
        rows, int(max_len), int(skip_le_blocks), int(block_positions), _ptr(keys),
        int(keys.stride(0)) if keys.dim() == 2 else 0,
        _ptr(dev_err), _stream(stream)))


def ci_publish_blocks(seq_len, max_len, keys, topk_blocks, blocks, nvalid, dev_err=None, stream=None):
    """Each row's candidate blocks, ascending, INT32_MAX padded (see include/ci.h)."""
    _expect(seq_len, torch.int32, "seq_len")
    _expect(keys, torch.float32, "keys")
    _expect(blocks, torch.int32, "blocks")
    _expect(nvalid, torch.int32, "nvalid")
    rows = int(seq_len.shape[0])
    _check("ci_publish_blocks", lib.ci_publish_blocks(
        _ptr(seq_len), rows, int(max_len), _ptr(keys), int(keys.stride(0)), int(topk_blocks), _ptr(blocks),
        int(blocks.stride(0)), _ptr(nvalid), _ptr(dev_err), _stream(stream)))


def ci_publish_blocks2(seq_len, max_len, keys, topk_blocks, blocks, nvalid, topk_blocks2, blocks2, nvalid2,
                       dev_err=None, stream=None):
    """Two block counts from the same keys in one pass (see include/ci.h)."""
    _expect(seq_len, torch.int32, "seq_len")
    _expect(keys, torch.float32, "keys")
    for t, n in ((blocks, "blocks"), (nvalid, "nvalid"), (blocks2, "blocks2"), (nvalid2, "nvalid2")):
        _expect(t, torch.int32, n)
    rows = int(seq_len.shape[0])
    _check("ci_publish_blocks2", lib.ci_publish_blocks2(
        _ptr(seq_len), rows, int(max_len), _ptr(keys), int(keys.stride(0)), int(topk_blocks), _ptr(blocks),
        int(blocks.stride(0)), _ptr(nvalid), int(topk_blocks2), _ptr(blocks2), int(blocks2.stride(0)), _ptr(nvalid2),
        _ptr(dev_err), _stream(stream)))


def ci_prefill_tail(req_start, tail_len, blocks, nvalid, out_row, out_blocks, out_nvalid, out_count, dev_err=None,
                    stream=None):
    """The published table of the last rows of each request (see include/ci.h)."""
    for t, n in ((req_start, "req_start"), (tail_len, "tail_len"), (blocks, "blocks"), (nvalid, "nvalid"),
                 (out_row, "out_row"), (out_blocks, "out_blocks"), (out_nvalid, "out_nvalid"),
                 (out_count, "out_count")):
        _expect(t, torch.int32, n)
    num_req = int(req_start.shape[0]) - 1
    if int(tail_len.shape[0]) != num_req:
        raise ValueError("tail_len needs one entry per request")
    _check("ci_prefill_tail", lib.ci_prefill_tail(
        _ptr(req_start), num_req, _ptr(tail_len), int(blocks.shape[0]), _ptr(blocks), int(blocks.stride(0)),
        _ptr(nvalid), int(blocks.shape[1]), _ptr(out_row), _ptr(out_blocks), int(out_blocks.stride(0)),
        _ptr(out_nvalid), _ptr(out_count), int(out_blocks.shape[0]), _ptr(dev_err), _stream(stream)))


def ci_select_sparse(q_fp4, q_sf, w, k_pool, page_table, layout, seq_len, max_len, blocks, nvalid, max_blocks, topk,
                     out_pos, out_score=None, dev_err=None, stream=None, req_start=None, block_positions=8):
    """A layer's top-k positions inside the candidate blocks (see include/ci.h)."""
    for t, d, n in ((q_fp4, torch.uint8, "q_fp4"), (q_sf, torch.uint8, "q_sf"), (w, torch.float32, "w"),
                    (k_pool, torch.uint8, "k_pool"), (page_table, torch.int32, "page_table"),
                    (seq_len, torch.int32, "seq_len"), (blocks, torch.int32, "blocks"),
                    (nvalid, torch.int32, "nvalid"), (out_pos, torch.int32, "out_pos")):
        _expect(t, d, n)
    if out_score is not None:
        _expect(out_score, torch.float32, "out_score")
    rows = int(seq_len.shape[0])
    _check("ci_select_sparse", lib.ci_select_sparse(
        _ptr(q_fp4), _ptr(q_sf), _ptr(w), _ptr(k_pool), int(k_pool.shape[0]), kv_format(k_pool), _ptr(page_table),
        int(page_table.shape[0]), int(page_table.shape[1]), int(layout), _req_start(layout, req_start), _ptr(seq_len),
        rows, int(max_len), _ptr(blocks), int(blocks.stride(0)), _ptr(nvalid), int(max_blocks), int(block_positions),
        int(topk), _ptr(out_pos),
        _ptr(out_score), int(out_pos.stride(0)), _ptr(dev_err), _stream(stream)))


def ci_select_sparse_layers(layers, page_table, layout, seq_len, max_len, topk, dev_err=None, stream=None,
                            req_start=None, block_positions=8):
    """Several layers' top-k positions in one launch (see include/ci.h).

    ``layers``: a sequence of dicts with the per-layer tensors q_fp4, q_sf, w,
    k_pool, blocks, nvalid, out_pos, the int max_blocks, and optionally
    out_score; every k_pool has the same format and page count, every out_pos
    the same row stride."""
    n = len(layers)
    if not 1 <= n <= 8:
        raise ValueError("1 to 8 layers per launch")
    for ly in layers:
        for key, d in (("q_fp4", torch.uint8), ("q_sf", torch.uint8), ("w", torch.float32), ("k_pool", torch.uint8),
                       ("blocks", torch.int32), ("nvalid", torch.int32), ("out_pos", torch.int32)):
            _expect(ly[key], d, key)
        if ly.get("out_score") is not None:
            _expect(ly["out_score"], torch.float32, "out_score")
    for t, d, name in ((page_table, torch.int32, "page_table"), (seq_len, torch.int32, "seq_len")):
        _expect(t, d, name)
    k0 = layers[0]["k_pool"]
    if any(kv_format(ly["k_pool"]) != kv_format(k0) or ly["k_pool"].shape[0] != k0.shape[0] for ly in layers):
        raise ValueError("every layer's pool needs the same page format and page count")
    stride = int(layers[0]["out_pos"].stride(0))
    if any(int(ly["out_pos"].stride(0)) != stride for ly in layers):
        raise ValueError("every layer's out_pos needs the same row stride")

    def arr(ctype, vals):
        return (ctype * n)(*vals)

    ptrs = lambda key: arr(_P, [_ptr(ly.get(key)) for ly in layers])  # noqa: E731
    scores = ptrs("out_score") if any(ly.get("out_score") is not None for ly in layers) else None
    rows = int(seq_len.shape[0])
    _check("ci_select_sparse_layers", lib.ci_select_sparse_layers(
        n, ptrs("q_fp4"), ptrs("q_sf"), ptrs("w"), ptrs("k_pool"), int(k0.shape[0]), kv_format(k0), _ptr(page_table),
        int(page_table.shape[0]), int(page_table.shape[1]), int(layout), _req_start(layout, req_start), _ptr(seq_len),
        rows, int(max_len), ptrs("blocks"), arr(_I64, [int(ly["blocks"].stride(0)) for ly in layers]), ptrs("nvalid"),
        arr(_I32, [int(ly["max_blocks"]) for ly in layers]), int(block_positions), int(topk), ptrs("out_pos"), scores,
        stride, _ptr(dev_err), _stream(stream)))


def ci_q_rope_quant(positions, q, cos_sin, w, softmax_scale, head_scale, is_neox, out_format, q_out, q_sf, w_out,
                    dev_err=None, stream=None):
    """The query producer: RoPE, quantization, head-weight scaling (see include/ci.h)."""
    _expect(positions, torch.int32, "positions")
    _expect(q, torch.bfloat16, "q")
    _expect(cos_sin, torch.float32, "cos_sin")
    _expect(w, torch.float32, "w")
    _expect(q_out, torch.uint8, "q_out")
    _expect(w_out, torch.float32, "w_out")
    if q_sf is not None:
        _expect(q_sf, torch.uint8, "q_sf")
    tokens = int(positions.shape[0])
    _check("ci_q_rope_quant", lib.ci_q_rope_quant(
        _ptr(positions), _ptr(q), _ptr(cos_sin), int(cos_sin.shape[0]), _ptr(w), float(softmax_scale),
        float(head_scale), int(bool(is_neox)), tokens, int(out_format), _ptr(q_out), _ptr(q_sf), _ptr(w_out),
        _ptr(dev_err), _stream(stream)))


def ci_dcp_merge_keys(keys_local, seq_len, max_len, skip_le_blocks, keys, dev_err=None, stream=None):
    """Shards' local block maxima ``keys_local[W, rows, stride]`` -> the global keys (see include/ci.h)."""
    _expect(keys_local, torch.float32, "keys_local")
    _expect(seq_len, torch.int32, "seq_len")
    _expect(keys, torch.float32, "keys")
    world, rows = int(keys_local.shape[0]), int(keys_local.shape[1])
    _check("ci_dcp_merge_keys", lib.ci_dcp_merge_keys(
        _ptr(keys_local), world, int(keys_local.stride(0)), int(keys_local.stride(1)), _ptr(seq_len), rows,
        int(max_len), int(skip_le_blocks), _ptr(keys), int(keys.stride(0)), _ptr(dev_err), _stream(stream)))


def ci_dcp_merge_topk(pos_local, score_local, out_pos, out_score=None, stream=None):
    """Shards' local top-k ``[W, rows, k]`` -> the global top-k (see include/ci.h)."""
    _expect(pos_local, torch.int32, "pos_local")
    _expect(score_local, torch.float32, "score_local")
    _expect(out_pos, torch.int32, "out_pos")
    world, rows, k = (int(x) for x in pos_local.shape)
    _check("ci_dcp_merge_topk", lib.ci_dcp_merge_topk(
        _ptr(pos_local), _ptr(score_local), world, int(pos_local.stride(0)), int(pos_local.stride(1)), rows, k,
        _ptr(out_pos), _ptr(out_score), int(out_pos.stride(0)), _stream(stream)))
