"""CPU oracle of the indexer's query producer: RoPE, quantization, weight scaling.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library.

The producer turns one token's projected indexer queries (bf16, 64 heads x
128 dims) into the quantized queries the indexer reads, and scales its head
weights (vLLM ``indexer.py`` page, ``rope_quant_q``, and the
``_fused_indexer_q_rope_quant_kernel`` of ``sparse_attn_indexer.py``):

* RoPE on the first 64 dims: the pair ``(x0, x1)`` -- dims ``(i, 32 + i)`` in
  the NeoX layout, ``(2i, 2i + 1)`` in the interleaved one -- becomes
  ``r0 = x0 cos - x1 sin``, ``r1 = x1 cos + x0 sin`` in fp32, each rounded to
  bf16 and back; dims 64..127 pass unrotated.  ``cos``/``sin`` are the 32 + 32
  values of the token's position row of the cos/sin cache.
* FP8 mode (as the pages print it): one scale per head,
  ``2^ceil(log2(max(amax, 1e-10) * (1/448)))`` over all 128 dims; the values
  are ``x / scale`` clamped to +-448 and rounded to e4m3; the head weight
  becomes ``w * scale * softmax_scale * head_scale``.
* MXFP4 mode (the indexer's query format; the pages call the producer with
  ``use_fp4`` and print only the FP8 body): the same scale rule per block of
  32 dims with 6, the largest e2m1 magnitude, in place of 448; the values are
  ``x / scale`` rounded to e2m1 (nearest, ties to the even code, saturating);
  the scale is stored as its ue8m0 code and the weight becomes
  ``w * softmax_scale * head_scale``.

All arithmetic is float32, one rounding per operation, in the order above, so
that every integer the producer writes (codes, scale bytes) is decided the
way the GPU decides it.  ``ceil(log2(v))`` is taken exactly from the bits of
``v`` (the plain definition; no approximate logarithm).
"""
from __future__ import annotations

import numpy as np

H = 64
D = 128
FP8_MAX = 448.0
FP4_MAX = 6.0
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """float32 -> nearest bf16 (ties to even), returned as float32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (r.astype(np.uint32) << 16).view(np.float32)


def ceil_log2(v) -> np.ndarray:
    """Exact ceil(log2(v)) of positive normal float32 values."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32)
    e = ((u >> 23) & 0xFF).astype(np.int64) - 127
    return e + ((u & 0x7FFFFF) != 0)


def pow2(e) -> np.ndarray:
    return np.ldexp(np.float32(1.0), np.asarray(e, dtype=np.int64)).astype(np.float32)


def rope_rows(q, cos, sin, is_neox: bool) -> np.ndarray:
    """q: float32 [..., 128] (bf16 values); cos, sin: float32 [..., 32] broadcast
    over heads.  Returns the float32 vectors after RoPE on dims 0..63."""
    q = np.asarray(q, dtype=np.float32)
    out = q.copy()
    if is_neox:
        x0, x1 = q[..., 0:32], q[..., 32:64]
    else:
        x0, x1 = q[..., 0:64:2], q[..., 1:64:2]
    r0 = round_to_bf16(np.float32(x0 * cos) - np.float32(x1 * sin))
    r1 = round_to_bf16(np.float32(x1 * cos) + np.float32(x0 * sin))
    if is_neox:
        out[..., 0:32], out[..., 32:64] = r0, r1
    else:
        out[..., 0:64:2], out[..., 1:64:2] = r0, r1
    return out


def _scale_exponent(amax, vmax):
    raw = np.maximum(np.asarray(amax, np.float32), np.float32(1e-10)) * np.float32(1.0 / vmax)
    return ceil_log2(raw.astype(np.float32))


def quantize_e2m1(y) -> np.ndarray:
    """float32 -> 4-bit e2m1 codes: nearest magnitude (ties to the even code),
    saturating at 6, sign kept (negative values that round to 0 give code 8)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), FP4_MAX)
    d = np.abs(a[..., None] - _E2M1_GRID)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # among equally near magnitudes take the even code
    codes = np.arange(8)
    pick = np.where(cand & (codes % 2 == 0), codes, 99).min(axis=-1)
    pick = np.where(pick == 99, np.argmax(cand, axis=-1), pick)
    return (pick + 8 * np.signbit(y)).astype(np.uint8)


def quantize_e4m3(y) -> np.ndarray:
    """float32 (|y| <= 448) -> e4m3 bytes, round to nearest even (torch's cast)."""
    import torch

    t = torch.from_numpy(np.asarray(y, dtype=np.float32).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def produce(positions, q_bits, cos_sin, w, softmax_scale, head_scale, is_neox, mode):
    """One batch of tokens through the producer.

    positions int [T]; q_bits uint16 [T, 64, 128] (bf16); cos_sin float32
    [max_pos, 64] (32 cos then 32 sin); w float32 [T, 64].  mode "mxfp4" gives
    (q_fp4 uint8 [T, 64, 64], q_sf uint8 [T, 64, 4], w_out float32 [T, 64]);
    mode "fp8" gives (q_fp8 uint8 [T, 64, 128], None, w_out).
    """
    q = bf16_bits_to_f32(q_bits)
    cs = np.asarray(cos_sin, dtype=np.float32)[np.asarray(positions, dtype=np.int64)]
    cos, sin = cs[:, None, 0:32], cs[:, None, 32:64]
    x = rope_rows(q, cos, sin, bool(is_neox))
    w = np.asarray(w, dtype=np.float32)
    ss, hs = np.float32(softmax_scale), np.float32(head_scale)
    if mode == "fp8":
        e = _scale_exponent(np.abs(x).max(axis=-1), FP8_MAX)  # [T, H]
        scale = pow2(e)
        y = np.clip(x / scale[..., None], -FP8_MAX, FP8_MAX).astype(np.float32)
        w_out = ((w * scale).astype(np.float32) * ss).astype(np.float32) * hs
        return quantize_e4m3(y), None, w_out.astype(np.float32)
    xb = x.reshape(x.shape[0], H, 4, 32)
    e = _scale_exponent(np.abs(xb).max(axis=-1), FP4_MAX)  # [T, H, 4]
    y = (xb / pow2(e)[..., None]).astype(np.float32)
    codes = quantize_e2m1(y).reshape(x.shape[0], H, D)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    q_sf = (e + 127).astype(np.uint8)
    w_out = (w * ss).astype(np.float32) * hs
    return packed, q_sf, w_out.astype(np.float32)
