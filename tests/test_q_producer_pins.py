"""Pins of the query-producer oracle against facts that do not come from it:
library roundings (torch's bf16 and e4m3 casts), the exact exponent of a
float from math.frexp, the OCP e2m1 grid, and closed forms of RoPE."""
import math

import numpy as np
import pytest
import torch

from oracle import q_producer as P
from oracle.ci_oracle import decode_e2m1, decode_e4m3


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 10, 5000), rng.normal(0, 1e-3, 1000), [0.0, -0.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8,
                                                                             -(1.0 + 2**-8), 65504.0, 3.0e38]])
    x = x.astype(np.float32)
    want = torch.tensor(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(P.round_to_bf16(x).view(np.uint32), want.view(np.uint32))


def test_ceil_log2_exact_against_frexp():
    rng = np.random.default_rng(2)
    v = np.concatenate([np.ldexp(1.0, rng.integers(-60, 60, 200)), rng.uniform(1e-12, 1e12, 2000)]).astype(np.float32)
    v = np.concatenate([v, np.nextafter(v, np.float32(np.inf)), np.nextafter(v, np.float32(0))])
    for x, got in zip(v.tolist(), P.ceil_log2(v).tolist()):
        m, e = math.frexp(x)  # x = m * 2^e, 0.5 <= m < 1
        assert got == (e - 1 if m == 0.5 else e), x


def test_e2m1_rounding_nearest_even_saturating():
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    y = np.concatenate([np.arange(-8, 8, 1 / 64), np.random.default_rng(3).uniform(-7, 7, 3000)]).astype(np.float32)
    codes = P.quantize_e2m1(y)
    dec = decode_e2m1(codes)
    for x, c, d in zip(y.tolist(), codes.tolist(), dec.tolist()):
        a = min(abs(x), 6.0)
        dist = np.abs(grid - a)
        assert abs(abs(d) - a) == dist.min(), x  # a nearest grid magnitude
        if np.sum(dist == dist.min()) > 1:
            assert c % 2 == 0, x                   # ties go to the even code
        assert (c >= 8) == (x < 0 or (x == 0 and math.copysign(1, x) < 0)), x  # sign kept
    # worked values from the rule
    hand = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7, -0.1: 8, -0.3: 9}
    for x, c in hand.items():
        assert int(P.quantize_e2m1(np.float32(x))) == c, x


def test_e4m3_cast_matches_torch_on_grid():
    y = np.linspace(-448, 448, 20001).astype(np.float32)
    got = decode_e4m3(P.quantize_e4m3(y))
    # the result is an e4m3 value within half a step of y
    assert np.all(np.abs(got - y) <= np.maximum(np.abs(y), 2**-6) * 2**-4 + 1e-12)


def test_rope_closed_forms():
    rng = np.random.default_rng(4)
    q = P.bf16_bits_to_f32(_bf16(rng.normal(0, 3, (2, 128))))
    one, zero = np.ones((1, 32), np.float32), np.zeros((1, 32), np.float32)
    for neox in (True, False):
        assert np.array_equal(P.rope_rows(q, one, zero, neox), q)  # angle 0: identity on bf16 inputs
        r = P.rope_rows(q, zero, one, neox)                          # angle 90 degrees
        x0, x1 = (q[:, 0:32], q[:, 32:64]) if neox else (q[:, 0:64:2], q[:, 1:64:2])
        r0, r1 = (r[:, 0:32], r[:, 32:64]) if neox else (r[:, 0:64:2], r[:, 1:64:2])
        assert np.array_equal(r0, -x1) and np.array_equal(r1, x0)
        assert np.array_equal(r[:, 64:], q[:, 64:])


def _inputs(tokens=3, seed=5, max_pos=50):
    rng = np.random.default_rng(seed)
    mag = 10.0 ** rng.uniform(-3, 3, (tokens, 64, 1))
    q = _bf16((rng.normal(0, 1, (tokens, 64, 128)) * mag).astype(np.float32))
    ang = rng.uniform(0, 2 * np.pi, (max_pos, 32))
    cos_sin = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    pos = rng.integers(0, max_pos, tokens)
    w = rng.normal(0, 0.125, (tokens, 64)).astype(np.float32)
    return pos, q, cos_sin, w


@pytest.mark.parametrize("neox", [True, False])
def test_mxfp4_mode_error_bound_and_block_maximum(neox):
    pos, q, cs, w = _inputs()
    packed, sf, w_out = P.produce(pos, q, cs, w, 0.0625, 0.125, neox, "mxfp4")
    x = P.rope_rows(P.bf16_bits_to_f32(q), cs[pos][:, None, :32], cs[pos][:, None, 32:], neox)
    codes = np.empty(packed.shape[:-1] + (128,), np.uint8)
    codes[..., 0::2], codes[..., 1::2] = packed & 15, packed >> 4
    scale = np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=-1)
    deq = decode_e2m1(codes) * scale
    y = np.abs(x) / scale
    gap = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))  # half the e2m1 step at that magnitude
    assert np.all(np.abs(deq - x) <= gap * scale)
    xb = np.abs(x).reshape(*x.shape[:-1], 4, 32)
    amax_code = np.take_along_axis(codes.reshape(*x.shape[:-1], 4, 32), xb.argmax(-1)[..., None], -1)[..., 0] & 7
    assert np.all(amax_code >= 5)  # amax / scale lies in (3, 6]: an exponent off by one breaks it
    assert np.array_equal(w_out, (w * np.float32(0.0625)) * np.float32(0.125))


@pytest.mark.parametrize("neox", [True, False])
def test_fp8_mode_scale_folded_into_weight(neox):
    pos, q, cs, w = _inputs(seed=6)
    q8, sf, w_out = P.produce(pos, q, cs, w, 0.0625, 0.125, neox, "fp8")
    assert sf is None
    x = P.rope_rows(P.bf16_bits_to_f32(q), cs[pos][:, None, :32], cs[pos][:, None, 32:], neox)
    ratio = w_out.astype(np.float64) / ((w.astype(np.float64) * 0.0625) * 0.125)
    e = np.log2(ratio)
    assert np.allclose(e, np.round(e), atol=1e-6)  # the folded scale is a power of two
    scale = np.ldexp(1.0, np.round(e).astype(np.int64))
    amax = np.abs(x).max(-1)
    assert np.all(amax / scale <= 448) and np.all(amax / scale > 224)
    deq = decode_e4m3(q8) * scale[..., None]
    assert np.all(np.abs(deq - x) <= np.abs(x) * 2**-4 + scale[..., None] * 2**-9)


def test_planted_rope_sign_is_caught(monkeypatch):
    good = P.rope_rows

    def flipped(q, cos, sin, is_neox):
        return good(q, cos, -sin, is_neox)
    monkeypatch.setattr(P, "rope_rows", flipped)
    with pytest.raises(AssertionError):
        test_rope_closed_forms()


def test_planted_scale_exponent_off_by_one_is_caught(monkeypatch):
    good = P.ceil_log2
    monkeypatch.setattr(P, "ceil_log2", lambda v: good(v) + 1)
    with pytest.raises(AssertionError):
        test_mxfp4_mode_error_bound_and_block_maximum(True)
