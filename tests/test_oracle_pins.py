"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of the oracle with something independent: a library
decoder, a closed form, a hand-worked fixture from the pages' definitions, a
brute-force count on tiny inputs, or an invariant the pages state.  The last
group plants mistakes in the oracle (on the CPU) and checks that a pin fails.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import ci_oracle as O
from two_level_sparse_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


# ----------------------------------------------------------------------------- decoders
def test_e4m3_decoder_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = O.decode_e4m3(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_ue8m0_decoder_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    got = O.decode_ue8m0(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_e2m1_decoder_via_e4m3_bit_fields():
    # e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.  Re-encode
    # every code as an e4m3 bit pattern (exponent rebiased to 7, mantissa moved
    # to the top mantissa bit) and decode that with torch.
    codes = np.arange(16)
    e4m3 = []
    for c in codes:
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        if e == 0:  # subnormal e2m1: m * 0.5 -> 0 or 2^-1
            byte = 0 if m == 0 else ((-1 + 7) << 3)
        else:
            byte = ((e - 1 + 7) << 3) | (m << 2)
        e4m3.append((s << 7) | byte)
    ref = torch.tensor(e4m3, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.decode_e2m1(codes), ref)


def test_fp4_nibble_order_low_first():
    # element 2i is the low nibble (reading of "2 values packed per byte")
    packed = np.array([[0x21, 0xF7]], dtype=np.uint8)
    assert O.unpack_fp4(packed).tolist() == [[1, 2, 7, 15]]
    assert O.decode_e2m1(O.unpack_fp4(packed)).tolist() == [[0.5, 1.0, 6.0, -6.0]]


def test_query_scale_applies_per_32_elements():
    q_fp4 = np.full((synth.H, synth.D // 2), 0x22, dtype=np.uint8)  # every element 1.0
    q_sf = np.tile(np.array([127, 128, 126, 130], dtype=np.uint8), (synth.H, 1))
    q = O.decode_query(q_fp4, q_sf)
    assert q.shape == (synth.H, synth.D)
    assert np.all(q[:, :32] == 1.0) and np.all(q[:, 32:64] == 2.0)
    assert np.all(q[:, 64:96] == 0.5) and np.all(q[:, 96:] == 8.0)


# ----------------------------------------------------------------------------- scores
def _pool_from_vectors(kbytes, kscale):
    """Pack [n, 128] e4m3 bytes and [n] scales into consecutive pages."""
    n = kbytes.shape[0]
    pages = (n + synth.PAGE - 1) // synth.PAGE
    pool = np.zeros((pages, synth.PAGE_BYTES), dtype=np.uint8)
    for s in range(n):
        p, o = divmod(s, synth.PAGE)
        pool[p, o * synth.D : (o + 1) * synth.D] = kbytes[s]
        pool[p, synth.PAGE_VALUE_BYTES + 4 * o : synth.PAGE_VALUE_BYTES + 4 * o + 4] = np.frombuffer(
            np.float32(kscale[s]).tobytes(), dtype=np.uint8)
    return pool


def test_scores_closed_form_all_ones():
    L = 70  # spans two pages
    k = np.full((L, synth.D), 0x38, dtype=np.uint8)  # e4m3 1.0
    ks = np.full(L, 2.0, dtype=np.float32)
    pool = _pool_from_vectors(k, ks)
    q = O.decode_query(np.full((synth.H, 64), 0x22, np.uint8), np.full((synth.H, 4), 127, np.uint8))
    w = np.linspace(-1, 1, synth.H)
    kk, kss = O.gather_keys(pool, np.arange(pool.shape[0]), np.arange(L))
    logit, tol = O.score_positions(q, w, kk, kss)
    # q_h . k = 128, times kscale 2 -> 256 for every head
    assert np.allclose(logit, 256.0 * w.sum(), rtol=0, atol=1e-9)
    assert np.allclose(tol, 256.0 * np.abs(w).sum(), rtol=0, atol=1e-9)


def test_scores_relu_zeroes_negative_heads_exactly():
    L = 9
    k = np.full((L, synth.D), 0x38, dtype=np.uint8)
    pool = _pool_from_vectors(k, np.ones(L, np.float32))
    q_fp4 = np.full((synth.H, 64), 0x22, np.uint8)
    q_fp4[1::2] = 0xAA  # odd heads are -1.0 everywhere
    q = O.decode_query(q_fp4, np.full((synth.H, 4), 127, np.uint8))
    w = np.ones(synth.H)
    w[::4] = -0.5
    kk, kss = O.gather_keys(pool, np.arange(pool.shape[0]), np.arange(L))
    logit, tol = O.score_positions(q, w, kk, kss)
    even = np.arange(0, synth.H, 2)
    assert np.all(logit == 128.0 * w[even].sum())
    assert np.all(tol == 128.0 * np.abs(w[even]).sum())
    # every head negative -> exactly zero score and zero tolerance
    q_neg = O.decode_query(np.full((synth.H, 64), 0xAA, np.uint8), np.full((synth.H, 4), 127, np.uint8))
    logit0, tol0 = O.score_positions(q_neg, w, kk, kss)
    assert np.all(logit0 == 0.0) and np.all(tol0 == 0.0)


def test_scores_match_bruteforce_loops():
    rng = np.random.default_rng(5)
    L = 5
    kbytes = rng.integers(0, 256, (L, synth.D), dtype=np.uint8)
    kbytes[(kbytes & 0x7F) == 0x7F] = 0x30  # avoid NaN codes
    ks = rng.uniform(0.5, 2.0, L).astype(np.float32)
    pool = _pool_from_vectors(kbytes, ks)
    q_fp4 = rng.integers(0, 256, (synth.H, 64), dtype=np.uint8)
    q_sf = rng.integers(123, 128, (synth.H, 4), dtype=np.uint8)
    w = rng.normal(0, 0.125, synth.H)
    kk, kss = O.gather_keys(pool, np.arange(pool.shape[0]), np.arange(L))
    logit, tol = O.score_positions(O.decode_query(q_fp4, q_sf), w, kk, kss)
    # brute force: every term written out with Python floats
    e2m1 = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}
    for s in range(L):
        total, mag = 0.0, 0.0
        for h in range(synth.H):
            acc = 0.0
            for d in range(synth.D):
                byte = int(q_fp4[h, d // 2])
                code = byte & 15 if d % 2 == 0 else byte >> 4
                qv = (-1.0 if code & 8 else 1.0) * e2m1[code & 7] * 2.0 ** (int(q_sf[h, d // 32]) - 127)
                kv = float(torch.tensor([int(kbytes[s, d])], dtype=torch.uint8).view(torch.float8_e4m3fn).item())
                acc += qv * kv
            x = acc * float(ks[s])
            total += w[h] * max(x, 0.0)
            mag += abs(w[h] * max(x, 0.0))
        assert math.isclose(total, logit[s], rel_tol=1e-12, abs_tol=1e-12)
        assert math.isclose(mag, tol[s], rel_tol=1e-12, abs_tol=1e-12)


def _e2m1_value(code):
    """OCP MX v1.0 FP4 E2M1: sign bit 3, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    mag = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}[code & 7]
    return -mag if code & 8 else mag


def test_mxfp4_pool_layout_hand_example():
    """One MXFP4 page built by hand: values then one scale word per position,
    byte j of the word scaling elements 32j .. 32j + 31; read through a page
    table that puts it second."""
    page = np.zeros(synth.PAGE_BYTES_MXFP4, dtype=np.uint8)
    page[0:64] = 0x71          # position 0: elements (0.5, 6.0) repeated
    page[63 * 64 : 64 * 64] = 0x9A  # position 63: elements (-1.0, -0.5) repeated
    base = synth.PAGE_VALUE_BYTES_MXFP4
    page[base : base + 4] = [127, 126, 128, 125]
    page[base + 4 * 63 : base + 4 * 64] = [120, 127, 127, 130]
    pool = np.stack([np.zeros_like(page), page])
    k, ks = O.gather_keys(pool, np.array([1]), np.array([0, 63]))
    assert np.all(ks == 1.0)
    blockscale0 = np.repeat([1.0, 0.5, 2.0, 0.25], 32)
    want0 = np.tile([0.5, 6.0], 64) * blockscale0
    blockscale63 = np.repeat([2.0**-7, 1.0, 1.0, 8.0], 32)
    want63 = np.tile([-1.0, -0.5], 64) * blockscale63
    assert np.array_equal(k[0], want0) and np.array_equal(k[1], want63)


def test_mxfp4_scores_match_bruteforce_loops():
    rng = np.random.default_rng(9)
    L = 70  # two pages
    pool = np.zeros((2, synth.PAGE_BYTES_MXFP4), dtype=np.uint8)
    pool[:, : synth.PAGE_VALUE_BYTES_MXFP4] = rng.integers(0, 256, (2, synth.PAGE_VALUE_BYTES_MXFP4))
    pool[:, synth.PAGE_VALUE_BYTES_MXFP4 :] = rng.integers(123, 128, (2, 256))
    q_fp4 = rng.integers(0, 256, (synth.H, 64), dtype=np.uint8)
    q_sf = rng.integers(123, 128, (synth.H, 4), dtype=np.uint8)
    w = rng.normal(0, 0.125, synth.H)
    prow = np.array([1, 0])  # logical page 0 is physical page 1
    kk, kss = O.gather_keys(pool, prow, np.arange(L))
    logit, tol = O.score_positions(O.decode_query(q_fp4, q_sf), w, kk, kss)
    for s in (0, 5, 63, 64, 69):
        phys, off = int(prow[s // 64]), s % 64
        total, mag = 0.0, 0.0
        for h in range(synth.H):
            acc = 0.0
            for d in range(synth.D):
                qb, kb = int(q_fp4[h, d // 2]), int(pool[phys, off * 64 + d // 2])
                qc = qb & 15 if d % 2 == 0 else qb >> 4
                kc = kb & 15 if d % 2 == 0 else kb >> 4
                qs = 2.0 ** (int(q_sf[h, d // 32]) - 127)
                kscale = 2.0 ** (int(pool[phys, synth.PAGE_VALUE_BYTES_MXFP4 + 4 * off + d // 32]) - 127)
                acc += _e2m1_value(qc) * qs * _e2m1_value(kc) * kscale
            total += w[h] * max(acc, 0.0)
            mag += abs(w[h] * max(acc, 0.0))
        assert math.isclose(total, logit[s], rel_tol=1e-12, abs_tol=1e-12)
        assert math.isclose(mag, tol[s], rel_tol=1e-12, abs_tol=1e-12)


def test_page_table_indirection_is_transparent():
    wl = synth.make_workload("t", synth.LAYOUT_DECODE, [150, 70], 4, seed=11, layers=1)
    layer = wl.layers[0]
    base = [O.dense_row_scores(layer, wl.page_table.numpy(), 0, t, int(L))[0] for t, L in enumerate(wl.seq_len)]
    # move every physical page to a new slot and rewrite the table accordingly
    n = layer.k_pool.shape[0]
    perm = np.random.default_rng(3).permutation(n)
    new_pool = np.empty_like(layer.k_pool.numpy())
    new_pool[perm] = layer.k_pool.numpy()
    pt = wl.page_table.numpy().copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    moved = synth.Layer(layer.q_fp4, layer.q_sf, layer.w, torch.from_numpy(new_pool))
    for t, L in enumerate(wl.seq_len.tolist()):
        assert np.array_equal(O.dense_row_scores(moved, pt, 0, t, L)[0], base[t])


def _concat_requests(a, b):
    """A two-request chunk made of two one-request workloads: rows of `a`
    then rows of `b`, b's pages moved after a's in one pool."""
    pa = a.layers[0].k_pool.shape[0]
    pta, ptb = a.page_table.numpy(), b.page_table.numpy()
    width = max(pta.shape[1], ptb.shape[1])
    pt = np.full((2, width), -1, dtype=np.int32)
    pt[0, : pta.shape[1]] = pta[0]
    pt[1, : ptb.shape[1]] = np.where(ptb[0] >= 0, ptb[0] + pa, -1)
    layers = [synth.Layer(torch.cat([la.q_fp4, lb.q_fp4]), torch.cat([la.q_sf, lb.q_sf]), torch.cat([la.w, lb.w]),
                          torch.cat([la.k_pool, lb.k_pool])) for la, lb in zip(a.layers, b.layers)]
    starts = torch.tensor([0, a.rows, a.rows + b.rows], dtype=torch.int32)
    return synth.Workload("ab", synth.LAYOUT_VARLEN, torch.cat([a.seq_len, b.seq_len]), torch.from_numpy(pt), layers,
                          a.topk_blocks, a.topk, starts)


def test_varlen_rows_read_their_own_request():
    # Rows of a multi-request chunk must score exactly as the same rows of
    # their own one-request chunk: wrong request or page-table row fails.
    a = synth.make_workload("a", synth.LAYOUT_PREFILL, [300, 301, 302], 8, seed=21, layers=2)
    b = synth.make_workload("b", synth.LAYOUT_PREFILL, [700, 701], 8, seed=22, layers=2)
    ab = _concat_requests(a, b)
    rr = ab.row_req()
    assert rr.tolist() == [0, 0, 0, 1, 1]
    pt = ab.page_table.numpy()
    for t in range(ab.rows):
        src, u = (a, t) if t < a.rows else (b, t - a.rows)
        L = int(src.seq_len[u])
        for j in range(2):
            want = O.dense_row_scores(src.layers[j], src.page_table.numpy(), synth.LAYOUT_PREFILL, u, L)[0]
            got = O.dense_row_scores(ab.layers[j], pt, synth.LAYOUT_VARLEN, t, L, rr)[0]
            assert np.array_equal(got, want), (t, j)


def test_varlen_builder_groups_rows_by_request():
    wl = synth.make_varlen_workload("v", [100, 3000, 20], [3, 5, 2], 16, seed=1, layers=1)
    assert wl.req_start.tolist() == [0, 3, 8, 10]
    assert wl.seq_len.tolist() == [101, 102, 103, 3001, 3002, 3003, 3004, 3005, 21, 22]
    pt = wl.page_table.numpy()
    used = np.concatenate([pt[r][pt[r] >= 0] for r in range(3)])
    assert len(set(used.tolist())) == used.size  # no page shared between requests
    assert [int((pt[r] >= 0).sum()) for r in range(3)] == [2, 47, 1]


@pytest.mark.parametrize("starts,tails,want", [
    ([0, 3, 8, 10], [1, 2, 5], [2, 6, 7, 8, 9]),      # tail longer than its request keeps all its rows
    ([0, 4, 4, 6], [0, 3, 1], [5]),                   # empty tail, empty request
    ([0, 2], [2], [0, 1]),
])
def test_prefill_tail_rows_definition(starts, tails, want):
    # brute force: a row is kept iff it is among the last tails[r] rows of its request
    brute = [t for r in range(len(starts) - 1) for t in range(starts[r], starts[r + 1])
             if t >= starts[r + 1] - max(tails[r], 0)]
    assert brute == want
    assert O.prefill_tail_rows(starts, tails).tolist() == want


# ----------------------------------------------------------------------------- level one
def test_block_keys_fixture():
    (L,), scores, expect = _read_fixture("amax8_contract.txt")
    keys, _ = O.block_keys(np.array(scores), int(L))
    assert keys.tolist() == expect


def _rank(keys, i):
    return sum(1 for j in range(len(keys)) if keys[j] > keys[i] or (keys[j] == keys[i] and j < i))


def test_select_blocks_bruteforce_ranks():
    rng = np.random.default_rng(0)
    for trial in range(300):
        nb = int(rng.integers(1, 12))
        K = int(rng.integers(1, 10))
        keys = rng.integers(0, 4, nb).astype(np.float64)  # many ties
        keys[-1] = np.inf
        blocks, nvalid = O.select_blocks(keys, nb, K)
        expect = [i for i in range(nb) if nb <= K or _rank(keys, i) < K]
        assert nvalid == min(nb, K)
        assert blocks[:nvalid].tolist() == expect
        assert np.all(blocks[nvalid:] == O.INT32_MAX)


def test_top_positions_bruteforce_ranks():
    rng = np.random.default_rng(1)
    for trial in range(300):
        n = int(rng.integers(0, 14))
        P = int(rng.integers(1, 9))
        pos = np.sort(rng.choice(100, n, replace=False))
        sc = rng.integers(0, 3, n).astype(np.float64)
        out = O.top_positions(sc, pos, P)
        expect = sorted(int(pos[i]) for i in range(n) if _rank(sc, i) < P)
        assert out[: len(expect)].tolist() == expect
        assert np.all(out[len(expect):] == -1)


def test_source_top_p_through_p_plus_1_blocks_equals_dense_top_p():
    """The source layer keeps its own top-(P + 1) blocks (newest pinned) and
    takes its top-P positions inside them; that equals the top-P over every
    position, ties toward the lower position included, because every block
    holding a position above the P-th score outranks the rest and the blocks
    of the tied positions taken come first in id order (sglang PR #40352,
    Design: the source's own top-512 through K' = P + 1 candidate blocks).
    Checked by brute force on rows of heavily tied integer scores."""
    rng = np.random.default_rng(7)
    for trial in range(800):
        L = int(rng.integers(1, 160))
        P = int(rng.integers(1, 14))
        sc = rng.integers(0, 3, L).astype(np.float64)
        nb = O.num_blocks(L)
        keys, _ = O.block_keys(sc, L)
        blocks, nvalid = O.select_blocks(keys, nb, P + 1)
        cand = O.candidate_positions(blocks, nvalid, L)
        two_level = O.top_positions(sc[cand], cand, P)
        dense = sorted(int(i) for i in range(L) if _rank(sc, i) < P)
        assert two_level[: len(dense)].tolist() == dense
        assert np.all(two_level[len(dense):] == -1)


def test_two_level_fixture():
    (L,), src, blocks_expect, cons, pos_expect = _read_fixture("two_level_example.txt")
    L = int(L)
    keys, _ = O.block_keys(np.array(src), L)
    blocks, nvalid = O.select_blocks(keys, O.num_blocks(L), 2)
    assert blocks[:nvalid].tolist() == blocks_expect
    cand = O.candidate_positions(blocks, nvalid, L)
    out = O.top_positions(np.array(cons)[cand], cand, 3)
    assert out.tolist() == pos_expect


# ----------------------------------------------------------------------------- invariants
@pytest.fixture(scope="module")
def tiny_decode():
    lens = [1500, 300, 9, 1024, 2049]
    return synth.make_workload("inv", synth.LAYOUT_DECODE, lens, topk_blocks=64, seed=21, layers=2,
                               dup_frac=0.05)


def test_invariants_on_tiny_workload(tiny_decode):
    wl = tiny_decode
    pt = wl.page_table.numpy()
    K, P = wl.topk_blocks, 40
    for t, L in enumerate(wl.seq_len.tolist()):
        src = O.source_row(wl.layers[0], pt, 0, t, L, K, P)
        nb = O.num_blocks(L)
        blocks = src["blocks"][: src["nvalid"]]
        assert nb - 1 in blocks  # (i) newest block always kept
        if nb <= K:  # (ii) keep-all rows
            assert blocks.tolist() == list(range(nb))
        top = src["top"][src["top"] >= 0]
        assert np.all(top < L)  # (iii)
        cons, cand, _, _ = O.select_row(wl.layers[1], pt, 0, t, L, src["blocks"], src["nvalid"], P)
        cons = cons[cons >= 0]
        assert np.all(cons < L) and set(cons.tolist()) <= set(cand.tolist())  # (iv)
        # (v) candidates covering every block -> two-level equals dense top-P
        allb, nall = O.select_blocks(src["keys"], nb, nb)
        same, _, _, _ = O.select_row(wl.layers[0], pt, 0, t, L, allb, nall, P)
        assert np.array_equal(same, src["top"])
        # (vi) dense top-P lies inside the top-(P+1) blocks
        bl, nv = O.select_blocks(src["keys"], nb, P + 1)
        assert set((top // O.BLOCK).tolist()) <= set(bl[:nv].tolist())


def test_duplicate_blocks_tie_and_lower_id_wins(tiny_decode):
    wl = tiny_decode
    pt = wl.page_table.numpy()
    vals, scales = O.page_values_and_scales(wl.layers[0].k_pool.numpy())
    found = 0
    for t, L in enumerate(wl.seq_len.tolist()):
        nb = O.num_blocks(L)
        logit, _ = O.dense_row_scores(wl.layers[0], pt, 0, t, L)
        keys, _ = O.block_keys(logit, L)
        sig = {}
        for b in range(nb - 1):
            p, o = pt[t, b // 8], (b % 8) * 8
            key = (vals[p, o : o + 8].tobytes(), scales[p, o : o + 8].tobytes())
            sig.setdefault(key, []).append(b)
        for dup in (v for v in sig.values() if len(v) > 1):
            found += 1
            assert len({keys[b] for b in dup}) == 1  # identical blocks tie exactly
            lo, hi = dup[0], dup[-1]
            # cut the ranking between the two copies: the lower id must win
            others = [b for b in range(nb) if keys[b] > keys[lo] or (keys[b] == keys[lo] and b < lo)]
            K = len(others) + 1
            blocks, nvalid = O.select_blocks(keys, nb, K)
            assert lo in blocks[:nvalid] and hi not in blocks[:nvalid]
    assert found > 0


# ----------------------------------------------------------------------------- planted mistakes
def test_planted_sign_error_is_caught(monkeypatch):
    good = O.decode_e2m1
    monkeypatch.setattr(O, "decode_e2m1", lambda c: np.abs(good(c)))
    with pytest.raises(AssertionError):
        test_e2m1_decoder_via_e4m3_bit_fields()


def test_planted_dropped_relu_is_caught(monkeypatch):
    def no_relu(q, w, k, ks):
        x = (q @ k.T) * ks[None, :]
        return np.asarray(w, np.float64) @ x, np.abs(np.asarray(w, np.float64)) @ np.abs(x)
    monkeypatch.setattr(O, "score_positions", no_relu)
    with pytest.raises(AssertionError):
        test_scores_relu_zeroes_negative_heads_exactly()


def test_planted_nibble_swap_is_caught(monkeypatch):
    def swapped(p):
        p = np.asarray(p, np.uint8)
        out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
        out[..., 0::2], out[..., 1::2] = p >> 4, p & 15
        return out
    monkeypatch.setattr(O, "unpack_fp4", swapped)
    with pytest.raises(AssertionError):
        test_fp4_nibble_order_low_first()


def test_planted_tie_rule_flip_is_caught(monkeypatch):
    def higher_id_wins(keys, nb, K):
        out = np.full(K, O.INT32_MAX, dtype=np.int64)
        if nb <= K:
            chosen = np.arange(nb)
        else:
            ids = np.arange(nb)
            chosen = np.sort(np.lexsort((-ids, -np.asarray(keys[:nb])))[:K])
        out[: len(chosen)] = chosen
        return out, min(nb, K)
    monkeypatch.setattr(O, "select_blocks", higher_id_wins)
    with pytest.raises(AssertionError):
        test_select_blocks_bruteforce_ranks()


def test_planted_transposed_key_index_is_caught(monkeypatch):
    def wrong_scale(q, w, k, ks):
        x = (q @ k.T) * ks[::-1][None, :]
        r = np.maximum(x, 0.0)
        return np.asarray(w) @ r, np.abs(np.asarray(w)) @ r
    monkeypatch.setattr(O, "score_positions", wrong_scale)
    with pytest.raises(AssertionError):
        test_scores_match_bruteforce_loops()


def test_planted_mxfp4_scale_byte_order_is_caught(monkeypatch):
    good = O.page_values_and_scales_mxfp4

    def reversed_bytes(pool):
        vals, scales = good(pool)
        return vals, scales[..., ::-1]
    monkeypatch.setattr(O, "page_values_and_scales_mxfp4", reversed_bytes)
    with pytest.raises(AssertionError):
        test_mxfp4_pool_layout_hand_example()
