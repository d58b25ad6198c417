"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small workloads are checked row by row in full; the five standard workloads
run at full size in the same launch configuration the benchmark uses and are
checked on sampled rows (every output of a sampled row: keys, published
blocks, the source's own top-512 and the four consumers' top-512).
"""
import math

import numpy as np
import pytest
import torch

from oracle import ci_oracle as O
from oracle import compare
from two_level_sparse_gb300 import synth

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
MX = synth.KV_MXFP4


@pytest.fixture(scope="module")
def ci():
    from two_level_sparse_gb300 import ci as mod

    return mod


def run_step(wl_cpu, device="cuda", with_scores=True, wl_dev=None):
    from two_level_sparse_gb300.step import IndexerStep

    step = IndexerStep(wl_dev if wl_dev is not None else wl_cpu.to(device), with_scores=with_scores)
    step.run()
    torch.cuda.synchronize()
    return step


def assert_ok(rep):
    assert rep.ok, rep


@needs_cuda
def test_tiny_decode_config_all_rows(ci):
    wl = synth.config_workload(0)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    rep = compare.check_step(wl, step.outputs_numpy())
    assert_ok(rep)


@needs_cuda
@pytest.mark.parametrize("lens,K,P", [
    ([0, 1, 7, 8, 9, 100, 2100, 20000], 128, 512),   # empty row, ragged tails, keep-all and selecting rows
    ([5000, 5001, 4096, 4095, 65], 64, 40),           # small top-k, selection on every long row
    ([1500, 3000], 600, 2048),                        # topk larger than every candidate set
])
def test_small_decode_all_rows(ci, lens, K, P):
    wl = synth.make_workload("dec", synth.LAYOUT_DECODE, lens, topk_blocks=K, seed=101, topk=P)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


@needs_cuda
@pytest.mark.parametrize("rows,base,K", [(7, 3000, 64), (4, 129, 8), (10, 2040, 200)])
def test_small_prefill_all_rows(ci, rows, base, K):
    # causal rows of one request; rows % 3 != 0 leaves a ragged last row group
    lens = [base + i for i in range(rows)]
    wl = synth.make_workload("pre", synth.LAYOUT_PREFILL, lens, topk_blocks=K, seed=202)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


def _four_vector_pools(wl, seed):
    """Every layer's pool rewritten so that each position holds one of four K
    vectors (values and scale bytes together; FP8 pools get one fp32 scale)."""
    rng = np.random.default_rng(seed)
    for ly in wl.layers:
        if O.is_mxfp4_pool(ly.k_pool.numpy()):
            pages = ly.k_pool.numpy().reshape(-1, O.PAGE_BYTES_MXFP4)  # shares the tensor's memory
            vals = pages[:, : O.PAGE_VALUE_BYTES_MXFP4].reshape(-1, O.PAGE, O.D // 2)
            scales = pages[:, O.PAGE_VALUE_BYTES_MXFP4 :].reshape(-1, O.PAGE, O.D // 32)
            pick = rng.integers(0, 4, size=vals.shape[:2])
            four_v, four_s = vals[0, :4].copy(), scales[0, :4].copy()
            vals[:] = four_v[pick]
            scales[:] = four_s[pick]
        else:
            pages = ly.k_pool.numpy().reshape(-1, O.PAGE_BYTES)
            vals = pages[:, : O.PAGE_VALUE_BYTES].reshape(-1, O.PAGE, O.D)
            four = vals[0, :4].copy()
            vals[:] = four[rng.integers(0, 4, size=vals.shape[:2])]
            pages[:, O.PAGE_VALUE_BYTES :].view("<f4")[:] = np.float32(0.75)


@needs_cuda
@pytest.mark.parametrize("case", ["decode", "prefill", "varlen", "decode_mxfp4", "prefill_mxfp4", "decode_dcp2",
                                  "prefill_dcp4"])
def test_position_ties_go_to_the_lower_position(ci, case):
    """Pools of four distinct K vectors: a row's scores take four values, so
    every top-512 cuts through a long run of bit-identical scores.  The
    source layer's positions must equal the dense definition's and each
    consumer's the oracle's top-512 of its candidates exactly: score
    descending, ties toward the lower position (sglang PR #40352, Design,
    "Level two"; the source keeps P + 1 blocks, so its top-P is the dense one
    even through ties).  The context-sharded cases take the same positions
    through the exact merge across shards (vLLM sparse_attn_indexer.py,
    _merge_dcp_topk_global: a stable top-k over (score, global id))."""
    kv = MX if case.endswith("mxfp4") else synth.KV_FP8
    if case.startswith("decode"):
        wl = synth.make_workload("ties", synth.LAYOUT_DECODE, [3000, 5001, 9000, 700], 128, seed=71, kv=kv)
    elif case.startswith("prefill"):
        wl = synth.make_workload("ties", synth.LAYOUT_PREFILL, [6000 + 37 * i for i in range(5)], 128, seed=73,
                                 kv=kv)
    else:
        wl = synth.make_varlen_workload("ties", (2000, 0, 7000), (2, 3, 2), 128, seed=75)
    _four_vector_pools(wl, 72)
    if "dcp" in case:
        from two_level_sparse_gb300.dcp import DcpStep

        step = DcpStep(wl.to("cuda"), int(case[-1]))
        step.run()
        torch.cuda.synchronize()
    else:
        step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    out = step.outputs_numpy()
    pt, row_req, P = wl.page_table.numpy(), wl.row_req(), wl.topk
    cut_ties = 0
    for t, L in enumerate(wl.seq_len.tolist()):
        logit, _ = O.dense_row_scores(wl.layers[0], pt, wl.layout, t, L, row_req)
        want = O.top_positions(logit, np.arange(L), P)
        np.testing.assert_array_equal(out["pos"][0][t], want, err_msg=f"row {t} layer 0")
        if L > P:
            kth = logit[want[want >= 0]].min()
            cut_ties += int(np.sum(logit == kth) > np.sum(logit[want[want >= 0]] == kth))
        blocks, nv = np.asarray(out["blocks"][t], dtype=np.int64), int(out["nvalid"][t])
        for j in range(1, len(wl.layers)):
            want_j, _, _, _ = O.select_row(wl.layers[j], pt, wl.layout, t, L, blocks, nv, P, row_req)
            np.testing.assert_array_equal(out["pos"][j][t], want_j, err_msg=f"row {t} layer {j}")
    assert cut_ties > 0  # the threshold did fall inside a run of ties
    assert_ok(compare.check_step(wl, out))


@needs_cuda
def test_duplicate_blocks_score_bit_identically(ci):
    # every copy of a block must get bit-identical keys (the tie rule needs it)
    wl = synth.make_workload("dup", synth.LAYOUT_DECODE, [4000, 3000], topk_blocks=16, seed=9, dup_frac=0.2)
    step = run_step(wl)
    keys = step.keys.cpu().numpy()
    vals, scales = O.page_values_and_scales(wl.layers[0].k_pool.numpy())
    pt = wl.page_table.numpy()
    pairs = 0
    for t, L in enumerate(wl.seq_len.tolist()):
        sig = {}
        for b in range(O.num_blocks(L) - 1):
            p, o = pt[t, b // 8], (b % 8) * 8
            sig.setdefault((vals[p, o:o + 8].tobytes(), scales[p, o:o + 8].tobytes()), []).append(b)
        for group in sig.values():
            if len(group) > 1:
                pairs += 1
                assert len({keys[t, b].tobytes() for b in group}) == 1
    assert pairs > 0


@needs_cuda
def test_dense_keys_equal_sparse_rescoring_bitwise(ci):
    # The sparse scorer reproduces the dense scorer's fp32 scores bit for bit,
    # which the source's own top-512 through its top-(P+1) blocks relies on:
    # with every block a candidate and topk >= L, select returns every position
    # with its score, and each block's maximum must equal its dense key.
    from two_level_sparse_gb300.step import IndexerStep

    lens = [2000, 2001, 2002, 2040]
    wl = synth.make_workload("lemma", synth.LAYOUT_PREFILL, lens, topk_blocks=64, seed=5)
    dev = wl.to("cuda")
    step = IndexerStep(dev)
    step.run()
    rows, L = wl.rows, max(lens)
    nb = O.num_blocks(L)
    allb = torch.arange(nb, dtype=torch.int32, device="cuda").repeat(rows, 1).contiguous()
    nv = torch.tensor([O.num_blocks(x) for x in lens], dtype=torch.int32, device="cuda")
    pos = torch.empty(rows, 2048, dtype=torch.int32, device="cuda")
    sc = torch.empty(rows, 2048, dtype=torch.float32, device="cuda")
    src = dev.layers[0]
    ci.ci_select_sparse(src.q_fp4, src.q_sf, src.w, src.k_pool, dev.page_table, dev.layout, dev.seq_len, L, allb, nv,
                        nb, 2048, pos, sc)
    torch.cuda.synchronize()
    keys = step.keys.cpu().numpy()
    pos, sc = pos.cpu().numpy(), sc.cpu().numpy()
    for t, Lt in enumerate(lens):
        assert pos[t, :Lt].tolist() == list(range(Lt)) and np.all(pos[t, Lt:] == -1)
        for b in range(O.num_blocks(Lt) - 1):
            assert keys[t, b].tobytes() == sc[t, 8 * b:8 * b + 8].max().tobytes(), (t, b)


@needs_cuda
def test_device_error_flags_bad_page_without_fault(ci):
    wl = synth.make_workload("bad", synth.LAYOUT_DECODE, [3000, 2000], topk_blocks=64, seed=3)
    dev = wl.to("cuda")
    dev.page_table[1, 3] = 10**6  # outside the pool: the kernel must skip it and flag
    from two_level_sparse_gb300.step import IndexerStep

    step = IndexerStep(dev)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) & ci.DEVERR_PAGE
    # row 0 is untouched by the corruption
    rep = compare.check_step(wl, step.outputs_numpy(), rows=[0])
    assert_ok(rep)


@needs_cuda
def test_device_error_flags_length_above_max(ci):
    wl = synth.make_workload("len", synth.LAYOUT_DECODE, [3000, 2000], topk_blocks=64, seed=4)
    dev = wl.to("cuda")
    keys = torch.zeros(2, 512, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = dev.layers[0]
    # claim max_len 2500 although row 0 has 3000 positions
    ci.ci_score_dense_amax8(src.q_fp4, src.q_sf, src.w, src.k_pool, dev.page_table, dev.layout, dev.seq_len, 2500, 8,
                            keys, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ci.DEVERR_LEN


@needs_cuda
def test_empty_batch_is_a_no_op(ci):
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    u8 = torch.empty(0, 64, 64, dtype=torch.uint8, device="cuda")
    pool = torch.zeros(1, synth.PAGE_BYTES, dtype=torch.uint8, device="cuda")
    pt = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    keys = torch.empty(0, 8, dtype=torch.float32, device="cuda")
    ci.ci_score_dense_amax8(u8, torch.empty(0, 64, 4, dtype=torch.uint8, device="cuda"),
                            torch.empty(0, 64, dtype=torch.float32, device="cuda"), pool, pt, 1, e, 0, 0, keys)
    torch.cuda.synchronize()


# ----------------------------------------------------------------------------- full-size workloads
SAMPLES = {
    1: [0, 1, 31, 62, 63],
    2: None,  # chosen below: short (keep-all) and long rows
    3: [0, 1, 2, 2047, 4093, 4094, 4095],
    4: [0, 1, 2, 5000, 9999, 16381, 16382, 16383],
}


@needs_cuda
@pytest.mark.parametrize("cid", [1, 2, 3, 4])
def test_full_size_config_sampled_rows(ci, cid):
    wl_dev = synth.config_workload(cid, device="cuda")
    step = run_step(None, wl_dev=wl_dev)
    assert int(step.dev_err.item()) == 0
    if cid == 2:
        lens = wl_dev.seq_len.cpu()
        short = [int(i) for i in torch.nonzero(lens <= 16384).flatten()[:2]]
        long = [int(i) for i in torch.nonzero(lens > 131072).flatten()[:3]]
        rows = short + long + [int(torch.argmax(lens))]
    else:
        rows = SAMPLES[cid]
    sub = subset_workload(wl_dev, rows)
    out = step.outputs_numpy()
    sub_out = {k: (v[:, rows] if k in ("pos", "score") else v[rows]) for k, v in out.items()}
    assert_ok(compare.check_step(sub, sub_out))


@needs_cuda
def test_full_size_prefill_chunk_more_rows(ci):
    """Sixteen more rows of the 16384-row chunk at 262144 positions, spread
    over the chunk with every residue mod 3 and mod 4 (the dense pass's
    three-row groups, the publish kernel's four row groups per CTA, the
    select's CTAs), against the oracle: keys, both block tables and every
    layer's top-512."""
    wl_dev = synth.config_workload(4, device="cuda")
    step = run_step(None, wl_dev=wl_dev)
    assert int(step.dev_err.item()) == 0
    rows = [1021 * i + (i % 3) for i in range(16)]
    assert len({r % 3 for r in rows}) == 3 and len({r % 4 for r in rows}) == 4
    sub = subset_workload(wl_dev, rows)
    out = step.outputs_numpy()
    sub_out = {k: (v[:, rows] if k in ("pos", "score") else v[rows]) for k, v in out.items()}
    assert_ok(compare.check_step(sub, sub_out))


def subset_workload(wl_dev, rows):
    """The sampled rows' operands on the CPU (the whole pool comes along)."""
    idx = torch.tensor(rows, dtype=torch.long, device=wl_dev.seq_len.device)
    layers = [synth.Layer(l.q_fp4[idx].cpu(), l.q_sf[idx].cpu(), l.w[idx].cpu(), l.k_pool.cpu()) for l in wl_dev.layers]
    if wl_dev.layout == synth.LAYOUT_VARLEN:
        # every sampled row becomes a one-row request that reads its own request's pages
        req = torch.as_tensor(wl_dev.row_req()[rows], dtype=torch.long)
        starts = torch.arange(len(rows) + 1, dtype=torch.int32)
        return synth.Workload(wl_dev.name, wl_dev.layout, wl_dev.seq_len[idx].cpu(), wl_dev.page_table.cpu()[req],
                              layers, wl_dev.topk_blocks, wl_dev.topk, starts)
    pt = wl_dev.page_table[idx].cpu() if wl_dev.layout == synth.LAYOUT_DECODE else wl_dev.page_table.cpu()
    return synth.Workload(wl_dev.name, wl_dev.layout, wl_dev.seq_len[idx].cpu(), pt, layers, wl_dev.topk_blocks,
                          wl_dev.topk)


@needs_cuda
@pytest.mark.parametrize("rows", [40, 400])
@pytest.mark.parametrize("K1,K2", [(2048, 513), (128, 513), (513, 64), (4096, 1000)])
def test_publish_pair_equals_two_single_publishes(ci, K1, K2, rows):
    """ci_publish_blocks2 returns exactly the two single selections, which
    equal the oracle's block selection (ties toward the lower block id), on
    few rows (one per CTA) and on many (four per SM)."""
    g = torch.Generator().manual_seed(7 + rows)
    lens = torch.randint(1, 40000, (rows,), generator=g, dtype=torch.int32)
    lens[:4] = torch.tensor([1, 8 * K1, 8 * K2 + 3, 8 * max(K1, K2) + 1], dtype=torch.int32)
    max_len = int(lens.max())
    stride = ((max_len + 7) // 8 + 7) // 8 * 8
    # few distinct values so that many keys tie
    keys = (torch.randint(0, 300, (rows, stride), generator=g).float() / 7.0 - 20.0)
    keys[5, :200] = -float("inf")
    dev = "cuda"
    kd, ld = keys.to(dev), lens.to(dev)
    b1 = torch.empty(rows, K1, dtype=torch.int32, device=dev)
    n1 = torch.empty(rows, dtype=torch.int32, device=dev)
    b2 = torch.empty(rows, K2, dtype=torch.int32, device=dev)
    n2 = torch.empty(rows, dtype=torch.int32, device=dev)
    s1, m1 = torch.empty_like(b1), torch.empty_like(n1)
    s2, m2 = torch.empty_like(b2), torch.empty_like(n2)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ci.ci_publish_blocks2(ld, max_len, kd, K1, b1, n1, K2, b2, n2, dev_err=err)
    ci.ci_publish_blocks(ld, max_len, kd, K1, s1, m1, dev_err=err)
    ci.ci_publish_blocks(ld, max_len, kd, K2, s2, m2, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(b1, s1) and torch.equal(n1, m1)
    assert torch.equal(b2, s2) and torch.equal(n2, m2)
    b1h, b2h = b1.cpu().numpy(), b2.cpu().numpy()
    for t in range(rows):
        nb = O.num_blocks(int(lens[t]))
        kr = keys[t, :nb].double().numpy()
        for K, out in ((K1, b1h), (K2, b2h)):
            ids, nv = O.select_blocks(kr, nb, K)
            assert nv == min(nb, K)
            assert np.array_equal(out[t, :nv], ids[:nv]), (t, K)
            assert np.all(out[t, nv:] == 0x7FFFFFFF)


def _publish_rows_against_oracle(ci, keys, lens, K1, K2):
    """ci_publish_blocks2 on the given keys against the oracle's selection."""
    rows, stride = keys.shape
    max_len = int(lens.max())
    dev = "cuda"
    kd, ld = keys.to(dev).contiguous(), lens.to(dev)
    b1 = torch.full((rows, K1), -5, dtype=torch.int32, device=dev)
    n1 = torch.empty(rows, dtype=torch.int32, device=dev)
    b2 = torch.full((rows, K2), -5, dtype=torch.int32, device=dev)
    n2 = torch.empty(rows, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ci.ci_publish_blocks2(ld, max_len, kd, K1, b1, n1, K2, b2, n2, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    b1h, b2h, n1h, n2h = b1.cpu().numpy(), b2.cpu().numpy(), n1.cpu().numpy(), n2.cpu().numpy()
    for t in range(rows):
        nb = O.num_blocks(int(lens[t]))
        kr = keys[t, :nb].double().numpy()
        for K, out, nv_out in ((K1, b1h, n1h), (K2, b2h, n2h)):
            ids, nv = O.select_blocks(kr, nb, K)
            assert int(nv_out[t]) == nv
            assert np.array_equal(out[t, :nv], ids[:nv]), (t, K)
            assert np.all(out[t, nv:] == 0x7FFFFFFF)


@needs_cuda
@pytest.mark.parametrize("rows", [24, 320])
@pytest.mark.parametrize("case", ["normal", "ties", "sample_adversarial", "mid_length", "wider_second"])
def test_publish_long_rows_match_the_oracle(ci, case, rows):
    """Rows of thousands of blocks, whose threshold the publish kernel brackets
    from a strided sample of the keys (with the radix path behind it when the
    sample's bound misses): the oracle's selection, ties toward the lower id,
    in every case -- random keys, keys with heavy ties at the threshold, keys
    whose every sampled position (each 16th block) outranks all the others so
    that the sample's bound fails, rows of 4096 - 8192 blocks, and a second
    selection wider than the first.  24 rows take the one-row-per-CTA kernel,
    320 rows (two per SM or more) the kernel with four rows per SM."""
    g = torch.Generator().manual_seed(91 + rows)
    L = 262144
    lens = torch.full((rows,), L, dtype=torch.int32)
    lens[1] = L - 5  # a ragged newest block
    K1, K2 = 2048, 513
    if case == "mid_length":
        lens = torch.randint(8 * 4096, 8 * 8192, (rows,), generator=g, dtype=torch.int32)
    stride = ((int(lens.max()) + 7) // 8 + 7) // 8 * 8
    keys = torch.randn(rows, stride, generator=g)
    if case == "ties":
        keys = torch.round(keys * 3.0) / 3.0  # a handful of distinct values: long runs of ties at the threshold
    elif case == "sample_adversarial":
        keys[:, ::16] += 50.0
    elif case == "wider_second":
        K1, K2 = 128, 513
    keys[2, : stride // 2] = -float("inf")
    _publish_rows_against_oracle(ci, keys, lens, K1, K2)



@needs_cuda
@pytest.mark.parametrize("cid", [1, 3])
def test_positions_without_scores_match_with_scores(ci, cid):
    """The benchmark runs the step without the optional score output; its
    positions must be exactly those of the scored run the oracle checks."""
    from two_level_sparse_gb300.step import IndexerStep

    dev = synth.config_workload(cid, device="cuda")
    a = IndexerStep(dev, with_scores=True)
    b = IndexerStep(dev, with_scores=False)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert int(a.dev_err.item()) == 0 and int(b.dev_err.item()) == 0
    assert torch.equal(a.pos, b.pos)
    assert torch.equal(a.blocks, b.blocks) and torch.equal(a.blocks_src, b.blocks_src)


@needs_cuda
@pytest.mark.parametrize("prefixes,rows_per_req,K", [
    ((300, 2040, 0, 5000), (4, 1, 2, 5), 64),     # requests of 1, 2, 4 and 5 rows: ragged row triples
    ((3000, 3000, 100), (3, 3, 3), 200),           # equal requests, one short enough to keep all its blocks
    ((20000,), (7,), 2048),                        # a single request through the several-requests layout
])
def test_varlen_prefill_all_rows(ci, prefixes, rows_per_req, K):
    wl = synth.make_varlen_workload("var", prefixes, rows_per_req, K, seed=303)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


@needs_cuda
def test_varlen_bad_row_starts_flag_without_fault(ci):
    wl = synth.make_varlen_workload("bad", (500, 700), (3, 3), 16, seed=7)
    dev = wl.to("cuda")
    dev.req_start[1] = 7  # beyond the rows: not a partition
    from two_level_sparse_gb300.step import IndexerStep

    step = IndexerStep(dev)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) & ci.DEVERR_REQ


@needs_cuda
def test_varlen_chunk_sampled_rows(ci):
    """A 16384-row chunk of four requests (prefixes 16 K - 240 K) in the
    benchmark's launch configuration, checked on rows at every request edge."""
    wl_dev = synth.varlen_chunk_workload(device="cuda")
    step = run_step(None, wl_dev=wl_dev)
    assert int(step.dev_err.item()) == 0
    starts = wl_dev.req_start.tolist()
    rows = sorted({r for s0 in starts[:-1] for r in (s0, s0 + 1, s0 + 2)} | {s1 - 1 for s1 in starts[1:]} | {9000})
    sub = subset_workload(wl_dev, rows)
    out = step.outputs_numpy()
    sub_out = {k: (v[:, rows] if k in ("pos", "score") else v[rows]) for k, v in out.items()}
    assert_ok(compare.check_step(sub, sub_out))



def run_tail(ci, rows_per_req, tail_lens, K, cap, seed):
    """ci_prefill_tail over a seeded table of block ids (any int32 values:
    the op only moves rows); returns the table, its counts and the outputs."""
    g = torch.Generator().manual_seed(seed)
    starts = torch.zeros(len(rows_per_req) + 1, dtype=torch.int32)
    starts[1:] = torch.cumsum(torch.as_tensor(rows_per_req, dtype=torch.int32), 0)
    rows = int(starts[-1])
    blocks = torch.randint(-2**31, 2**31 - 1, (rows, K), generator=g, dtype=torch.int32)
    nvalid = torch.randint(0, K + 1, (rows,), generator=g, dtype=torch.int32)
    dev = dict(req_start=starts.cuda(), tail_len=torch.as_tensor(tail_lens, dtype=torch.int32).cuda(),
               blocks=blocks.cuda(), nvalid=nvalid.cuda())
    out_row = torch.full((cap,), 12345, dtype=torch.int32, device="cuda")
    out_blocks = torch.full((cap, K), 12345, dtype=torch.int32, device="cuda")
    out_nvalid = torch.full((cap,), 12345, dtype=torch.int32, device="cuda")
    out_count = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ci.ci_prefill_tail(dev["req_start"], dev["tail_len"], dev["blocks"], dev["nvalid"], out_row, out_blocks, out_nvalid,
                       out_count, dev_err=dev_err)
    torch.cuda.synchronize()
    return (starts.numpy(), blocks.numpy(), nvalid.numpy(), out_row.cpu().numpy(), out_blocks.cpu().numpy(),
            out_nvalid.cpu().numpy(), int(out_count.item()), int(dev_err.item()))


@needs_cuda
@pytest.mark.parametrize("rows_per_req,tail_lens,K,extra", [
    ((5, 1, 0, 7, 300), (2, 3, 4, 7, 129), 16, 0),        # tail shorter, longer, empty request, whole, long
    ((4, 4, 4), (0, -3, 4), 2048, 5),                     # nothing kept, negative length, spare capacity padded
    ((1,) * 4096, tuple(i % 2 for i in range(4096)), 64, 3),  # the most requests: every other one kept
    ((16384,), (4096,), 2048, 0),                         # one long request, the tail a quarter of it
    ((3, 5, 2), (2, 4, 9), 13, 2),                        # rows of 13 ids: 4-byte copies, no 16-byte path
])
def test_prefill_tail_gathers_tail_rows_bit_exact(ci, rows_per_req, tail_lens, K, extra):
    starts, blocks, nvalid, _, _, _, _, _ = run_tail(ci, rows_per_req, tail_lens, K, 0, seed=11)
    want = O.prefill_tail_rows(starts, tail_lens)
    cap = len(want) + extra
    _, _, _, out_row, out_blocks, out_nvalid, count, err = run_tail(ci, rows_per_req, tail_lens, K, cap, seed=11)
    assert err == 0 and count == len(want)
    np.testing.assert_array_equal(out_row[:count], want)
    np.testing.assert_array_equal(out_blocks[:count], blocks[want])
    np.testing.assert_array_equal(out_nvalid[:count], nvalid[want])
    assert (out_row[count:] == -1).all() and (out_nvalid[count:] == 0).all()
    assert (out_blocks[count:] == 0x7FFFFFFF).all()


@needs_cuda
def test_prefill_tail_short_capacity_flags_and_writes_the_first_rows(ci):
    rows_per_req, tail_lens = (10, 20, 30), (5, 10, 15)
    starts, blocks, nvalid, out_row, out_blocks, out_nvalid, count, err = run_tail(ci, rows_per_req, tail_lens, 32, 12,
                                                                                   seed=3)
    want = O.prefill_tail_rows(starts, tail_lens)
    assert count == len(want) == 30 and err & ci.DEVERR_REQ
    np.testing.assert_array_equal(out_row, want[:12])
    np.testing.assert_array_equal(out_blocks, blocks[want[:12]])
    np.testing.assert_array_equal(out_nvalid, nvalid[want[:12]])


@needs_cuda
def test_prefill_tail_after_a_varlen_step_matches_the_oracle(ci):
    """The tail of a real multi-request chunk: the gathered candidate blocks of
    each tail row are the oracle's selection for that row."""
    wl = synth.make_varlen_workload("tail", (300, 2040, 5000), (4, 9, 5), 64, seed=21)
    dev = wl.to("cuda")
    step = run_step(None, wl_dev=dev)
    tail_lens = torch.tensor([2, 9, 0], dtype=torch.int32, device="cuda")
    want = O.prefill_tail_rows(wl.req_start.numpy(), tail_lens.cpu().numpy()).tolist()
    n = len(want)
    out_row = torch.empty(n, dtype=torch.int32, device="cuda")
    out_blocks = torch.empty(n, step.blocks.shape[1], dtype=torch.int32, device="cuda")
    out_nvalid = torch.empty(n, dtype=torch.int32, device="cuda")
    out_count = torch.empty(1, dtype=torch.int32, device="cuda")
    ci.ci_prefill_tail(dev.req_start, tail_lens, step.blocks, step.nvalid, out_row, out_blocks, out_nvalid, out_count,
                       dev_err=step.dev_err)
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0 and int(out_count.item()) == n
    assert out_row.cpu().tolist() == want
    sub = subset_workload(dev, want)
    out = step.outputs_numpy()
    sub_out = {k: (v[:, want] if k in ("pos", "score") else v[want]) for k, v in out.items()}
    sub_out["blocks"] = out_blocks.cpu().numpy()
    sub_out["nvalid"] = out_nvalid.cpu().numpy()
    assert_ok(compare.check_step(sub, sub_out))


# ----------------------------------------------------------------------------- MXFP4 index-K


@needs_cuda
def test_mxfp4_tiny_decode_config_all_rows(ci):
    wl = synth.config_workload(0, kv=MX)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


@needs_cuda
@pytest.mark.parametrize("layout,lens,K,P", [
    (synth.LAYOUT_DECODE, [0, 1, 7, 8, 9, 100, 2100, 20000], 128, 512),
    (synth.LAYOUT_DECODE, [5000, 5001, 4096, 4095, 65], 64, 40),
    (synth.LAYOUT_PREFILL, [3000 + i for i in range(7)], 64, 512),
    (synth.LAYOUT_PREFILL, [2040 + i for i in range(10)], 200, 512),
])
def test_mxfp4_small_all_rows(ci, layout, lens, K, P):
    wl = synth.make_workload("mx", layout, lens, topk_blocks=K, seed=404, topk=P, kv=MX)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


@needs_cuda
def test_mxfp4_varlen_prefill_all_rows(ci):
    wl = synth.make_varlen_workload("mxv", (300, 2040, 0, 5000), (4, 1, 2, 5), 64, seed=505, kv=MX)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


@needs_cuda
def test_mxfp4_dense_keys_equal_sparse_rescoring_bitwise(ci):
    """The lemma's premise for MXFP4 pools: the sparse scorer's scores equal
    the dense scorer's bit for bit (every block a candidate, topk >= L)."""
    from two_level_sparse_gb300.step import IndexerStep

    lens = [2000, 2001, 2002, 2040]
    wl = synth.make_workload("lemma4", synth.LAYOUT_PREFILL, lens, topk_blocks=64, seed=6, kv=MX)
    dev = wl.to("cuda")
    step = IndexerStep(dev)
    step.run()
    rows, L = wl.rows, max(lens)
    nb = O.num_blocks(L)
    allb = torch.arange(nb, dtype=torch.int32, device="cuda").repeat(rows, 1).contiguous()
    nv = torch.tensor([O.num_blocks(x) for x in lens], dtype=torch.int32, device="cuda")
    pos = torch.empty(rows, 2048, dtype=torch.int32, device="cuda")
    sc = torch.empty(rows, 2048, dtype=torch.float32, device="cuda")
    src = dev.layers[0]
    ci.ci_select_sparse(src.q_fp4, src.q_sf, src.w, src.k_pool, dev.page_table, dev.layout, dev.seq_len, L, allb, nv,
                        nb, 2048, pos, sc)
    torch.cuda.synchronize()
    keys = step.keys.cpu().numpy()
    pos, sc = pos.cpu().numpy(), sc.cpu().numpy()
    for t, Lt in enumerate(lens):
        assert pos[t, :Lt].tolist() == list(range(Lt)) and np.all(pos[t, Lt:] == -1)
        for b in range(O.num_blocks(Lt) - 1):
            assert keys[t, b].tobytes() == sc[t, 8 * b:8 * b + 8].max().tobytes(), (t, b)


@needs_cuda
@pytest.mark.parametrize("cid", [2, 4])
def test_mxfp4_full_size_config_sampled_rows(ci, cid):
    """The long-decode batch and the 16384-row chunk with MXFP4 pools, in the
    benchmark's launch configuration, checked on sampled rows."""
    wl_dev = synth.config_workload(cid, device="cuda", kv=MX)
    step = run_step(None, wl_dev=wl_dev)
    assert int(step.dev_err.item()) == 0
    if cid == 2:
        lens = wl_dev.seq_len.cpu()
        rows = [int(i) for i in torch.nonzero(lens <= 16384).flatten()[:1]] + [int(torch.argmax(lens))]
    else:
        rows = [0, 2, 9999, 16383]
    sub = subset_workload(wl_dev, rows)
    out = step.outputs_numpy()
    sub_out = {k: (v[:, rows] if k in ("pos", "score") else v[rows]) for k, v in out.items()}
    assert_ok(compare.check_step(sub, sub_out))


# ----------------------------------------------------------------------------- query producer
def _producer_inputs(tokens, seed, max_pos=4096):
    from oracle import q_producer as QP

    g = torch.Generator().manual_seed(seed)
    mag = 10.0 ** (torch.rand(tokens, 64, 1, generator=g) * 6 - 3)
    q = (torch.randn(tokens, 64, 128, generator=g) * mag).to(torch.bfloat16)
    q[0, 0] = 0  # an all-zero head
    q[0, 1, 5] = -0.0
    ang = torch.rand(max_pos, 32, generator=g, dtype=torch.float64) * 2 * math.pi
    cos_sin = torch.cat([torch.cos(ang), torch.sin(ang)], 1).float()
    pos = torch.randint(0, max_pos, (tokens,), generator=g, dtype=torch.int32)
    w = torch.randn(tokens, 64, generator=g) * 0.125
    return pos, q, cos_sin, w, QP


def _run_producer(ci, pos, q, cos_sin, w, neox, fmt, dev_err=None):
    t = q.shape[0]
    d = "cuda"
    q_out = torch.empty(t, 64, 128 if fmt == ci.Q_FP8 else 64, dtype=torch.uint8, device=d)
    q_sf = torch.empty(t, 64, 4, dtype=torch.uint8, device=d) if fmt == ci.Q_MXFP4 else None
    w_out = torch.empty(t, 64, dtype=torch.float32, device=d)
    ci.ci_q_rope_quant(pos.to(d), q.to(d), cos_sin.to(d), w.to(d), 0.0625, 0.125, neox, fmt, q_out, q_sf, w_out,
                       dev_err=dev_err)
    torch.cuda.synchronize()
    return q_out.cpu().numpy(), None if q_sf is None else q_sf.cpu().numpy(), w_out.cpu().numpy()


@needs_cuda
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("fmt", ["mxfp4", "fp8"])
def test_q_producer_bit_exact(ci, neox, fmt):
    pos, q, cos_sin, w, QP = _producer_inputs(3000, seed=17)
    code = ci.Q_MXFP4 if fmt == "mxfp4" else ci.Q_FP8
    got = _run_producer(ci, pos, q, cos_sin, w, neox, code)
    want = QP.produce(pos.numpy(), q.view(torch.uint16).numpy(), cos_sin.numpy(), w.numpy(), 0.0625, 0.125, neox, fmt)
    np.testing.assert_array_equal(got[0], want[0])
    if fmt == "mxfp4":
        np.testing.assert_array_equal(got[1], want[1])
    np.testing.assert_array_equal(got[2].view(np.uint32), want[2].view(np.uint32))


@needs_cuda
def test_q_producer_bad_position_flags_without_fault(ci):
    pos, q, cos_sin, w, QP = _producer_inputs(40, seed=3, max_pos=100)
    pos[7] = 100
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_out, q_sf, _ = _run_producer(ci, pos, q, cos_sin, w, True, ci.Q_MXFP4, dev_err=err)
    assert int(err.item()) & ci.DEVERR_POS
    assert not q_out[7].any()


@needs_cuda
def test_q_producer_feeds_the_indexer(ci):
    """bf16 queries -> producer -> indexer step, against the producer oracle
    followed by the indexer oracle: the path from the step before it."""
    lens = [3000 + i for i in range(7)]
    base = synth.make_workload("prod", synth.LAYOUT_PREFILL, lens, topk_blocks=64, seed=77)
    layers = []
    for j, l in enumerate(base.layers):
        pos, q, cos_sin, w, QP = _producer_inputs(len(lens), seed=900 + j)
        q_fp4, q_sf, w_out = _run_producer(ci, pos, q, cos_sin, w, True, ci.Q_MXFP4)
        want = QP.produce(pos.numpy(), q.view(torch.uint16).numpy(), cos_sin.numpy(), w.numpy(), 0.0625, 0.125, True,
                          "mxfp4")
        np.testing.assert_array_equal(q_fp4, want[0])
        layers.append(synth.Layer(torch.from_numpy(q_fp4), torch.from_numpy(q_sf), torch.from_numpy(w_out), l.k_pool))
    wl = synth.Workload("prod", base.layout, base.seq_len, base.page_table, layers, base.topk_blocks, base.topk)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))


# ----------------------------------------------------------------------------- context sharding (one device)
@needs_cuda
@pytest.mark.parametrize("world", [2, 4, 8])
@pytest.mark.parametrize("case", ["decode", "prefill", "varlen"])
def test_dcp_step_equals_unsharded_step_bitwise(ci, world, case):
    """W context shards (interleave 1): local block maxima merged across shards,
    local top-512 merged across shards -- the oracle's keys, blocks, positions
    and scores (vLLM sparse_attn_indexer.py: the MAX-reduce of block scores
    with the global newest block pinned, and _merge_dcp_topk_global's exact
    merge), and bit for bit the unsharded step's."""
    from two_level_sparse_gb300.dcp import DcpStep
    from two_level_sparse_gb300.step import IndexerStep

    if case == "decode":
        wl = synth.make_workload("dcp", synth.LAYOUT_DECODE, [0, 1, 7, 8, 9, 100, 2100, 20000], 128, seed=31)
    elif case == "prefill":
        wl = synth.make_workload("dcp", synth.LAYOUT_PREFILL, [3000 + i for i in range(7)], 64, seed=32)
    else:
        wl = synth.make_varlen_workload("dcp", (300, 2040, 0, 5000), (4, 1, 2, 5), 64, seed=33)
    dev = wl.to("cuda")
    ref = IndexerStep(dev, with_scores=True)
    ref.run()
    d = DcpStep(dev, world)
    d.run()
    torch.cuda.synchronize()
    assert int(d.dev_err.item()) == 0 and int(ref.dev_err.item()) == 0
    a, b = ref.outputs_numpy(), d.outputs_numpy()
    assert_ok(compare.check_step(wl, b))
    for k in ("blocks", "nvalid", "blocks_src", "nvalid_src", "pos"):
        np.testing.assert_array_equal(b[k], a[k], err_msg=k)
    np.testing.assert_array_equal(b["score"].view(np.uint32), a["score"].view(np.uint32))
    nb = (wl.seq_len.numpy() + 7) // 8
    for t in np.nonzero(nb > min(wl.topk_blocks, wl.topk + 1))[0]:
        np.testing.assert_array_equal(b["keys"][t, : nb[t]].view(np.uint32), a["keys"][t, : nb[t]].view(np.uint32))


@needs_cuda
def test_dcp_full_size_prefill_chunk_sampled_rows(ci):
    """The 16384-row chunk at 262144 positions as 2 context shards: the merged
    keys, published blocks and every layer's top-512 of sampled rows against
    the oracle (the exact merge of vLLM sparse_attn_indexer.py,
    _merge_dcp_topk_global)."""
    from two_level_sparse_gb300.dcp import DcpStep

    wl_dev = synth.config_workload(4, device="cuda")
    d = DcpStep(wl_dev, 2)
    d.run()
    torch.cuda.synchronize()
    assert int(d.dev_err.item()) == 0
    rows = [0, 8191, 16383]
    out = d.outputs_numpy()
    sub_out = {k: (v[:, rows] if k in ("pos", "score") else v[rows]) for k, v in out.items()}
    del d
    assert_ok(compare.check_step(subset_workload(wl_dev, rows), sub_out))


@needs_cuda
def test_decode_batch_all_rows(ci):
    """The 64-row decode batch at full size against the oracle on every row."""
    wl_dev = synth.config_workload(1, device="cuda")
    step = run_step(None, wl_dev=wl_dev)
    assert int(step.dev_err.item()) == 0
    rows = list(range(wl_dev.rows))
    assert_ok(compare.check_step(subset_workload(wl_dev, rows), step.outputs_numpy()))


@needs_cuda
@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_select_layers_equals_one_launch_per_layer(ci, case):
    """One ci_select_sparse_layers launch over every layer (the source with
    its top-(P+1) blocks, the consumers with the published K) writes bit for
    bit what one ci_select_sparse launch per layer writes, scores for some
    layers and not others included."""
    from two_level_sparse_gb300.step import IndexerStep

    if case == "decode":  # 5 x 7 (layer, row) units on a grid of 35 CTAs
        wl = synth.make_workload("sl", synth.LAYOUT_DECODE, [9000, 3001, 20000, 64, 4096, 700, 15000], 96, seed=51,
                                 topk=60)
    else:  # 5 x 300 units on one CTA per SM: layer boundaries inside every CTA's sequence
        wl = synth.make_workload("sl", synth.LAYOUT_PREFILL, [2500 + 7 * i for i in range(300)], 48, seed=52, topk=40)
    dev = wl.to("cuda")
    step = IndexerStep(dev, with_scores=True)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0
    for j, layer in enumerate(dev.layers):
        blocks, nvalid, mb = (step.blocks_src, step.nvalid_src, step.Kp) if j == 0 else (step.blocks, step.nvalid,
                                                                                        step.K)
        pos = torch.full_like(step.pos[j], -9)
        score = torch.full_like(step.score[j], 7.0) if j % 2 == 0 else None
        ci.ci_select_sparse(layer.q_fp4, layer.q_sf, layer.w, layer.k_pool, dev.page_table, dev.layout, dev.seq_len,
                            dev.max_len, blocks, nvalid, mb, step.P, pos, score, dev_err=step.dev_err)
        torch.cuda.synchronize()
        assert torch.equal(pos, step.pos[j]), j
        if score is not None:
            assert torch.equal(score.view(torch.int32), step.score[j].view(torch.int32)), j
    # scores for layer 1 only, positions for all: the other layers' score rows stay untouched
    out_pos = torch.full_like(step.pos, -9)
    out_score = torch.full_like(step.score, 7.0)
    layers = []
    for j, layer in enumerate(dev.layers):
        blocks, nvalid, mb = (step.blocks_src, step.nvalid_src, step.Kp) if j == 0 else (step.blocks, step.nvalid,
                                                                                        step.K)
        layers.append(dict(q_fp4=layer.q_fp4, q_sf=layer.q_sf, w=layer.w, k_pool=layer.k_pool, blocks=blocks,
                           nvalid=nvalid, max_blocks=mb, out_pos=out_pos[j], out_score=out_score[j] if j == 1 else None))
    ci.ci_select_sparse_layers(layers, dev.page_table, dev.layout, dev.seq_len, dev.max_len, step.P,
                               dev_err=step.dev_err)
    torch.cuda.synchronize()
    assert torch.equal(out_pos, step.pos)
    assert torch.equal(out_score[1].view(torch.int32), step.score[1].view(torch.int32))
    assert bool((out_score[0] == 7.0).all()) and bool((out_score[2:] == 7.0).all())
    assert int(step.dev_err.item()) == 0


@needs_cuda
def test_select_pools_beyond_l2_one_launch_per_layer(ci):
    """The 64-row decode batch, whose pools do not fit in L2 (so the FP8 K
    scales are fetched tiles ahead): one ci_select_sparse launch per layer
    writes bit for bit what the step's single all-layer launch wrote (and
    test_decode_batch_all_rows checks that one against the oracle)."""
    from two_level_sparse_gb300.step import IndexerStep

    dev = synth.config_workload(1, device="cuda")
    pool_bytes = dev.layers[0].k_pool.numel()
    assert pool_bytes > torch.cuda.get_device_properties(0).L2_cache_size // 2
    step = IndexerStep(dev, with_scores=True)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_err.item()) == 0
    for j, layer in enumerate(dev.layers):
        blocks, nvalid, mb = (step.blocks_src, step.nvalid_src, step.Kp) if j == 0 else (step.blocks, step.nvalid,
                                                                                        step.K)
        pos = torch.full_like(step.pos[j], -9)
        score = torch.full_like(step.score[j], 7.0)
        ci.ci_select_sparse(layer.q_fp4, layer.q_sf, layer.w, layer.k_pool, dev.page_table, dev.layout, dev.seq_len,
                            dev.max_len, blocks, nvalid, mb, step.P, pos, score, dev_err=step.dev_err)
        torch.cuda.synchronize()
        assert torch.equal(pos, step.pos[j]), j
        assert torch.equal(score.view(torch.int32), step.score[j].view(torch.int32)), j
    assert int(step.dev_err.item()) == 0


@needs_cuda
@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_run_host_moves_the_same_results(ci, case):
    """IndexerStep.run_host (pinned host in, pinned host out, copies overlapped
    with the kernels) returns exactly what run() leaves on the device."""
    from two_level_sparse_gb300.step import IndexerStep

    if case == "decode":  # fewer rows than SMs: the select launch spreads every layer's rows over the SMs
        wl = synth.make_workload("rh", synth.LAYOUT_DECODE, [5000, 5001, 4096, 4095, 65], 64, seed=41, topk=40)
    else:
        wl = synth.make_workload("rh", synth.LAYOUT_PREFILL, [3000 + i for i in range(200)], 64, seed=42)
    dev = wl.to("cuda")
    step = IndexerStep(dev)
    step.run()
    torch.cuda.synchronize()
    want = [step.blocks.cpu(), step.nvalid.cpu()] + [step.pos[j].cpu() for j in range(len(wl.layers))]
    shared, layers = step.device_inputs()
    host_shared = [t.cpu().pin_memory() for t in shared]
    host_layers = [[t.cpu().pin_memory() for t in l] for l in layers]
    for t in shared + [x for l in layers for x in l]:
        t.zero_()  # the inputs must come from the host copies
    for j in range(len(wl.layers)):
        step.pos[j].fill_(-7)
    host_out = [torch.empty(w.shape, dtype=w.dtype, pin_memory=True) for w in want]
    step.run_host(host_shared, host_layers, host_out, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for got, exp in zip(host_out, want):
        assert torch.equal(got, exp)


@needs_cuda
@pytest.mark.parametrize("cid", [0])
def test_graph_replay_equals_eager_step(ci, cid):
    """The step captured as a CUDA graph reproduces the eager step's outputs."""
    from two_level_sparse_gb300.step import IndexerStep

    wl = synth.config_workload(cid, device="cuda")
    step = IndexerStep(wl, with_scores=True)
    s = torch.cuda.Stream()
    step.run(s)
    torch.cuda.synchronize()
    want = step.outputs_numpy()
    g = step.capture(s)
    step.pos.fill_(-9)
    step.blocks.fill_(-9)
    g.replay()
    torch.cuda.synchronize()
    got = step.outputs_numpy()
    for k in ("blocks", "nvalid", "pos"):
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    np.testing.assert_array_equal(got["score"].view(np.uint32), want["score"].view(np.uint32))


@needs_cuda
def test_maximum_sizes(ci):
    """The largest supported sizes in one step: a row of 393216 positions
    (the publish limit), 2176 candidate blocks per consumer row (the select
    limit), top-2048 positions (the top-k limit, so the source selects within
    its top 2049 blocks), beside a 17-position row."""
    wl = synth.make_workload("max", synth.LAYOUT_DECODE, [393216, 17], 2176, seed=55, topk=2048)
    step = run_step(wl)
    assert int(step.dev_err.item()) == 0
    assert_ok(compare.check_step(wl, step.outputs_numpy()))
