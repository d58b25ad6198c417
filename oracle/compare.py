"""Acceptance rules for GPU results against the oracle (test infrastructure).

Scores: ``|gpu - oracle| <= 1e-4 * tolmag`` per element, where ``tolmag =
sum_h |w_h * ReLU(q_h . k)|`` of that position.  Index sets: identical, except
for swaps at the selection boundary: every element in the symmetric difference
must have an oracle score within its own tolerance of the oracle's k-th score
(for blocks: the block key, with the tolerance of its arg-max position).  The
consumer layers are judged on the candidate blocks the GPU published, fed to
the oracle, so a legal swap at level one does not cascade.
"""
from __future__ import annotations

import numpy as np

from . import ci_oracle as O

REL_TOL = 1e-4


class Report:
    def __init__(self):
        self.errors = []
        self.stats = {"rows": 0, "key_checks": 0, "block_swaps": 0, "pos_swaps": 0, "score_checks": 0}

    def fail(self, msg):
        if len(self.errors) < 50:
            self.errors.append(msg)

    @property
    def ok(self):
        return not self.errors

    def __repr__(self):
        return f"Report(ok={self.ok}, stats={self.stats}, errors={self.errors[:5]})"


def check_keys(rep, tag, gpu_keys, L, logit, tolmag):
    """Every key of a scored row against the oracle's block maximum."""
    keys, arg = O.block_keys(logit, L)
    nb = keys.shape[0]
    g = np.asarray(gpu_keys[:nb], dtype=np.float64)
    if nb and not np.isposinf(g[nb - 1]):
        rep.fail(f"{tag}: newest key {g[nb - 1]} is not +inf")
    if nb > 1:
        ref = keys[: nb - 1]
        tol = REL_TOL * tolmag[arg[: nb - 1]]
        bad = np.nonzero(~(np.abs(g[: nb - 1] - ref) <= tol))[0]
        for b in bad[:3]:
            rep.fail(f"{tag}: key[{b}] gpu {g[b]!r} oracle {ref[b]!r} tol {tol[b]!r}")
    rep.stats["key_checks"] += max(nb - 1, 0)
    return keys, arg


def check_blocks(rep, tag, gpu_blocks, gpu_nvalid, keys, key_arg, tolmag, nb, K):
    """Published blocks: ascending, padded, the right count, the oracle's set up
    to boundary swaps within tolerance."""
    expect_nv = min(nb, K)
    if int(gpu_nvalid) != expect_nv:
        rep.fail(f"{tag}: nvalid {gpu_nvalid} != {expect_nv}")
        return
    gb = np.asarray(gpu_blocks[:K], dtype=np.int64)
    if np.any(gb[expect_nv:] != O.INT32_MAX):
        rep.fail(f"{tag}: padding is not INT32_MAX")
    sel = gb[:expect_nv]
    if np.any(np.diff(sel) <= 0):
        rep.fail(f"{tag}: blocks not strictly ascending")
        return
    ref, _ = O.select_blocks(keys, nb, K)
    ref = ref[:expect_nv]
    if np.array_equal(sel, ref):
        return
    if np.any(sel < 0) or np.any(sel >= nb):
        rep.fail(f"{tag}: block id out of range")
        return
    diff = np.setxor1d(sel, ref)
    kth = keys[ref].min()
    for b in diff:
        tol = REL_TOL * tolmag[key_arg[b]]
        if not abs(keys[b] - kth) <= tol:
            rep.fail(f"{tag}: block {b} swapped with key {keys[b]!r} vs floor {kth!r} (tol {tol!r})")
            return
    rep.stats["block_swaps"] += len(diff) // 2


def check_positions(rep, tag, gpu_pos, gpu_score, cand, scores, tolmag, P):
    """Selected positions (and their GPU scores when given) against the
    oracle's top-P over the candidate positions ``cand``."""
    n_take = min(P, cand.shape[0])
    gp = np.asarray(gpu_pos[:P], dtype=np.int64)
    if np.any(gp[n_take:] != -1):
        rep.fail(f"{tag}: padding is not -1 past {n_take}")
    sel = gp[:n_take]
    if np.any(np.diff(sel) <= 0):
        rep.fail(f"{tag}: positions not strictly ascending")
        return
    index = {int(p): i for i, p in enumerate(cand.tolist())}
    missing = [p for p in sel.tolist() if p not in index]
    if missing:
        rep.fail(f"{tag}: positions {missing[:4]} are not candidates")
        return
    ref = O.top_positions(scores, cand, P)[:n_take]
    if gpu_score is not None:
        gs = np.asarray(gpu_score[:n_take], dtype=np.float64)
        idx = np.array([index[int(p)] for p in sel], dtype=np.int64)
        tol = REL_TOL * tolmag[idx]
        bad = np.nonzero(~(np.abs(gs - scores[idx]) <= tol))[0]
        for i in bad[:3]:
            rep.fail(f"{tag}: score at {sel[i]} gpu {gs[i]!r} oracle {scores[idx[i]]!r} tol {tol[i]!r}")
        rep.stats["score_checks"] += n_take
    if np.array_equal(sel, ref):
        return
    diff = np.setxor1d(sel, ref)
    ref_idx = np.array([index[int(p)] for p in ref], dtype=np.int64)
    kth = scores[ref_idx].min()
    for p in diff:
        i = index[int(p)]
        tol = REL_TOL * tolmag[i]
        if not abs(scores[i] - kth) <= tol:
            rep.fail(f"{tag}: position {p} swapped, score {scores[i]!r} vs floor {kth!r} (tol {tol!r})")
            return
    rep.stats["pos_swaps"] += len(diff) // 2


def check_step(wl, out, rows=None, rep=None):
    """Check one indexer step.

    ``wl``: the CPU workload; ``out``: numpy arrays from the GPU step with keys
    ``keys`` [rows, stride], ``blocks`` / ``nvalid`` (topk_blocks),
    ``blocks_src`` / ``nvalid_src`` (the source's own top P+1 blocks), ``pos``
    [layers, rows, P] and optionally ``score`` [layers, rows, P].
    """
    rep = rep or Report()
    pt = wl.page_table.numpy()
    layout = wl.layout
    K, P = wl.topk_blocks, wl.topk
    Kp = P + 1
    rows = range(wl.rows) if rows is None else rows
    seq = wl.seq_len.numpy()
    row_req = wl.row_req()
    for t in rows:
        L = int(seq[t])
        nb = O.num_blocks(L)
        logit, tolmag = O.dense_row_scores(wl.layers[0], pt, layout, t, L, row_req)
        if nb > min(K, Kp):
            keys, arg = check_keys(rep, f"row {t} keys", out["keys"][t], L, logit, tolmag)
        else:
            keys, arg = O.block_keys(logit, L)
        check_blocks(rep, f"row {t} blocks", out["blocks"][t], out["nvalid"][t], keys, arg, tolmag, nb, K)
        check_blocks(rep, f"row {t} src-blocks", out["blocks_src"][t], out["nvalid_src"][t], keys, arg, tolmag, nb,
                     Kp)
        score = out.get("score")
        # the source layer's own top-P: dense definition over every position
        check_positions(rep, f"row {t} layer 0", out["pos"][0][t], None if score is None else score[0][t],
                        np.arange(L), logit, tolmag, P)
        # consumers: judged on the GPU's published candidates
        blocks = np.asarray(out["blocks"][t], dtype=np.int64)
        nv = int(out["nvalid"][t])
        for j in range(1, len(wl.layers)):
            _, cand, sc, tm = O.select_row(wl.layers[j], pt, layout, t, L, blocks, nv, P, row_req)
            check_positions(rep, f"row {t} layer {j}", out["pos"][j][t], None if score is None else score[j][t],
                            cand, sc, tm, P)
        rep.stats["rows"] += 1
    return rep
