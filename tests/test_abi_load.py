"""The C-ABI library builds, loads, exports every declared symbol, and rejects
bad arguments on the host (no GPU needed: these checks run before any CUDA
call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ci.h")


@pytest.fixture(scope="module")
def ci():
    from two_level_sparse_gb300 import build

    if not os.path.exists(os.path.join(ROOT, "two_level_sparse_gb300", "libci.so")):
        build.build()
    from two_level_sparse_gb300 import ci as mod

    return mod


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(ci_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_symbols() == sorted(
        ["ci_dcp_merge_keys", "ci_dcp_merge_topk", "ci_prefill_tail", "ci_publish_blocks", "ci_publish_blocks2",
         "ci_q_rope_quant", "ci_score_dense_amax8", "ci_select_sparse", "ci_select_sparse_layers", "ci_strerror",
         "ci_version"])


def test_library_exports_every_declared_symbol(ci):
    lib = ctypes.CDLL(ci.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(ci.SIGNATURES) == set(declared_symbols())


def test_status_names(ci):
    assert ci.version() == 301
    assert ci.strerror(0) == "ok"
    for code in ci.CI_ERR:
        assert ci.strerror(code) != "unknown status"


P = ctypes.c_void_p(0x1000)  # never dereferenced: host checks fail first
N = None


def test_dense_host_checks(ci):
    f = ci.lib.ci_score_dense_amax8
    # rows == 0: nothing to do, even with null pointers
    assert f(N, N, N, N, 1, 0, N, 0, 1, 0, N, N, 0, 0, 0, 8, N, 8, N, N) == 0
    # null pointer
    assert f(N, P, P, P, 1, 0, P, 2, 1, 0, N, P, 2, 64, 0, 8, P, 8, N, N) == -1
    # bad layout
    assert f(P, P, P, P, 1, 0, P, 2, 1, 7, N, P, 2, 64, 0, 8, P, 8, N, N) == -5
    # decode needs one request per row
    assert f(P, P, P, P, 1, 0, P, 3, 1, 0, N, P, 2, 64, 0, 8, P, 8, N, N) == -2
    # prefill needs exactly one request
    assert f(P, P, P, P, 1, 0, P, 2, 1, 1, N, P, 2, 64, 0, 8, P, 8, N, N) == -2
    # several requests: row starts required, 1..4096 requests
    assert f(P, P, P, P, 1, 0, P, 2, 1, 2, N, P, 2, 64, 0, 8, P, 8, N, N) == -1
    assert f(P, P, P, P, 1, 0, P, 0, 1, 2, P, P, 2, 64, 0, 8, P, 8, N, N) == -4
    assert f(P, P, P, P, 1, 0, P, 5000, 1, 2, P, P, 2, 64, 0, 8, P, 8, N, N) == -4
    # max_len beyond the page table
    assert f(P, P, P, P, 1, 0, P, 2, 1, 0, N, P, 2, 65, 0, 8, P, 16, N, N) == -2
    # keys stride not a multiple of 8 / too short
    assert f(P, P, P, P, 1, 0, P, 2, 2, 0, N, P, 2, 128, 0, 8, P, 12, N, N) == -2
    assert f(P, P, P, P, 1, 0, P, 2, 4, 0, N, P, 2, 256, 0, 8, P, 8, N, N) == -2
    # misaligned pool
    assert f(P, P, P, ctypes.c_void_p(0x1001), 1, 0, P, 2, 1, 0, N, P, 2, 64, 0, 8, P, 8, N, N) == -3
    # unknown K page format
    assert f(P, P, P, P, 1, 2, P, 2, 1, 0, N, P, 2, 64, 0, 8, P, 8, N, N) == -5
    # block size other than 8, 4, 2, 1; local blocks need FP8 pages
    assert f(P, P, P, P, 1, 0, P, 2, 1, 0, N, P, 2, 64, 0, 3, P, 8, N, N) == -4
    assert f(P, P, P, P, 1, 1, P, 2, 1, 0, N, P, 2, 64, 0, 4, P, 8, N, N) == -5
    # negative skip
    assert f(P, P, P, P, 1, 0, P, 2, 1, 0, N, P, 2, 64, -1, 8, P, 8, N, N) == -4


def test_publish_host_checks(ci):
    f = ci.lib.ci_publish_blocks
    assert f(N, 0, 0, N, 8, 16, N, 16, N, N, N) == 0
    assert f(P, 2, 64, P, 8, 0, P, 16, P, N, N) == -4  # topk_blocks < 1
    assert f(P, 2, 64, P, 8, 16, P, 15, P, N, N) == -2  # blocks stride < topk
    assert f(P, 2, 64, N, 8, 16, P, 16, P, N, N) == -1
    assert f(P, 2, 400000, P, 50000, 16, P, 16, P, N, N) == -4  # longer than supported
    assert f(P, 2, 64, ctypes.c_void_p(0x1004), 8, 16, P, 16, P, N, N) == -3


def test_publish_pair_host_checks(ci):
    f = ci.lib.ci_publish_blocks2
    assert f(N, 0, 0, N, 8, 16, N, 16, N, 4, N, 4, N, N, N) == 0
    assert f(P, 2, 64, P, 8, 16, P, 16, P, 0, P, 16, P, N, N) == -4  # topk_blocks2 < 1
    assert f(P, 2, 64, P, 8, 16, P, 16, P, 20, P, 16, P, N, N) == -2  # blocks2 stride < topk_blocks2
    assert f(P, 2, 64, P, 8, 16, P, 16, P, 4, P, 4, N, N, N) == -1  # nvalid2 missing
    assert f(P, 2, 64, P, 8, 0, P, 16, P, 4, N, 4, N, N, N) == -4  # first selection checked as before
    # the two tables may not share a byte (the second is read back from the first while it is written)
    assert f(P, 2, 64, P, 8, 16, P, 16, P, 4, P, 4, P, N, N) == -2  # the same table twice
    inside = ctypes.c_void_p(0x1000 + 4 * 20)  # row 1 of a [2][16] table
    assert f(P, 2, 64, P, 8, 16, P, 16, P, 4, inside, 4, P, N, N) == -2
    below = ctypes.c_void_p(0x1000 - 4 * 10)  # a [2][4] table whose last row runs into the first table
    assert f(P, 2, 64, P, 8, 16, P, 16, P, 4, below, 8, P, N, N) == -2


def test_prefill_tail_host_checks(ci):
    f = ci.lib.ci_prefill_tail
    ok_args = [P, 2, P, 64, P, 16, P, 16, P, P, 16, P, P, 8, N, N]
    bad = list(ok_args)
    bad[1] = 0  # no request
    assert f(*bad) == -4
    bad = list(ok_args)
    bad[1] = 4097  # too many requests
    assert f(*bad) == -4
    bad = list(ok_args)
    bad[7] = 0  # topk_blocks < 1
    assert f(*bad) == -4
    bad = list(ok_args)
    bad[13] = -1  # negative capacity
    assert f(*bad) == -2
    bad = list(ok_args)
    bad[10] = 8  # output stride < topk_blocks
    assert f(*bad) == -2
    bad = list(ok_args)
    bad[5] = 8  # input stride < topk_blocks
    assert f(*bad) == -2
    bad = list(ok_args)
    bad[0] = N  # no row starts
    assert f(*bad) == -1
    bad = list(ok_args)
    bad[12] = N  # no count
    assert f(*bad) == -1
    bad = list(ok_args)
    bad[9] = N  # capacity but no output table
    assert f(*bad) == -1


def test_q_rope_quant_host_checks(ci):
    f = ci.lib.ci_q_rope_quant
    ok_args = [P, P, P, 100, P, 0.125, 0.125, 1, 4, 0, P, P, P, N, N]
    assert f(*ok_args[:8], 0, *ok_args[9:]) == 0  # no tokens
    bad = list(ok_args)
    bad[9] = 2  # unknown output format
    assert f(*bad) == -5
    bad = list(ok_args)
    bad[11] = N  # MXFP4 needs the scale output
    assert f(*bad) == -1
    bad = list(ok_args)
    bad[1] = N
    assert f(*bad) == -1
    bad = list(ok_args)
    bad[11] = ctypes.c_void_p(0x1002)  # scale output not 4-byte aligned
    assert f(*bad) == -3
    bad = list(ok_args)
    bad[8] = -1
    assert f(*bad) == -2


def test_select_host_checks(ci):
    f = ci.lib.ci_select_sparse
    ok_args = [P, P, P, P, 1, 0, P, 2, 1, 0, N, P, 2, 64, P, 16, P, 16, 8, 8, P, N, 8, N, N]
    assert f(*ok_args[:12], 0, *ok_args[13:]) == 0  # rows == 0
    bad = list(ok_args)
    bad[19] = 0  # topk < 1
    assert f(*bad) == -4
    bad = list(ok_args)
    bad[17] = 5000  # max_blocks too large
    assert f(*bad) == -4
    bad = list(ok_args)
    bad[22] = 4  # out stride < topk
    assert f(*bad) == -2
    bad = list(ok_args)
    bad[20] = N  # no output
    assert f(*bad) == -1
    bad = list(ok_args)
    bad[9] = 2  # several requests without row starts
    assert f(*bad) == -1
    bad = list(ok_args)
    bad[5] = 3  # unknown K page format
    assert f(*bad) == -5
    bad = list(ok_args)
    bad[18] = 16  # block size other than 8, 4, 2, 1
    assert f(*bad) == -4


def test_select_layers_host_checks(ci):
    f = ci.lib.ci_select_sparse_layers
    n = 2
    ptrs = (ctypes.c_void_p * n)(0x1000, 0x2000)
    i64 = (ctypes.c_int64 * n)(16, 16)
    i32 = (ctypes.c_int32 * n)(16, 16)

    def args(num_layers=n, mb=i32, outs=ptrs, rows=2, topk=8, kv=0):
        return [num_layers, ptrs, ptrs, ptrs, ptrs, 1, kv, P, 2, 1, 0, N, P, rows, 64, ptrs, i64, ptrs, mb, 8, topk,
                outs, N, 8, N, N]

    assert f(*args(rows=0)) == 0  # nothing to do
    assert f(*args(num_layers=0)) == -4
    assert f(*args(num_layers=9)) == -4
    assert f(*args(mb=(ctypes.c_int32 * n)(16, 5000))) == -4  # the second layer's max_blocks too large
    assert f(*args(outs=(ctypes.c_void_p * n)(0x1000, None))) == -1  # the second layer has no output
    assert f(*args(topk=0)) == -4
    assert f(*args(kv=3)) == -5
    bad = args()
    bad[1] = N  # no q array
    assert f(*bad) == -1
    bad = args()
    bad[23] = 4  # out stride < topk
    assert f(*bad) == -2


def test_select_layers_binding_checks_the_layer_count(ci):
    with pytest.raises(ValueError):
        ci.ci_select_sparse_layers([], None, 0, None, 0, 8)
    with pytest.raises(ValueError):
        ci.ci_select_sparse_layers([{}] * 9, None, 0, None, 0, 8)


def test_dcp_merge_host_checks(ci):
    fk, ft = ci.lib.ci_dcp_merge_keys, ci.lib.ci_dcp_merge_topk
    assert fk(P, 3, 64, 8, P, 4, 64, 0, P, 8, N, N) == -4   # world not 2, 4 or 8
    assert fk(P, 2, 16, 8, P, 4, 64, 0, P, 8, N, N) == -2   # shards overlap
    assert fk(P, 2, 0, 8, P, 0, 64, 0, P, 8, N, N) == 0     # no rows
    assert fk(N, 2, 64, 8, P, 4, 64, 0, P, 8, N, N) == -1
    assert ft(P, P, 8, 4096, 1024, 4, 1024, P, N, 1024, N) == -4  # 8 x 1024 candidates
    assert ft(P, P, 2, 4096, 512, 8, 600, P, N, 600, N) == -2   # local stride < topk
