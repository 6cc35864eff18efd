"""The C-ABI library builds, loads, exports every declared symbol and rejects bad
arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from int8_kv_top_gb300 import build as qbuild
from int8_kv_top_gb300 import qsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qsa.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"QSA_API\s+[\w\s\*]+?\b(qsa_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"qsa_flash_prefill", "qsa_select", "qsa_merge", "qsa_decode_partial", "qsa_prep_quantize"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(qsa.EXPORTS) <= names


FAKE = 1 << 20  # aligned, never dereferenced: every call below fails validation first


def test_null_and_misaligned_pointers(lib):
    P = ctypes.c_void_p
    rc = lib.qsa_flash_prefill(None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), 10, 4, 0, None, P(FAKE), None, 0, None, None)
    assert rc == qsa.QSA_ERR_INVALID_ARG and b"q is NULL" in lib.qsa_last_error()
    rc = lib.qsa_flash_prefill(P(FAKE + 8), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 10, 4, 0, None, P(FAKE), None, 0, None, None)
    assert rc == qsa.QSA_ERR_INVALID_ARG and b"aligned" in lib.qsa_last_error()
    rc = lib.qsa_merge(P(FAKE), None, 1, 33, P(FAKE), None)
    assert rc == qsa.QSA_ERR_INVALID_ARG


def test_bad_sizes(lib):
    P = ctypes.c_void_p
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE))
    assert lib.qsa_flash_prefill(*args, 100, 0, 0, None, P(FAKE), None, 0, None, None) == qsa.QSA_ERR_INVALID_ARG   # T = 0
    assert lib.qsa_flash_prefill(*args, 100, 4, -1, None, P(FAKE), None, 0, None, None) == qsa.QSA_ERR_INVALID_ARG  # pos0 < 0
    assert lib.qsa_flash_prefill(*args, 100, 4, 97, None, P(FAKE), None, 0, None, None) == qsa.QSA_ERR_INVALID_ARG  # cache small
    assert b"cache too small" in lib.qsa_last_error()
    # tokens above the threshold need ids, then a workspace
    assert lib.qsa_flash_prefill(*args, 3000, 4, 2500, None, P(FAKE), None, 0, None, None) == qsa.QSA_ERR_INVALID_ARG
    need = lib.qsa_flash_prefill_workspace_bytes(4, 2500, 3000, None)
    assert need == 2 * 2504 * 2 * 256 * 2
    assert lib.qsa_flash_prefill(*args, 3000, 4, 2500, P(FAKE), P(FAKE), P(FAKE), need - 16, None, None) == \
        qsa.QSA_ERR_WORKSPACE
    assert lib.qsa_flash_prefill_workspace_bytes(4, 0, 100, None) == 2 * 4 * 2 * 256 * 2  # the fp16 mirror
    assert lib.qsa_merge(P(FAKE), P(FAKE), 0, 33, P(FAKE), None) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_merge(P(FAKE), P(FAKE), 1, 2000, P(FAKE), None) == qsa.QSA_ERR_UNSUPPORTED
    # decode: chunk_cap too small for the default set size (2051 cells -> 33 chunks)
    rc = lib.qsa_decode_partial(*args, 600, 1, 512, None, P(FAKE), P(FAKE), 32, None, None)
    assert rc == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_prep_quantize(P(FAKE), -1, P(FAKE), P(FAKE), None) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_prep_quantize(None, 0, None, None, None) == qsa.QSA_OK


def test_bad_params(lib):
    P = ctypes.c_void_p
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 100, 4, 0, None, P(FAKE), None, 0)
    for bad in [(0, 2051, 0.0625), (2053, 2051, 0.0625), (4, 0, 0.0625), (4, 8, 0.0), (4, 8, -1.0),
                (4, 8, float("inf"))]:
        p = qsa.qsa_params(*bad)
        assert lib.qsa_flash_prefill(*args, ctypes.byref(p), None) == qsa.QSA_ERR_INVALID_ARG, bad
    assert lib.qsa_select_workspace_bytes(4, 0, 100, None) == 0   # no token above the threshold


def test_select_rejects_missing_workspace(lib):
    P = ctypes.c_void_p
    need = lib.qsa_select_workspace_bytes(64, 2040, 2104, None)
    rc = lib.qsa_select(P(FAKE), P(FAKE), P(FAKE), 2104, 64, 2040, P(FAKE), None, 0, None, None)
    assert rc in (qsa.QSA_ERR_WORKSPACE, qsa.QSA_ERR_UNSUPPORTED)
    # a smaller workspace is taken in chunks of tokens, down to one token per chunk: below what the
    # last single-token chunk needs, the call is refused
    need1 = lib.qsa_select_workspace_bytes(1, 2040 + 63, 2104, None)
    assert 0 < need1 < need
    rc = lib.qsa_select(P(FAKE), P(FAKE), P(FAKE), 2104, 64, 2040, P(FAKE), P(FAKE), need1 - 16, None, None)
    assert rc == qsa.QSA_ERR_WORKSPACE
    assert b"in chunks of one token" in lib.qsa_last_error()
    # under the threshold nothing is needed or launched
    assert lib.qsa_select(P(FAKE), P(FAKE), P(FAKE), 100, 4, 0, None, None, 0, None, None) == qsa.QSA_OK


def test_select_workspace_covers_the_score_rows(lib):
    # the workspace holds (at least) the fp16 score row of every selected token and group, one row
    # per token whose n_kv = pos0 + t + 1 exceeds identity_max, padded to whole 256-cell blocks;
    # it grows with T and pos0, and is a whole number of 1 KB blocks
    prev = {}
    for pos0 in (2040, 8192, 30000):
        for T in (1, 8, 9, 64, 512, 1984):
            n = pos0 + T
            need = lib.qsa_select_workspace_bytes(T, pos0, n, None)
            t_sel = max(0, 2051 - pos0)
            T_sel = max(0, T - t_sel)
            n_pad = -(-n // 256) * 256
            assert need >= 2 * T_sel * n_pad * 2, (T, pos0)
            assert need % 1024 == 0
            if pos0 in prev:
                assert need >= prev[pos0], (T, pos0)
            prev[pos0] = need
    assert lib.qsa_select_workspace_bytes(512, 30000, 30512, None) >= lib.qsa_select_workspace_bytes(512, 8192, 8704, None)


def test_decode_layer_and_gated_calls_validate_on_the_host(lib):
    P = ctypes.c_void_p
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE))
    # qsa_decode_layer(q, kq, vq, ksc, vsc, n_cells, N, pos0, ids, gate, xp, params, stream)
    assert lib.qsa_decode_layer(*args, 100, 0, 0, None, None, P(FAKE), None, None) == qsa.QSA_ERR_INVALID_ARG  # N = 0
    assert lib.qsa_decode_layer(*args, 100, 4, 97, None, None, P(FAKE), None, None) == qsa.QSA_ERR_INVALID_ARG
    assert b"cache too small" in lib.qsa_last_error()
    assert lib.qsa_decode_layer(*args, 100, 4, 0, None, None, None, None, None) == qsa.QSA_ERR_INVALID_ARG  # xp
    assert lib.qsa_decode_layer(*args, 100, 4, 0, None, P(FAKE + 2), P(FAKE), None, None) == qsa.QSA_ERR_INVALID_ARG
    assert b"gate" in lib.qsa_last_error()
    # qsa_decode_layer_batched(q, kq, vq, ksc, vsc, n_pool, seqs, n_seq, n_tok, max_n_kv, ids, gate, xp, params, stream)
    assert lib.qsa_decode_layer_batched(*args, 100, None, 1, 1, 100, None, None, P(FAKE), None, None) == \
        qsa.QSA_ERR_INVALID_ARG                                                     # seqs NULL
    assert lib.qsa_decode_layer_batched(*args, 100, P(FAKE), 3, 2, 100, None, None, P(FAKE), None, None) == \
        qsa.QSA_ERR_INVALID_ARG                                                     # more sequences than tokens
    assert lib.qsa_decode_layer_batched(*args, 0, P(FAKE), 1, 1, 100, None, None, P(FAKE), None, None) == \
        qsa.QSA_ERR_INVALID_ARG                                                     # empty pool
    # gated prefill and merge: a misaligned gate is refused before anything else runs
    assert lib.qsa_flash_prefill_gated(*args, 100, 4, 0, None, P(FAKE + 2), P(FAKE), P(FAKE), 1 << 20, None,
                                       None) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_merge_gated(P(FAKE), P(FAKE), 1, 33, P(FAKE + 2), P(FAKE), None) == qsa.QSA_ERR_INVALID_ARG


def test_batched_prefill_validates_on_the_host(lib):
    P = ctypes.c_void_p
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE))
    # workspace: a 256-byte-rounded work list, then K^ and V^ of round_up(min(2051, max_n_kv), 128)
    # rows per sequence, 2 groups x 256 fp16 each
    assert lib.qsa_flash_prefill_batched_workspace_bytes(3, 10, 100, None) == 256 + 2 * 3 * 128 * 2 * 256 * 2
    assert lib.qsa_flash_prefill_batched_workspace_bytes(2, 1000, 9000, None) == \
        (1 + 1000 // 64 + 2) * 16 // 256 * 256 + 256 + 2 * 2 * 2176 * 2 * 256 * 2
    assert lib.qsa_flash_prefill_batched_workspace_bytes(0, 10, 100, None) == 0
    ws = 1 << 24
    # qsa_flash_prefill_batched(q, kq, vq, ksc, vsc, n_pool, seqs, n_seq, n_tok, max_n_kv, ids, gate, out, ws,
    #                           ws_bytes, params, stream)
    call = lib.qsa_flash_prefill_batched
    assert call(*args, 100, None, 1, 1, 100, None, None, P(FAKE), P(FAKE), ws, None, None) == qsa.QSA_ERR_INVALID_ARG
    assert call(*args, 100, P(FAKE), 1, 1, 100, None, None, None, P(FAKE), ws, None, None) == qsa.QSA_ERR_INVALID_ARG
    assert call(*args, 100, P(FAKE), 0, 1, 100, None, None, P(FAKE), P(FAKE), ws, None, None) == qsa.QSA_ERR_INVALID_ARG
    assert call(*args, 100, P(FAKE), 1, 1, 100, None, P(FAKE + 2), P(FAKE), P(FAKE), ws, None, None) == \
        qsa.QSA_ERR_INVALID_ARG                                                      # misaligned gate
    assert call(*args, 100, P(FAKE), 1, 70000, 100, None, None, P(FAKE), P(FAKE), ws, None, None) == \
        qsa.QSA_ERR_UNSUPPORTED                                                      # n_tok > 65535
    assert call(*args, 100, P(FAKE), 1, 1, 0, None, None, P(FAKE), P(FAKE), ws, None, None) == qsa.QSA_ERR_UNSUPPORTED
    assert call(*args, 100, P(FAKE), 1, 1, 100, None, None, P(FAKE), P(FAKE), 1000, None, None) == \
        qsa.QSA_ERR_WORKSPACE                                                        # too small
    assert call(*args, 100, P(FAKE), 1, 1, 100, None, None, P(FAKE), P(FAKE + 8), ws, None, None) == \
        qsa.QSA_ERR_INVALID_ARG                                                      # misaligned ws


def test_wait_probe_rejects_budgets_outside_its_range(lib):
    assert lib.qsa_debug_wait_probe(10, None) == qsa.QSA_ERR_INVALID_ARG
    assert lib.qsa_debug_wait_probe(10_000_000_000, None) == qsa.QSA_ERR_INVALID_ARG
