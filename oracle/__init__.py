"""CPU oracle for the QSA layer: float64 C code behind ctypes.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  The library never imports it, and it imports nothing from the
library (inputs arrive as numpy arrays from the seeded generator).

Every function here is a thin marshalling layer over ``qsa_oracle.c``; the arithmetic,
with its citations, lives there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

NG, HPG, NH, HD, NB, PSTRIDE, CHUNK = 2, 12, 24, 256, 4, 258, 64


def build(force: bool = False) -> str:
    """Compile qsa_oracle.c with gcc (OpenMP when available) into an in-tree .so."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off", _SRC, "-o",
            _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I, D64 = ctypes.c_int, ctypes.c_double
        _lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        _lib.oracle_half_to_double.restype = D64
        _lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        _lib.oracle_float_to_half.restype = ctypes.c_uint16
        _lib.oracle_quantize.argtypes = [P, ctypes.c_int64, P, P]
        _lib.oracle_exact_key_parts.argtypes = [P, P, P, ctypes.c_int64, I, P, P]
        _lib.oracle_cell_set.argtypes = [P, P, P, ctypes.c_int64, I, I, I, D64, P, P]
        _lib.oracle_cell_set.restype = I
        _lib.oracle_attend.argtypes = [P, P, P, P, P, I, P, I, D64, P]
        _lib.oracle_partials.argtypes = [P, P, P, P, P, I, P, I, D64, P]
        _lib.oracle_partials.restype = I
        _lib.oracle_merge_f32.argtypes = [P, P, I, I, P]
        _lib.oracle_merge_group.argtypes = [P, I, P]
        _lib.oracle_prefill.argtypes = [P, P, P, P, P, I, I, P, I, I, I, D64, P, P, P, P]
        _lib.oracle_decode.argtypes = [P, P, P, P, P, I, I, I, I, D64, I, P, P, P, P, P]
        _lib.oracle_apply_gate.argtypes = [P, P, ctypes.c_int64]
        _lib.oracle_prep.argtypes = [P, P, P, P, P, I, I, D64, I, D64, P, P, P]
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float16
    return a.view(np.uint16)


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(int(bits))


def float_to_half_bits(x: float) -> int:
    return int(lib().oracle_float_to_half(float(x)))


def quantize(x: np.ndarray):
    """fp16 rows [..., 256] -> (int8 codes [..., 256], fp16 scales [..., 4])."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    rows = x.reshape(-1, HD)
    xq = np.zeros(rows.shape, dtype=np.int8)
    xsc = np.zeros((rows.shape[0], NB), dtype=np.uint16)
    lib().oracle_quantize(_p(rows.view(np.uint16)), rows.shape[0], _p(xq), _p(xsc))
    return xq.reshape(x.shape), xsc.view(np.float16).reshape(x.shape[:-1] + (NB,))


def exact_key(q_tok: np.ndarray, kq: np.ndarray, ksc: np.ndarray, c: int, g: int) -> int:
    """Exact selection key (16 * 2^48 * score) of cell c, group g, as a Python int."""
    hi = ctypes.c_int64()
    lo = ctypes.c_uint64()
    lib().oracle_exact_key_parts(_p(_bits(q_tok)), _p(np.ascontiguousarray(kq)), _p(_bits(ksc)), int(c), int(g),
                                 ctypes.byref(hi), ctypes.byref(lo))
    return (hi.value << 64) | lo.value


def cell_set(q_tok, kq, ksc, n_kv: int, g: int, topk=2048, identity_max=2051, sm_scale=1 / 16,
             with_f64_check=False):
    """Ascending cell set of one (token, group); returns (cells, f64_ranking_differs)."""
    cap = max(n_kv, topk, identity_max, 1)
    cells = np.zeros(cap, dtype=np.int32)
    diff = ctypes.c_int(0)
    n = lib().oracle_cell_set(_p(_bits(q_tok)), _p(np.ascontiguousarray(kq)), _p(_bits(ksc)), int(n_kv), int(g),
                              int(topk), int(identity_max), float(sm_scale), _p(cells),
                              ctypes.byref(diff) if with_f64_check else None)
    return cells[:n].copy(), bool(diff.value)


def attend(q_tok, kq, vq, ksc, vsc, g: int, cells, sm_scale=1 / 16) -> np.ndarray:
    """Attention of group g's 12 heads over `cells`: [12][256] float64."""
    cells = np.ascontiguousarray(cells, dtype=np.int32)
    out = np.zeros((HPG, HD), dtype=np.float64)
    lib().oracle_attend(_p(_bits(q_tok)), _p(np.ascontiguousarray(kq)), _p(np.ascontiguousarray(vq)),
                        _p(_bits(ksc)), _p(_bits(vsc)), int(g), _p(cells), len(cells), float(sm_scale), _p(out))
    return out


def partials(q_tok, kq, vq, ksc, vsc, g: int, cells, sm_scale=1 / 16) -> np.ndarray:
    """Split partials of group g: [n_chunks][12][258] float64 (o[256], m, l)."""
    cells = np.ascontiguousarray(cells, dtype=np.int32)
    nc = (len(cells) + CHUNK - 1) // CHUNK
    part = np.zeros((max(nc, 1), HPG, PSTRIDE), dtype=np.float64)
    lib().oracle_partials(_p(_bits(q_tok)), _p(np.ascontiguousarray(kq)), _p(np.ascontiguousarray(vq)),
                          _p(_bits(ksc)), _p(_bits(vsc)), int(g), _p(cells), len(cells), float(sm_scale), _p(part))
    return part[:nc]


def merge_group(part: np.ndarray) -> np.ndarray:
    """Merge [n_chunks][12][258] float64 partials -> [12][256]."""
    part = np.ascontiguousarray(part, dtype=np.float64)
    out = np.zeros((HPG, HD), dtype=np.float64)
    lib().oracle_merge_group(_p(part), part.shape[0], _p(out))
    return out


def merge_f32(part: np.ndarray, n_chunks) -> np.ndarray:
    """Merge float32 partials [N][cap][24][258] with chunk counts [N] -> [N][24][256] float64."""
    part = np.ascontiguousarray(part, dtype=np.float32)
    n_chunks = np.ascontiguousarray(n_chunks, dtype=np.int32)
    N, cap = part.shape[0], part.shape[1]
    out = np.zeros((N, NH, HD), dtype=np.float64)
    lib().oracle_merge_f32(_p(part), _p(n_chunks), N, cap, _p(out))
    return out


def prefill(inp: dict, T: int, pos0: int, toks=None, topk=2048, identity_max=2051, sm_scale=1 / 16,
            f64_check=False):
    """Prefill oracle over tokens `toks` (default all): (out [n][24][256], ids [n][2][topk], n_set [n][2], differs)."""
    toks = np.arange(T, dtype=np.int32) if toks is None else np.ascontiguousarray(toks, dtype=np.int32)
    # the cache contract: every token's causal cells exist (the C code reads cells 0 .. pos0 + t)
    assert inp["kq"].shape[0] >= pos0 + T and inp["q"].shape[0] >= T, "cache or query rows too short"
    n = len(toks)
    out = np.zeros((n, NH, HD), dtype=np.float64)
    ids = np.zeros((n, NG, topk), dtype=np.int32)
    n_set = np.zeros((n, NG), dtype=np.int32)
    differs = np.zeros((n, NG), dtype=np.int32)
    lib().oracle_prefill(_p(_bits(inp["q"])), _p(np.ascontiguousarray(inp["kq"])), _p(np.ascontiguousarray(inp["vq"])),
                         _p(_bits(inp["ksc"])), _p(_bits(inp["vsc"])), int(T), int(pos0), _p(toks), n, int(topk),
                         int(identity_max), float(sm_scale), _p(out), _p(ids), _p(n_set),
                         _p(differs) if f64_check else None)
    return out, ids, n_set, differs


def chunk_cap_for(topk=2048, identity_max=2051) -> int:
    return (max(topk, identity_max) + CHUNK - 1) // CHUNK


def decode(inp: dict, N: int, P: int, topk=2048, identity_max=2051, sm_scale=1 / 16):
    """Decode oracle: (part [N][cap][24][258], n_chunks [N], merged [N][24][256], direct [N][24][256], ids [N][2][topk])."""
    assert inp["kq"].shape[0] >= P + N and inp["q"].shape[0] >= N, "cache or query rows too short"
    cap = chunk_cap_for(topk, identity_max)
    part = np.full((N, cap, NH, PSTRIDE), np.nan, dtype=np.float64)
    n_chunks = np.zeros(N, dtype=np.int32)
    out = np.zeros((N, NH, HD), dtype=np.float64)
    direct = np.zeros((N, NH, HD), dtype=np.float64)
    ids = np.zeros((N, NG, topk), dtype=np.int32)
    lib().oracle_decode(_p(_bits(inp["q"])), _p(np.ascontiguousarray(inp["kq"])), _p(np.ascontiguousarray(inp["vq"])),
                        _p(_bits(inp["ksc"])), _p(_bits(inp["vsc"])), int(N), int(P), int(topk), int(identity_max),
                        float(sm_scale), cap, _p(part), _p(n_chunks), _p(out), _p(direct), _p(ids))
    return part, n_chunks, out, direct, ids


def decode_batch(pool: dict, seqs, topk=2048, identity_max=2051, sm_scale=1 / 16):
    """Decode oracle for many sequences sharing one cell pool (the batched decode contract).

    pool: {"q": [n_tok][24][256], "kq"/"vq": [n_pool][2][256], "ksc"/"vsc": [n_pool][2][4]};
    seqs: rows (first pool cell, n_cells, pos0, first token row), first rows increasing from 0.
    Sequence s is decode() over its own cells and token rows.  Returns (merged [n_tok][24][256],
    ids [n_tok][2][topk], with -1 in the rows of identity tokens)."""
    seqs = np.asarray(seqs, dtype=np.int64).reshape(-1, 4)
    n_tok = pool["q"].shape[0]
    out = np.zeros((n_tok, NH, HD), dtype=np.float64)
    ids = np.full((n_tok, NG, topk), -1, dtype=np.int32)
    for s, (c0, n, pos0, t0) in enumerate(seqs):
        t1 = int(seqs[s + 1][3]) if s + 1 < len(seqs) else n_tok
        sub = {"q": np.ascontiguousarray(pool["q"][t0:t1])}
        for k in ("kq", "vq", "ksc", "vsc"):
            sub[k] = np.ascontiguousarray(pool[k][c0:c0 + n])
        _, _, merged, _, sid = decode(sub, int(t1 - t0), int(pos0), topk=topk, identity_max=identity_max,
                                      sm_scale=sm_scale)
        out[t0:t1] = merged
        ids[t0:t1] = sid
    return out, ids


def prefill_batch(pool: dict, seqs, topk=2048, identity_max=2051, sm_scale=1 / 16):
    """Prefill oracle for many sequences sharing one cell pool (the batched prefill contract, the
    same seqs table as decode_batch): sequence s is prefill() over its own cells and token rows.
    Returns (out [n_tok][24][256] float64, ids [n_tok][2][topk], with -1 in the rows of identity
    tokens)."""
    seqs = np.asarray(seqs, dtype=np.int64).reshape(-1, 4)
    n_tok = pool["q"].shape[0]
    out = np.zeros((n_tok, NH, HD), dtype=np.float64)
    ids = np.full((n_tok, NG, topk), -1, dtype=np.int32)
    for s, (c0, n, pos0, t0) in enumerate(seqs):
        t1 = int(seqs[s + 1][3]) if s + 1 < len(seqs) else n_tok
        if t1 <= t0:
            continue
        sub = {"q": np.ascontiguousarray(pool["q"][t0:t1])}
        for k in ("kq", "vq", "ksc", "vsc"):
            sub[k] = np.ascontiguousarray(pool[k][c0:c0 + n])
        o, sid, _, _ = prefill(sub, int(t1 - t0), int(pos0), topk=topk, identity_max=identity_max, sm_scale=sm_scale)
        out[t0:t1] = o
        sel = (pos0 + np.arange(t1 - t0) + 1) > identity_max
        ids[t0:t1][sel] = sid[sel]
    return out, ids


def apply_gate(out: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """Output gate: out * sigmoid(gate), elementwise in float64 (a new array; gate fp16, out's shape)."""
    res = np.ascontiguousarray(out, dtype=np.float64).copy()
    g = _bits(np.ascontiguousarray(gate, dtype=np.float16))
    assert g.size == res.size
    lib().oracle_apply_gate(_p(res), _p(g), res.size)
    return res


def prep(q_raw, k_raw, q_gamma, k_gamma, T: int, pos0: int, pos3=None, base=10000.0, rotary_dim=256, eps=1e-6,
         sections=(32, 48, 48)):
    """Fused prep oracle: (qcur [T][24][256], kcur [T][2][256]) float64 (RMS norm with gain, then
    rotary embedding at positions pos0 + t, or the mrope positions pos3 [T][3])."""
    qc = np.zeros((T, NH, HD), dtype=np.float64)
    kc = np.zeros((T, NG, HD), dtype=np.float64)
    qg = np.ascontiguousarray(q_gamma, dtype=np.float64)
    kg = np.ascontiguousarray(k_gamma, dtype=np.float64)
    sec = np.ascontiguousarray(sections, dtype=np.int32)
    p3 = None if pos3 is None else np.ascontiguousarray(pos3, dtype=np.int32)
    lib().oracle_prep(_p(_bits(q_raw)), _p(_bits(k_raw)), _p(qg), _p(kg), None if p3 is None else _p(p3), int(T),
                      int(pos0), float(base), int(rotary_dim), float(eps), _p(sec), _p(qc), _p(kc))
    return qc, kc
