"""Python binding of libqsa (the C ABI in include/qsa.h): argument marshalling only.

Every function has the name of the C entry point it calls, takes torch tensors that live
on the current CUDA device (plus plain ints), passes their device pointers and the current
torch stream, and raises QSAError when the call returns a non-zero status.  No step of the
layer runs here: all arithmetic is in the CUDA kernels behind the library.  Loading fails
loudly if libqsa.so has not been built; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")

QSA_OK = 0
QSA_ERR_INVALID_ARG = -1
QSA_ERR_UNSUPPORTED = -2
QSA_ERR_WORKSPACE = -3
QSA_ERR_CUDA = -4
QSA_ERR_TIMEOUT = -5
QSA_ERR_DEVICE = -6

N_GROUPS, HEADS_PER_GROUP, N_HEADS, HEAD_DIM, CHUNK, PART_STRIDE = 2, 12, 24, 256, 64, 258

# every symbol include/qsa.h declares
EXPORTS = ("qsa_last_error", "qsa_prep_quantize", "qsa_prep", "qsa_select_workspace_bytes", "qsa_select",
           "qsa_flash_prefill_workspace_bytes", "qsa_flash_prefill",
           "qsa_flash_prefill_gated", "qsa_decode_partial", "qsa_merge", "qsa_merge_gated", "qsa_decode_layer",
           "qsa_decode_layer_batched", "qsa_flash_prefill_batched_workspace_bytes", "qsa_flash_prefill_batched",
           "qsa_check_device_status", "qsa_select_noalloc", "qsa_debug_wait_probe")


class QSAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"QSA error {code}: {msg}")
        self.code = code


class qsa_params(ctypes.Structure):
    _fields_ = [("topk", ctypes.c_int), ("identity_max", ctypes.c_int), ("sm_scale", ctypes.c_float)]


class qsa_rope(ctypes.Structure):
    _fields_ = [("base", ctypes.c_float), ("rotary_dim", ctypes.c_int), ("eps", ctypes.c_float),
                ("sections", ctypes.c_int * 3)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqsa.so (raises if it is missing: build it with int8_kv_top_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not built; run `python -m int8_kv_top_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    PP = ctypes.POINTER(qsa_params)
    lib.qsa_last_error.argtypes = []
    lib.qsa_last_error.restype = ctypes.c_char_p
    lib.qsa_prep_quantize.argtypes = [P, I64, P, P, P]
    lib.qsa_prep.argtypes = [P, P, P, P, P, P, ctypes.POINTER(qsa_rope), I, I, I, P, P, P, P, P, P, P]
    lib.qsa_select_workspace_bytes.argtypes = [I, I, I, PP]
    lib.qsa_select_workspace_bytes.restype = SZ
    lib.qsa_select.argtypes = [P, P, P, I, I, I, P, P, SZ, PP, P]
    lib.qsa_flash_prefill_workspace_bytes.argtypes = [I, I, I, PP]
    lib.qsa_flash_prefill_workspace_bytes.restype = SZ
    lib.qsa_flash_prefill.argtypes = [P, P, P, P, P, I, I, I, P, P, P, SZ, PP, P]
    lib.qsa_decode_partial.argtypes = [P, P, P, P, P, I, I, I, P, P, P, I, PP, P]
    lib.qsa_merge.argtypes = [P, P, I, I, P, P]
    lib.qsa_flash_prefill_gated.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P, SZ, PP, P]
    lib.qsa_merge_gated.argtypes = [P, P, I, I, P, P, P]
    lib.qsa_decode_layer.argtypes = [P, P, P, P, P, I, I, I, P, P, P, PP, P]
    lib.qsa_decode_layer_batched.argtypes = [P, P, P, P, P, I64, P, I, I, I, P, P, P, PP, P]
    lib.qsa_flash_prefill_batched_workspace_bytes.argtypes = [I, I, I, PP]
    lib.qsa_flash_prefill_batched_workspace_bytes.restype = SZ
    lib.qsa_flash_prefill_batched.argtypes = [P, P, P, P, P, I64, P, I, I, I, P, P, P, P, SZ, PP, P]
    lib.qsa_check_device_status.argtypes = [P]
    lib.qsa_debug_wait_probe.argtypes = [ctypes.c_uint64, P]
    lib.qsa_select_noalloc.argtypes = [P, P, P, I, I, I, P, PP, P]
    for name in EXPORTS:
        if name not in ("qsa_last_error", "qsa_select_workspace_bytes", "qsa_flash_prefill_workspace_bytes",
                        "qsa_flash_prefill_batched_workspace_bytes"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _params(params):
    if params is None:
        return None
    if isinstance(params, qsa_params):
        return ctypes.byref(params)
    topk, identity_max, sm_scale = params
    return ctypes.byref(qsa_params(int(topk), int(identity_max), float(sm_scale)))


def _check(rc: int):
    if rc != QSA_OK:
        raise QSAError(rc, load().qsa_last_error().decode(errors="replace"))


def qsa_last_error() -> str:
    return load().qsa_last_error().decode(errors="replace")


def qsa_prep_quantize(x, xq, xsc, stream=None):
    n_rows = x.numel() // HEAD_DIM
    _check(load().qsa_prep_quantize(_ptr(x), n_rows, _ptr(xq), _ptr(xsc), _stream(stream)))


def qsa_prep(q_raw, k_raw, v_raw, q_gamma, k_gamma, T: int, pos0: int, n_cells: int, qcur, kcur, kq, ksc, vq, vsc,
             pos3=None, rope=None, stream=None):
    """Fused prep: norm + rotary of q and k, qcur / kcur and the new tokens' int8 cache rows.
    rope: None or (base, rotary_dim, eps, (s0, s1, s2))."""
    r = None
    if rope is not None:
        base, rd, eps, sec = rope
        r = ctypes.byref(qsa_rope(float(base), int(rd), float(eps), (ctypes.c_int * 3)(*sec)))
    _check(load().qsa_prep(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(q_gamma), _ptr(k_gamma), _ptr(pos3), r, T,
                           pos0, n_cells, _ptr(qcur), _ptr(kcur), _ptr(kq), _ptr(ksc), _ptr(vq), _ptr(vsc),
                           _stream(stream)))


def qsa_select_workspace_bytes(T: int, pos0: int, n_cells: int, params=None) -> int:
    return int(load().qsa_select_workspace_bytes(T, pos0, n_cells, _params(params)))


def qsa_select(q, kq, ksc, n_cells: int, T: int, pos0: int, ids, ws, params=None, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().qsa_select(_ptr(q), _ptr(kq), _ptr(ksc), n_cells, T, pos0, _ptr(ids), _ptr(ws), ws_bytes,
                             _params(params), _stream(stream)))


def qsa_select_noalloc(q, kq, ksc, n_cells: int, T: int, pos0: int, ids, params=None, stream=None):
    """qsa_select on the library's built-in scratch (for callers that cannot allocate)."""
    _check(load().qsa_select_noalloc(_ptr(q), _ptr(kq), _ptr(ksc), n_cells, T, pos0, _ptr(ids), _params(params),
                                     _stream(stream)))


def qsa_flash_prefill_workspace_bytes(T: int, pos0: int, n_cells: int, params=None) -> int:
    return int(load().qsa_flash_prefill_workspace_bytes(T, pos0, n_cells, _params(params)))


def qsa_flash_prefill(q, kq, vq, ksc, vsc, n_cells: int, T: int, pos0: int, ids, out, ws=None, params=None,
                      stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().qsa_flash_prefill(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_cells, T, pos0, _ptr(ids),
                                    _ptr(out), _ptr(ws), ws_bytes, _params(params), _stream(stream)))


def qsa_decode_partial(q, kq, vq, ksc, vsc, n_cells: int, N: int, pos0: int, ids, part, n_chunks,
                       chunk_cap: int, params=None, stream=None):
    _check(load().qsa_decode_partial(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_cells, N, pos0, _ptr(ids),
                                     _ptr(part), _ptr(n_chunks), chunk_cap, _params(params), _stream(stream)))


def qsa_merge(part, n_chunks, N: int, chunk_cap: int, xp, stream=None):
    _check(load().qsa_merge(_ptr(part), _ptr(n_chunks), N, chunk_cap, _ptr(xp), _stream(stream)))


def qsa_flash_prefill_gated(q, kq, vq, ksc, vsc, n_cells: int, T: int, pos0: int, ids, gate, out, ws=None,
                            params=None, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().qsa_flash_prefill_gated(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_cells, T, pos0,
                                          _ptr(ids), _ptr(gate), _ptr(out), _ptr(ws), ws_bytes, _params(params),
                                          _stream(stream)))


def qsa_merge_gated(part, n_chunks, N: int, chunk_cap: int, gate, xp, stream=None):
    _check(load().qsa_merge_gated(_ptr(part), _ptr(n_chunks), N, chunk_cap, _ptr(gate), _ptr(xp), _stream(stream)))


def qsa_decode_layer(q, kq, vq, ksc, vsc, n_cells: int, N: int, pos0: int, ids, xp, params=None, stream=None,
                     gate=None):
    """One decode step (select, attend, merge) in one launch; ids and gate may be None."""
    _check(load().qsa_decode_layer(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_cells, N, pos0, _ptr(ids),
                                   _ptr(gate), _ptr(xp), _params(params), _stream(stream)))


def qsa_decode_layer_batched(q, kq, vq, ksc, vsc, n_pool: int, seqs, n_seq: int, n_tok: int, max_n_kv: int, ids, xp,
                             params=None, stream=None, gate=None):
    """Decode steps of many sequences in one launch; seqs is a device int32 tensor [n_seq][4]."""
    _check(load().qsa_decode_layer_batched(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_pool, _ptr(seqs),
                                           n_seq, n_tok, max_n_kv, _ptr(ids), _ptr(gate), _ptr(xp), _params(params),
                                           _stream(stream)))


def qsa_flash_prefill_batched_workspace_bytes(n_seq: int, n_tok: int, max_n_kv: int, params=None) -> int:
    return int(load().qsa_flash_prefill_batched_workspace_bytes(n_seq, n_tok, max_n_kv, _params(params)))


def qsa_flash_prefill_batched(q, kq, vq, ksc, vsc, n_pool: int, seqs, n_seq: int, n_tok: int, max_n_kv: int, ids,
                              out, ws, params=None, stream=None, gate=None):
    """Prefill of many sequences in one call (selection included); seqs is a device int32 tensor [n_seq][4]."""
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().qsa_flash_prefill_batched(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_pool, _ptr(seqs),
                                            n_seq, n_tok, max_n_kv, _ptr(ids), _ptr(gate), _ptr(out), _ptr(ws),
                                            ws_bytes, _params(params), _stream(stream)))


def qsa_debug_wait_probe(budget_ns: int, stream=None):
    """Test hook: a bounded device wait that can only give up after budget_ns (sets the status word)."""
    _check(load().qsa_debug_wait_probe(int(budget_ns), _stream(stream)))


def qsa_check_device_status(stream=None):
    _check(load().qsa_check_device_status(_stream(stream)))


def chunk_cap_for(topk: int = 2048, identity_max: int = 2051) -> int:
    return (max(topk, identity_max) + CHUNK - 1) // CHUNK
