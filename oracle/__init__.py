"""fp64 CPU oracle for the multi-LoRA fused MoE layer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs import this package.  The product path never does: it shares no
code with the CUDA library.

``oracle.c`` is the plain definition in C (fp64, OpenMP over tokens);
``brute.py`` is a second, independent numpy restatement used to pin it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("T", "H", "I", "E", "k", "L", "r")]


def load_library(path: str):
    """Open an oracle build at ``path`` with its argument types declared."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_forward.restype = ctypes.c_long
    lib.oracle_forward.argtypes = [ctypes.POINTER(_Dims)] + [P] * 10 + [P, ctypes.c_int, P, ctypes.c_int]
    lib.oracle_forward_w8.restype = ctypes.c_long
    lib.oracle_forward_w8.argtypes = [ctypes.POINTER(_Dims)] + [P] * 12 + [P, ctypes.c_int, P, ctypes.c_int]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_pair.restype = ctypes.c_int
    lib.oracle_pair.argtypes = [ctypes.POINTER(_Dims)] + [P] * 9 + [ctypes.c_long] + [P] * 5
    lib.oracle_align.restype = ctypes.c_long
    lib.oracle_align.argtypes = [ctypes.c_int] * 5 + [P, P, P, ctypes.c_long] + [P] * 5
    lib.oracle_align_capacity.restype = ctypes.c_long
    lib.oracle_align_capacity.argtypes = [ctypes.c_int] * 5
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _args(layer):
    d = _Dims(layer.T, layer.H, layer.I, layer.E, layer.k, layer.L, layer.r)
    arrs = dict(
        x=_c(layer.x, np.uint16), topk_ids=_c(layer.topk_ids, np.int32),
        topk_weights=_c(layer.topk_weights, np.float32), lora_ids=_c(layer.lora_ids, np.int32),
        W1=_c(layer.W1, np.uint16), W2=_c(layer.W2, np.uint16),
        A1=_c(layer.A1, np.uint16), B1=_c(layer.B1, np.uint16),
        A2=_c(layer.A2, np.uint16), B2=_c(layer.B2, np.uint16))
    return d, arrs


def forward(layer, tokens=None, n_threads: int | None = None, lib=None):
    """fp64 layer output [n][H] for the given token indices (default: all).

    Returns (out, n_invalid_pairs)."""
    lib = lib or _load()
    d, a = _args(layer)
    if tokens is None:
        tok = None
        n = layer.T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tok.size
    out = np.zeros((n, layer.H), dtype=np.float64)
    nt = n_threads or default_threads()
    inv = lib.oracle_forward(ctypes.byref(d), _ptr(a["x"]), _ptr(a["topk_ids"]), _ptr(a["topk_weights"]),
                             _ptr(a["lora_ids"]), _ptr(a["W1"]), _ptr(a["W2"]), _ptr(a["A1"]),
                             _ptr(a["B1"]), _ptr(a["A2"]), _ptr(a["B2"]), _ptr(tok), n, _ptr(out), nt)
    if inv < 0:
        raise ValueError("oracle_forward: bad arguments")
    return out, int(inv)


def forward_w8(layer, tokens=None, n_threads: int | None = None, lib=None):
    """fp64 layer output with FP8 base expert weights (layer.w8: E4M3 codes and
    per-output-row scales, weight = scale * value(code)); the LoRA matrices
    are the layer's bf16 ones.  Returns (out, n_invalid_pairs)."""
    lib = lib or _load()
    q = layer.w8
    if q is None:
        raise ValueError("forward_w8: the layer has no FP8 weights")
    d, a = _args(layer)
    if tokens is None:
        tok = None
        n = layer.T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = tok.size
    W1q, W2q = _c(q.W1q, np.uint8), _c(q.W2q, np.uint8)
    W1s, W2s = _c(q.W1s, np.float32), _c(q.W2s, np.float32)
    out = np.zeros((n, layer.H), dtype=np.float64)
    nt = n_threads or default_threads()
    inv = lib.oracle_forward_w8(ctypes.byref(d), _ptr(a["x"]), _ptr(a["topk_ids"]), _ptr(a["topk_weights"]),
                                _ptr(a["lora_ids"]), _ptr(W1q), _ptr(W1s), _ptr(W2q), _ptr(W2s),
                                _ptr(a["A1"]), _ptr(a["B1"]), _ptr(a["A2"]), _ptr(a["B2"]), _ptr(tok), n,
                                _ptr(out), nt)
    if inv < 0:
        raise ValueError("oracle_forward_w8: bad arguments")
    return out, int(inv)


def e4m3(code: int, lib=None) -> float:
    """Value of one E4M3 code by the oracle's decoder."""
    return float((lib or _load()).oracle_e4m3(int(code)))


def pair(layer, p: int, lib=None):
    """Intermediates of pair p: dict(z1, g, act, z2, d, valid)."""
    lib = lib or _load()
    d, a = _args(layer)
    res = dict(z1=np.zeros(layer.r), g=np.zeros(2 * layer.I), act=np.zeros(layer.I),
               z2=np.zeros(layer.r), d=np.zeros(layer.H))
    rc = lib.oracle_pair(ctypes.byref(d), _ptr(a["x"]), _ptr(a["topk_ids"]), _ptr(a["lora_ids"]),
                         _ptr(a["W1"]), _ptr(a["W2"]), _ptr(a["A1"]), _ptr(a["B1"]), _ptr(a["A2"]),
                         _ptr(a["B2"]), int(p), _ptr(res["z1"]), _ptr(res["g"]), _ptr(res["act"]),
                         _ptr(res["z2"]), _ptr(res["d"]))
    if rc < 0:
        raise ValueError("oracle_pair: bad arguments")
    res["valid"] = rc == 0
    return res


def align_capacity(T: int, k: int, E: int, L: int, bm: int) -> int:
    return int(_load().oracle_align_capacity(T, k, E, L, bm))


def align(topk_ids, lora_ids, E: int, L: int, bm: int):
    """Expert x adapter bucketing; returns a dict of numpy arrays and counts."""
    lib = _load()
    topk = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = topk.shape
    lora = np.ascontiguousarray(lora_ids, dtype=np.int32)
    cap = align_capacity(T, k, E, L, bm)
    NB = E * (L + 1)
    sorted_ids = np.full(max(cap, 1), -7, dtype=np.int32)
    tiles = max(cap // bm, 1)
    tile_expert = np.full(tiles, -7, dtype=np.int32)
    tile_lora = np.full(tiles, -7, dtype=np.int32)
    npp = np.zeros(1, dtype=np.int32)
    cnt = np.zeros(NB, dtype=np.int32)
    off = np.zeros(NB + 1, dtype=np.int32)
    inv = lib.oracle_align(T, k, E, L, bm, _ptr(topk), _ptr(lora), _ptr(sorted_ids), cap,
                           _ptr(tile_expert), _ptr(tile_lora), _ptr(npp), _ptr(cnt), _ptr(off))
    if inv < 0:
        raise ValueError(f"oracle_align failed: {inv}")
    n = int(npp[0])
    return dict(sorted_ids=sorted_ids[:n].copy(), tile_expert=tile_expert[:n // bm].copy(),
                tile_lora=tile_lora[:n // bm].copy(), num_post_padded=n, bucket_count=cnt,
                bucket_offset=off, invalid=int(inv), capacity=cap)
