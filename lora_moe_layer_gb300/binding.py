"""Thin ctypes binding of libmoelora.so (include/moe_lora.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, turns tensors into device pointers and the stream into a
cudaStream_t, and returns the C status code.  All compute runs in the CUDA
library; if the library is missing this module raises instead of falling
back to anything.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoelora.so")

MOELORA_OK = 0
MOELORA_EINVAL = -1
MOELORA_ENOSPC = -2
MOELORA_EUNSUPPORTED = -3
MOELORA_ECUDA = -4
MOELORA_EDEVICE_ID = -5
MOELORA_ETIMEOUT = -6

# every symbol the header declares
EXPORTED = ("moe_lora_strerror", "moe_lora_version", "moe_lora_align_capacity",
            "moe_lora_workspace_bytes", "moe_lora_align", "moe_lora_forward",
            "moe_lora_get_status", "moe_lora_workspace_layout", "moe_lora_forward_traced",
            "moe_lora_forward_noalloc", "moe_lora_selftest_wait", "moe_lora_forward_w8",
            "moe_lora_forward_w8_traced")
MOELORA_NOALLOC_SCRATCH_BYTES = 16 << 20
MOELORA_TRACE_EVENTS = 6
# kernel slots of one forward, in launch order
KERNEL_SLOTS = ("align", "gather_x", "gate_up_gemm", "down_gemm", "topk_reduce")


class MoeLoraError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: status {code} ({moe_lora_strerror(code)})")


class moe_lora_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "E", "k", "L", "r", "block_m", "options",
                                                     "sm_count")]


class moe_lora_ws_layout(ctypes.Structure):
    _fields_ = [("compact_ids", ctypes.c_size_t), ("compact_offset", ctypes.c_size_t),
                ("z1", ctypes.c_size_t), ("act", ctypes.c_size_t), ("z2", ctypes.c_size_t),
                ("pair_out", ctypes.c_size_t), ("s1", ctypes.c_int32), ("s2", ctypes.c_int32),
                ("down_splits", ctypes.c_int32), ("launches", ctypes.c_int32), ("gemm_ctas", ctypes.c_int32),
                ("tc_expand", ctypes.c_int32), ("pair_out_bf16", ctypes.c_int32), ("total", ctypes.c_size_t)]


_lib = None


def library_path() -> str:
    return LIB_PATH


def load(path: Optional[str] = None):
    """Open libmoelora.so (built in-tree by lora_moe_layer_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with lora_moe_layer_gb300.build.build() "
                           "(the layer has no non-CUDA implementation)")
    lib = ctypes.CDLL(p)
    V, SZ, I32, I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
    D = ctypes.POINTER(moe_lora_dims)
    lib.moe_lora_strerror.restype = ctypes.c_char_p
    lib.moe_lora_strerror.argtypes = [I32]
    lib.moe_lora_version.restype = I32
    lib.moe_lora_version.argtypes = []
    lib.moe_lora_align_capacity.restype = I64
    lib.moe_lora_align_capacity.argtypes = [D]
    lib.moe_lora_workspace_bytes.restype = SZ
    lib.moe_lora_workspace_bytes.argtypes = [D]
    lib.moe_lora_align.restype = I32
    lib.moe_lora_align.argtypes = [D, V, V, V, V, V, V, V, V, V, SZ, V]
    lib.moe_lora_forward.restype = I32
    lib.moe_lora_forward.argtypes = [D] + [V] * 12 + [SZ, V]
    lib.moe_lora_forward_traced.restype = I32
    lib.moe_lora_forward_traced.argtypes = [D] + [V] * 12 + [SZ, V, ctypes.POINTER(V), ctypes.c_int32]
    lib.moe_lora_forward_w8.restype = I32
    lib.moe_lora_forward_w8.argtypes = [D] + [V] * 14 + [SZ, V]
    lib.moe_lora_forward_w8_traced.restype = I32
    lib.moe_lora_forward_w8_traced.argtypes = [D] + [V] * 14 + [SZ, V, ctypes.POINTER(V), ctypes.c_int32]
    lib.moe_lora_forward_noalloc.restype = I32
    lib.moe_lora_forward_noalloc.argtypes = [D] + [V] * 12
    lib.moe_lora_get_status.restype = I32
    lib.moe_lora_get_status.argtypes = [V, V]
    lib.moe_lora_selftest_wait.restype = I32
    lib.moe_lora_selftest_wait.argtypes = [I32, V, V]
    lib.moe_lora_workspace_layout.restype = I32
    lib.moe_lora_workspace_layout.argtypes = [D, ctypes.POINTER(moe_lora_ws_layout)]
    if path is None:
        _lib = lib
    return lib


# ---------------------------------------------------------------- marshalling

MOELORA_OPT_SINGLE_CTA = 1


def dims(T: int, H: int, I: int, E: int, k: int, L: int, r: int, block_m: int = 0,
         options: int = 0, sm_count: int = 0) -> moe_lora_dims:
    return moe_lora_dims(T, H, I, E, k, L, r if L > 0 else 0, block_m, options, sm_count)


def _ptr(t) -> Optional[int]:
    """Device pointer of a tensor (or pass an int address / None through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- entry points

def moe_lora_strerror(code: int) -> str:
    return load().moe_lora_strerror(code).decode()


def moe_lora_version() -> int:
    return load().moe_lora_version()


def moe_lora_align_capacity(d: moe_lora_dims) -> int:
    return load().moe_lora_align_capacity(ctypes.byref(d))


def moe_lora_workspace_bytes(d: moe_lora_dims) -> int:
    return load().moe_lora_workspace_bytes(ctypes.byref(d))


def moe_lora_workspace_layout(d: moe_lora_dims) -> dict:
    out = moe_lora_ws_layout()
    st = load().moe_lora_workspace_layout(ctypes.byref(d), ctypes.byref(out))
    if st != MOELORA_OK:
        raise MoeLoraError(st, "moe_lora_workspace_layout")
    return {name: getattr(out, name) for name, _ in moe_lora_ws_layout._fields_}


def moe_lora_align(d: moe_lora_dims, topk_ids, token_lora_ids, sorted_ids, tile_expert, tile_lora,
                   num_post_padded, bucket_count, bucket_offset, workspace, stream=None,
                   workspace_bytes: Optional[int] = None) -> int:
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return load().moe_lora_align(ctypes.byref(d), _ptr(topk_ids), _ptr(token_lora_ids), _ptr(sorted_ids),
                                 _ptr(tile_expert), _ptr(tile_lora), _ptr(num_post_padded),
                                 _ptr(bucket_count), _ptr(bucket_offset), _ptr(workspace), wb,
                                 _stream(stream))


def moe_lora_forward(d: moe_lora_dims, x, topk_ids, topk_weights, token_lora_ids, W1, W2, A1, B1, A2, B2,
                     out, workspace, stream=None, workspace_bytes: Optional[int] = None) -> int:
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return load().moe_lora_forward(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                   _ptr(token_lora_ids), _ptr(W1), _ptr(W2), _ptr(A1), _ptr(B1),
                                   _ptr(A2), _ptr(B2), _ptr(out), _ptr(workspace), wb, _stream(stream))


def _event_handles(events):
    """cudaEvent_t handles of torch.cuda.Event objects (or raw ints), as a C array."""
    handles = []
    for ev in events:
        if isinstance(ev, int):
            handles.append(ev)
        else:
            if ev.cuda_event == 0:  # torch creates the event lazily
                ev.record()
            handles.append(ev.cuda_event)
    return (ctypes.c_void_p * len(handles))(*handles), len(handles)


def moe_lora_forward_traced(d: moe_lora_dims, x, topk_ids, topk_weights, token_lora_ids, W1, W2, A1, B1, A2,
                            B2, out, workspace, events, stream=None,
                            workspace_bytes: Optional[int] = None) -> int:
    """events: MOELORA_TRACE_EVENTS torch.cuda.Event objects (or raw cudaEvent_t ints)."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    arr, n = _event_handles(events)
    return load().moe_lora_forward_traced(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                          _ptr(token_lora_ids), _ptr(W1), _ptr(W2), _ptr(A1), _ptr(B1),
                                          _ptr(A2), _ptr(B2), _ptr(out), _ptr(workspace), wb,
                                          _stream(stream), arr, n)


def moe_lora_forward_w8(d: moe_lora_dims, x, topk_ids, topk_weights, token_lora_ids, W1q, W1s, W2q, W2s, A1, B1,
                        A2, B2, out, workspace, stream=None, workspace_bytes: Optional[int] = None) -> int:
    """The forward with FP8 (E4M3) base expert weights and per-row fp32 scales."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return load().moe_lora_forward_w8(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                      _ptr(token_lora_ids), _ptr(W1q), _ptr(W1s), _ptr(W2q), _ptr(W2s), _ptr(A1),
                                      _ptr(B1), _ptr(A2), _ptr(B2), _ptr(out), _ptr(workspace), wb,
                                      _stream(stream))


def moe_lora_forward_w8_traced(d: moe_lora_dims, x, topk_ids, topk_weights, token_lora_ids, W1q, W1s, W2q, W2s,
                               A1, B1, A2, B2, out, workspace, events, stream=None,
                               workspace_bytes: Optional[int] = None) -> int:
    """moe_lora_forward_w8 with the timing marks of moe_lora_forward_traced."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    arr, n = _event_handles(events)
    return load().moe_lora_forward_w8_traced(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                             _ptr(token_lora_ids), _ptr(W1q), _ptr(W1s), _ptr(W2q), _ptr(W2s),
                                             _ptr(A1), _ptr(B1), _ptr(A2), _ptr(B2), _ptr(out), _ptr(workspace), wb,
                                             _stream(stream), arr, n)


def moe_lora_forward_noalloc(d: moe_lora_dims, x, topk_ids, topk_weights, token_lora_ids, W1, W2, A1, B1, A2,
                             B2, out, stream=None) -> int:
    """moe_lora_forward on the library's built-in 16 MiB scratch buffer, for callers that
    cannot allocate device memory (see include/moe_lora.h for the sharing rules)."""
    return load().moe_lora_forward_noalloc(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                           _ptr(token_lora_ids), _ptr(W1), _ptr(W2), _ptr(A1), _ptr(B1),
                                           _ptr(A2), _ptr(B2), _ptr(out), _stream(stream))


def moe_lora_selftest_wait(kind: int, workspace, stream=None) -> int:
    return load().moe_lora_selftest_wait(kind, _ptr(workspace), _stream(stream))


def moe_lora_get_status(workspace, stream=None) -> int:
    return load().moe_lora_get_status(_ptr(workspace), _stream(stream))


def check(status: int, where: str = "moe_lora") -> None:
    if status != MOELORA_OK:
        raise MoeLoraError(status, where)
