"""Python binding of libgdn_gb300.so (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: it turns torch tensors into device pointers and the
current torch stream into a cudaStream_t, calls the library, and raises
GdnError on a nonzero return code.  There is no CPU fallback: if the library
cannot be built or loaded, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_MISALIGNED = -3
GDN_ERR_WORKSPACE = -4
GDN_ERR_CUDA = -5
GDN_ACT_NONE = 0
GDN_ACT_SILU = 1
GDN_COMMIT_RECOMPUTE = 0
GDN_COMMIT_SNAPSHOT = 1
GDN_COMMIT_DEFERRED = 2
GDN_VERIFY_OVERLAP = 0x100
GDN_VERIFY_OVERLAP_STATE = 0x200
GDN_STATUS_TIMEOUT = 2
GDN_STATUS_BAD_KEEP = 1
GDN_STATUS_BAD_ROW = 4
GDN_MAX_LAYERS = 256
GDN_NOALLOC_WS_BYTES = 4 << 20

EXPORTS = ("gdn_version", "gdn_last_error", "gdn_layer_workspace_bytes", "gdn_conv_verify",
           "gdn_commit", "gdn_prefill_workspace_bytes", "gdn_prefill_chunked", "gdn_get_status",
           "gdn_conv_verify_noalloc", "gdn_flush", "gdn_accept_workspace_bytes", "gdn_accept_greedy",
           "gdn_conv_verify_gated", "gdn_move_rows", "gdn_test_verify_timeout")


class GdnError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


class gdn_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "T", "T_max", "H_k", "H_v", "d_k", "d_v", "width", "act")]


def dims(B, T, H_k, H_v, d, T_max=None, width=4, act=GDN_ACT_SILU) -> gdn_dims:
    """gdn_dims for one cohort: B rows, T positions per verify (T_max >= T sizes
    the conv ring), H_k key and H_v value heads of size d, width-4 conv."""
    return gdn_dims(B, T, T if T_max is None else T_max, H_k, H_v, d, d, width, act)


def dims_of(geom) -> gdn_dims:
    """gdn_dims from a synth.Geometry."""
    return dims(geom.B, geom.T, geom.H_k, geom.H_v, geom.d, geom.tmax, geom.width, geom.act)


_P = ctypes.c_void_p
_lock = threading.Lock()
_lib = None


def _declare(lib):
    D = ctypes.POINTER(gdn_dims)
    lib.gdn_version.restype = ctypes.c_char_p
    lib.gdn_version.argtypes = []
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_layer_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_layer_workspace_bytes.argtypes = [D, ctypes.c_int]
    lib.gdn_conv_verify.restype = ctypes.c_int
    lib.gdn_conv_verify.argtypes = [D, ctypes.c_int] + [_P] * 10 + [ctypes.c_size_t, _P]
    lib.gdn_commit.restype = ctypes.c_int
    lib.gdn_commit.argtypes = [D, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_P), ctypes.POINTER(_P),
                               ctypes.POINTER(_P), _P, _P, _P, _P]
    lib.gdn_flush.restype = ctypes.c_int
    lib.gdn_flush.argtypes = [D, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_P), ctypes.POINTER(_P), _P]
    lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_prefill_workspace_bytes.argtypes = [D, ctypes.c_int]
    lib.gdn_prefill_chunked.restype = ctypes.c_int
    lib.gdn_prefill_chunked.argtypes = [D, ctypes.c_int] + [_P] * 9 + [ctypes.c_size_t, _P]
    lib.gdn_conv_verify_noalloc.restype = ctypes.c_int
    lib.gdn_conv_verify_noalloc.argtypes = [D, ctypes.c_int] + [_P] * 9 + [ctypes.POINTER(_P), _P]
    lib.gdn_test_verify_timeout.restype = ctypes.c_int
    lib.gdn_test_verify_timeout.argtypes = [D, ctypes.c_int] + [_P] * 10 + [ctypes.c_size_t, ctypes.c_uint32, _P]
    lib.gdn_get_status.restype = ctypes.c_int
    lib.gdn_get_status.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)]
    lib.gdn_conv_verify_gated.restype = ctypes.c_int
    lib.gdn_conv_verify_gated.argtypes = [D, ctypes.c_int] + [_P] * 10 + [ctypes.c_float, _P, _P, ctypes.c_size_t, _P]
    PP = ctypes.POINTER(_P)
    lib.gdn_move_rows.restype = ctypes.c_int
    lib.gdn_move_rows.argtypes = [D, D, ctypes.c_int, ctypes.c_int, PP, PP, _P, PP, PP, _P, PP, _P, _P,
                                  ctypes.c_int, _P]
    lib.gdn_accept_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_accept_workspace_bytes.argtypes = [ctypes.c_int] * 3
    lib.gdn_accept_greedy.restype = ctypes.c_int
    lib.gdn_accept_greedy.argtypes = [ctypes.c_int] * 3 + [_P] * 6 + [ctypes.c_size_t, _P]


def library_path() -> str:
    """Where build() puts libgdn_gb300.so."""
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load (building first if missing or stale) and return the ctypes library."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or _build.build()
            if not os.path.exists(p):
                raise RuntimeError(f"libgdn_gb300.so not found at {p}")
            lib = ctypes.CDLL(p)
            _declare(lib)
            if path is not None:
                return lib
            _lib = lib
    return _lib


# ------------------------------------------------------------------ marshalling
def _ptr(t, what, dtype=None):
    """Device pointer of a tensor (or a raw int pointer / None)."""
    if t is None or isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what}: expected a torch.Tensor or an int pointer")
    if not t.is_cuda:
        raise ValueError(f"{what}: tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{what}: tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc, fn):
    if rc != GDN_OK:
        raise GdnError(rc, fn, load().gdn_last_error().decode())


def _t():
    import torch
    return torch


def gdn_version() -> str:
    """Library name, version and target architecture."""
    return load().gdn_version().decode()


def gdn_last_error() -> str:
    """Text of the last error returned on this thread."""
    return load().gdn_last_error().decode()


def gdn_layer_workspace_bytes(d: gdn_dims, mode: int) -> int:
    """Bytes of per-layer workspace gdn_conv_verify fills and gdn_commit reads
    in commit mode `mode` (0 for invalid dims or mode)."""
    return int(load().gdn_layer_workspace_bytes(ctypes.byref(d), mode))


def gdn_conv_verify(d: gdn_dims, mode, x, conv_w, g, beta, state, ring, offsets, active, out,
                    layer_ws, layer_ws_bytes=None, stream=None):
    """Verify one layer (gdn.h, gdn_conv_verify).  CUDA tensors: x [B][T][C]
    bf16, conv_w [C][4] bf16, g and beta [B][T][H_v] fp32, state
    [B][H_v][d][d] fp32, ring [B][R][C] bf16, offsets [B] int32 (may be
    None), active [B] uint8, out [B][T][H_v][d] bf16, layer_ws uint8 of
    gdn_layer_workspace_bytes.  `mode` may carry GDN_VERIFY_OVERLAP.
    Runs on `stream` (default: torch's current stream)."""
    torch = _t()
    if layer_ws_bytes is None:
        layer_ws_bytes = layer_ws.numel() * layer_ws.element_size()
    rc = load().gdn_conv_verify(
        ctypes.byref(d), mode, _ptr(x, "x", torch.bfloat16), _ptr(conv_w, "conv_w", torch.bfloat16),
        _ptr(g, "g", torch.float32), _ptr(beta, "beta", torch.float32), _ptr(state, "state", torch.float32),
        _ptr(ring, "ring", torch.bfloat16), _ptr(offsets, "offsets", torch.int32),
        _ptr(active, "active", torch.uint8), _ptr(out, "out", torch.bfloat16), _ptr(layer_ws, "layer_ws"),
        int(layer_ws_bytes), _stream(stream))
    _check(rc, "gdn_conv_verify")


def gdn_conv_verify_gated(d: gdn_dims, mode, x, conv_w, g, beta, state, ring, offsets, active, gate_z, norm_w,
                          eps, out, layer_ws, layer_ws_bytes=None, stream=None):
    """gdn_conv_verify with the gated RMSNorm of the output fused in:
    out = o / sqrt(mean(o^2) + eps) * norm_w * silu(gate_z) per (row, position, head)."""
    torch = _t()
    if layer_ws_bytes is None:
        layer_ws_bytes = layer_ws.numel() * layer_ws.element_size()
    rc = load().gdn_conv_verify_gated(
        ctypes.byref(d), mode, _ptr(x, "x", torch.bfloat16), _ptr(conv_w, "conv_w", torch.bfloat16),
        _ptr(g, "g", torch.float32), _ptr(beta, "beta", torch.float32), _ptr(state, "state", torch.float32),
        _ptr(ring, "ring", torch.bfloat16), _ptr(offsets, "offsets", torch.int32),
        _ptr(active, "active", torch.uint8), _ptr(gate_z, "gate_z", torch.bfloat16),
        _ptr(norm_w, "norm_w", torch.bfloat16), float(eps), _ptr(out, "out", torch.bfloat16),
        _ptr(layer_ws, "layer_ws"), int(layer_ws_bytes), _stream(stream))
    _check(rc, "gdn_conv_verify_gated")


def gdn_conv_verify_noalloc(d: gdn_dims, mode, x, conv_w, g, beta, state, ring, offsets, active, out,
                            stream=None) -> int:
    """gdn_conv_verify with the library's built-in scratch as the workspace.

    For callers that cannot allocate device memory.  Returns the scratch's
    device address, to be passed as this layer's workspace to gdn_commit
    before the next call of this function on the device.
    """
    torch = _t()
    used = _P(0)
    rc = load().gdn_conv_verify_noalloc(
        ctypes.byref(d), mode, _ptr(x, "x", torch.bfloat16), _ptr(conv_w, "conv_w", torch.bfloat16),
        _ptr(g, "g", torch.float32), _ptr(beta, "beta", torch.float32), _ptr(state, "state", torch.float32),
        _ptr(ring, "ring", torch.bfloat16), _ptr(offsets, "offsets", torch.int32),
        _ptr(active, "active", torch.uint8), _ptr(out, "out", torch.bfloat16), ctypes.byref(used),
        _stream(stream))
    _check(rc, "gdn_conv_verify_noalloc")
    return int(used.value)


def gdn_test_verify_timeout(d: gdn_dims, mode, x, conv_w, g, beta, state, ring, offsets, active, out, layer_ws,
                            wait_limit, layer_ws_bytes=None, stream=None):
    """gdn_conv_verify with its bounded-wait failure path forced for the CTA of
    (row 0, head 0), giving up after `wait_limit` polls (gdn.h, test hook)."""
    torch = _t()
    if layer_ws_bytes is None:
        layer_ws_bytes = layer_ws.numel() * layer_ws.element_size()
    rc = load().gdn_test_verify_timeout(
        ctypes.byref(d), mode, _ptr(x, "x", torch.bfloat16), _ptr(conv_w, "conv_w", torch.bfloat16),
        _ptr(g, "g", torch.float32), _ptr(beta, "beta", torch.float32), _ptr(state, "state", torch.float32),
        _ptr(ring, "ring", torch.bfloat16), _ptr(offsets, "offsets", torch.int32),
        _ptr(active, "active", torch.uint8), _ptr(out, "out", torch.bfloat16), _ptr(layer_ws, "layer_ws"),
        int(layer_ws_bytes), int(wait_limit), _stream(stream))
    _check(rc, "gdn_test_verify_timeout")


def _layer_ptrs(seq, what, dtype=None):
    return (_P * max(len(seq), 1))(*[_ptr(t, f"{what}[{i}]", dtype) for i, t in enumerate(seq)])


def gdn_commit(d: gdn_dims, mode, states, rings, layer_ws, keep, active, offsets, stream=None):
    """states / rings / layer_ws: sequences (one per layer) of tensors or int device pointers."""
    torch = _t()
    n = len(states)
    if len(layer_ws) != n or len(rings) != n:
        raise ValueError("states, rings and layer_ws must have one entry per layer")
    rc = load().gdn_commit(ctypes.byref(d), mode, n, _layer_ptrs(states, "state", torch.float32),
                           _layer_ptrs(rings, "ring", torch.bfloat16), _layer_ptrs(layer_ws, "layer_ws"),
                           _ptr(keep, "keep", torch.int32), _ptr(active, "active", torch.uint8),
                           _ptr(offsets, "offsets", torch.int32), _stream(stream))
    _check(rc, "gdn_commit")


def gdn_flush(d: gdn_dims, mode, states, layer_ws, stream=None):
    """Materialise commits a DEFERRED cycle left pending (no-op in other modes)."""
    torch = _t()
    if len(layer_ws) != len(states):
        raise ValueError("states and layer_ws must have one entry per layer")
    rc = load().gdn_flush(ctypes.byref(d), mode, len(states), _layer_ptrs(states, "state", torch.float32),
                          _layer_ptrs(layer_ws, "layer_ws"), _stream(stream))
    _check(rc, "gdn_flush")


def gdn_prefill_workspace_bytes(d: gdn_dims, L: int) -> int:
    """Bytes of scratch gdn_prefill_chunked needs for an L-token prompt."""
    return int(load().gdn_prefill_workspace_bytes(ctypes.byref(d), L))


def gdn_prefill_chunked(d: gdn_dims, L, x, conv_w, g, beta, state, ring, offsets, out, ws,
                        ws_bytes=None, stream=None):
    """Prime state, ring and offsets over an L-token prompt (gdn.h,
    gdn_prefill_chunked): x [B][L][C] bf16, g and beta [B][L][H_v] fp32,
    out [B][L][H_v][d] bf16, ws of gdn_prefill_workspace_bytes; the other
    tensors as in gdn_conv_verify."""
    torch = _t()
    if ws_bytes is None:
        ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().gdn_prefill_chunked(
        ctypes.byref(d), L, _ptr(x, "x", torch.bfloat16), _ptr(conv_w, "conv_w", torch.bfloat16),
        _ptr(g, "g", torch.float32), _ptr(beta, "beta", torch.float32), _ptr(state, "state", torch.float32),
        _ptr(ring, "ring", torch.bfloat16), _ptr(offsets, "offsets", torch.int32),
        _ptr(out, "out", torch.bfloat16), _ptr(ws, "ws"), int(ws_bytes), _stream(stream))
    _check(rc, "gdn_prefill_chunked")


def gdn_move_rows(src_d: gdn_dims, dst_d: gdn_dims, mode, src_states, src_rings, src_offsets, dst_states,
                  dst_rings, dst_offsets, dst_layer_ws, src_rows, dst_rows, stream=None):
    """Copy rows src_rows[i] of one cohort into rows dst_rows[i] of another,
    every layer: state, conv cache and committed offset (device index arrays)."""
    torch = _t()
    n = len(src_states)
    ws = None if dst_layer_ws is None else _layer_ptrs(dst_layer_ws, "dst_layer_ws")
    rc = load().gdn_move_rows(
        ctypes.byref(src_d), ctypes.byref(dst_d), mode, n, _layer_ptrs(src_states, "src_state", torch.float32),
        _layer_ptrs(src_rings, "src_ring", torch.bfloat16), _ptr(src_offsets, "src_offsets", torch.int32),
        _layer_ptrs(dst_states, "dst_state", torch.float32), _layer_ptrs(dst_rings, "dst_ring", torch.bfloat16),
        _ptr(dst_offsets, "dst_offsets", torch.int32), ws, _ptr(src_rows, "src_rows", torch.int32),
        _ptr(dst_rows, "dst_rows", torch.int32), int(src_rows.numel()), _stream(stream))
    _check(rc, "gdn_move_rows")


def gdn_accept_workspace_bytes(B: int, T: int, V: int) -> int:
    """Bytes of workspace gdn_accept_greedy needs (0 for invalid sizes)."""
    return int(load().gdn_accept_workspace_bytes(B, T, V))


def gdn_accept_greedy(logits, draft, active, keep, nxt, ws, stream=None):
    """Greedy acceptance on the device: logits [B][T][V] bf16, draft [B][T]
    int32, active [B] uint8 -> keep [B], nxt [B] int32 (written in place).
    ws: gdn_accept_workspace_bytes(B, T, V) bytes, zero-filled once."""
    torch = _t()
    B, T, V = logits.shape
    rc = load().gdn_accept_greedy(B, T, V, _ptr(logits, "logits", torch.bfloat16), _ptr(draft, "draft", torch.int32),
                                  _ptr(active, "active", torch.uint8), _ptr(keep, "keep", torch.int32),
                                  _ptr(nxt, "next", torch.int32), _ptr(ws, "ws"),
                                  ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "gdn_accept_greedy")


def gdn_get_status(clear: bool = False) -> int:
    """The sticky device status word (GDN_STATUS_* bits); synchronises the
    device.  clear=True resets it after reading."""
    v = ctypes.c_uint32(0)
    rc = load().gdn_get_status(1 if clear else 0, ctypes.byref(v))
    _check(rc, "gdn_get_status")
    return int(v.value)
