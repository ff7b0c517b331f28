"""CPU oracle for the GDN speculative transaction -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around ``gdn_oracle.c`` (plain sequential fp64 C).  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product library never does, and it
has no CPU fallback.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against something other than itself (numpy's convolution, a dense
matrix-product form of the recurrence, closed forms, an fp64 chunked/WY
reformulation, and a hand-worked example under ``tests/golden/``).  The pieces
pinned only to a reading rather than to the pages are listed in the design
notes: the SiLU activation, the 1e-6 L2-norm epsilon and the key-head mapping.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)
_F = ctypes.POINTER(ctypes.c_float)
_I = ctypes.POINTER(ctypes.c_int32)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_int = ctypes.c_int


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library (plain C11, no FMA contraction)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library in ``oracle/_build`` if it is missing or stale."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
            compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _p(a, ct):
    return a.ctypes.data_as(ct)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_causal_conv.argtypes = [_int, _int, _int, _D, _D, _D, _D]
        lib.oracle_causal_conv.restype = None
        lib.oracle_verify.argtypes = [_int] * 7 + [_D, _D, _D, _D, _D, _F, _U8, _D, _D]
        lib.oracle_verify.restype = _int
        lib.oracle_commit.argtypes = [_int] * 6 + [_I, _U8, _D, _D, _F, _D, _I, _I]
        lib.oracle_commit.restype = None
        lib.oracle_prefill.argtypes = [_int] * 7 + [_D, _D, _D, _D, _D, _F, _D, _I]
        lib.oracle_prefill.restype = _int
        lib.oracle_accept.argtypes = [_int] * 3 + [_D, _I, _U8, _I, _I]
        lib.oracle_accept.restype = _int
        lib.oracle_gated_rmsnorm.argtypes = [_int, _int, _D, _D, _D, ctypes.c_double, _D]
        lib.oracle_gated_rmsnorm.restype = None
        self.lib = lib
        self.path = lib_path

    def causal_conv(self, hist, x, w, act=1):
        """hist [C][3], x [n][C], w [C][4] -> y [n][C] (fp64)."""
        hist, x, w = _f64(hist), _f64(x), _f64(w)
        n, C = x.shape
        y = np.empty((n, C), dtype=np.float64)
        self.lib.oracle_causal_conv(n, C, act, _p(hist, _D), _p(x, _D), _p(w, _D), _p(y, _D))
        return y

    def verify(self, x, w, win, g, beta, S0, active, H_k, act=1, want_states=True):
        """Sequential verify from the pre-verification state.

        x [B][T][C], w [C][4], win [B][C][3], g/beta [B][T][H_v],
        S0 float32 [B][H_v][d][d], active uint8 [B].
        Returns (o [B][T][H_v][d] fp64, Sall [B][T][H_v][d][d] fp64 or None).
        """
        x, w, win, g, beta = map(_f64, (x, w, win, g, beta))
        S0 = np.ascontiguousarray(S0, dtype=np.float32)
        active = np.ascontiguousarray(active, dtype=np.uint8)
        B, T, C = x.shape
        H_v, dv, dk = S0.shape[1:]
        o = np.empty((B, T, H_v, dv), dtype=np.float64)
        Sall = np.empty((B, T, H_v, dv, dk), dtype=np.float64) if want_states else None
        rc = self.lib.oracle_verify(B, T, H_k, H_v, dk, dv, act, _p(x, _D), _p(w, _D), _p(win, _D),
                                    _p(g, _D), _p(beta, _D), _p(S0, _F), _p(active, _U8), _p(o, _D),
                                    _p(Sall, _D) if want_states else None)
        if rc:
            raise MemoryError("oracle_verify allocation failed")
        return o, Sall

    def commit(self, keep, active, Sall, x, S, win, offsets):
        """Accepted-prefix commit, in place on S (fp32), win (fp64) and offsets (int32).

        Returns the status word (bit 0: an active row had keep outside [0, T]).
        """
        for a, dt in ((S, np.float32), (win, np.float64), (offsets, np.int32)):
            if a.dtype != dt or not a.flags.c_contiguous:
                raise TypeError("commit updates S, win and offsets in place: pass contiguous arrays")
        keep = np.ascontiguousarray(keep, dtype=np.int32)
        active = np.ascontiguousarray(active, dtype=np.uint8)
        Sall, x = _f64(Sall), _f64(x)
        B, T, H_v, dv, dk = Sall.shape
        C = x.shape[2]
        status = np.zeros(1, dtype=np.int32)
        self.lib.oracle_commit(B, T, H_v, dk, dv, C, _p(keep, _I), _p(active, _U8), _p(Sall, _D),
                               _p(x, _D), _p(S, _F), _p(win, _D), _p(offsets, _I), _p(status, _I))
        return int(status[0])

    def prefill(self, x, w, win, g, beta, S, offsets, H_k, act=1):
        """Sequential priming over L tokens; updates S (fp32), win, offsets in place.

        x [B][L][C], g/beta [B][L][H_v].  Returns o [B][L][H_v][d] (fp64).
        """
        for a, dt in ((S, np.float32), (win, np.float64), (offsets, np.int32)):
            if a.dtype != dt or not a.flags.c_contiguous:
                raise TypeError("prefill updates S, win and offsets in place: pass contiguous arrays")
        x, w, g, beta = map(_f64, (x, w, g, beta))
        B, L, C = x.shape
        H_v, dv, dk = S.shape[1:]
        o = np.empty((B, L, H_v, dv), dtype=np.float64)
        rc = self.lib.oracle_prefill(B, L, H_k, H_v, dk, dv, act, _p(x, _D), _p(w, _D), _p(win, _D),
                                     _p(g, _D), _p(beta, _D), _p(S, _F), _p(o, _D), _p(offsets, _I))
        if rc:
            raise MemoryError("oracle_prefill allocation failed")
        return o


    def accept(self, logits, draft, active):
        """Greedy acceptance: logits [B][T][V] (values as given), draft [B][T]
        int32, active [B] -> (keep [B], next [B]) int32."""
        logits = _f64(logits)
        B, T, V = logits.shape
        draft = np.ascontiguousarray(draft, dtype=np.int32)
        active = np.ascontiguousarray(active, dtype=np.uint8)
        keep = np.empty(B, dtype=np.int32)
        nxt = np.empty(B, dtype=np.int32)
        if self.lib.oracle_accept(B, T, V, _p(logits, _D), _p(draft, _I), _p(active, _U8), _p(keep, _I),
                                  _p(nxt, _I)):
            raise MemoryError("oracle_accept allocation failed")
        return keep, nxt


    def gated_rmsnorm(self, o, z, w, eps=1e-6):
        """y = o / sqrt(mean(o^2) + eps) * w * silu(z) over the last axis (fp64)."""
        o, z, w = _f64(o), _f64(z), _f64(w)
        d = o.shape[-1]
        y = np.empty_like(o)
        self.lib.oracle_gated_rmsnorm(int(o.size // d), d, _p(o, _D), _p(z, _D), _p(w, _D), float(eps), _p(y, _D))
        return y


_default = None


def default() -> Oracle:
    """The oracle built from ``gdn_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        path = build()
        with _lock:
            if _default is None:
                _default = Oracle(path)
    return _default


def causal_conv(*a, **k):
    return default().causal_conv(*a, **k)


def verify(*a, **k):
    return default().verify(*a, **k)


def commit(*a, **k):
    return default().commit(*a, **k)


def prefill(*a, **k):
    return default().prefill(*a, **k)


def accept(*a, **k):
    return default().accept(*a, **k)


def gated_rmsnorm(*a, **k):
    return default().gated_rmsnorm(*a, **k)
