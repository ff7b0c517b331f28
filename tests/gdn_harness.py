"""Shared machinery for the GPU parity tests: the same seeded inputs go to the
CUDA library (through the C ABI) and to the CPU oracle, and the results are
compared element by element with the tolerances stated for this path:

* outputs o (bf16): max |o_gpu - o_ref| <= 2e-2, and max |diff| / max |o_ref|
  <= 1e-2 (a scale-aware bound, since |o| is often well below 1);
* fp32 state: per (layer, row, head) tile, max |dS| <= 1e-3 * max |S_ref| + 1e-6;
* offsets, conv windows, restored and inactive rows: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth

OUT_ABS_TOL = 2e-2
OUT_REL_TOL = 1e-2
STATE_REL_TOL = 1e-3
STATE_ABS_FLOOR = 1e-6


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_to_f32(bits).astype(np.float64)


def ring_window(ring_bits: np.ndarray) -> np.ndarray:
    """Committed conv window [B][C][3] (oldest first) of a ring [B][R][C]: the
    window lives in slots 0..2."""
    return f64(np.ascontiguousarray(np.transpose(ring_bits[:, :3, :], (0, 2, 1))))


def check_out(o_gpu: torch.Tensor, o_ref: np.ndarray, what: str):
    og = o_gpu.float().cpu().numpy().astype(np.float64)
    err = float(np.abs(og - o_ref).max()) if og.size else 0.0
    scale = float(np.abs(o_ref).max()) if og.size else 0.0
    assert np.isfinite(og).all(), f"{what}: non-finite outputs"
    assert err <= OUT_ABS_TOL, f"{what}: max abs err {err:.3e} > {OUT_ABS_TOL}"
    assert err <= OUT_REL_TOL * max(scale, 1e-3), f"{what}: err {err:.3e} vs scale {scale:.3e}"
    return err, scale


def check_state(S_gpu: np.ndarray, S_ref: np.ndarray, what: str):
    """S [..][d][d] compared per trailing (d, d) tile."""
    a = S_gpu.reshape(-1, S_gpu.shape[-2] * S_gpu.shape[-1]).astype(np.float64)
    r = S_ref.reshape(-1, S_ref.shape[-2] * S_ref.shape[-1]).astype(np.float64)
    err = np.abs(a - r).max(axis=1)
    bound = STATE_REL_TOL * np.abs(r).max(axis=1) + STATE_ABS_FLOOR
    assert np.isfinite(a).all(), f"{what}: non-finite state"
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, f"{what}: {bad.size} tiles out of tolerance, worst {float((err / bound).max()):.2f}x"
    return float((err / bound).max())


class GpuStack:
    """Device tensors of an n-layer GDN stack plus the verify/commit calls."""

    def __init__(self, geom: synth.Geometry, st: dict, active: np.ndarray, mode: int, n_layers: int):
        self.geom, self.mode, self.n = geom, mode, n_layers
        self.dims = L.dims_of(geom)
        self.state = torch.from_numpy(st["state"]).cuda()
        self.ring = dev_bf16(st["ring"])
        self.w = dev_bf16(st["conv_w"])
        self.offsets = torch.from_numpy(st["offsets"].copy()).cuda()
        self.active = torch.from_numpy(active.copy()).cuda()
        nbytes = L.gdn_layer_workspace_bytes(self.dims, mode)
        # zero-filled once: required by DEFERRED, harmless for the other modes
        self.ws = [torch.zeros(nbytes, dtype=torch.uint8, device="cuda") for _ in range(n_layers)]
        g = geom
        self.out = torch.empty((n_layers, g.B, g.T, g.H_v, g.d), dtype=torch.bfloat16, device="cuda")

    def verify(self, layer: int, x_bits, g, beta, overlap=False):
        mode = self.mode | (L.GDN_VERIFY_OVERLAP if overlap else 0)
        L.gdn_conv_verify(self.dims, mode, dev_bf16(x_bits), self.w[layer],
                          torch.from_numpy(np.ascontiguousarray(g)).cuda(),
                          torch.from_numpy(np.ascontiguousarray(beta)).cuda(),
                          self.state[layer], self.ring[layer], self.offsets, self.active,
                          self.out[layer], self.ws[layer])

    def commit(self, keep):
        L.gdn_commit(self.dims, self.mode, [self.state[l] for l in range(self.n)],
                     [self.ring[l] for l in range(self.n)], self.ws,
                     torch.from_numpy(np.asarray(keep, np.int32)).cuda(), self.active, self.offsets)

    def flush(self):
        """Materialise pending DEFERRED commits so `state` holds the committed state."""
        L.gdn_flush(self.dims, self.mode, [self.state[l] for l in range(self.n)], self.ws)


class OracleStack:
    """The oracle's mirror of a GpuStack: fp32 states, fp64 windows, offsets."""

    def __init__(self, geom: synth.Geometry, st: dict, active: np.ndarray, n_layers: int):
        self.geom, self.n = geom, n_layers
        self.S = st["state"].copy()
        self.w = [f64(st["conv_w"][l]) for l in range(n_layers)]
        self.win = [ring_window(st["ring"][l]) for l in range(n_layers)]
        self.offsets = st["offsets"].copy()
        self.active = active.copy()
        self.pending = [None] * n_layers

    def verify(self, layer, x_bits, g, beta):
        x = f64(x_bits)
        o, Sall = oracle.verify(x, self.w[layer], self.win[layer], g, beta, self.S[layer], self.active,
                                H_k=self.geom.H_k, act=self.geom.act)
        self.pending[layer] = (Sall, x)
        return o

    def commit(self, keep):
        status = 0
        new_off = None
        for l in range(self.n):
            Sall, x = self.pending[l]
            off = self.offsets.copy()
            Sl = np.ascontiguousarray(self.S[l])
            status |= oracle.commit(keep, self.active, Sall, x, Sl, self.win[l], off)
            self.S[l] = Sl
            new_off = off
        self.offsets = new_off
        return status


def unit_channels(geom: synth.Geometry, h: int) -> np.ndarray:
    """Conv channels one value head reads: q and k of its key head, then its v."""
    d, rep = geom.d, geom.H_v // geom.H_k
    hk = h // rep
    return np.concatenate([np.arange(hk * d, hk * d + d),
                           np.arange(geom.H_k * d + hk * d, geom.H_k * d + hk * d + d),
                           np.arange(2 * geom.H_k * d + h * d, 2 * geom.H_k * d + h * d + d)])


class OracleUnit:
    """The oracle on one (layer, row, value head) of a large stack: a B=1,
    H_k=1, H_v=1 problem sliced out of the full inputs (rows and heads are
    independent, so this is the same arithmetic the full problem does)."""

    def __init__(self, geom, st, layer, b, h):
        self.geom, self.layer, self.b, self.h = geom, layer, b, h
        self.ch = unit_channels(geom, h)
        self.S = np.ascontiguousarray(st["state"][layer, b:b + 1, h:h + 1]).copy()
        self.w = f64(st["conv_w"][layer][self.ch])
        win = ring_window(st["ring"][layer][b:b + 1])
        self.win = np.ascontiguousarray(win[:, self.ch])
        self.offset = np.array([st["offsets"][b]], np.int32)

    def verify(self, x_bits_layer, g_layer, beta_layer, active_b):
        x = f64(x_bits_layer[self.b:self.b + 1][:, :, self.ch])
        g = g_layer[self.b:self.b + 1, :, self.h:self.h + 1]
        beta = beta_layer[self.b:self.b + 1, :, self.h:self.h + 1]
        act = np.array([active_b], np.uint8)
        o, Sall = oracle.verify(x, self.w, self.win, g, beta, self.S, act, H_k=1, act=self.geom.act)
        self._pending = (Sall, x, act)
        return o[0, :, 0]

    def commit(self, keep_b):
        Sall, x, act = self._pending
        return oracle.commit(np.array([keep_b], np.int32), act, Sall, x, self.S, self.win, self.offset)
