"""Seeded synthetic inputs for the GDN speculative transaction.

This module is the one piece shared by the CUDA path's tests/bench and by the
CPU oracle's callers.  It draws random numbers and lays them out; it holds none
of the method's arithmetic (no convolution, normalisation, gating or delta rule).

Random numbers come from SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", 2014) used as a counter-based generator:
value i of stream (seed, name) is mix64(key(seed, name) + (i + 1) * golden),
and normals come from the Box-Muller transform.  Everything is numpy, so the
same seed gives the same arrays on x86 and Arm hosts (up to libm's last ulp in
log/cos, which only matters after bf16 rounding in rare ties).

Distributions follow the workloads named for this path (MTP depth-one verify
cohorts of hybrid Qwen models):

* raw pre-conv q|k|v inputs x ~ N(0, 1), rounded to bf16;
* conv weights ~ N(0, 0.5^2) (std 0.5), rounded to bf16;
* log-decay g = -softplus(N(0, 1)) * 0.5  (so g <= 0, alpha = e^g in (0, 1]);
* write strength beta = sigmoid(N(0, 1));
* recurrent state S0 ~ N(0, 0.1^2) (std 0.1), fp32;
* primed conv window ~ N(0, 1) bf16 in ring slots 0..2; the verify slots 3..
  hold bf16 NaN so that any read outside the window poisons the result;
* committed offsets (bookkeeping only) uniform in [3, 1000);
* keep per row uniform in {0..T}.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
BF16_NAN = np.uint16(0x7FC0)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, name: str) -> np.uint64:
    tag = zlib.crc32(name.encode()) & 0xFFFFFFFF
    base = np.array([(seed & 0xFFFFFFFF) << 32 | tag], dtype=np.uint64)
    return _mix64(base)[0]


def uniform(seed: int, name: str, n: int, start: int = 0) -> np.ndarray:
    """Doubles start .. start+n-1 of stream (seed, name), in the open interval (0, 1)."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix64(_key(seed, name) + i * _GOLDEN)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


_BLOCK = 1 << 22  # normals generated per block (bounds temporary memory)


def _normal_block(seed, name, start, n, std):
    u = uniform(seed, name, 2 * n, 2 * start)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    return std * r * np.cos(2.0 * np.pi * u[1::2])


def normal(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """fp64 normals N(0, std^2) of the given shape (Box-Muller, cosine branch).

    Value i uses uniforms 2i and 2i+1 of the stream, so blocks of any size give
    the same array."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for s0 in range(0, n, _BLOCK):
        m = min(_BLOCK, n - s0)
        out[s0:s0 + m] = _normal_block(seed, name, s0, m, std)
    return out.reshape(shape)


def normal_bf16(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """normal() rounded to bf16 bits, generated block by block (for large arrays)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s0 in range(0, n, _BLOCK):
        m = min(_BLOCK, n - s0)
        out[s0:s0 + m] = bf16_bits(_normal_block(seed, name, s0, m, std))
    return out.reshape(shape)


def integers(seed: int, name: str, shape, lo: int, hi: int) -> np.ndarray:
    """int32 uniform in [lo, hi)."""
    n = int(np.prod(shape))
    u = uniform(seed, name, n)
    return (lo + np.floor(u * (hi - lo))).astype(np.int32).reshape(shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32/fp64 values to bf16 (round to nearest even); return uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact fp32 values of bf16 bit patterns."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Geometry:
    """Shape of one GDN layer's speculative transaction.

    B rows, T positions per verify, ring capacity for up to T_max positions,
    H_k key heads, H_v value heads, head size d (= d_k = d_v), conv width 4.
    """

    B: int
    T: int
    H_k: int
    H_v: int
    d: int
    T_max: int | None = None
    width: int = 4
    act: int = 1  # 1 = SiLU after the conv, 0 = none

    @property
    def tmax(self) -> int:
        return self.T if self.T_max is None else self.T_max

    @property
    def C(self) -> int:
        return 2 * self.H_k * self.d + self.H_v * self.d

    @property
    def R(self) -> int:
        return self.width - 1 + self.tmax


# Named workloads.  TINY is small enough for pure-Python checks; COHORT is the
# depth-one MTP verify cohort (8 rows, 2 positions, Qwen-style 16/32 heads of 128).
TINY = Geometry(B=1, T=2, H_k=2, H_v=4, d=32)
COHORT = Geometry(B=8, T=2, H_k=16, H_v=32, d=128)


def softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, z)


def layer_state(geom: Geometry, seed: int, n_layers: int = 1, offsets=None) -> dict:
    """Persistent per-layer tensors: conv weights, state, ring and row offsets.

    Returns numpy arrays:
      conv_w  uint16 bf16 [n_layers][C][4]
      state   float32     [n_layers][B][H_v][d_v][d_k]
      ring    uint16 bf16 [n_layers][B][R][C]  conv cache: slots 0..2 hold the
              committed window (oldest first), slots 3.. are verify scratch
      offsets int32       [B]  committed tokens per row (shared by all layers)
    """
    g = geom
    w = bf16_bits(normal(seed, "conv_w", (n_layers, g.C, g.width), std=0.5))
    s0 = normal(seed, "state", (n_layers, g.B, g.H_v, g.d, g.d), std=0.1).astype(np.float32)
    if offsets is None:
        offsets = integers(seed, "offsets", (g.B,), 3, 1000)
    offsets = np.asarray(offsets, dtype=np.int32)
    ring = np.full((n_layers, g.B, g.R, g.C), BF16_NAN, dtype=np.uint16)
    ring[:, :, : g.width - 1, :] = bf16_bits(normal(seed, "window", (n_layers, g.B, g.width - 1, g.C)))
    return {"conv_w": w, "state": s0, "ring": ring, "offsets": offsets}


def cycle_inputs(geom: Geometry, seed: int, cycle: int, n_layers: int = 1) -> dict:
    """Per-cycle verify inputs for every layer plus the cycle's keep[] draw.

      x     uint16 bf16 [n_layers][B][T][C]  raw pre-conv q|k|v
      g     float32     [n_layers][B][T][H_v] log-decay (<= 0)
      beta  float32     [n_layers][B][T][H_v]
      keep  int32       [B] uniform in {0..T}
    """
    g = geom
    tag = f"c{cycle}"
    x = normal_bf16(seed, "x" + tag, (n_layers, g.B, g.T, g.C))
    gl = (-softplus(normal(seed, "g" + tag, (n_layers, g.B, g.T, g.H_v))) * 0.5).astype(np.float32)
    bz = normal(seed, "beta" + tag, (n_layers, g.B, g.T, g.H_v))
    beta = (1.0 / (1.0 + np.exp(-bz))).astype(np.float32)
    keep = integers(seed, "keep" + tag, (g.B,), 0, g.T + 1)
    return {"x": x, "g": gl, "beta": beta, "keep": keep}


def active_mask(B: int, inactive=()) -> np.ndarray:
    a = np.ones(B, dtype=np.uint8)
    for r in inactive:
        a[r] = 0
    return a


def prompt_inputs(geom: Geometry, seed: int, L: int) -> dict:
    """A prompt of L tokens for state priming (B rows, all active).

      x    uint16 bf16 [B][L][C],  g, beta float32 [B][L][H_v]
    """
    g = geom
    x = normal_bf16(seed, "px", (g.B, L, g.C))
    gl = (-softplus(normal(seed, "pg", (g.B, L, g.H_v))) * 0.5).astype(np.float32)
    bz = normal(seed, "pbeta", (g.B, L, g.H_v))
    beta = (1.0 / (1.0 + np.exp(-bz))).astype(np.float32)
    return {"x": x, "g": gl, "beta": beta}


def keep_draws(geom: Geometry, seed: int, n_cycles: int) -> np.ndarray:
    """keep[] for n consecutive cycles, int32 [n_cycles][B], uniform in {0..T}.

    Long runs draw x/g/beta from a pool of cycle_inputs() (pool index = cycle
    mod pool size) but re-draw keep every cycle from this stream.
    """
    return integers(seed, "keeps", (n_cycles, geom.B), 0, geom.T + 1)


# ---------------------------------------------------------------------------
# The same streams drawn with torch on a device, for workloads too large to
# draw on the host in reasonable time (benchmark cohorts of many rows and
# layers).  Integer parts are bit-identical to the numpy generator (int64
# wrap-around arithmetic and logical shifts reproduce the uint64 steps); the
# Box-Muller floats can differ from the host's in the last ulp of log/cos,
# which after rounding to bf16 or fp32 changes a value only in rare ties.
# ---------------------------------------------------------------------------
def _i64(u: int) -> int:
    """A 64-bit pattern as a signed int64 value."""
    return u - (1 << 64) if u >= (1 << 63) else u


_GOLDEN_I = _i64(int(_GOLDEN))
_M1_I = _i64(int(_M1))
_M2_I = _i64(int(_M2))
_DBLOCK = 1 << 24  # values drawn per device block


def _lsr(z, s: int):
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64_t(z):
    z = (z ^ _lsr(z, 30)) * _M1_I
    z = (z ^ _lsr(z, 27)) * _M2_I
    return z ^ _lsr(z, 31)


def uniform_dev(seed: int, name: str, n: int, start: int, device):
    """uniform() as a float64 torch tensor on `device`."""
    import torch
    key = _i64(int(_key(seed, name)))
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = _mix64_t(i * _GOLDEN_I + key)
    return (_lsr(z, 11).to(torch.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal_dev(seed: int, name: str, shape, std: float = 1.0, device="cpu", dtype=None):
    """normal() as a torch tensor on `device` (float64, or `dtype` after rounding)."""
    import torch
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=dtype or torch.float64, device=device)
    for s0 in range(0, n, _DBLOCK):
        m = min(_DBLOCK, n - s0)
        u = uniform_dev(seed, name, 2 * m, 2 * s0, device)
        v = std * torch.sqrt(-2.0 * torch.log(u[0::2])) * torch.cos(2.0 * np.pi * u[1::2])
        out[s0:s0 + m] = v.to(out.dtype)
    return out.reshape(shape)


def integers_dev(seed: int, name: str, shape, lo: int, hi: int, device="cpu"):
    import torch
    n = int(np.prod(shape))
    u = uniform_dev(seed, name, n, 0, device)
    return (lo + torch.floor(u * (hi - lo))).to(torch.int32).reshape(shape)


def layer_state_dev(geom: Geometry, seed: int, n_layers: int, device, offsets=None) -> dict:
    """layer_state() drawn on `device`: torch tensors conv_w / ring as bfloat16,
    state float32, offsets int32."""
    import torch
    g = geom
    w = normal_dev(seed, "conv_w", (n_layers, g.C, g.width), 0.5, device, torch.bfloat16)
    s0 = normal_dev(seed, "state", (n_layers, g.B, g.H_v, g.d, g.d), 0.1, device, torch.float32)
    if offsets is None:
        offsets = integers_dev(seed, "offsets", (g.B,), 3, 1000, device)
    else:
        offsets = torch.as_tensor(np.asarray(offsets, dtype=np.int32)).to(device)
    ring = torch.full((n_layers, g.B, g.R, g.C), float("nan"), dtype=torch.bfloat16, device=device)
    ring[:, :, : g.width - 1, :] = normal_dev(seed, "window", (n_layers, g.B, g.width - 1, g.C), 1.0, device,
                                              torch.bfloat16)
    return {"conv_w": w, "state": s0, "ring": ring, "offsets": offsets}


def cycle_inputs_dev(geom: Geometry, seed: int, cycle: int, n_layers: int, device) -> dict:
    """cycle_inputs() drawn on `device` (x bfloat16, g and beta float32, keep int32)."""
    import torch
    g = geom
    tag = f"c{cycle}"
    x = normal_dev(seed, "x" + tag, (n_layers, g.B, g.T, g.C), 1.0, device, torch.bfloat16)
    gz = normal_dev(seed, "g" + tag, (n_layers, g.B, g.T, g.H_v), 1.0, device)
    gl = (-torch.nn.functional.softplus(gz) * 0.5).to(torch.float32)
    bz = normal_dev(seed, "beta" + tag, (n_layers, g.B, g.T, g.H_v), 1.0, device)
    beta = (1.0 / (1.0 + torch.exp(-bz))).to(torch.float32)
    keep = integers_dev(seed, "keep" + tag, (g.B,), 0, g.T + 1, device)
    return {"x": x, "g": gl, "beta": beta, "keep": keep}
