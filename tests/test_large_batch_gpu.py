"""GPU parity at the batch/draft sweep's large cohorts (B = 64 at T = 2 and 8,
B = 32 at T = 5; 32 value heads of 128), in the launch configuration the
benchmark times (layers after the first flagged GDN_VERIFY_OVERLAP, the first
GDN_VERIFY_OVERLAP_STATE in DEFERRED mode).

Three layers over three cycles, the last B/4 rows inactive, keep ~ U{0..T}.
Every cycle: sampled (layer, row, head) units against the oracle (each unit
recomputed on its own, rows and heads being independent), the offsets, and
every row's committed conv window bit for bit against its definition (the
last three raw inputs of window ++ x[:keep']).  After the last cycle (and a
flush in DEFERRED mode) the sampled units' states."""
import functools

import numpy as np
import pytest
import torch

from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import GpuStack, OracleUnit, check_out, check_state, dev_bf16, host_bits
from tests.test_verify_commit_gpu import bench_verify_mode

pytestmark = pytest.mark.gpu
N_LAYERS, N_CYCLES = 3, 3


@functools.lru_cache(maxsize=2)
def _state(B, T, seed):
    return synth.layer_state(synth.Geometry(B=B, T=T, H_k=16, H_v=32, d=128), seed, N_LAYERS)


CASES = [(64, 2, L.GDN_COMMIT_RECOMPUTE), (64, 2, L.GDN_COMMIT_DEFERRED), (64, 8, L.GDN_COMMIT_RECOMPUTE),
         (64, 8, L.GDN_COMMIT_DEFERRED), (32, 5, L.GDN_COMMIT_DEFERRED)]


@pytest.mark.parametrize("B,T,mode", CASES, ids=lambda v: str(v))
def test_large_cohort_sampled_parity(gdn, B, T, mode):
    geom = synth.Geometry(B=B, T=T, H_k=16, H_v=32, d=128)
    seed = 60 + T
    st = _state(B, T, seed)
    inactive = tuple(range(B - B // 4, B))
    active = synth.active_mask(B, inactive)
    gpu = GpuStack(geom, st, active, mode, N_LAYERS)
    last_active = B - B // 4 - 1
    picks = [(0, 0, 0), (1, B // 2 - 1, 31), (2, last_active, 17), (0, B - 1, 0), (2, 1, 31), (1, last_active, 5)]
    if B >= 48:
        picks.append((1, 47, 31))
    units = [OracleUnit(geom, st, l, b, h) for (l, b, h) in picks]
    keeps = synth.keep_draws(geom, seed, N_CYCLES)
    win = [np.ascontiguousarray(st["ring"][l][:, :3, :]).copy() for l in range(N_LAYERS)]  # [B][3][C] bits
    offsets = st["offsets"].copy()
    for c in range(N_CYCLES):
        cy = synth.cycle_inputs(geom, seed, c, N_LAYERS)
        for l in range(N_LAYERS):
            vmode = bench_verify_mode(mode, l)
            L.gdn_conv_verify(gpu.dims, vmode, dev_bf16(cy["x"][l]), gpu.w[l], torch.from_numpy(cy["g"][l]).cuda(),
                              torch.from_numpy(cy["beta"][l]).cuda(), gpu.state[l], gpu.ring[l], gpu.offsets,
                              gpu.active, gpu.out[l], gpu.ws[l])
        torch.cuda.synchronize()
        for u in units:
            o = u.verify(cy["x"][u.layer], cy["g"][u.layer], cy["beta"][u.layer], active[u.b])
            check_out(gpu.out[u.layer, u.b, :, u.h], o, f"cycle {c} unit {(u.layer, u.b, u.h)}")
        assert torch.all(gpu.out[:, B - B // 4:] == 0), "inactive rows give zero outputs"
        keep = keeps[c]
        gpu.commit(keep)
        for u in units:
            u.commit(keep[u.b])
        kp = np.where((active == 1) & (keep >= 0) & (keep <= T), keep, 0)
        offsets = offsets + kp.astype(np.int32)
        torch.cuda.synchronize()
        assert np.array_equal(gpu.offsets.cpu().numpy(), offsets), f"cycle {c} offsets"
        ring = host_bits(gpu.ring)
        for l in range(N_LAYERS):
            seq = np.concatenate([win[l], cy["x"][l]], axis=1)  # [B][3+T][C]: window ++ new raw inputs
            for b in range(B):
                if kp[b] >= 1:
                    win[l][b] = seq[b, kp[b]:kp[b] + 3]
            assert np.array_equal(ring[l][:, :3, :], win[l]), f"cycle {c} layer {l} conv windows"
    if mode == L.GDN_COMMIT_DEFERRED:
        gpu.flush()
    torch.cuda.synchronize()
    for u in units:
        check_state(gpu.state[u.layer, u.b, u.h].cpu().numpy()[None], u.S[0], f"unit {(u.layer, u.b, u.h)} state")
    assert L.gdn_get_status(clear=True) == 0
