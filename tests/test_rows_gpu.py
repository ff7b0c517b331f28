"""gdn_move_rows: rows of one cohort copied into another, bit for bit, and a
row primed by gdn_prefill_chunked (B = 1) joined into a B = 4 cohort that
then verifies and commits in parity with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import GpuStack, OracleStack, check_out, check_state, dev_bf16, f64, host_bits, ring_window

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_DEFERRED], ids=["recompute", "deferred"])
def test_move_rows_bit_exact(gdn, mode):
    n_layers = 3
    g_src = synth.Geometry(B=3, T=2, H_k=2, H_v=4, d=64)
    g_dst = synth.Geometry(B=8, T=2, H_k=2, H_v=4, d=64)
    src = GpuStack(g_src, synth.layer_state(g_src, 80, n_layers), synth.active_mask(3), mode, n_layers)
    dst = GpuStack(g_dst, synth.layer_state(g_dst, 81, n_layers), synth.active_mask(8), mode, n_layers)
    if mode == L.GDN_COMMIT_DEFERRED:
        for w in dst.ws:  # pending keeps that the move must clear for its rows
            w.view(torch.int32)[: g_dst.B * g_dst.H_v] = 2
    before = (dst.state.clone(), host_bits(dst.ring).copy(), dst.offsets.clone())
    src_rows = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    dst_rows = torch.tensor([5, 1], dtype=torch.int32, device="cuda")
    L.gdn_move_rows(src.dims, dst.dims, mode, [src.state[l] for l in range(n_layers)],
                    [src.ring[l] for l in range(n_layers)], src.offsets, [dst.state[l] for l in range(n_layers)],
                    [dst.ring[l] for l in range(n_layers)], dst.offsets,
                    dst.ws if mode == L.GDN_COMMIT_DEFERRED else None, src_rows, dst_rows)
    torch.cuda.synchronize()
    s_ring, d_ring = host_bits(src.ring), host_bits(dst.ring)
    for sr, dr in ((2, 5), (0, 1)):
        assert torch.equal(dst.state[:, dr], src.state[:, sr])
        assert np.array_equal(d_ring[:, dr], s_ring[:, sr])
        assert dst.offsets[dr].item() == src.offsets[sr].item()
    for r in (0, 2, 3, 4, 6, 7):
        assert torch.equal(dst.state[:, r], before[0][:, r])
        assert np.array_equal(d_ring[:, r], before[1][:, r])
        assert dst.offsets[r].item() == before[2][r].item()
    if mode == L.GDN_COMMIT_DEFERRED:
        for w in dst.ws:
            pend = w.view(torch.int32)[: g_dst.B * g_dst.H_v].view(g_dst.B, g_dst.H_v).cpu().numpy()
            assert (pend[[5, 1]] == 0).all() and (pend[[0, 2, 3, 4, 6, 7]] == 2).all()
    assert L.gdn_get_status(clear=True) == 0


def test_move_rows_bad_index_skipped(gdn):
    g = synth.Geometry(B=3, T=2, H_k=1, H_v=2, d=32)
    src = GpuStack(g, synth.layer_state(g, 82, 1), synth.active_mask(3), L.GDN_COMMIT_RECOMPUTE, 1)
    dst = GpuStack(g, synth.layer_state(g, 83, 1), synth.active_mask(3), L.GDN_COMMIT_RECOMPUTE, 1)
    before = dst.state.clone()
    L.gdn_get_status(clear=True)
    L.gdn_move_rows(src.dims, dst.dims, L.GDN_COMMIT_RECOMPUTE, [src.state[0]], [src.ring[0]], src.offsets,
                    [dst.state[0]], [dst.ring[0]], dst.offsets, None,
                    torch.tensor([7], dtype=torch.int32, device="cuda"),
                    torch.tensor([1], dtype=torch.int32, device="cuda"))
    assert L.gdn_get_status(clear=True) & L.GDN_STATUS_BAD_ROW
    assert torch.equal(dst.state, before)


def test_primed_row_joins_cohort(gdn):
    """Prime one row over a 150-token prompt on its own (B = 1), move it into
    row 3 of a B = 4 cohort, then run two verify + commit cycles; the oracle
    does the same with its own sequential priming."""
    geom1 = synth.Geometry(B=1, T=2, H_k=2, H_v=4, d=128)
    geom4 = synth.Geometry(B=4, T=2, H_k=2, H_v=4, d=128)
    Lp = 150
    st1 = synth.layer_state(geom1, 84, 1, offsets=np.zeros(1, np.int32))
    st1["state"][:] = 0
    st1["ring"][:] = 0
    pr = synth.prompt_inputs(geom1, 84, Lp)
    prim = GpuStack(geom1, st1, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
    ws = torch.empty(L.gdn_prefill_workspace_bytes(prim.dims, Lp), dtype=torch.uint8, device="cuda")
    out_p = torch.empty((1, Lp, geom1.H_v, geom1.d), dtype=torch.bfloat16, device="cuda")
    st4 = synth.layer_state(geom4, 85, 1)
    st4["conv_w"] = st1["conv_w"]  # one layer's weights shared by both cohorts
    active = synth.active_mask(4)
    cohort = GpuStack(geom4, st4, active, L.GDN_COMMIT_RECOMPUTE, 1)
    L.gdn_prefill_chunked(prim.dims, Lp, dev_bf16(pr["x"]), prim.w[0], torch.from_numpy(pr["g"]).cuda(),
                          torch.from_numpy(pr["beta"]).cuda(), prim.state[0], prim.ring[0], prim.offsets, out_p, ws)
    L.gdn_move_rows(prim.dims, cohort.dims, L.GDN_COMMIT_RECOMPUTE, [prim.state[0]], [prim.ring[0]], prim.offsets,
                    [cohort.state[0]], [cohort.ring[0]], cohort.offsets, None,
                    torch.tensor([0], dtype=torch.int32, device="cuda"),
                    torch.tensor([3], dtype=torch.int32, device="cuda"))
    # the oracle primes its own copy of the row and places it in its cohort
    S1 = st1["state"][0].copy()
    win1 = ring_window(st1["ring"][0]).copy()
    off1 = st1["offsets"].copy()
    oracle.prefill(f64(pr["x"]), f64(st1["conv_w"][0]), win1, pr["g"], pr["beta"], S1, off1, H_k=2)
    orc = OracleStack(geom4, st4, active, 1)
    orc.S[0][3] = S1[0]
    orc.win[0][3] = win1[0]
    orc.offsets[3] = off1[0]
    torch.cuda.synchronize()
    assert cohort.offsets[3].item() == Lp
    for c, keep in enumerate(([2, 1, 0, 2], [1, 2, 2, 1])):
        cy = synth.cycle_inputs(geom4, 86, c, 1)
        cohort.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
        check_out(cohort.out[0], orc.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0]), f"cycle {c} outputs")
        cohort.commit(np.array(keep, np.int32))
        orc.commit(np.array(keep, np.int32))
        torch.cuda.synchronize()
        check_state(cohort.state.cpu().numpy(), orc.S, f"cycle {c} state")
        assert np.array_equal(cohort.offsets.cpu().numpy(), orc.offsets)
