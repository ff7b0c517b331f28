"""GPU parity of gdn_conv_verify + gdn_commit against the CPU oracle.

All calls go through the C ABI (the ctypes binding); inputs are the seeded
synthetic workloads of ``synth``.  Covers the tiny configuration, the B8/T2
cohort, a sweep of head sizes and T up to 8, multi-cycle runs with mixed keep,
exact restore, inert rows, bad keep, fresh rows, row separability, guard
regions, and the 30-layer stack over 256 cycles on sampled units.
"""
import numpy as np
import pytest
import torch

from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import (GpuStack, OracleStack, OracleUnit, check_out, check_state, dev_bf16,
                               host_bits, ring_window)

pytestmark = pytest.mark.gpu
MODES = [L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_SNAPSHOT, L.GDN_COMMIT_DEFERRED]
MODE_IDS = ["recompute", "snapshot", "deferred"]


def run_cycles(geom, seed, active, mode, n_layers, n_cycles, keeps=None, offsets=None, flush_every=None):
    """Cycles of verify (every layer) + grouped commit against the oracle.

    Outputs, offsets and conv windows are compared every cycle.  The state is
    compared every cycle in the eager modes; in DEFERRED mode (where the state
    buffer lags until the next verify) after a flush every `flush_every`
    cycles and at the end, so that the apply-in-verify path runs in between."""
    st = synth.layer_state(geom, seed, n_layers, offsets=offsets)
    gpu = GpuStack(geom, st, active, mode, n_layers)
    orc = OracleStack(geom, st, active, n_layers)
    deferred = mode == L.GDN_COMMIT_DEFERRED
    for c in range(n_cycles):
        cy = synth.cycle_inputs(geom, seed, c, n_layers)
        keep = cy["keep"] if keeps is None else np.asarray(keeps[c], np.int32)
        for l in range(n_layers):
            gpu.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l])
            o_ref = orc.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l])
            check_out(gpu.out[l], o_ref, f"cycle {c} layer {l} outputs")
            inactive = np.nonzero(active == 0)[0]
            if inactive.size:
                assert torch.all(gpu.out[l][torch.from_numpy(inactive).cuda()] == 0)
        gpu.commit(keep)
        status = orc.commit(keep)
        last = c == n_cycles - 1
        if deferred and (last or (flush_every and c % flush_every == flush_every - 1)):
            gpu.flush()
        torch.cuda.synchronize()
        assert np.array_equal(gpu.offsets.cpu().numpy(), orc.offsets), f"cycle {c} offsets"
        if not deferred or last or (flush_every and c % flush_every == flush_every - 1):
            check_state(gpu.state.cpu().numpy(), orc.S, f"cycle {c} state")
        ring = host_bits(gpu.ring)
        for l in range(n_layers):
            win = ring_window(ring[l])
            assert np.array_equal(win, orc.win[l]), f"cycle {c} layer {l} conv window"
        assert L.gdn_get_status(clear=True) == status
    return gpu, orc


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_tiny_configuration(gdn, mode):
    geom = synth.TINY
    keeps = [[0], [1], [2], [2], [1]]
    run_cycles(geom, 0, synth.active_mask(1), mode, 1, len(keeps), keeps)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_cohort_b8_t2(gdn, mode):
    geom = synth.COHORT
    keeps = [[2, 1, 0, 2, 1, 0, 2, 2], [0, 2, 2, 1, 1, 2, 0, 1], [1, 1, 2, 0, 2, 2, 1, 0]]
    run_cycles(geom, 1, synth.active_mask(8, (6, 7)), mode, 1, 3, keeps)


SWEEP = [  # (B, T, T_max, H_k, H_v, d)
    (3, 1, 1, 2, 4, 32), (2, 3, 4, 1, 3, 32), (4, 4, 4, 2, 2, 64), (3, 5, 8, 2, 6, 64),
    (2, 6, 6, 1, 2, 128), (2, 7, 8, 2, 4, 128), (3, 8, 8, 2, 4, 128), (5, 2, 3, 3, 6, 128),
    (2, 8, 8, 4, 4, 32), (3, 4, 4, 2, 4, 128), (2, 5, 8, 1, 4, 128), (2, 1, 2, 2, 2, 128),
]


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", SWEEP, ids=lambda s: "B{}T{}Tm{}Hk{}Hv{}d{}".format(*s))
def test_shape_sweep(gdn, shape, mode):
    B, T, T_max, H_k, H_v, d = shape
    geom = synth.Geometry(B=B, T=T, H_k=H_k, H_v=H_v, d=d, T_max=T_max)
    active = synth.active_mask(B, (B - 1,) if B > 2 else ())
    keeps = [[(b + c) % (T + 1) for b in range(B)] for c in range(4)]
    run_cycles(geom, 10 + T, active, mode, 2, 4, keeps, flush_every=2)


@pytest.mark.parametrize("mode", [L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_DEFERRED], ids=["recompute", "deferred"])
def test_deep_draft_cohort_b8_t8(gdn, mode):
    """The deep-draft cohort at full head count (B = 8, T = 8, H_v = 32,
    d = 128: the tensor-core dot products), two layers over three cycles
    with rows 6 and 7 inactive, keeps from 0 to 8."""
    geom = synth.Geometry(B=8, T=8, H_k=16, H_v=32, d=128)
    keeps = [[8, 0, 3, 5, 1, 8, 2, 7], [2, 8, 0, 6, 4, 1, 8, 8], [5, 5, 8, 0, 7, 3, 0, 1]]
    run_cycles(geom, 41, synth.active_mask(8, (6, 7)), mode, 2, 3, keeps)


def test_no_activation(gdn):
    geom = synth.Geometry(B=2, T=2, H_k=2, H_v=4, d=64, act=0)
    run_cycles(geom, 5, synth.active_mask(2), L.GDN_COMMIT_RECOMPUTE, 1, 2, [[1, 2], [2, 0]])


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_keep_zero_restores_bit_exact(gdn, mode):
    geom = synth.Geometry(B=4, T=3, H_k=2, H_v=4, d=128)
    st = synth.layer_state(geom, 7, 2)
    gpu = GpuStack(geom, st, synth.active_mask(4, (1,)), mode, 2)
    before_state = gpu.state.clone()
    before_ring = host_bits(gpu.ring)
    cy = synth.cycle_inputs(geom, 7, 0, 2)
    for l in range(2):
        gpu.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l])
    torch.cuda.synchronize()
    assert torch.equal(gpu.state, before_state), "verify must not write the state"
    gpu.commit(np.zeros(4, np.int32))
    torch.cuda.synchronize()
    assert torch.equal(gpu.state, before_state), "keep=0 must leave state bytes untouched"
    if mode == L.GDN_COMMIT_DEFERRED:
        gpu.flush()
        torch.cuda.synchronize()
        assert torch.equal(gpu.state, before_state), "a keep=0 commit leaves nothing pending"
    assert np.array_equal(gpu.offsets.cpu().numpy(), st["offsets"])
    ring = host_bits(gpu.ring)
    for l in range(2):
        assert np.array_equal(ring_window(ring[l]), ring_window(before_ring[l]))
    # the inactive row's ring bytes are untouched entirely, not just its window
    assert np.array_equal(ring[:, 1], before_ring[:, 1])


def test_inactive_rows_inert_under_full_accept(gdn):
    geom = synth.Geometry(B=4, T=2, H_k=2, H_v=4, d=64)
    st = synth.layer_state(geom, 8, 1)
    gpu = GpuStack(geom, st, synth.active_mask(4, (0, 3)), L.GDN_COMMIT_RECOMPUTE, 1)
    before_state = gpu.state.clone()
    before_ring = host_bits(gpu.ring)
    cy = synth.cycle_inputs(geom, 8, 0, 1)
    gpu.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    gpu.commit(np.full(4, 2, np.int32))
    torch.cuda.synchronize()
    for b in (0, 3):
        assert torch.equal(gpu.state[:, b], before_state[:, b])
        assert np.array_equal(host_bits(gpu.ring)[:, b], before_ring[:, b])
        assert gpu.offsets[b].item() == st["offsets"][b]
        assert torch.all(gpu.out[0, b] == 0)
    for b in (1, 2):
        assert gpu.offsets[b].item() == st["offsets"][b] + 2


@pytest.mark.parametrize("bad", [-1, 3, 1 << 30])
def test_bad_keep_sets_status_and_restores(gdn, bad):
    geom = synth.Geometry(B=3, T=2, H_k=1, H_v=2, d=32)
    st = synth.layer_state(geom, 9, 1)
    gpu = GpuStack(geom, st, synth.active_mask(3), L.GDN_COMMIT_RECOMPUTE, 1)
    L.gdn_get_status(clear=True)
    before = gpu.state.clone()
    cy = synth.cycle_inputs(geom, 9, 0, 1)
    gpu.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    gpu.commit(np.array([bad, 0, 1], np.int32))
    assert L.gdn_get_status(clear=True) & L.GDN_STATUS_BAD_KEEP
    assert L.gdn_get_status() == 0, "clear must reset the sticky word"
    assert torch.equal(gpu.state[0, 0], before[0, 0]), "a bad keep commits nothing"
    assert gpu.offsets[0].item() == st["offsets"][0]
    assert gpu.offsets[2].item() == st["offsets"][2] + 1


def test_fresh_rows_small_offsets(gdn):
    """Rows at offsets 0, 1, 2 read a window that reaches before the first token."""
    geom = synth.Geometry(B=3, T=2, H_k=2, H_v=4, d=64)
    offsets = np.array([0, 1, 2], np.int32)
    run_cycles(geom, 11, synth.active_mask(3), L.GDN_COMMIT_RECOMPUTE, 1, 4,
               [[2, 1, 0], [1, 2, 2], [0, 0, 1], [2, 2, 2]], offsets=offsets)


def test_row_separability_bit_exact(gdn):
    """A row of a B8 cohort equals a B1 run of that row, bit for bit."""
    geom = synth.COHORT
    st = synth.layer_state(geom, 12, 1)
    cy = synth.cycle_inputs(geom, 12, 0, 1)
    keep = np.array([2, 1, 0, 2, 1, 2, 0, 1], np.int32)
    big = GpuStack(geom, st, synth.active_mask(8), L.GDN_COMMIT_RECOMPUTE, 1)
    big.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    big.commit(keep)
    g1 = synth.Geometry(B=1, T=2, H_k=16, H_v=32, d=128)
    for b in (0, 3, 6):
        st1 = {"state": st["state"][:, b:b + 1].copy(), "ring": st["ring"][:, b:b + 1].copy(),
               "conv_w": st["conv_w"], "offsets": st["offsets"][b:b + 1].copy()}
        one = GpuStack(g1, st1, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
        one.verify(0, cy["x"][0][b:b + 1], cy["g"][0][b:b + 1], cy["beta"][0][b:b + 1])
        one.commit(keep[b:b + 1])
        torch.cuda.synchronize()
        assert torch.equal(one.out[0, 0].view(torch.int16), big.out[0, b].view(torch.int16))
        assert torch.equal(one.state[0, 0], big.state[0, b])


def test_guard_regions_untouched(gdn):
    """Every buffer sits inside a larger allocation whose margins must not change."""
    geom = synth.Geometry(B=3, T=3, H_k=2, H_v=4, d=64, T_max=4)
    st = synth.layer_state(geom, 13, 1)
    cy = synth.cycle_inputs(geom, 13, 0, 1)
    pad = 4096

    def guarded(t):
        flat = t.reshape(-1).view(torch.uint8)
        big = torch.full((flat.numel() + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
        big[pad:pad + flat.numel()] = flat
        return big, big[pad:pad + flat.numel()].view(t.dtype).view(t.shape)

    g_state, state = guarded(torch.from_numpy(st["state"][0]).cuda())
    g_ring, ring = guarded(dev_bf16(st["ring"][0]))
    g_out, out = guarded(torch.zeros((3, 3, 4, 64), dtype=torch.bfloat16, device="cuda"))
    d = L.dims_of(geom)
    nbytes = L.gdn_layer_workspace_bytes(d, L.GDN_COMMIT_RECOMPUTE)
    g_ws, ws = guarded(torch.zeros(nbytes, dtype=torch.uint8, device="cuda"))
    offs = torch.from_numpy(st["offsets"].copy()).cuda()
    act = torch.ones(3, dtype=torch.uint8, device="cuda")
    L.gdn_conv_verify(d, L.GDN_COMMIT_RECOMPUTE, dev_bf16(cy["x"][0]), dev_bf16(st["conv_w"][0]),
                      torch.from_numpy(cy["g"][0]).cuda(), torch.from_numpy(cy["beta"][0]).cuda(),
                      state, ring, offs, act, out, ws)
    L.gdn_commit(d, L.GDN_COMMIT_RECOMPUTE, [state], [ring], [ws], torch.tensor([3, 1, 2], dtype=torch.int32).cuda(),
                 act, offs)
    torch.cuda.synchronize()
    for big in (g_state, g_ring, g_out, g_ws):
        assert torch.all(big[:pad] == 0xA5) and torch.all(big[-pad:] == 0xA5)


@pytest.mark.parametrize("mode", [L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_DEFERRED], ids=["recompute", "deferred"])
def test_stack_30_layers_256_cycles_sampled(gdn, mode):
    """The B8/T2 cohort over a 30-layer stack for 256 consecutive cycles, keep
    re-drawn every cycle and offsets tracked, checked on sampled (layer, row,
    head) units every cycle (the oracle recomputes each unit on its own), in
    the launch configuration the benchmark times."""
    geom = synth.COHORT
    n_layers, n_cycles, pool = 30, 256, 16
    seed = 2
    active = synth.active_mask(8, (6, 7))
    st = synth.layer_state(geom, seed, n_layers)
    keeps = synth.keep_draws(geom, seed, n_cycles)
    gpu = GpuStack(geom, st, active, mode, n_layers)
    units = [OracleUnit(geom, st, l, b, h) for (l, b, h) in
             [(0, 0, 0), (7, 1, 31), (13, 2, 5), (29, 5, 17), (21, 3, 10), (4, 6, 3), (29, 4, 30), (16, 5, 1)]]
    pool_in = [synth.cycle_inputs(geom, seed, p, n_layers) for p in range(pool)]
    dev_pool = [(dev_bf16(c["x"]), torch.from_numpy(c["g"]).cuda(), torch.from_numpy(c["beta"]).cuda())
                for c in pool_in]
    offsets = st["offsets"].copy()
    for c in range(n_cycles):
        cy = pool_in[c % pool]
        xd, gd, bd = dev_pool[c % pool]
        for l in range(n_layers):
            # the launch configuration the benchmark times: layers after the
            # first stage their state while the previous layer's verify ends;
            # in DEFERRED mode the first stages its state beside the commit
            vmode = bench_verify_mode(gpu.mode, l)
            L.gdn_conv_verify(gpu.dims, vmode, xd[l], gpu.w[l], gd[l], bd[l], gpu.state[l], gpu.ring[l],
                              gpu.offsets, gpu.active, gpu.out[l], gpu.ws[l])
        o_units = [u.verify(cy["x"][u.layer], cy["g"][u.layer], cy["beta"][u.layer], active[u.b]) for u in units]
        out = gpu.out
        for u, o in zip(units, o_units):
            check_out(out[u.layer, u.b, :, u.h], o, f"cycle {c} unit {(u.layer, u.b, u.h)}")
        gpu.commit(keeps[c])
        for u in units:
            u.commit(keeps[c][u.b])
        offsets += np.where(active == 1, keeps[c], 0).astype(np.int32)
        assert np.array_equal(gpu.offsets.cpu().numpy(), offsets), f"cycle {c} offsets"
        if c % 32 == 31 or c == n_cycles - 1:
            if mode == L.GDN_COMMIT_DEFERRED:
                gpu.flush()
            for u in units:
                check_state(gpu.state[u.layer, u.b, u.h].cpu().numpy()[None], u.S[0], f"cycle {c} unit state")
                ring = host_bits(gpu.ring[u.layer, u.b:u.b + 1])
                win = ring_window(ring)[:, u.ch]
                assert np.array_equal(win, u.win), f"cycle {c} unit window"
    assert L.gdn_get_status(clear=True) == 0


def test_overlap_flag_is_bit_identical(gdn):
    """GDN_VERIFY_OVERLAP changes only when the state tile is fetched, never a value."""
    geom = synth.COHORT
    st = synth.layer_state(geom, 14, 3)
    cy = synth.cycle_inputs(geom, 14, 0, 3)
    keep = np.array([2, 1, 0, 2, 1, 2, 0, 1], np.int32)
    runs = []
    for overlap in (False, True):
        gpu = GpuStack(geom, st, synth.active_mask(8, (6, 7)), L.GDN_COMMIT_RECOMPUTE, 3)
        for l in range(3):
            gpu.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l], overlap=overlap and l > 0)
        gpu.commit(keep)
        torch.cuda.synchronize()
        runs.append((gpu.out.clone(), gpu.state.clone(), host_bits(gpu.ring), gpu.offsets.clone()))
    a, b = runs
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1]) and np.array_equal(a[2], b[2]) and torch.equal(a[3], b[3])


def bench_verify_mode(mode, layer):
    """The flags the benchmark puts on layer `layer` of a cycle."""
    if layer > 0:
        return mode | L.GDN_VERIFY_OVERLAP
    return mode | (L.GDN_VERIFY_OVERLAP_STATE if mode == L.GDN_COMMIT_DEFERRED else 0)


@pytest.mark.parametrize("T", [2, 8], ids=["T2", "T8"])
def test_overlap_state_flag_is_bit_identical(gdn, T):
    """DEFERRED cycles with the first layer flagged GDN_VERIFY_OVERLAP_STATE
    (and the others GDN_VERIFY_OVERLAP) give the same bytes as unflagged
    calls: outputs every cycle, then the flushed state, rings and offsets."""
    geom = synth.Geometry(B=4, T=T, H_k=2, H_v=4, d=128)
    st = synth.layer_state(geom, 15, 3)
    active = synth.active_mask(4, (3,))
    runs = []
    for flagged in (False, True):
        gpu = GpuStack(geom, st, active, L.GDN_COMMIT_DEFERRED, 3)
        outs = []
        for c in range(4):
            cy = synth.cycle_inputs(geom, 15, c, 3)
            for l in range(3):
                mode = bench_verify_mode(gpu.mode, l) if flagged else gpu.mode
                L.gdn_conv_verify(gpu.dims, mode, dev_bf16(cy["x"][l]), gpu.w[l],
                                  torch.from_numpy(cy["g"][l]).cuda(), torch.from_numpy(cy["beta"][l]).cuda(),
                                  gpu.state[l], gpu.ring[l], gpu.offsets, gpu.active, gpu.out[l], gpu.ws[l])
            outs.append(gpu.out.clone())
            gpu.commit(cy["keep"])
        gpu.flush()
        torch.cuda.synchronize()
        runs.append((outs, gpu.state.clone(), host_bits(gpu.ring), gpu.offsets.clone()))
    (oa, sa, ra, fa), (ob, sb, rb, fb) = runs
    for c, (a, b) in enumerate(zip(oa, ob)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"cycle {c} outputs"
    assert torch.equal(sa, sb) and np.array_equal(ra, rb) and torch.equal(fa, fb)
    assert L.gdn_get_status(clear=True) == 0


def test_unknown_mode_flag_rejected(gdn):
    geom = synth.TINY
    st = synth.layer_state(geom, 0, 1)
    gpu = GpuStack(geom, st, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
    cy = synth.cycle_inputs(geom, 0, 0, 1)
    with pytest.raises(L.GdnError) as ei:
        L.gdn_conv_verify(gpu.dims, 0x400, dev_bf16(cy["x"][0]), gpu.w[0],
                          torch.from_numpy(cy["g"][0]).cuda(), torch.from_numpy(cy["beta"][0]).cuda(),
                          gpu.state[0], gpu.ring[0], gpu.offsets, gpu.active, gpu.out[0], gpu.ws[0])
    assert ei.value.code == L.GDN_ERR_INVALID_ARG


def _cycle_runs(geom, st, masks, keeps, n_layers, mode, overlap_all=False, repeat_verify=False):
    """Outputs of every cycle, then the (flushed) state, offsets and rings."""
    gpu = GpuStack(geom, st, masks[0], mode, n_layers)
    outs = []
    for c, keep in enumerate(keeps):
        gpu.active.copy_(torch.from_numpy(masks[c]))
        cy = synth.cycle_inputs(geom, 30, c, n_layers)
        for l in range(n_layers):
            # flagged except after the commit (layer 0) and on a repeated
            # verify of a layer (its first pass may have written the state)
            for rep in range(2 if repeat_verify else 1):
                flag = overlap_all and rep == 0 and l > 0
                gpu.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l], overlap=flag)
        outs.append(gpu.out.clone())
        gpu.commit(np.asarray(keep, np.int32))
    if mode == L.GDN_COMMIT_DEFERRED:
        gpu.flush()
    torch.cuda.synchronize()
    return outs, gpu.state.clone(), host_bits(gpu.ring), gpu.offsets.clone()


@pytest.mark.parametrize("T", [3, 8], ids=["T3", "T8"])
@pytest.mark.parametrize("repeat_verify", [False, True], ids=["once", "repeated"])
def test_deferred_bit_identical_to_recompute(gdn, repeat_verify, T):
    """DEFERRED applies a commit inside the next verify with the arithmetic of
    the eager commit: every output, and the flushed state, equals RECOMPUTE bit
    for bit.  Rows switch between active and inactive with commits pending, and
    every layer's verify after the first is flagged GDN_VERIFY_OVERLAP in
    DEFERRED mode, so those apply their pending commit before the PDL wait."""
    geom = synth.Geometry(B=4, T=T, H_k=2, H_v=4, d=128, T_max=max(T, 4))
    st = synth.layer_state(geom, 30, 3)
    masks = [synth.active_mask(4), synth.active_mask(4, (1,)), synth.active_mask(4, (1,)),
             synth.active_mask(4, (1, 2)), synth.active_mask(4, (3,)), synth.active_mask(4)]
    keeps = [[min(k, T) for k in row] for row in
             [[3, 2, 1, 0], [1, 3, 3, 2], [2, 0, 3, 1], [0, 1, 2, 3], [2, 2, 0, 3], [3, 0, 1, 1]]]
    if T == 8:  # deep keeps as well
        keeps[1], keeps[4] = [8, 5, 7, 0], [6, 8, 0, 4]
    ref = _cycle_runs(geom, st, masks, keeps, 3, L.GDN_COMMIT_RECOMPUTE, repeat_verify=repeat_verify)
    dfr = _cycle_runs(geom, st, masks, keeps, 3, L.GDN_COMMIT_DEFERRED, overlap_all=True,
                      repeat_verify=repeat_verify)
    for c, (a, b) in enumerate(zip(ref[0], dfr[0])):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"cycle {c} outputs"
    assert torch.equal(ref[1], dfr[1]), "flushed state"
    assert np.array_equal(ref[2], dfr[2]) and torch.equal(ref[3], dfr[3])
    assert L.gdn_get_status(clear=True) == 0


def test_deferred_flush_idempotent(gdn):
    geom = synth.Geometry(B=3, T=2, H_k=1, H_v=2, d=64)
    st = synth.layer_state(geom, 31, 2)
    gpu = GpuStack(geom, st, synth.active_mask(3), L.GDN_COMMIT_DEFERRED, 2)
    cy = synth.cycle_inputs(geom, 31, 0, 2)
    for l in range(2):
        gpu.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l])
    gpu.commit(np.array([2, 0, 1], np.int32))
    torch.cuda.synchronize()
    assert torch.equal(gpu.state, torch.from_numpy(st["state"]).cuda()), "DEFERRED commit writes no state"
    gpu.flush()
    torch.cuda.synchronize()
    once = gpu.state.clone()
    assert not torch.equal(once[:, 0], torch.from_numpy(st["state"][:, 0]).cuda())
    assert torch.equal(once[:, 1], torch.from_numpy(st["state"][:, 1]).cuda()), "keep=0 row unchanged"
    gpu.flush()
    torch.cuda.synchronize()
    assert torch.equal(gpu.state, once), "a second flush applies nothing"
    # and the next verify must not apply the commit again
    orc_state = once.clone()
    cy1 = synth.cycle_inputs(geom, 31, 1, 2)
    gpu.verify(0, cy1["x"][0], cy1["g"][0], cy1["beta"][0])
    torch.cuda.synchronize()
    assert torch.equal(gpu.state[0], orc_state[0])


def test_deferred_rejected_by_noalloc(gdn):
    geom = synth.TINY
    st = synth.layer_state(geom, 0, 1)
    gpu = GpuStack(geom, st, synth.active_mask(1), L.GDN_COMMIT_DEFERRED, 1)
    cy = synth.cycle_inputs(geom, 0, 0, 1)
    with pytest.raises(L.GdnError) as ei:
        L.gdn_conv_verify_noalloc(gpu.dims, L.GDN_COMMIT_DEFERRED, dev_bf16(cy["x"][0]), gpu.w[0],
                                  torch.from_numpy(cy["g"][0]).cuda(), torch.from_numpy(cy["beta"][0]).cuda(),
                                  gpu.state[0], gpu.ring[0], gpu.offsets, gpu.active, gpu.out[0])
    assert ei.value.code in (L.GDN_ERR_INVALID_ARG, L.GDN_ERR_UNSUPPORTED)
