"""GPU parity of gdn_prefill_chunked (chunked WY/UT form) against the
sequential CPU oracle, and of the verify/commit cycle that follows priming.

"MTP inference: review and commit structure", Verification and limits: the
chunked recurrence differs from the sequential one only in rounding, so the
chunked GPU result is held to the same tolerances as verify.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import (GpuStack, OracleStack, check_out, check_state, dev_bf16, f64, host_bits,
                               ring_window, unit_channels)

pytestmark = pytest.mark.gpu


def gpu_prefill(stack: GpuStack, layer: int, pr: dict, Lp: int):
    d = stack.dims
    nbytes = L.gdn_prefill_workspace_bytes(d, Lp)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    g = stack.geom
    out = torch.empty((g.B, Lp, g.H_v, g.d), dtype=torch.bfloat16, device="cuda")
    L.gdn_prefill_chunked(d, Lp, dev_bf16(pr["x"]), stack.w[layer], torch.from_numpy(pr["g"]).cuda(),
                          torch.from_numpy(pr["beta"]).cuda(), stack.state[layer], stack.ring[layer],
                          stack.offsets, out, ws)
    return out


def fresh_state(geom, seed):
    """A row that has seen no tokens: zero state, zero conv window, offset 0."""
    st = synth.layer_state(geom, seed, 1, offsets=np.zeros(geom.B, np.int32))
    st["state"][:] = 0
    st["ring"][:] = 0
    return st


SHAPES = [  # (B, L, H_k, H_v, d)
    (2, 1, 1, 2, 32), (2, 2, 2, 4, 64), (1, 5, 2, 4, 128), (2, 64, 2, 4, 64), (2, 150, 2, 4, 128),
    (1, 200, 1, 1, 32), (3, 129, 2, 6, 64),
    # d = 128 prompts of 24+ chunks run as chunk ranges whose state pass
    # overlaps the next range's products: two ranges, and three with an odd tail
    (1, 1536, 1, 2, 128), (2, 1600, 2, 4, 128),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}L{}Hk{}Hv{}d{}".format(*s))
def test_prefill_matches_sequential_oracle(gdn, shape):
    B, Lp, H_k, H_v, d = shape
    geom = synth.Geometry(B=B, T=2, H_k=H_k, H_v=H_v, d=d)
    st = synth.layer_state(geom, 40 + Lp, 1)
    pr = synth.prompt_inputs(geom, 40 + Lp, Lp)
    gpu = GpuStack(geom, st, synth.active_mask(B), L.GDN_COMMIT_RECOMPUTE, 1)
    out = gpu_prefill(gpu, 0, pr, Lp)
    S = st["state"][0].copy()
    win = ring_window(st["ring"][0])
    off = st["offsets"].copy()
    o_ref = oracle.prefill(f64(pr["x"]), f64(st["conv_w"][0]), win, pr["g"], pr["beta"], S, off, H_k=H_k)
    torch.cuda.synchronize()
    check_out(out, o_ref, "prefill outputs")
    check_state(gpu.state[0].cpu().numpy(), S, "prefill final state")
    assert np.array_equal(gpu.offsets.cpu().numpy(), off)
    assert np.array_equal(ring_window(host_bits(gpu.ring[0])), win), "primed conv window"


def test_prefill_then_verify_commit(gdn):
    """Priming leaves state, ring and offsets ready for the next verify cycle."""
    geom = synth.Geometry(B=2, T=2, H_k=2, H_v=4, d=128)
    st = fresh_state(geom, 50)
    Lp = 100
    pr = synth.prompt_inputs(geom, 50, Lp)
    active = synth.active_mask(2)
    gpu = GpuStack(geom, st, active, L.GDN_COMMIT_RECOMPUTE, 1)
    gpu_prefill(gpu, 0, pr, Lp)
    orc = OracleStack(geom, st, active, 1)
    orc.prefill_o = oracle.prefill(f64(pr["x"]), orc.w[0], orc.win[0], pr["g"], pr["beta"], orc.S[0],
                                   orc.offsets, H_k=2)
    for c, keep in enumerate(([2, 1], [0, 2], [1, 1])):
        cy = synth.cycle_inputs(geom, 50, c, 1)
        gpu.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
        check_out(gpu.out[0], orc.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0]), f"cycle {c} outputs")
        gpu.commit(np.array(keep, np.int32))
        orc.commit(np.array(keep, np.int32))
        torch.cuda.synchronize()
        check_state(gpu.state.cpu().numpy(), orc.S, f"cycle {c} state")
        assert np.array_equal(gpu.offsets.cpu().numpy(), orc.offsets)


def _unit_prefill(st, pr, geom, b, h):
    """Oracle priming of one (row, value head), sliced out of the full inputs."""
    ch = unit_channels(geom, h)
    S = np.ascontiguousarray(st["state"][0, b:b + 1, h:h + 1]).copy()
    win = ring_window(st["ring"][0][b:b + 1])[:, ch].copy()
    off = st["offsets"][b:b + 1].copy()
    o = oracle.prefill(f64(pr["x"][b:b + 1][:, :, ch]), f64(st["conv_w"][0][ch]), win,
                       pr["g"][b:b + 1, :, h:h + 1], pr["beta"][b:b + 1, :, h:h + 1], S, off, H_k=1)
    return o[0, :, 0], S[0, 0]


@pytest.mark.parametrize("Lp,heads", [(4096, None), (32768, (0, 17))], ids=["L4096_all_heads", "L32768_sampled"])
def test_prime_long_prompt(gdn, Lp, heads):
    """A fresh B=1 row primed over a long prompt (chunk 64), then one T=2 verify
    and commit on the primed state."""
    geom = synth.Geometry(B=1, T=2, H_k=16, H_v=32, d=128)
    st = fresh_state(geom, 60)
    pr = synth.prompt_inputs(geom, 60, Lp)
    active = synth.active_mask(1)
    gpu = GpuStack(geom, st, active, L.GDN_COMMIT_RECOMPUTE, 1)
    out = gpu_prefill(gpu, 0, pr, Lp)
    torch.cuda.synchronize()
    heads = range(geom.H_v) if heads is None else heads
    S_after = {}
    for h in heads:
        o_ref, S_ref = _unit_prefill(st, pr, geom, 0, h)
        check_out(out[0, :, h], o_ref, f"head {h} prompt outputs")
        check_state(gpu.state[0, 0, h].cpu().numpy()[None], S_ref[None], f"head {h} primed state")
        S_after[h] = S_ref
    assert gpu.offsets[0].item() == Lp
    win = ring_window(host_bits(gpu.ring[0]))[0]
    assert np.array_equal(win, f64(pr["x"][0, Lp - 3:Lp]).T), "primed window = last three prompt inputs"
    # one verify + commit on the primed state, against the oracle continuing
    # from its own primed state
    st2 = {"state": gpu.state.cpu().numpy().copy(), "ring": host_bits(gpu.ring).copy(),
           "conv_w": st["conv_w"], "offsets": gpu.offsets.cpu().numpy().copy()}
    for h in heads:
        st2["state"][0, 0, h] = S_after[h].astype(np.float32)  # oracle continues from its own state
    orc = OracleStack(geom, st2, active, 1)
    cy = synth.cycle_inputs(geom, 60, 0, 1)
    gpu.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    o_ref = orc.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    keep = np.array([2], np.int32)
    gpu.commit(keep)
    orc.commit(keep)
    torch.cuda.synchronize()
    hs = list(heads)
    check_out(gpu.out[0][:, :, hs], o_ref[:, :, hs], "verify after priming")
    check_state(gpu.state[0, :, hs].cpu().numpy(), orc.S[0][:, hs], "commit after priming")
    assert gpu.offsets[0].item() == Lp + 2


def test_prefill_rejects_bad_arguments(gdn):
    geom = synth.Geometry(B=1, T=2, H_k=2, H_v=4, d=64)
    st = fresh_state(geom, 70)
    gpu = GpuStack(geom, st, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
    pr = synth.prompt_inputs(geom, 70, 10)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    out = torch.empty((1, 10, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.GdnError) as ei:
        L.gdn_prefill_chunked(gpu.dims, 10, dev_bf16(pr["x"]), gpu.w[0], torch.from_numpy(pr["g"]).cuda(),
                              torch.from_numpy(pr["beta"]).cuda(), gpu.state[0], gpu.ring[0], gpu.offsets,
                              out, small)
    assert ei.value.code == L.GDN_ERR_WORKSPACE
    assert gpu.offsets[0].item() == 0


def test_ranged_prefill_in_a_cuda_graph_is_bit_identical(gdn):
    """A d = 128 prompt long enough for the ranged schedule (its state pass on
    the library's internal stream) captured into a CUDA graph and replayed
    gives the same bits as the direct call: the internal stream joins the
    capture and is joined back."""
    geom = synth.Geometry(B=1, T=2, H_k=2, H_v=4, d=128)
    Lp = 1600
    st = synth.layer_state(geom, 81, 1)
    pr = synth.prompt_inputs(geom, 81, Lp)
    direct = GpuStack(geom, st, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
    out_direct = gpu_prefill(direct, 0, pr, Lp)
    torch.cuda.synchronize()

    cap = GpuStack(geom, st, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
    d = cap.dims
    ws = torch.empty(L.gdn_prefill_workspace_bytes(d, Lp), dtype=torch.uint8, device="cuda")
    out = torch.empty((geom.B, Lp, geom.H_v, geom.d), dtype=torch.bfloat16, device="cuda")
    x, g, beta = dev_bf16(pr["x"]), torch.from_numpy(pr["g"]).cuda(), torch.from_numpy(pr["beta"]).cuda()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        L.gdn_prefill_chunked(d, Lp, x, cap.w[0], g, beta, cap.state[0], cap.ring[0], cap.offsets, out, ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_direct.view(torch.int16)), "prompt outputs"
    assert torch.equal(cap.state, direct.state), "primed state"
    assert np.array_equal(host_bits(cap.ring), host_bits(direct.ring)), "primed window"
    assert torch.equal(cap.offsets, direct.offsets)
