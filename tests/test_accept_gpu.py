"""GPU parity of gdn_accept_greedy (on-device greedy acceptance) against the
oracle, and a verify -> accept -> commit cycle in one CUDA graph with keep
never leaving the device ("Add request-owned eight-way MTP serving for Qwen
35B": acceptance taken off the host so the decode cycle needs no host
synchronisation).  keep and next are integers: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import GpuStack, OracleStack, check_out, check_state, dev_bf16, f64

pytestmark = pytest.mark.gpu

BF16_NAN = np.uint16(0x7FC0)


def make_case(seed, B, T, V, p_inactive=0.2):
    """bf16 logits ~ N(0,1); drafts that repeat the targets for a random
    number of leading positions (targets from numpy's argmax, used only to
    build the inputs; the expected keep comes from the oracle)."""
    bits = synth.normal_bf16(seed, "accept_logits", B * T * V).reshape(B, T, V)
    tgt = np.argmax(f64(bits), axis=2)
    rng = np.random.default_rng(seed)
    draft = rng.integers(0, V, size=(B, T)).astype(np.int32)
    for b in range(B):
        n = int(rng.integers(0, T))
        draft[b, 1:1 + n] = tgt[b, :n]
    active = (rng.random(B) >= p_inactive).astype(np.uint8)
    return bits, draft, active


def run_gpu(bits, draft, active, ws=None):
    B, T, V = bits.shape
    if ws is None:
        ws = torch.zeros(L.gdn_accept_workspace_bytes(B, T, V), dtype=torch.uint8, device="cuda")
    keep = torch.full((B,), -99, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -99, dtype=torch.int32, device="cuda")
    L.gdn_accept_greedy(dev_bf16(bits), torch.from_numpy(draft).cuda(), torch.from_numpy(active).cuda(), keep, nxt, ws)
    torch.cuda.synchronize()
    return keep.cpu().numpy(), nxt.cpu().numpy(), ws


@pytest.mark.parametrize("shape", [(8, 2, 151936), (3, 5, 1003), (64, 8, 32000), (2, 1, 7), (5, 4, 8192 * 3 + 8)],
                         ids=lambda s: "B{}T{}V{}".format(*s))
def test_accept_matches_oracle(gdn, shape):
    B, T, V = shape
    bits, draft, active = make_case(sum(shape), B, T, V)
    keep, nxt, _ = run_gpu(bits, draft, active)
    k_ref, n_ref = oracle.accept(f64(bits), draft, active)
    assert np.array_equal(keep, k_ref), (keep, k_ref)
    assert np.array_equal(nxt, n_ref), (nxt, n_ref)
    if active.any():
        assert keep[active == 1].max() > 1 or T == 1, "the planted prefixes produced no accepted draft"


def test_accept_ties_nan_and_repeat(gdn):
    """Equal maxima in different vocabulary slices (the first index wins), NaN
    entries and an all-NaN position, and a second call on the same workspace."""
    B, T, V = 4, 3, 20000
    bits, draft, active = make_case(3, B, T, V, p_inactive=0.0)
    big = np.uint16(0x4120)  # 10.0
    bits[0, 0, 15000] = big
    bits[0, 0, 900] = big        # tie across slices: 900 must win
    bits[1, 1, 5] = BF16_NAN
    bits[1, 1, 17] = BF16_NAN
    bits[2, 0, :] = BF16_NAN     # all NaN: target 0
    draft[0, 1] = 900
    draft[2, 1] = 0
    keep, nxt, ws = run_gpu(bits, draft, active)
    k_ref, n_ref = oracle.accept(f64(bits), draft, active)
    assert np.array_equal(keep, k_ref) and np.array_equal(nxt, n_ref), (keep, k_ref, nxt, n_ref)
    assert keep[0] >= 2 and keep[2] >= 2, "the planted ties/NaN rows accept their first draft"
    keep2, nxt2, _ = run_gpu(bits, draft, active, ws)  # the workspace is ready again
    assert np.array_equal(keep2, k_ref) and np.array_equal(nxt2, n_ref)


def test_accept_rejects_bad_arguments(gdn):
    logits = torch.zeros((2, 3, 16), dtype=torch.bfloat16, device="cuda")
    draft = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    active = torch.ones(2, dtype=torch.uint8, device="cuda")
    keep = torch.zeros(2, dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(L.GdnError) as ei:
        L.gdn_accept_greedy(logits, draft, active, keep, keep.clone(), small)
    assert ei.value.code == L.GDN_ERR_WORKSPACE


def test_verify_accept_commit_one_graph(gdn):
    """One cycle per CUDA graph: verify (two layers), accept on the device,
    commit with the device keep; three cycles against the oracle doing the
    same with its own acceptance."""
    geom = synth.Geometry(B=4, T=3, H_k=2, H_v=4, d=128)
    n_layers, V = 2, 4096
    st = synth.layer_state(geom, 40, n_layers)
    active = synth.active_mask(4, (2,))
    for mode in (L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_DEFERRED):
        gpu = GpuStack(geom, st, active, mode, n_layers)
        orc = OracleStack(geom, st, active, n_layers)
        ws_a = torch.zeros(L.gdn_accept_workspace_bytes(geom.B, geom.T, V), dtype=torch.uint8, device="cuda")
        keep = torch.zeros(geom.B, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(geom.B, dtype=torch.int32, device="cuda")
        for c in range(3):
            cy = synth.cycle_inputs(geom, 40, c, n_layers)
            bits, draft, _ = make_case(100 + c, geom.B, geom.T, V)
            dl, dd = dev_bf16(bits), torch.from_numpy(draft).cuda()
            x = [dev_bf16(cy["x"][l]) for l in range(n_layers)]
            g = [torch.from_numpy(cy["g"][l]).cuda() for l in range(n_layers)]
            be = [torch.from_numpy(cy["beta"][l]).cuda() for l in range(n_layers)]
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for l in range(n_layers):
                    L.gdn_conv_verify(gpu.dims, mode, x[l], gpu.w[l], g[l], be[l], gpu.state[l], gpu.ring[l],
                                      gpu.offsets, gpu.active, gpu.out[l], gpu.ws[l])
                L.gdn_accept_greedy(dl, dd, gpu.active, keep, nxt, ws_a)
                L.gdn_commit(gpu.dims, mode, [gpu.state[l] for l in range(n_layers)],
                             [gpu.ring[l] for l in range(n_layers)], gpu.ws, keep, gpu.active, gpu.offsets)
            graph.replay()
            torch.cuda.synchronize()
            for l in range(n_layers):
                o_ref = orc.verify(l, cy["x"][l], cy["g"][l], cy["beta"][l])
                check_out(gpu.out[l], o_ref, f"cycle {c} layer {l}")
            k_ref, n_ref = oracle.accept(f64(bits), draft, active)
            assert np.array_equal(keep.cpu().numpy(), k_ref) and np.array_equal(nxt.cpu().numpy(), n_ref)
            orc.commit(k_ref)
        if mode == L.GDN_COMMIT_DEFERRED:
            gpu.flush()
        torch.cuda.synchronize()
        check_state(gpu.state.cpu().numpy(), orc.S, "state after three graph cycles")
        assert np.array_equal(gpu.offsets.cpu().numpy(), orc.offsets)
