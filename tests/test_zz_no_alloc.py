"""gdn_conv_verify_noalloc: the verify entry point for callers that cannot
allocate device memory (a plug-in whose host framework owns every allocation,
or a serving loop that may not call cudaMalloc once it is running).

It must give the same outputs as gdn_conv_verify with a caller-allocated
workspace, bit for bit (the same kernel on the same inputs), on consecutive
calls that reuse its built-in scratch, and its scratch address must serve
gdn_commit like any workspace.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import GpuStack, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def _inputs(cy, layer):
    return (dev_bf16(cy["x"][layer]), torch.from_numpy(cy["g"][layer]).cuda(),
            torch.from_numpy(cy["beta"][layer]).cuda())


NOALLOC_CASES = [  # (geometry, mode, inactive rows): all fit the built-in scratch
    (synth.COHORT, L.GDN_COMMIT_RECOMPUTE, (6, 7)),                                      # the B8/T2 cohort
    (synth.Geometry(B=8, T=8, H_k=16, H_v=32, d=128), L.GDN_COMMIT_RECOMPUTE, (6, 7)),  # deep drafts
    (synth.Geometry(B=2, T=2, H_k=2, H_v=4, d=64), L.GDN_COMMIT_SNAPSHOT, ()),           # snapshots, small
]


@pytest.mark.parametrize("geom,mode,inactive", NOALLOC_CASES, ids=["B8T2-recompute", "B8T8-recompute",
                                                                   "B2T2d64-snapshot"])
def test_noalloc_matches_allocated_workspace_two_calls(gdn, geom, mode, inactive):
    """The same kernel on the same inputs: outputs, rings, committed states and
    offsets equal bit for bit, on two calls in a row that reuse the scratch."""
    assert L.gdn_layer_workspace_bytes(L.dims_of(geom), mode) <= L.GDN_NOALLOC_WS_BYTES
    st = synth.layer_state(geom, 31, 1)
    active = synth.active_mask(geom.B, inactive)
    ref = GpuStack(geom, st, active, mode, 1)   # caller-allocated workspace
    new = GpuStack(geom, st, active, mode, 1)   # built-in scratch
    for call in range(2):
        cy = synth.cycle_inputs(geom, 31, call, 1)
        keep = np.asarray(cy["keep"], np.int32)
        x, g, beta = _inputs(cy, 0)
        L.gdn_conv_verify(ref.dims, ref.mode, x, ref.w[0], g, beta, ref.state[0], ref.ring[0], ref.offsets,
                          ref.active, ref.out[0], ref.ws[0])
        scratch = L.gdn_conv_verify_noalloc(new.dims, new.mode, x, new.w[0], g, beta, new.state[0], new.ring[0],
                                            new.offsets, new.active, new.out[0])
        assert scratch != 0
        torch.cuda.synchronize()
        assert torch.equal(new.out.view(torch.int16), ref.out.view(torch.int16)), f"call {call} outputs"
        assert np.array_equal(host_bits(new.ring), host_bits(ref.ring)), f"call {call} ring"
        L.gdn_commit(ref.dims, ref.mode, [ref.state[0]], [ref.ring[0]], ref.ws, torch.from_numpy(keep).cuda(),
                     ref.active, ref.offsets)
        L.gdn_commit(new.dims, new.mode, [new.state[0]], [new.ring[0]], [scratch], torch.from_numpy(keep).cuda(),
                     new.active, new.offsets)
        torch.cuda.synchronize()
        assert torch.equal(new.state, ref.state), f"call {call} committed state"
        assert torch.equal(new.offsets, ref.offsets)
        assert np.array_equal(host_bits(new.ring), host_bits(ref.ring)), f"call {call} committed window"


def test_noalloc_rejects_shapes_beyond_its_scratch(gdn):
    geom = synth.COHORT  # SNAPSHOT needs T * |S| = 32 MiB of workspace here
    st = synth.layer_state(geom, 32, 1)
    gpu = GpuStack(geom, st, synth.active_mask(8), L.GDN_COMMIT_RECOMPUTE, 1)
    assert L.gdn_layer_workspace_bytes(gpu.dims, L.GDN_COMMIT_SNAPSHOT) > L.GDN_NOALLOC_WS_BYTES
    before = gpu.out.clone()
    cy = synth.cycle_inputs(geom, 32, 0, 1)
    x, g, beta = _inputs(cy, 0)
    with pytest.raises(L.GdnError) as ei:
        L.gdn_conv_verify_noalloc(gpu.dims, L.GDN_COMMIT_SNAPSHOT, x, gpu.w[0], g, beta, gpu.state[0],
                                  gpu.ring[0], gpu.offsets, gpu.active, gpu.out[0])
    assert ei.value.code == L.GDN_ERR_WORKSPACE and "scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.equal(gpu.out.view(torch.int16), before.view(torch.int16)), "nothing may run on rejection"
