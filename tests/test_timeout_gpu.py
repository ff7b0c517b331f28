"""The bounded-wait failure path of the d = 128 verify, forced without any
GPU fault: gdn_test_verify_timeout makes one CTA's state-tile barrier expect
more bytes than its copy delivers, so that CTA's bounded waits run out.  The
kernel must return, flag GDN_STATUS_TIMEOUT, leave that (row, head)'s output
and the state untouched, and the next ordinary call must match the oracle."""
import numpy as np
import pytest
import torch

from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import GpuStack, OracleStack, check_out, check_state, dev_bf16

pytestmark = pytest.mark.gpu
SENTINEL = 0x7BCD  # a bf16 pattern no verify writes here (a large finite value)


@pytest.mark.parametrize("mode", [L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_DEFERRED], ids=["recompute", "deferred"])
def test_bounded_wait_runs_out_and_recovers(gdn, mode):
    geom = synth.Geometry(B=3, T=2, H_k=2, H_v=4, d=128)
    st = synth.layer_state(geom, 50, 1)
    active = synth.active_mask(3)
    gpu = GpuStack(geom, st, active, mode, 1)
    orc = OracleStack(geom, st, active, 1)
    cy = synth.cycle_inputs(geom, 50, 0, 1)
    L.gdn_get_status(clear=True)
    before = gpu.state.clone()
    gpu.out.view(torch.int16).fill_(SENTINEL)
    x, g, beta = dev_bf16(cy["x"][0]), torch.from_numpy(cy["g"][0]).cuda(), torch.from_numpy(cy["beta"][0]).cuda()
    L.gdn_test_verify_timeout(gpu.dims, mode, x, gpu.w[0], g, beta, gpu.state[0], gpu.ring[0], gpu.offsets,
                              gpu.active, gpu.out[0], gpu.ws[0], wait_limit=4000)
    torch.cuda.synchronize()
    assert L.gdn_get_status(clear=True) & L.GDN_STATUS_TIMEOUT, "the bounded wait must run out and be flagged"
    assert torch.equal(gpu.state, before), "a timed-out verify writes no state"
    o00 = gpu.out[0, 0, :, 0].contiguous().view(torch.int16)
    assert torch.all(o00 == SENTINEL), "the timed-out (row 0, head 0) writes no output"
    # every other (row, head) completed: compare with the oracle
    o_ref = orc.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    for b in range(geom.B):
        for h in range(geom.H_v):
            if (b, h) != (0, 0):
                check_out(gpu.out[0, b, :, h], o_ref[b, :, h], f"row {b} head {h} beside the timed-out CTA")
    # the next ordinary call on the same buffers recomputes everything
    gpu.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
    keep = np.array([2, 1, 0], np.int32)
    gpu.commit(keep)
    orc.commit(keep)
    if mode == L.GDN_COMMIT_DEFERRED:
        gpu.flush()
    torch.cuda.synchronize()
    check_out(gpu.out[0], o_ref, "the verify after the timeout")
    check_state(gpu.state.cpu().numpy(), orc.S, "state after the recovered cycle")
    assert np.array_equal(gpu.offsets.cpu().numpy(), orc.offsets)
    assert L.gdn_get_status(clear=True) == 0
