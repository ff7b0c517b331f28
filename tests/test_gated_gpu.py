"""GPU parity of gdn_conv_verify_gated (verify with the gated RMSNorm of the
output fused in) against the oracle's verify followed by its gated RMSNorm,
over two cycles so the captures the fused kernel leaves for the commit are
checked through the committed state as well."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gated_gdn_gb300 import lib as L
from speculative_decode_gated_gdn_gb300 import synth
from tests.gdn_harness import GpuStack, OracleStack, check_out, check_state, dev_bf16, f64

pytestmark = pytest.mark.gpu

CASES = [  # (B, T, H_k, H_v, d, inactive rows)
    (1, 2, 2, 4, 32, ()), (8, 2, 16, 32, 128, (6, 7)), (3, 5, 2, 4, 64, (1,)), (2, 8, 1, 2, 128, ()),
]


@pytest.mark.parametrize("mode", [L.GDN_COMMIT_RECOMPUTE, L.GDN_COMMIT_DEFERRED], ids=["recompute", "deferred"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}Hk{}Hv{}d{}".format(*c[:5]))
def test_gated_verify_matches_oracle(gdn, case, mode):
    B, T, H_k, H_v, d, inactive = case
    geom = synth.Geometry(B=B, T=T, H_k=H_k, H_v=H_v, d=d)
    seed = 70 + B + T + d
    st = synth.layer_state(geom, seed, 1)
    active = synth.active_mask(B, inactive)
    gpu = GpuStack(geom, st, active, mode, 1)
    orc = OracleStack(geom, st, active, 1)
    eps = 1e-6
    w_bits = synth.normal_bf16(seed, "norm_w", d, std=0.5)
    w_dev = dev_bf16(w_bits)
    for c in range(2):
        cy = synth.cycle_inputs(geom, seed, c, 1)
        z_bits = synth.normal_bf16(seed + c, "gate_z", B * T * H_v * d).reshape(B, T, H_v, d)
        L.gdn_conv_verify_gated(gpu.dims, mode, dev_bf16(cy["x"][0]), gpu.w[0], torch.from_numpy(cy["g"][0]).cuda(),
                                torch.from_numpy(cy["beta"][0]).cuda(), gpu.state[0], gpu.ring[0], gpu.offsets,
                                gpu.active, dev_bf16(z_bits), w_dev, eps, gpu.out[0], gpu.ws[0])
        o_ref = orc.verify(0, cy["x"][0], cy["g"][0], cy["beta"][0])
        y_ref = oracle.gated_rmsnorm(o_ref, f64(z_bits), f64(w_bits), eps)
        torch.cuda.synchronize()
        check_out(gpu.out[0], y_ref, f"cycle {c} gated outputs")
        if inactive:
            assert torch.all(gpu.out[0][torch.tensor(list(inactive)).cuda()] == 0)
        keep = np.array([(b + c) % (T + 1) for b in range(B)], np.int32)
        gpu.commit(keep)
        orc.commit(keep)
    if mode == L.GDN_COMMIT_DEFERRED:
        gpu.flush()
    torch.cuda.synchronize()
    check_state(gpu.state.cpu().numpy(), orc.S, "state after two gated cycles")
    assert np.array_equal(gpu.offsets.cpu().numpy(), orc.offsets)


def test_gated_verify_rejects_missing_gate(gdn):
    geom = synth.TINY
    st = synth.layer_state(geom, 0, 1)
    gpu = GpuStack(geom, st, synth.active_mask(1), L.GDN_COMMIT_RECOMPUTE, 1)
    cy = synth.cycle_inputs(geom, 0, 0, 1)
    w_dev = torch.ones(geom.d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.GdnError) as ei:
        L.gdn_conv_verify_gated(gpu.dims, L.GDN_COMMIT_RECOMPUTE, dev_bf16(cy["x"][0]), gpu.w[0],
                                torch.from_numpy(cy["g"][0]).cuda(), torch.from_numpy(cy["beta"][0]).cuda(),
                                gpu.state[0], gpu.ring[0], gpu.offsets, gpu.active, None, w_dev, 1e-6,
                                gpu.out[0], gpu.ws[0])
    assert ei.value.code == L.GDN_ERR_INVALID_ARG
