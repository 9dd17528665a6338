"""Device-side failure reporting.  Every wait inside the kernels is bounded; a
wait that gives up sets the workspace's device error flag, which
qmoe_check_device_error reads and clears.  These tests make no wait give up
(no GPU fault, trap or hang is ever provoked): they check that normal calls
leave the flag clear, and that a flag set by hand in the workspace (standing in
for a kernel whose wait gave up) is reported once and then cleared."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import to_dev

pytestmark = pytest.mark.gpu


def test_kernels_run_the_sm103a_image(qgpu):
    assert qgpu.binary_version() == 103


def _forward(qgpu, wl, d, ws):
    return qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"],
                            wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit, workspace=ws)


@pytest.mark.parametrize("wl", [syn.WORKLOADS["nvfp4_mtp_decode"],
                                syn.small("pf_err", T=40, E=16, k=4, H=256, I=128)], ids=lambda w: w.name)
def test_flag_stays_clear_after_normal_calls(qgpu, wl):
    d = to_dev(syn.layer(wl, seed=0))
    ws = torch.zeros(qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt), dtype=torch.uint8,
                     device="cuda")
    for _ in range(3):
        _forward(qgpu, wl, d, ws)
    qgpu.check_device_error(ws)
    assert int(ws[4:8].view(torch.int32).item()) == 0


def test_flag_set_is_reported_once_then_cleared(qgpu):
    wl = syn.WORKLOADS["nvfp4_mtp_decode"]
    ws = torch.zeros(qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt), dtype=torch.uint8,
                     device="cuda")
    ws[4:8].view(torch.int32).fill_(1)   # what a kernel does when a bounded wait gives up
    with pytest.raises(qgpu.QMoEError) as ei:
        qgpu.check_device_error(ws)
    assert ei.value.status == 6 and "bounded wait" in str(ei.value)
    qgpu.check_device_error(ws)          # cleared by the first check
    assert int(ws[4:8].view(torch.int32).item()) == 0


def test_primed_decode_keeps_a_set_flag(qgpu):
    """With a primed workspace the decode kernel never resets the flag: a flag
    left by an earlier call survives later calls until it is checked."""
    wl = syn.WORKLOADS["nvfp4_mtp_decode"]
    d = to_dev(syn.layer(wl, seed=1))
    fmt = wl.fmt | qgpu.WORKSPACE_PRIMED
    ws = torch.zeros(qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, fmt), dtype=torch.uint8,
                     device="cuda")
    ws[4:8].view(torch.int32).fill_(1)
    qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"], fmt, wl.k,
                     wl.normalize, workspace=ws)
    with pytest.raises(qgpu.QMoEError):
        qgpu.check_device_error(ws)
    # the counters behind the flag are back at zero
    assert np.all(ws[8:64].cpu().numpy() == 0)
