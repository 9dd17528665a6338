"""Decode calls on a primed workspace (QMOE_WORKSPACE_PRIMED): no per-call
header reset, programmatic dependent launch behind the previous kernel.  The
results must equal those of the default calls bit for bit (the kernel is
deterministic), the header must be zero again after every call, whatever ran
on the workspace in between (prefill calls included), eagerly and replayed
from a CUDA graph."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu

CHAIN = [("nvfp4_mtp_decode", 0), ("tiny_nvfp4_decode", 1), ("nvfp4_mtp_decode", 2),
         ("mxfp4_decode", 3), ("nvfp4_verify_edge", 4), ("nvfp4_mtp_decode", 5)]


def _call(q, d, wl, fmt, ws, out):
    q.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"], fmt, wl.k,
                  wl.normalize, wl.alpha, wl.beta, wl.limit, out=out, workspace=ws)


def _header(ws):
    return ws[: 64].view(torch.int32).cpu().numpy()


def _layers():
    res = []
    for name, seed in CHAIN:
        wl = syn.WORKLOADS[name]
        res.append((wl, to_dev(syn.layer(wl, seed))))
    return res


def _ws_bytes(q, layers, fmt_flags=0):
    return max(q.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt | fmt_flags) for wl, _ in layers)


def test_primed_chain_matches_default_calls(qgpu):
    layers = _layers()
    need = _ws_bytes(qgpu, layers)
    outs_ref = []
    for wl, d in layers:
        o = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        _call(qgpu, d, wl, wl.fmt, torch.empty(need, dtype=torch.uint8, device="cuda"), o)
        outs_ref.append(o)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda") for wl, _ in layers]
    for _ in range(3):  # back to back on one stream, three rounds
        for (wl, d), o in zip(layers, outs):
            _call(qgpu, d, wl, wl.fmt | qgpu.WORKSPACE_PRIMED, ws, o)
    torch.cuda.synchronize()
    assert not _header(ws).any(), _header(ws)
    for a, b in zip(outs, outs_ref):
        assert np.array_equal(bf16_tensor_bits(a), bf16_tensor_bits(b))


def test_primed_header_survives_prefill_calls(qgpu, oracle):
    """A prefill call on the same workspace leaves the decode header alone."""
    dec = syn.WORKLOADS["nvfp4_mtp_decode"]
    pre = syn.small("pre", T=40, E=16, k=4, H=256, I=128)   # T * k = 160 > 64: prefill path
    Ld, Lp = syn.layer(dec, 7), syn.layer(pre, 8)
    dd, dp = to_dev(Ld), to_dev(Lp)
    need = max(qgpu.forward_workspace_bytes(dec.T, dec.H, dec.I, dec.E, dec.k, dec.fmt),
               qgpu.forward_workspace_bytes(pre.T, pre.H, pre.I, pre.E, pre.k, pre.fmt))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    od = torch.empty((dec.T, dec.H), dtype=torch.bfloat16, device="cuda")
    op = torch.empty((pre.T, pre.H), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        _call(qgpu, dd, dec, dec.fmt | qgpu.WORKSPACE_PRIMED, ws, od)
        _call(qgpu, dp, pre, pre.fmt | qgpu.WORKSPACE_PRIMED, ws, op)
    _call(qgpu, dd, dec, dec.fmt | qgpu.WORKSPACE_PRIMED, ws, od)
    torch.cuda.synchronize()
    assert not _header(ws).any(), _header(ws)
    for wl, L, o in ((dec, Ld, od), (pre, Lp, op)):
        ref = oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                                 wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit)
        err, _ = row_rel_l2(bf16_tensor_bits(o), ref)
        assert err <= OUTPUT_RTOL, (wl.name, err)


def test_primed_chain_in_cuda_graph(qgpu):
    """Captured primed calls (programmatic edges in the graph) replay to the
    same outputs as eager default calls, and leave the header at zero."""
    layers = _layers()
    need = _ws_bytes(qgpu, layers)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda") for wl, _ in layers]
    s = torch.cuda.Stream()
    # inputs and the workspace were written on the current stream: order them first
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for (wl, d), o in zip(layers, outs):  # warm-up, outside the capture
            _call(qgpu, d, wl, wl.fmt | qgpu.WORKSPACE_PRIMED, ws, o)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (wl, d), o in zip(layers, outs):
            _call(qgpu, d, wl, wl.fmt | qgpu.WORKSPACE_PRIMED, ws, o)
    torch.cuda.synchronize()
    for o in outs:
        o.fill_(0)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert not _header(ws).any(), _header(ws)
    for (wl, d), o in zip(layers, outs):
        ref = torch.empty_like(o)
        _call(qgpu, d, wl, wl.fmt, torch.empty(need, dtype=torch.uint8, device="cuda"), ref)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_tensor_bits(o), bf16_tensor_bits(ref)), wl.name


def test_default_call_resets_a_dirty_header(qgpu):
    """Without the flag the header is reset by the call itself: a header left
    nonzero by anything else changes nothing."""
    wl = syn.WORKLOADS["nvfp4_mtp_decode"]
    d = to_dev(syn.layer(wl, 9))
    need = qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt)
    a = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    _call(qgpu, d, wl, wl.fmt, torch.zeros(need, dtype=torch.uint8, device="cuda"), a)
    dirty = torch.zeros(need, dtype=torch.uint8, device="cuda")
    dirty[:64] = 0x5A
    _call(qgpu, d, wl, wl.fmt, dirty, b)
    torch.cuda.synchronize()
    assert not _header(dirty).any()
    assert np.array_equal(bf16_tensor_bits(a), bf16_tensor_bits(b))


@pytest.mark.parametrize("name,kmajor", [("nvfp4_mtp_decode", True), ("mxfp4_decode", False),
                                         ("nvfp4_verify_edge", False), ("tiny_nvfp4_decode", True)])
def test_primed_long_chain_keeps_the_flag_clear(qgpu, name, kmajor):
    """Many primed calls of one workload back to back (eagerly and replayed
    from a CUDA graph): every launch is chained to the previous one by
    programmatic dependent launch, and no bounded wait may give up (the
    device error flag stays clear) while the results equal the default
    calls' bit for bit."""
    import importlib
    bench = importlib.import_module("bench")
    dev = torch.device("cuda", 0)
    wl, layers = bench.make_layers(4, 99, dev, name)
    fmt = wl.fmt
    if kmajor:
        for L in layers:
            L["s1"], L["s2"] = qgpu.scales_kmajor(L["s1"], wl.fmt), qgpu.scales_kmajor(L["s2"], wl.fmt)
        fmt |= qgpu.SCALES_KMAJOR
    need = qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, fmt)
    refs = []
    for L in layers:
        o = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
        _call(qgpu, L, wl, fmt, torch.empty(need, dtype=torch.uint8, device=dev), o)
        refs.append(bf16_tensor_bits(o))
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev) for _ in layers]
    stream = torch.cuda.Stream()
    # inputs and the workspace were written on the current stream: order them first
    stream.wait_stream(torch.cuda.current_stream())

    def chain():
        for _ in range(6):
            for L, o in zip(layers, outs):
                _call(qgpu, L, wl, fmt | qgpu.WORKSPACE_PRIMED, ws, o)

    with torch.cuda.stream(stream):
        chain()
    torch.cuda.synchronize()
    qgpu.check_device_error(ws, stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        chain()
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    qgpu.check_device_error(ws, stream)
    assert not _header(ws).any(), _header(ws)
    for o, r in zip(outs, refs):
        assert np.array_equal(bf16_tensor_bits(o), r)
