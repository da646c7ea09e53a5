"""Bitwise reproducibility under concurrent HBM traffic from another stream.

The kernels' pipelines wait on barriers and counters whose completion order
depends on memory timing; traffic from a second stream reorders load
completions.  Every repetition must reproduce the first result exactly."""
import pytest
import torch

from gpu_common import need_cuda
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu

# DeepSeek-V3 row widths (H = 7168, I = 2048) with a few experts, skewed so that
# some experts are hot and some empty.
W = synth.Workload("stress", N=1024, H=7168, I=2048, E=16, k=4, S=8, dtype="mxfp8", skew=3.0)


def _noise():
    buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    return buf, torch.cuda.Stream()


def test_forward_staged_and_fused_bitwise_under_traffic():
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    layer = MoeLayer(W, synth.make_inputs(W, device="cuda"))
    first = layer.forward().clone()
    assert torch.equal(layer.forward(fused=True), first)
    buf, side = _noise()
    for rep in range(8):
        with torch.cuda.stream(side):
            buf.fill_(rep)
        staged = layer.forward()
        with torch.cuda.stream(side):
            buf.fill_(rep + 1)
        fused = layer.forward(fused=True)
        torch.cuda.synchronize()
        assert torch.equal(staged, first), rep
        assert torch.equal(fused, first), rep
    assert layer.device_status() == 0


def test_backward_bitwise_under_traffic():
    need_cuda()
    from token_dispatch_expert_top_gb300.layer import MoeLayer
    layer = MoeLayer(W, synth.make_inputs(W, device="cuda"), train=True)
    dout = torch.randn((W.N, W.H), generator=torch.Generator(device="cuda").manual_seed(2),
                       device="cuda").to(torch.bfloat16)
    layer.forward_train()
    layer.backward(dout)
    ref = [t.clone() for t in (layer.dx, layer.dw_router, layer.dbias, layer.dw_gate_up, layer.dw_down)]
    buf, side = _noise()
    for rep in range(6):
        with torch.cuda.stream(side):
            buf.fill_(rep)
        layer.forward_train()
        layer.backward(dout)
        torch.cuda.synchronize()
        got = (layer.dx, layer.dw_router, layer.dbias, layer.dw_gate_up, layer.dw_down)
        for name, a, b in zip(("dx", "dw_router", "dbias", "dw_gate_up", "dw_down"), got, ref):
            assert torch.equal(a, b), (rep, name)
    assert layer.device_status() == 0 and layer.backward_status() == 0
