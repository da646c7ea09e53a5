"""The expert-parallel cut of the layer (ep.py) run rank by rank on one GPU
through the C ABI: every rank pulls its own slot range ([MoK-2.37x] = "Cursor's
MoK achieves 2.37x performance boost on NVIDIA GB300 NVL72", section 02: the
expert side pulls the rows its schedule lists) and runs the FFN of its own
experts, then one combine brings every output row back to its token.  The
result must equal the staged moe_forward bit for bit: each expert's rows meet
the same tiles in the same order whichever experts share the launch."""
import numpy as np
import pytest
import torch

from gpu_common import need_cuda, to_np
from token_dispatch_expert_top_gb300 import ep, synth

pytestmark = pytest.mark.gpu

CASES = [
    (synth.Workload("ep_mx", N=512, H=512, I=256, E=16, k=4, S=4, dtype="mxfp8"), 2),
    (synth.Workload("ep_mx", N=512, H=512, I=256, E=16, k=4, S=4, dtype="mxfp8"), 4),
    (synth.Workload("ep_bf16_skew", N=768, H=1024, I=384, E=12, k=3, S=6, dtype="bf16", skew=1.0), 3),
]


@pytest.mark.parametrize("w,R", CASES, ids=[f"{c[0].name}-R{c[1]}" for c in CASES])
def test_expert_parallel_ranks_on_one_gpu_equal_staged(w, R):
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe as M
    from token_dispatch_expert_top_gb300.layer import MoeLayer, quantize_mxfp8
    layer = MoeLayer(w, synth.make_inputs(w, device="cpu"))
    staged = layer.forward().clone()
    assert layer.device_status() == 0
    mx = w.dtype == "mxfp8"
    shape, ws, dev = layer.shape, layer.ws, layer.x.device
    T, rows = w.T, w.rows_per_shard
    i32 = dict(dtype=torch.int32, device=dev)
    counts, offsets = torch.empty(w.E, **i32), torch.empty(w.E + 1, **i32)
    sched, inv = torch.empty((T, 2), **i32), torch.empty((w.N, w.k), **i32)
    M.moe_layout(layer.idx, shape, counts, offsets, sched, inv, ws)   # every rank's choices
    off, sch = to_np(offsets).astype(np.int64), to_np(sched)
    # the source rows every rank serves: the MXFP8 copy of x (or x), S shards of N/S rows
    src, src_sf = quantize_mxfp8(layer.x) if mx else (layer.x, None)
    row_bytes = w.H * (1 if mx else 2)
    tab = torch.tensor([src.data_ptr() + s * rows * row_bytes for s in range(w.S)], dtype=torch.int64,
                       device=dev)
    tab_sf = None if not mx else torch.tensor(
        [src_sf.data_ptr() + s * rows * (w.H // 32) for s in range(w.S)], dtype=torch.int64, device=dev)
    ring = torch.empty((T, row_bytes), dtype=torch.uint8, device=dev)
    ring_sf = torch.empty((T, w.H // 32), dtype=torch.uint8, device=dev) if mx else None
    y = torch.zeros((T, w.H), dtype=torch.bfloat16, device=dev)
    covered = 0
    for r in range(R):
        first, cnt = ep.slot_range(off, w.E, R, r)
        if w.S % R == 0:     # the pull schedule names the rank that holds each source row
            ps = ep.pull_schedule(sch, off, w.E, R, w.S, r)
            np.testing.assert_array_equal(ps[:, 0] * (w.S // R) + ps[:, 1], sch[first:first + cnt, 0])
            np.testing.assert_array_equal(ps[:, 2], sch[first:first + cnt, 1])
        M.moe_dispatch_pull(tab, tab_sf, shape, sched, None, first, cnt, ring, ring_sf, T, ws)
        # this rank's experts only: every other expert's segment is empty
        off_r = torch.from_numpy(np.clip(off, first, first + cnt).astype(np.int32)).to(dev)
        M.moe_expert_ffn(ring, ring_sf, off_r, layer.wgu, layer.wgu_sf, layer.wd, layer.wd_sf, shape, y, ws)
        covered += cnt
    assert covered == T
    out = torch.empty_like(staged)
    M.moe_combine(y, inv, layer.gate, shape, out, ws)
    assert M.moe_last_device_status(ws) == 0
    assert torch.equal(out, staged)
