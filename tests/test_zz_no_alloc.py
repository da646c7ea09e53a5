"""moe_layout_noalloc: the layout entry point for callers that cannot allocate
device memory (under a host that forbids allocation after start-up),
whose scratch is the library's fixed device array instead of a workspace.

It must give exactly what moe_layout gives, on two calls in a row through the C
ABI (the second call reuses the array the first one left behind).  This file is
collected last so that a run stopping at the first failure has run everything
else first; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(M, idx, shape, ws=None):
    N, k = idx.shape
    E = shape.E
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    sched = torch.full((N * k, 2), -1, dtype=torch.int32, device="cuda")
    inv = torch.full((N, k), -1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    if ws is None:
        rc = M.lib().moe_layout_noalloc(idx.data_ptr(), ctypes.byref(shape), counts.data_ptr(),
                                        offsets.data_ptr(), sched.data_ptr(), inv.data_ptr(), st)
    else:
        rc = M.lib().moe_layout(idx.data_ptr(), ctypes.byref(shape), counts.data_ptr(),
                                offsets.data_ptr(), sched.data_ptr(), inv.data_ptr(),
                                ws.data_ptr(), ws.numel(), st)
    assert rc == 0, M.status_name(rc)
    torch.cuda.synchronize()
    return counts.cpu(), offsets.cpu(), sched.cpu(), inv.cpu()


def test_layout_noalloc_matches_layout_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_expert_top_gb300 import moe as M
    cases = [  # (N, E, k, S): a full DeepSeek-V3-sized batch, then a different smaller one
        (8192, 256, 8, 64),
        (1000, 33, 5, 10),
    ]
    for call, (N, E, k, S) in enumerate(cases):
        rng = np.random.default_rng(100 + call)
        idx = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)).cuda()
        shape = M.Shape.of(synth.Workload("noalloc", N=N, H=256, I=128, E=E, k=k, S=S, dtype="bf16"))
        ws = torch.empty(M.moe_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
        M.moe_workspace_init(ws)
        ref = _run(M, idx, shape, ws=ws)
        got = _run(M, idx, shape)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_layout_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_expert_top_gb300 import moe as M
    shape = M.Shape(N=131072, H=256, I=128, E=512, k=8, S=64, dtype=1)   # 4096 chunks x 512 experts
    rc = M.lib().moe_layout_noalloc(None, ctypes.byref(shape), None, None, None, None, None)
    assert rc == M.MOE_ERR_INVALID_ARG or rc == M.MOE_ERR_WORKSPACE
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    rc = M.lib().moe_layout_noalloc(p, ctypes.byref(shape), p, p, p, p, None)
    assert rc == M.MOE_ERR_WORKSPACE
