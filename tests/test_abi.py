"""CPU-side checks of the C ABI: the library loads, exports every function that
include/moe.h declares, and its host-only logic (workspace sizing, argument
checks, the minibatch wave rule) behaves as documented.  No kernel is launched."""
import ctypes
import os
import re

import pytest

from token_dispatch_expert_top_gb300 import moe as M
from token_dispatch_expert_top_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_entry_points():
    decl = declared_functions()
    assert set(decl) == set(M.ENTRY_POINTS), set(decl) ^ set(M.ENTRY_POINTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(os.path.join(ROOT, "token_dispatch_expert_top_gb300", "libmoe.so"))
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    assert M.status_name(0) == "MOE_OK"
    assert M.status_name(M.MOE_ERR_TIMEOUT) == "MOE_ERR_TIMEOUT"
    assert M.status_name(99) == "MOE_ERR_UNKNOWN"


def test_workspace_bytes_grows_with_shape_and_rejects_bad_shapes():
    small = M.Shape.of(synth.WORKLOADS["tiny_f32"])
    big = M.Shape.of(synth.WORKLOADS["dsv3_mxfp8"])
    b_small = M.moe_workspace_bytes(small)
    b_big = M.moe_workspace_bytes(big)
    assert 0 < b_small < b_big
    # config-3 staged forward: ring (T x 7392 B) + h + y (T x 14336 B) dominate
    T = 8192 * 8
    assert b_big > T * (7168 + 224 + 2048 + 64 + 2 * 7168)
    for bad in [dict(k=9, E=8), dict(N=65, S=2), dict(H=100), dict(dtype=7), dict(E=0)]:
        d = dict(N=64, H=128, I=256, E=8, k=2, S=2, dtype=0)
        d.update(bad)
        assert M.moe_workspace_bytes(M.Shape(**d)) == 0, bad
    # tensor-core dtypes need H % 256 == 0 and I % 128 == 0
    assert M.moe_workspace_bytes(M.Shape(N=64, H=128, I=256, E=8, k=2, S=2, dtype=1)) == 0


def test_argument_errors_return_before_any_launch():
    bad = M.Shape(N=64, H=128, I=256, E=8, k=9, S=2, dtype=0)
    lib = M.lib()
    assert lib.moe_layout(None, ctypes.byref(bad), None, None, None, None, None, 0, None) == M.MOE_ERR_INVALID_ARG
    ok = M.Shape.of(synth.WORKLOADS["tiny_f32"])
    # missing workspace
    assert lib.moe_layout(1, ctypes.byref(ok), 1, 1, 1, 1, None, 0, None) == M.MOE_ERR_WORKSPACE
    assert lib.moe_expert_ffn(None, None, None, None, None, None, None, ctypes.byref(ok), None, 32,
                              1 << 40, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_mxfp8(None, 1, 4, 33, None, None, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_nvfp4(None, 1, 4, 24, None, None, None, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_nvfp4(None, 1, 4, 32, None, None, None, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_pull(1, None, ctypes.byref(ok), 1, None, 100, 100, 1, None, 8, 16, 256,
                                 None) == M.MOE_ERR_INVALID_ARG   # slots past T


def test_minibatch_wave_rule_golden():
    path = os.path.join(ROOT, "tests", "golden", "minibatch_waves.txt")
    rows = [l.split("#")[0].split() for l in open(path)]
    rows = [r for r in rows if r]
    assert rows
    for waves, sms, bm, bn, I, expect in rows:
        assert M.moe_min_minibatch(int(waves), int(sms), int(bm), int(bn), int(I)) == int(expect)


def test_backward_host_checks():
    lib = M.lib()
    f32 = M.Shape.of(synth.WORKLOADS["tiny_f32"])
    mx = M.Shape.of(synth.WORKLOADS["dsv3_mxfp8"])
    # the backward has no FP32 path
    assert M.moe_backward_workspace_bytes(f32) == 0
    assert lib.moe_reverse_combine(1, 1, 1, 1, ctypes.byref(f32), 1, None, 1, 1, 1, 1, 32, 1 << 20,
                                   None) == M.MOE_ERR_UNSUPPORTED
    # workspace: dy codes + scales, du|dv in BF16 and MXFP8, da, per-slot floats
    T, H, I = 8192 * 8, 7168, 2048
    need = T * (H + H // 32 + 4 * I + 2 * I + 2 * I // 32 + 2 * H + 16)
    assert M.moe_backward_workspace_bytes(mx) >= need
    # MXFP8 reverse combine needs dy scales; a null dout is an argument error
    assert lib.moe_reverse_combine(16, 16, 16, 16, ctypes.byref(mx), 16, None, 16, 16, 16, 16, 32,
                                   1 << 20, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_reverse_combine(None, 16, 16, 16, ctypes.byref(mx), 16, 16, 16, 16, 16, 16, 32,
                                   1 << 20, None) == M.MOE_ERR_INVALID_ARG
    # router wgrad needs the backward workspace
    assert lib.moe_router_wgrad(16, 16, 16, 16, ctypes.byref(mx), 16, 16, 32, 1 << 20,
                                None) == M.MOE_ERR_WORKSPACE
    # the training forward needs every saved buffer
    sv = M.Saved(16, 16, 16, 16, 16, 32, None)
    assert lib.moe_forward_train(16, 16, None, 16, 16, 16, 16, ctypes.byref(mx), None, 16,
                                 ctypes.byref(sv), 32, 1 << 40, None) == M.MOE_ERR_INVALID_ARG
    # misaligned du|dv output
    assert lib.moe_expert_ffn_dgrad(16, 16, 32, 16, 16, 16, 16, 16, ctypes.byref(mx), 48, 32, 16, 32,
                                    32, 1 << 20, None) == M.MOE_ERR_INVALID_ARG


def test_macrobatch_host_checks():
    """Macrobatch workspace sizing and argument errors, decided on the host."""
    w = synth.Workload("mb", N=512, H=512, I=256, E=16, k=4, S=4, dtype="mxfp8")
    shape = M.Shape.of(w)
    one = M.moe_workspace_bytes(M.Shape.of(w.scaled(N=256)), None)
    assert M.moe_macro_workspace_bytes(shape, None, 2) == 2 * ((one + 255) // 256 * 256)
    assert M.moe_macro_workspace_bytes(shape, None, 3) == 0      # 512 is not a multiple of 3 * 4
    assert M.moe_macro_workspace_bytes(shape, None, 0) == 0
    lib = M.lib()
    args = [None] * 7 + [ctypes.byref(shape), None]
    assert lib.moe_forward_macrobatched(*args, 0, None, None, 0, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_macrobatched(*args, 3, None, None, 0, None) == M.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_macrobatched(*args, 2, None, None, 0, None) == M.MOE_ERR_WORKSPACE
    # the reverse-ring flag sits at the end of moe_params_t; it leaves the workspace unchanged
    p = M.Params(0, 0, 0, 0, 0, 0, 1)
    assert M.moe_workspace_bytes(shape, p) == M.moe_workspace_bytes(shape, M.Params(0, 0, 0, 0, 0, 0, 0))


def test_layout_noalloc_checks_shapes_as_layout_does():
    """moe_layout_noalloc rejects exactly the shapes moe_layout rejects, with the
    same status, before it touches the device."""
    lib = M.lib()
    bad = [
        dict(N=64, H=100, I=128, E=8, k=2, S=2, dtype=1),     # H not a multiple of 32
        dict(N=64, H=256, I=96, E=8, k=2, S=2, dtype=2),      # MXFP8: I not a multiple of 128
        dict(N=64, H=256, I=128, E=8, k=2, S=2, dtype=7),     # no such dtype
        dict(N=64, H=256, I=128, E=8, k=9, S=2, dtype=1),     # k > E
        dict(N=63, H=256, I=128, E=8, k=2, S=2, dtype=1),     # N not a multiple of S
        dict(N=64, H=256, I=128, E=2048, k=2, S=2, dtype=1),  # too many experts
    ]
    for d in bad:
        shape = M.Shape(**d)
        a = lib.moe_layout(None, ctypes.byref(shape), None, None, None, None, None, 0, None)
        b = lib.moe_layout_noalloc(None, ctypes.byref(shape), None, None, None, None, None)
        assert a == b != 0, (d, M.status_name(a), M.status_name(b))
