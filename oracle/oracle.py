"""The oracle: a plain, slow FP64 CPU forward MoE layer.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline / reference legs may import this module.  It shares no code with the
CUDA library.

The element-wise and combinatorial steps (number formats, softmax/top-k/gates,
layout, SwiGLU, combine) are plain C loops in ``moe_oracle.c``; the contractions
(router logits, expert GEMMs) use numpy's FP64 matmul as a library primitive.
Steps run in the order the pages give for the layer ([MoK-2.37x] = "Cursor's MoK
achieves 2.37x performance boost on NVIDIA GB300 NVL72", section 03: schedule,
dispatch, expert FFN, combine, final weighted merge):

  1. logits  = x . W_r (+ b)                          FP64 over the stored values
  2. p = softmax(logits); top-k; g = p_sel / sum p_sel
  3. layout: counts, offsets, (shard, row) schedule, inverse map
  4. dispatch: each slot takes its token's row (MXFP8-quantised along H for the
     MXFP8 workloads)
  5. expert FFN: u = a . W_gate, v = a . W_up, h = silu(u) * v, h rounded to the
     workload's intermediate format, y = h . W_down rounded to the staging format
  6. combine: out[n] = sum_j g[n,j] * y[slot(n,j)] in j order, rounded once.

The backward (``backward``) is the exact derivative of that forward, taken in FP64
with every rounding point passed straight through and the top-k choice held fixed;
its two element-wise steps (SwiGLU derivative, gate Jacobian) are C loops too.

Rounding points per workload dtype:
  f64   : nothing rounded (the smooth layer the derivative pins perturb)
  f32   : operands FP32 values; h, y and out rounded to FP32
  bf16  : operands BF16 values; h, y and out rounded to BF16
  mxfp8 : x, W_gate/W_up (along H) and W_down (along I) MXFP8-quantised; h
          MXFP8-quantised along I per slot row; y and out rounded to BF16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the C oracle (plain -O2, IEEE semantics, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.orc_round_bf16.restype = ctypes.c_double
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_round_f32.restype = ctypes.c_double
        L.orc_round_f32.argtypes = [ctypes.c_double]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_round_bf16_array.argtypes = [_f64p, _i64, _f64p]
        L.orc_round_f32_array.argtypes = [_f64p, _i64, _f64p]
        L.orc_e4m3_encode_array.argtypes = [_f64p, _i64, _u8p]
        L.orc_quantize_mxfp8.argtypes = [_f64p, _i64, _i64, _u8p, _u8p]
        L.orc_dequantize_mxfp8.argtypes = [_u8p, _u8p, _i64, _i64, _f64p]
        L.orc_route_topk.argtypes = [_f64p, _i64, _int, _int, _i32p, _f64p, ctypes.c_void_p]
        L.orc_layout.argtypes = [_i32p, _i64, _int, _int, _int, _i32p, _i32p, _i32p, _i32p]
        L.orc_swiglu.argtypes = [_f64p, _f64p, _i64, _f64p]
        L.orc_combine.argtypes = [_f64p, _i32p, _f64p, _i64, _int, _i64, _f64p]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_double]
        L.orc_nvfp4_tensor_scale.restype = ctypes.c_double
        L.orc_nvfp4_tensor_scale.argtypes = [_f64p, _i64]
        L.orc_quantize_nvfp4.argtypes = [_f64p, _i64, _i64, ctypes.c_double, _u8p, _u8p]
        L.orc_dequantize_nvfp4.argtypes = [_u8p, _u8p, _i64, _i64, ctypes.c_double, _f64p]
        L.orc_swiglu_backward.argtypes = [_f64p, _f64p, _f64p, _i64, _f64p, _f64p]
        L.orc_gate_backward.argtypes = [_f64p, _f64p, _i64, _int, _f64p]
        _lib = L
    return _lib


def _f64(a) -> np.ndarray:
    """Host FP64 copy of a numpy array or torch tensor (exact for f32/bf16 values)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        if str(a.dtype) == "torch.bfloat16":
            a = a.float()
        a = a.numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# --------------------------------------------------------------------------- formats
def round_bf16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty_like(a)
    lib().orc_round_bf16_array(a.ravel(), a.size, out.ravel())
    return out


def round_f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty_like(a)
    lib().orc_round_f32_array(a.ravel(), a.size, out.ravel())
    return out


def e4m3_encode(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(a.ravel(), a.size, out.ravel())
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    f = lib().orc_e4m3_decode
    table = np.array([f(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def quantize_mxfp8(a: np.ndarray):
    """[rows, K] FP64 -> (codes [rows, K] u8, scales [rows, K/32] u8)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    rows, K = a.shape
    assert K % 32 == 0
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    lib().orc_quantize_mxfp8(a, rows, K, codes, scales)
    return codes, scales


def dequantize_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, K = codes.shape
    out = np.empty((rows, K), dtype=np.float64)
    lib().orc_dequantize_mxfp8(codes, scales, rows, K, out)
    return out


def mxfp8_values(a: np.ndarray) -> np.ndarray:
    """The values an MXFP8 operand holds after quantising a along its last axis."""
    return dequantize_mxfp8(*quantize_mxfp8(a))


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    f = lib().orc_e2m1_decode
    table = np.array([f(c) for c in range(16)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8) & 15]


def e2m1_encode(a) -> np.ndarray:
    f = lib().orc_e2m1_encode
    a = np.asarray(a, dtype=np.float64)
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def quantize_nvfp4(a: np.ndarray):
    """[rows, K] FP32 values -> (codes [rows, K/2] u8 (two E2M1 per byte, lower
    element in the low nibble), scales [rows, K/16] E4M3 u8, tensor scale float)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    rows, K = a.shape
    assert K % 16 == 0
    st = lib().orc_nvfp4_tensor_scale(a.ravel(), a.size)
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 16), dtype=np.uint8)
    lib().orc_quantize_nvfp4(a, rows, K, st, codes, scales)
    return codes, scales, st


def dequantize_nvfp4(codes: np.ndarray, scales: np.ndarray, st: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, K), dtype=np.float64)
    lib().orc_dequantize_nvfp4(codes, scales, rows, K, float(st), out)
    return out


def round_to(a: np.ndarray, fmt: str) -> np.ndarray:
    """Round an FP64 array to the storage format of a tensor: f64 (kept as is), f32,
    bf16, mxfp8."""
    if fmt == "f64":
        return np.array(a, dtype=np.float64)
    if fmt == "f32":
        return round_f32(a)
    if fmt == "bf16":
        return round_bf16(a)
    if fmt == "mxfp8":
        return mxfp8_values(a)
    raise ValueError(fmt)


# --------------------------------------------------------------------------- steps
def router_logits(x, w_router, bias=None) -> np.ndarray:
    """logits[n, e] = sum_h x[n, h] W_r[h, e] (+ b_e), FP64 (w_router stored [E, H])."""
    lg = _f64(x) @ _f64(w_router).T
    if bias is not None:
        lg = lg + _f64(bias)[None, :]
    return np.ascontiguousarray(lg)


def route_topk(logits: np.ndarray, k: int, want_probs: bool = False):
    """Softmax, top-k (descending logit, lower index first on ties), renormalised gates."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    n, E = logits.shape
    idx = np.empty((n, k), dtype=np.int32)
    gate = np.empty((n, k), dtype=np.float64)
    probs = np.empty((n, E), dtype=np.float64) if want_probs else None
    lib().orc_route_topk(logits, n, E, k, idx, gate,
                         None if probs is None else probs.ctypes.data_as(ctypes.c_void_p))
    return (idx, gate, probs) if want_probs else (idx, gate)


def topk_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: k-th largest logit minus the (k+1)-th (inf when k == E).  Used to
    set aside near-ties, where FP32 and FP64 logits may pick different experts."""
    E = logits.shape[1]
    if k >= E:
        return np.full(logits.shape[0], np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


def layout(idx: np.ndarray, E: int, S: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    sched = np.empty((N * k, 2), dtype=np.int32)
    inv = np.empty((N, k), dtype=np.int32)
    lib().orc_layout(idx, N, k, E, S, counts, offsets, sched, inv)
    return counts, offsets, sched, inv


def swiglu(u: np.ndarray, v: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    h = np.empty_like(u)
    lib().orc_swiglu(u.ravel(), v.ravel(), u.size, h.ravel())
    return h


def combine(y: np.ndarray, inv: np.ndarray, gate: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float64)
    inv = np.ascontiguousarray(inv, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    n, k = inv.shape
    H = y.shape[1]
    out = np.empty((n, H), dtype=np.float64)
    lib().orc_combine(y, inv, gate, n, k, H, out)
    return out


# Storage formats of the FFN operands and outputs per workload dtype.
FORMATS = {
    #          operands  h        y       out
    "f64":   ("f64",     "f64",   "f64",  "f64"),     # unrounded: smooth, for derivative pins
    "f32":   ("f32",     "f32",   "f32",  "f32"),
    "bf16":  ("bf16",    "bf16",  "bf16", "bf16"),
    "mxfp8": ("mxfp8",   "mxfp8", "bf16", "bf16"),
}


def expert_operands(w_gate_up_e, w_down_e, dtype: str):
    """FP64 values of one expert's weights as the GEMMs see them: (Wg^T [I,H],
    Wu^T [I,H], Wd^T [H,I]); MXFP8 quantises each output column along K."""
    wgu = _f64(w_gate_up_e)
    wd = _f64(w_down_e)
    I = wgu.shape[0] // 2
    if dtype == "mxfp8":
        wgu = mxfp8_values(wgu)
        wd = mxfp8_values(wd)
    return wgu[:I], wgu[I:], wd


def expert_ffn(a: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, dtype: str) -> np.ndarray:
    """y = round_y( round_h( silu(a Wg) * (a Wu) ) Wd ) for the rows a of one expert."""
    _, fmt_h, fmt_y, _ = FORMATS[dtype]
    u = a @ wg.T
    v = a @ wu.T
    h = round_to(swiglu(u, v), fmt_h)
    return round_to(h @ wd.T, fmt_y)


def forward(inp: dict, E: int, k: int, S: int, dtype: str, tokens=None, expert_fn=None,
            weights=None) -> dict:
    """The forward layer on the oracle.

    inp: dict with x [N,H], w_router [E,H], bias [E] or None, w_gate_up [E,2I,H],
         w_down [E,H,I] (numpy arrays or torch tensors; values are read as stored).
    tokens: optional list of token indices; only their outputs are computed
         (routing and layout always cover all N tokens).
    expert_fn: optional hook (e, a) -> y replacing the SwiGLU FFN (closed-form tests).
    weights: optional callable e -> (wg, wu, wd) FP64 operand values (lets callers
         stream experts); defaults to expert_operands over inp's tensors.
    Returns dict(logits, idx, gate, gap, counts, offsets, sched, inv, tokens, out).
    """
    fmt_a, _, _, fmt_out = FORMATS[dtype]
    x = _f64(inp["x"])
    N = x.shape[0]
    logits = router_logits(x, inp["w_router"], inp.get("bias"))
    idx, gate = route_topk(logits, k)
    counts, offsets, sched, inv = layout(idx, E, S)
    toks = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)

    # dispatch: the operand rows the experts read (MXFP8: quantised along H per row)
    a_rows = x[toks]
    if fmt_a == "mxfp8":
        a_rows = mxfp8_values(a_rows)

    # expert FFN, one expert at a time, over the (token, choice) pairs of toks
    pair_tok, pair_j = np.meshgrid(np.arange(len(toks)), np.arange(k), indexing="ij")
    pair_e = idx[toks][:, :k]
    H = x.shape[1]
    y = np.zeros((len(toks) * k, H), dtype=np.float64)
    for e in np.unique(pair_e):
        sel = np.nonzero(pair_e.ravel() == e)[0]
        a = a_rows[pair_tok.ravel()[sel]]
        if expert_fn is not None:
            y[sel] = expert_fn(int(e), a)
        else:
            wg, wu, wd = weights(int(e)) if weights is not None else expert_operands(
                inp["w_gate_up"][int(e)], inp["w_down"][int(e)], dtype)
            y[sel] = expert_ffn(a, wg, wu, wd, dtype)

    # combine: y rows of this call are numbered token-major (t*k + j)
    local_inv = (np.arange(len(toks) * k, dtype=np.int32)).reshape(len(toks), k)
    out = combine(y, local_inv, gate[toks])
    out = round_to(out, fmt_out)
    return dict(logits=logits, idx=idx, gate=gate, gap=topk_gap(logits, k), counts=counts,
                offsets=offsets, sched=sched, inv=inv, tokens=toks, out=out, y=y)


# --------------------------------------------------------------------------- backward
def swiglu_backward(u: np.ndarray, v: np.ndarray, dh: np.ndarray):
    """(du, dv) for h = silu(u) * v, given dh."""
    u = np.ascontiguousarray(u, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    dh = np.ascontiguousarray(dh, dtype=np.float64)
    du = np.empty_like(u)
    dv = np.empty_like(u)
    lib().orc_swiglu_backward(u.ravel(), v.ravel(), dh.ravel(), u.size, du.ravel(), dv.ravel())
    return du, dv


def gate_backward(gate: np.ndarray, dgate: np.ndarray) -> np.ndarray:
    """Gradient of the renormalised top-k gates w.r.t. the selected logits, [n, k]."""
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    dgate = np.ascontiguousarray(dgate, dtype=np.float64)
    n, k = gate.shape
    out = np.empty_like(gate)
    lib().orc_gate_backward(gate, dgate, n, k, out)
    return out


# Storage formats of the backward's dgrad operands and intermediates per workload
# dtype: dy (the first dgrad GEMM's A operand, along H), the kept pre-activations
# u|v, du|dv (the second dgrad GEMM's A operand, along I), da, and dh as it is
# kept between the first dgrad GEMM and the SwiGLU derivative.  The dgrad
# weights are the masters in the GEMM format quantised along the dgrad K
# (``expert_operands_dgrad``).
BWD_FORMATS = {
    #          dy        uv      duv      da      dh
    "f64":   ("f64",    "f64",  "f64",   "f64",  "f64"),
    "f32":   ("f32",    "f32",  "f32",   "f32",  "f32"),
    "bf16":  ("bf16",   "bf16", "bf16",  "bf16", "bf16"),
    "mxfp8": ("mxfp8",  "bf16", "mxfp8", "bf16", "bf16"),
}


# Format of the wgrad GEMM operands (quantised along the expert's slots, which
# those GEMMs reduce over) and of the weight gradients; None: the exact
# straight-through formulas on the forward's own values.
WGRAD_FORMATS = {"f64": None, "f32": None, "bf16": "bf16", "mxfp8": "mxfp8"}


def round_along_slots(m: np.ndarray, fmt: str) -> np.ndarray:
    """Round the rows of one expert's slot segment [slots, C] as a wgrad operand:
    MXFP8 blocks of 32 consecutive slots from the segment's first slot (the last
    block zero-padded), or element-wise for the other formats."""
    if fmt != "mxfp8":
        return round_to(m, fmt)
    R = m.shape[0]
    pad = (-R) % 32
    mp = np.vstack([m, np.zeros((pad, m.shape[1]))]) if pad else m
    return np.ascontiguousarray(mxfp8_values(np.ascontiguousarray(mp.T)).T[:R])


def round_dgrad_operand(m: np.ndarray, fmt: str) -> np.ndarray:
    """A dgrad GEMM's token-side operand m [slots, K] in its storage format: each
    slot row on its own, MXFP8 blocks of 32 consecutive elements along K, the
    GEMM's reduction axis (dy: K = H; du and dv: K = I)."""
    return round_to(m, fmt)


def expert_operands_dgrad(w_gate_up_e, w_down_e, dtype: str):
    """FP64 values of one expert's weights as the dgrad GEMMs see them: (Wg [I,H],
    Wu [I,H], Wd [H,I]) with the reduction running over I (gate/up) and over H
    (down).  MXFP8 quantises the masters along that reduction axis: W_gate_up
    down its 2I rows (blocks split at I), W_down down its H rows."""
    wgu = _f64(w_gate_up_e)
    wd = _f64(w_down_e)
    I = wgu.shape[0] // 2
    if dtype == "mxfp8":
        wgu = mxfp8_values(wgu.T).T
        wd = mxfp8_values(wd.T).T
    return wgu[:I], wgu[I:], wd


def expert_ffn_backward(a: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray,
                        dy: np.ndarray, dtype: str, wb=None, a_master=None,
                        want_wgrad: bool = True) -> dict:
    """Backward of one expert's SwiGLU FFN over its rows a, given dy = dL/dy.

    Forward as ``expert_ffn``: u = a Wg^T, v = a Wu^T, h = round_h(silu(u) v),
    y = round_y(h Wd^T).  Each rounding point's derivative is taken as 1, so
      dh = round_dh(dy_b Wd_b),  (du, dv) = swiglu_backward(u_s, v_s, dh),
      da = round_da(du_b Wg_b + dv_b Wu_b),
      dWg = du^T a,  dWu = dv^T a,  dWd = dy^T h   (h after its rounding),
    where _b marks a dgrad GEMM operand in its storage format (BWD_FORMATS, each
    slot row quantised along K by round_dgrad_operand; the weights ``wb`` =
    expert_operands_dgrad, default the forward's values) and
    u_s, v_s the kept pre-activations.  With a wgrad format (WGRAD_FORMATS) the
    weight gradients are GEMMs over the slots too, each operand rounded along the
    slots (round_along_slots) and the result rounded to BF16:
      dWg = (du_s)^T a_w,  dWu = (dv_s)^T a_w,  dWd = (dy)^T h_w
    with du_s, dv_s the BF16 copies of du, dv, a_w the master rows a_master (x,
    unquantised), h_w = silu(u_s) v_s recomputed from the kept u|v, every one of
    them then rounded along the slots.  For "f64" nothing is rounded and this is
    the exact derivative.  want_wgrad=False skips the weight gradients (None).
    Returns dict(u, v, h, y, dh, du, dv, da, dwg, dwu, dwd)."""
    _, fmt_h, fmt_y, _ = FORMATS[dtype]
    f_dy, f_uv, f_duv, f_da, f_dh = BWD_FORMATS[dtype]
    wg_b, wu_b, wd_b = (wg, wu, wd) if wb is None else wb
    u = a @ wg.T
    v = a @ wu.T
    h = round_to(swiglu(u, v), fmt_h)
    y = round_to(h @ wd.T, fmt_y)
    u_s, v_s = round_to(u, f_uv), round_to(v, f_uv)
    dh = round_to(round_dgrad_operand(dy, f_dy) @ wd_b, f_dh)
    du, dv = swiglu_backward(u_s, v_s, dh)
    da = round_to(round_dgrad_operand(du, f_duv) @ wg_b + round_dgrad_operand(dv, f_duv) @ wu_b,
                  f_da)
    if not want_wgrad:
        dwg = dwu = dwd = None
    elif WGRAD_FORMATS[dtype] is None:
        dwg, dwu, dwd = du.T @ a, dv.T @ a, dy.T @ h
    else:
        dwg, dwu, dwd = expert_wgrad(a if a_master is None else a_master, round_bf16(du),
                                     round_bf16(dv), dy, u_s, v_s, dtype)
    return dict(u=u, v=v, h=h, y=y, dh=dh, du=du, dv=dv, da=da, dwg=dwg, dwu=dwu, dwd=dwd)


def expert_wgrad(a: np.ndarray, du: np.ndarray, dv: np.ndarray, dy: np.ndarray, u: np.ndarray,
                 v: np.ndarray, dtype: str):
    """One expert's weight gradients as GEMMs over its slots (rows in slot order):
      dWg = du^T a,  dWu = dv^T a,  dWd = dy^T h,  h = silu(u) v,
    every operand rounded along the slots in the wgrad format (round_along_slots)
    and each result rounded to BF16.  a: master x rows; du, dv, u, v: the values
    as stored (BF16 copies); dy: g * dout."""
    q = lambda m: round_along_slots(m, WGRAD_FORMATS[dtype])
    a_w = q(a)
    h_w = q(swiglu(u, v))
    return (round_bf16(q(du).T @ a_w), round_bf16(q(dv).T @ a_w), round_bf16(q(dy).T @ h_w))


def backward(inp: dict, E: int, k: int, S: int, dtype: str, dout, tokens=None, experts=None,
             weights=None, router_experts=None) -> dict:
    """Gradients of the forward layer, L = sum(dout * out), on the oracle.

    The backward the pages describe for the layer ([MoK-2.37x] section 01: training
    adds two exchanges in the opposite direction; section 02: a pulled reverse
    combine and a pushed reverse dispatch) undoes the combine by bringing dout back
    to every slot, differentiates the expert FFN, and undoes the dispatch by adding
    every slot's input gradient back to its token.  Here it is the exact derivative
    of ``forward`` with two readings the pages leave open:
      * every rounding point (MXFP8 / BF16 / FP32 storage of x, the weights, h, y
        and out) is passed straight through: its derivative is taken as 1, and the
        values after rounding are the ones used wherever the forward used them;
      * the top-k choice is piecewise constant, so only the k selected logits of a
        token get a gradient, through the renormalised gates.

    For the rounded dtypes the dgrad GEMMs also round their operands the way the
    layer's configuration fixes for every expert GEMM (MXFP8: each operand
    quantised along that GEMM's reduction axis; BWD_FORMATS, expert_operands_dgrad),
    the kept pre-activations u, v are BF16, da is BF16 and dx is rounded once.

    Per (token n, choice j) pair, with slot expert e = idx[n, j], gate g = gate[n, j]:
      dy     = g * dout[n]                            reverse combine, pulled by slot
      dgate  = <dout[n], y>                           y as the forward stored it
      dh     = dy . Wd                                (y = h . Wd^T)
      du, dv = dh * v * silu'(u), dh * silu(u)       (h = silu(u) * v)
      da     = du . Wg + dv . Wu                      (u = a . Wg^T, v = a . Wu^T)
    Per expert: dWg = sum du^T a, dWu = sum dv^T a, dWd = sum dy^T h over its pairs.
    Per token: dx_ffn = sum_j da (reverse dispatch); dlogit of the selected experts
    = g_j (dgate_j - sum_i g_i dgate_i); dx_router = dlogit . W_r; dx = both summed.
    Router: dW_r = sum_n dlogit^T x (x as stored, which is what the logits read),
    dbias = sum_n dlogit.

    tokens:  optional token subset for dx and the per-pair outputs of those tokens.
    experts: optional expert subset for dW_gate_up and dW_down.
    router_experts: optional expert subset for the dW_r rows and dbias entries
             (default: ``experts``).
    Without them, every output covers the whole layer.  The per-pair arrays cover
    the pairs listed in ``pairs`` (pair id = n*k + j): all pairs of ``tokens``, of
    the tokens routed to ``router_experts`` (their dlogit needs every choice's
    dgate) and every pair routed to ``experts``.  The FFN backward (dh, du, dv,
    da) is taken for the pairs where ``full`` is set: those of ``tokens`` and
    those routed to ``experts``; the other listed pairs only need the forward's y
    for their dgate, and hold zeros in dh, du, dv and da.
    Returns dict(idx, gate, inv, counts, offsets, pairs, full, dy, dgate, dh, du, dv,
    da, tokens, dx_ffn, dx_router, dx, dlogit, experts, router_experts, dw_router,
    dbias, dw_gate_up, dw_down).
    """
    fmt_a = FORMATS[dtype][0]
    x = _f64(inp["x"])
    wr = _f64(inp["w_router"])
    dY = _f64(dout)
    N, H = x.shape
    logits = router_logits(x, inp["w_router"], inp.get("bias"))
    idx, gate = route_topk(logits, k)
    counts, offsets, sched, inv = layout(idx, E, S)
    pair_e = idx.ravel().astype(np.int64)
    toks = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)
    exps = np.arange(E) if experts is None else np.asarray(experts, dtype=np.int64)
    rexps = exps if router_experts is None else np.asarray(router_experts, dtype=np.int64)

    # the tokens whose dlogit is needed, the pairs whose FFN gradient is needed
    # (full), and the pairs that only need y for their dgate
    routed = np.isin(idx, rexps).any(axis=1)
    need_tok = np.union1d(toks, np.nonzero(routed)[0])
    full_ids = np.union1d((toks[:, None] * k + np.arange(k)[None, :]).ravel(),
                          np.nonzero(np.isin(pair_e, exps))[0])
    pairs = np.union1d((need_tok[:, None] * k + np.arange(k)[None, :]).ravel(), full_ids)
    full = np.isin(pairs, full_ids)
    pos = {int(p): i for i, p in enumerate(pairs)}
    ptok = pairs // k
    P = len(pairs)

    a_rows = x[ptok]
    if fmt_a == "mxfp8":
        a_rows = mxfp8_values(a_rows)
    dy = gate.ravel()[pairs][:, None] * dY[ptok]           # reverse combine
    dgate_p = np.empty(P)
    I = _f64(inp["w_down"][0]).shape[1] if weights is None else weights(int(pair_e[0]))[2].shape[1]
    dh = np.zeros((P, I))
    du = np.zeros((P, I))
    dv = np.zeros((P, I))
    da = np.zeros((P, H))
    dwgu = np.zeros((len(exps), 2 * I, H))
    dwd = np.zeros((len(exps), H, I))
    exp_pos = {int(e): i for i, e in enumerate(exps)}
    for e in np.unique(pair_e[pairs]):
        on_e = pair_e[pairs] == e
        wg, wu, wd = weights(int(e)) if weights is not None else expert_operands(
            inp["w_gate_up"][int(e)], inp["w_down"][int(e)], dtype)
        fwd_only = np.nonzero(on_e & ~full)[0]
        if len(fwd_only):
            y_f = expert_ffn(a_rows[fwd_only], wg, wu, wd, dtype)
            dgate_p[fwd_only] = np.einsum("ph,ph->p", dY[ptok[fwd_only]], y_f)
        sel = np.nonzero(on_e & full)[0]
        if not len(sel):
            continue
        wb = expert_operands_dgrad(inp["w_gate_up"][int(e)], inp["w_down"][int(e)], dtype)
        r = expert_ffn_backward(a_rows[sel], wg, wu, wd, dy[sel], dtype, wb, x[ptok[sel]],
                                want_wgrad=int(e) in exp_pos)
        dgate_p[sel] = np.einsum("ph,ph->p", dY[ptok[sel]], r["y"])
        dh[sel], du[sel], dv[sel], da[sel] = r["dh"], r["du"], r["dv"], r["da"]
        if int(e) in exp_pos:
            i = exp_pos[int(e)]
            dwgu[i, :I] = r["dwg"]
            dwgu[i, I:] = r["dwu"]
            dwd[i] = r["dwd"]

    # reverse dispatch: each token adds the input gradients of its k slots, j order
    tok_pairs = np.array([[pos[int(n * k + j)] for j in range(k)] for n in toks],
                         dtype=np.int32).reshape(len(toks), k)
    dx_ffn = combine(da, tok_pairs, np.ones((len(toks), k)))
    f_dx = FORMATS[dtype][3]

    # router: dlogit over the tokens that need it (zero for unselected experts)
    dgate_full = np.zeros((N, k))
    have = np.zeros((N, k), dtype=bool)
    dgate_full.ravel()[pairs] = dgate_p
    have.ravel()[pairs] = True
    assert have[need_tok].all()
    dlsel = gate_backward(gate[need_tok], dgate_full[need_tok])
    dlogit = np.zeros((N, E))
    rows = np.repeat(need_tok, k)
    dlogit[rows, idx[need_tok].ravel()] = dlsel.ravel()
    dx_router = dlogit[toks] @ wr
    dw_router = dlogit[:, rexps].T @ x
    dbias = dlogit[:, rexps].sum(axis=0)
    return dict(idx=idx, gate=gate, inv=inv, counts=counts, offsets=offsets, pairs=pairs,
                full=full, dy=dy, dgate=dgate_full, dh=dh, du=du, dv=dv, da=da, tokens=toks,
                dx_ffn=dx_ffn, dx_router=dx_router, dx=round_to(dx_ffn + dx_router, f_dx),
                dlogit=dlogit, experts=exps, router_experts=rexps, dw_router=dw_router,
                dbias=dbias, dw_gate_up=dwgu, dw_down=dwd)
