"""Pins of the axis along which the oracle's MXFP8 backward quantises each GEMM operand.

The layer's configuration makes every expert GEMM an MXFP8 GEMM: each operand is
quantised in blocks of 32 along that GEMM's reduction axis.  In the backward those
axes are
  * dgrad, token side: dy along H (dh = dy . W_down), du and dv along I
    (da = du . W_gate + dv . W_up), every slot row on its own;
  * dgrad, weight side: W_gate_up down its 2I rows, W_down down its H rows;
  * wgrad: every operand along the expert's slots (dW = X^T Y sums over slots).

Two kinds of input pin the axis without re-deriving the quantiser:
  * matrices built so that every 32-block along the intended axis is exactly
    representable (E4M3 values times a power of two the block shares, one element
    in the top binade) while the power of two jumps by up to 2^20 along the other
    axis: quantising along the intended axis must leave them unchanged, and the
    test checks that quantising along the other axis would not;
  * one hand-worked block, from the E4M3 definition (three mantissa bits, smallest
    subnormal 2^-9) and the MX scale rule (scale = 2^(floor(log2 amax) - 8)):
      along the intended axis the block is [2, 1.0625]: amax 2 gives scale 2^-7,
      1.0625 * 2^7 = 136 lies half way between the E4M3 neighbours 128 and 144 and
      goes to the even one, 128, so the element reads back as 1.0;
      along the other axis the element shares a block with 2^20: scale 2^12,
      1.0625 * 2^-12 is below half of 2^-9 and reads back as 0;
      kept in BF16 (not MXFP8) it stays 1.0625.
    Each of the three outcomes differs, so the expected 1.0 tells a wrong axis and
    a missing quantisation apart from the right one.
The identity-like weights and one-hot operands below turn each GEMM into a
selection, so every gradient entry is one quantised operand entry.
"""
import numpy as np
import pytest
import torch

import oracle as O


def _e4m3_magnitudes():
    """The positive finite E4M3 values, decoded by torch's float8_e4m3fn."""
    codes = torch.arange(1, 0x7F, dtype=torch.uint8)           # 0x7F is NaN
    vals = codes.view(torch.float8_e4m3fn).double().numpy()
    return vals[vals > 0]


def _representable_along(rows, cols, axis, seed, spread=20):
    """rows x cols values whose MXFP8 blocks of 32 along `axis` (0: down the rows of
    each column, 1: along each row) are exactly representable: an E4M3 value times
    2^g, g shared by the block and drawn from [-spread, spread], with one element per
    block forced into the top binade [256, 448] so that the block's scale is 2^g."""
    rng = np.random.default_rng(seed)
    mags = _e4m3_magnitudes()
    top = mags[(mags >= 256) & (mags <= 448)]
    if axis == 1:
        return np.ascontiguousarray(_representable_along(cols, rows, 0, seed, spread).T)
    nb = -(-rows // 32)
    c = rng.choice(mags, size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
    for b in range(nb):
        r0, r1 = 32 * b, min(rows, 32 * b + 32)
        at = rng.integers(r0, r1, size=cols)
        c[at, np.arange(cols)] = rng.choice(top, size=cols) * rng.choice([-1.0, 1.0], size=cols)
    g = rng.integers(-spread, spread + 1, size=(nb, cols))
    return c * np.exp2(np.repeat(g, 32, axis=0)[:rows])


def _along_rows(m):
    return O.mxfp8_values(np.ascontiguousarray(m))


def _along_cols(m):
    return np.ascontiguousarray(O.mxfp8_values(np.ascontiguousarray(m.T)).T)


def test_constructed_blocks_discriminate_the_axis():
    """The inputs below have teeth: exact along their axis, changed along the other."""
    for axis, same, other in ((0, _along_cols, _along_rows), (1, _along_rows, _along_cols)):
        m = _representable_along(64, 96, axis, seed=axis)
        np.testing.assert_array_equal(same(m), m)
        assert np.mean(other(m) != m) > 0.3
    # bf16-exact too (E4M3 significands have 4 bits), so no other rounding point moves them
    m = _representable_along(64, 96, 1, seed=3)
    np.testing.assert_array_equal(O.round_bf16(m), m)


def _hand_block(rows, cols, along_rows):
    """The hand-worked block: [2, 1.0625] along the intended axis, 2^20 beside
    1.0625 along the other; returns (input, expected after quantising along the
    intended axis)."""
    m = np.zeros((rows, cols))
    if along_rows:               # blocks along each row
        m[1, 0], m[1, 1], m[0, 1] = 2.0, 1.0625, 2.0 ** 20
        q = m.copy()
        q[1, 1] = 1.0
    else:                        # blocks down each column
        m[0, 1], m[1, 1], m[1, 0] = 2.0, 1.0625, 2.0 ** 20
        q = m.copy()
        q[1, 1] = 1.0
    return m, q


def test_hand_block_reads_back_as_worked_out():
    m, q = _hand_block(32, 32, along_rows=True)
    np.testing.assert_array_equal(_along_rows(m), q)
    assert _along_cols(m)[1, 1] == 0.0 and O.round_bf16(m)[1, 1] == 1.0625


# ------------------------------------------------------------------ dgrad weights
def test_dgrad_weights_are_quantised_down_their_reduction_axis():
    """expert_operands_dgrad: W_gate_up [2I, H] in blocks down its 2I rows (dgrad
    reduces over I), W_down [H, I] in blocks down its H rows."""
    H, I = 96, 64
    wgu = _representable_along(2 * I, H, 0, seed=10)
    wd = _representable_along(H, I, 0, seed=11)
    wg, wu, wdd = O.expert_operands_dgrad(wgu, wd, "mxfp8")
    np.testing.assert_array_equal(wg, wgu[:I])
    np.testing.assert_array_equal(wu, wgu[I:])
    np.testing.assert_array_equal(wdd, wd)
    # the hand-worked block, once in W_gate (rows 0..31), once in W_up, once in W_down
    for which in range(3):
        m, q = _hand_block(32, 32, along_rows=False)
        wgu = np.zeros((2 * I, H))
        wd = np.zeros((H, I))
        if which == 0:
            wgu[:32, :32] = m
        elif which == 1:
            wgu[I:I + 32, :32] = m
        else:
            wd[:32, :32] = m
        wg, wu, wdd = O.expert_operands_dgrad(wgu, wd, "mxfp8")
        got = (wg[:32, :32], wu[:32, :32], wdd[:32, :32])[which]
        np.testing.assert_array_equal(got, q)


# ------------------------------------------------------------------ dgrad token side
def _dgrad_selectors(H, I):
    """Weights that make dh = dy[:, :I] and da = [du_q | dv_q] (H = 2I)."""
    wd_b = np.zeros((H, I))
    wd_b[np.arange(I), np.arange(I)] = 1.0
    wg_b = np.zeros((I, H))
    wg_b[np.arange(I), np.arange(I)] = 1.0
    wu_b = np.zeros((I, H))
    wu_b[np.arange(I), I + np.arange(I)] = 1.0
    return wg_b, wu_b, wd_b


@pytest.mark.parametrize("case", ["random", "hand"])
def test_dgrad_dy_is_quantised_along_H_per_slot(case):
    """dh = dy_q . W_down: with W_down selecting dy's first I columns and the forward
    operands zero (so du = dv = 0), dh is exactly the quantised dy's columns."""
    P, I = 64, 32
    H = 2 * I
    if case == "random":
        dy = _representable_along(P, H, 1, seed=20)
        q = dy
    else:
        dy, q = _hand_block(P, H, along_rows=True)
    z = np.zeros
    r = O.expert_ffn_backward(z((P, H)), z((I, H)), z((I, H)), z((H, I)), dy, "mxfp8",
                              _dgrad_selectors(H, I), z((P, H)))
    np.testing.assert_array_equal(r["dh"], q[:, :I])


@pytest.mark.parametrize("case", ["random", "hand"])
def test_dgrad_du_dv_are_quantised_along_I_per_slot(case):
    """da = du_q . W_gate + dv_q . W_up.  The forward operand a makes u = 64 (where
    silu(u) = u and silu'(u) = 1 hold exactly in FP64) and v = V, and dy = 1 makes
    dh = 1; so du = V and dv = 64, and the selectors give da = [du_q | dv_q]."""
    P, I = 64, 32
    H = 2 * I
    if case == "random":
        V = _representable_along(P, I, 1, seed=30, spread=12)
        q = V
    else:
        V, q = _hand_block(P, I, along_rows=True)
    a = np.zeros((P, H))
    a[:, 0] = 64.0
    a[:, 1:1 + I] = V
    wg = np.zeros((I, H))
    wg[:, 0] = 1.0                      # u = 64
    wu = np.zeros((I, H))
    wu[np.arange(I), 1 + np.arange(I)] = 1.0   # v = V
    dy = np.zeros((P, H))
    dy[:, :I] = 1.0                     # dh = 1
    r = O.expert_ffn_backward(a, wg, wu, np.zeros((H, I)), dy, "mxfp8",
                              _dgrad_selectors(H, I), a)
    np.testing.assert_array_equal(r["du"], V)
    np.testing.assert_array_equal(r["da"][:, :I], q)
    np.testing.assert_array_equal(r["da"][:, I:], np.full((P, I), 64.0))


# ------------------------------------------------------------------ wgrad
@pytest.mark.parametrize("P", [64, 40])
@pytest.mark.parametrize("case", ["random", "hand"])
def test_wgrad_operands_are_quantised_along_the_slots(P, case):
    """dW_gate = du_q^T a_q, dW_up = dv_q^T a_q, dW_down = dy_q^T h_q, each operand
    quantised down the expert's slots.  One-hot partners turn each product into one
    operand: first a is the subject (du = dv = one-hot, h = one-hot), then du, dv and
    h are (a = dy = one-hot).  40 slots leave a partial second block."""
    H, I = 64, 32
    u = np.full((P, I), 64.0)           # silu(64) = 64 exactly, so h = 64 v
    eye_pi = np.eye(P, I)
    eye_ph = np.eye(P, H)

    def subject(cols, seed):
        if case == "random":
            m = _representable_along(P, cols, 0, seed=seed)
            return m, m
        m, q = _hand_block(P, cols, along_rows=False)
        return m, q

    A, Aq = subject(H, 40)
    dWg, dWu, dWd = O.expert_wgrad(A, eye_pi, eye_pi, A, u, eye_pi / 64.0, "mxfp8")
    n = min(P, I)
    np.testing.assert_array_equal(dWg[:n], O.round_bf16(Aq[:n]))
    np.testing.assert_array_equal(dWu[:n], O.round_bf16(Aq[:n]))
    np.testing.assert_array_equal(dWd[:, :n], O.round_bf16(Aq[:n].T))

    D, Dq = subject(I, 41)
    dWg, dWu, dWd = O.expert_wgrad(eye_ph, D, D, eye_ph, u, D / 64.0, "mxfp8")
    np.testing.assert_array_equal(dWg[:, :P], O.round_bf16(Dq.T))
    np.testing.assert_array_equal(dWu[:, :P], O.round_bf16(Dq.T))
    np.testing.assert_array_equal(dWd[:P], O.round_bf16(Dq))
