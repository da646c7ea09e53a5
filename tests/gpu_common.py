"""Helpers shared by the GPU parity tests: the error metric and small builders.
No step of the layer's arithmetic lives here."""
import numpy as np
import torch

TOL = {"f32": 1e-5, "bf16": 2e-2, "mxfp8": 6e-2}   # max per-row relative error vs FP64
TIE_TAU = 1e-4                                      # logit gap below which FP32 may pick differently


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per row: max_h |got - ref| / max_h |ref|."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(got - ref).max(axis=1)
    den = np.abs(ref).max(axis=1)
    den[den == 0] = 1.0
    return num / den


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def need_cuda():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def check_routing(g_idx, ref_idx, ref_logits, gap, tau=TIE_TAU):
    """Routing of every token away from selection near-ties: the selected expert
    set equals the oracle's (unique), and the kernel's order is descending in the
    FP64 logits up to tau (the order of near-equal selected logits is not unique).
    Returns the fraction of tokens checked."""
    import numpy as np
    ok = gap >= tau
    np.testing.assert_array_equal(np.sort(g_idx[ok], axis=1), np.sort(ref_idx[ok], axis=1))
    lg = np.take_along_axis(ref_logits, g_idx.astype(np.int64), axis=1)
    assert np.all(np.diff(lg[ok], axis=1) <= tau)
    return ok.mean()
