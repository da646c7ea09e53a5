"""GPU parity of the NVFP4 quantiser through the C ABI against the oracle:
E2M1 codes, E4M3 block scales and the FP32 tensor scale, bit-exact."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import need_cuda, to_np
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe
    return moe


def _run(M, x: torch.Tensor):
    rows, K = x.shape
    codes = torch.full((rows, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows, K // 16), 0xAB, dtype=torch.uint8, device="cuda")
    st = torch.full((2,), -1.0, dtype=torch.float32, device="cuda")
    M.moe_quantize_nvfp4(x, codes, scales, st)
    torch.cuda.synchronize()
    return codes, scales, st


def _check(M, x: torch.Tensor):
    codes, scales, st = _run(M, x.cuda())
    ref = x.float().cpu().numpy().astype(np.float64)
    oc, os_, ost = O.quantize_nvfp4(ref)
    assert float(st[0]) == ost
    assert float(st[1]) == np.abs(ref).max()
    np.testing.assert_array_equal(to_np(scales), os_)
    np.testing.assert_array_equal(to_np(codes), oc)
    return oc, os_


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_nvfp4_bit_exact_mixed_magnitudes(M, dtype):
    """Block magnitudes spread over E4M3's normal and subnormal scale range, a ragged
    row count, zero blocks, an underflowing row, negative zeros."""
    rng = np.random.default_rng(5)
    rows, K = 333, 272                  # 17 blocks of 16 per row
    v = rng.standard_normal((rows, K)) * np.exp2(rng.integers(-14, 1, size=(rows, K // 16)).repeat(16, 1))
    v[3, :16] = 0.0                     # zero block
    v[4] *= 1e-9                        # block scales underflow to zero
    v[5, 16:32] = -0.0                  # negative-zero block
    v[6, 40] = 50.0                     # the tensor amax
    x = torch.from_numpy(v.astype(np.float32)).to(dtype)
    oc, os_ = _check(M, x)
    assert (os_[4] == 0).all() and (os_ > 0).mean() > 0.9


def test_nvfp4_bit_exact_on_ties(M):
    """Elements that land exactly halfway between E2M1 values round to even: the
    tensor amax is 24 = 6 * 4, so the top block's scale unit is exactly 4.  A row
    scaled by 0.9999999 sits just below the ties."""
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    row = np.concatenate([[6.0], ties, [-0.0], -ties])
    v = np.stack([row * 4.0, row * 0.5, row * 4.0 * 0.9999999]).astype(np.float32)
    oc, _ = _check(M, torch.from_numpy(v))
    lo, hi = oc[0] & 15, oc[0] >> 4
    # 6, .25, .75, 1.25 | 1.75, 2.5, 3.5, 5 -> 6, 0, 1, 1 | 2, 2, 4, 4 (codes 7 0 2 2 4 4 6 6)
    assert list(lo[:4]) == [7, 2, 4, 6] and list(hi[:4]) == [0, 2, 4, 6]
    assert list(lo[4:]) == [8, 10, 12, 14] and list(hi[4:]) == [8, 10, 12, 14]


def test_nvfp4_bit_exact_all_bf16_values(M):
    """Every finite BF16 value, shuffled into blocks of 16 (most block scales
    underflow against the largest BF16 tensor amax), and the same values folded
    into two binades of the amax."""
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    rng = np.random.default_rng(0)
    rng.shuffle(f)
    f = np.concatenate([f, np.zeros((-len(f)) % 16, np.float32)]).reshape(-1, 16)
    _check(M, torch.from_numpy(f).to(torch.bfloat16))
    m, e = np.frexp(f.astype(np.float64))
    folded = np.ldexp(m, np.mod(e, 2)).astype(np.float32)   # mantissas kept, exponents in {0, 1}
    _check(M, torch.from_numpy(folded).to(torch.bfloat16))


def test_nvfp4_shapes_and_empty(M):
    _check(M, torch.randn(1, 16))
    _check(M, torch.zeros(7, 48, dtype=torch.bfloat16))
    codes = torch.empty(0, dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.float32, device="cuda")
    M.moe_quantize_nvfp4(torch.empty((0, 64), device="cuda"), codes, codes, st)
    torch.cuda.synchronize()
    assert st.tolist() == [1.0, 0.0]


def test_nvfp4_full_size_activations_and_one_expert(M):
    """The 8192 x 7168 BF16 token matrix of the DeepSeek-V3-shaped layer and one
    expert's [4096][7168] gate/up weights."""
    w = synth.WORKLOADS["dsv3_mxfp8"]
    inp = synth.make_inputs(w, device="cuda", with_weights=False)
    _check(M, inp["x"])
    gen = torch.Generator(device="cuda").manual_seed(7)
    wgu = (torch.randn((2 * w.I, w.H), generator=gen, device="cuda") / w.H ** 0.5).to(torch.bfloat16)
    _check(M, wgu)
