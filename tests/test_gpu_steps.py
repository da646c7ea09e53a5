"""GPU parity of each step of the layer through the C ABI against the oracle:
MXFP8 quantisation, router top-k, layout, pull dispatch, expert FFN, combine."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import TIE_TAU, TOL, check_routing, need_cuda, row_rel_err, to_np
from token_dispatch_expert_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    need_cuda()
    from token_dispatch_expert_top_gb300 import moe
    return moe


def _ws(M, shape, params=None):
    ws = torch.empty(M.moe_workspace_bytes(shape, params), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    return ws


# ------------------------------------------------------------------------ quantise
def test_quantize_bit_exact_all_bf16_values(M):
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    rng = np.random.default_rng(0)
    rng.shuffle(f)
    pad = (-len(f)) % 32
    f = np.concatenate([f, np.zeros(pad, np.float32)]).reshape(-1, 32)
    x = torch.from_numpy(f).to(torch.bfloat16)
    codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty((x.shape[0], 1), dtype=torch.uint8, device="cuda")
    M.moe_quantize_mxfp8(x.cuda(), codes, scales)
    oc, os_ = O.quantize_mxfp8(x.float().numpy().astype(np.float64))
    np.testing.assert_array_equal(to_np(scales), os_)
    np.testing.assert_array_equal(to_np(codes), oc)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_bit_exact_mixed_magnitudes(M, dtype):
    rng = np.random.default_rng(1)
    rows, K = 333, 512
    v = rng.standard_normal((rows, K)) * np.exp2(rng.integers(-60, 60, size=(rows, K // 32)).repeat(32, 1))
    v[3, :32] = 0.0                       # zero block
    v[4, :32] = 1e-40                     # subnormal-only block (f32)
    v[5, 0] = 3e38                        # near the top of the range
    v[6, 5] = -500.0                      # saturating element
    x = torch.from_numpy(v.astype(np.float32)).to(dtype)
    codes = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    M.moe_quantize_mxfp8(x.cuda(), codes, scales)
    oc, os_ = O.quantize_mxfp8(x.float().numpy().astype(np.float64))
    np.testing.assert_array_equal(to_np(scales), os_)
    np.testing.assert_array_equal(to_np(codes), oc)


# -------------------------------------------------------------------------- router
ROUTE_CASES = [
    synth.WORKLOADS["tiny_f32"],
    synth.WORKLOADS["small_bf16"],
    synth.Workload("route_skew", N=1024, H=512, I=128, E=64, k=8, S=4, dtype="bf16", skew=3.0),
    synth.Workload("route_e256", N=640, H=256, I=128, E=256, k=8, S=5, dtype="mxfp8"),
    # 48-expert halves of the pair's partial logits (three 16-column loads each),
    # ragged last token tile
    synth.Workload("route_e96", N=257, H=512, I=128, E=96, k=6, S=1, dtype="mxfp8"),
    synth.Workload("route_e64_bf16", N=300, H=256, I=128, E=64, k=4, S=3, dtype="bf16"),
    # k > 8: the 16- and 32-entry top-k lists (two column ranges per quarter for k > 16)
    synth.Workload("route_k12", N=384, H=512, I=128, E=256, k=12, S=3, dtype="bf16"),
    synth.Workload("route_k20", N=200, H=512, I=128, E=128, k=20, S=1, dtype="mxfp8"),
]


@pytest.mark.parametrize("w", ROUTE_CASES, ids=lambda w: w.name)
def test_route_topk(M, w):
    inp = synth.make_inputs(w, device="cpu", with_weights=False)
    shape = M.Shape.of(w)
    x, wr = inp["x"].cuda(), inp["w_router"].cuda()
    bias = None if inp["bias"] is None else inp["bias"].cuda()
    idx = torch.empty((w.N, w.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((w.N, w.k), dtype=torch.float32, device="cuda")
    logits = torch.empty((w.N, w.E), dtype=torch.float32, device="cuda")
    M.moe_route_topk(x, wr, bias, shape, idx, gate, logits)
    g_logits, g_idx, g_gate = to_np(logits).astype(np.float64), to_np(idx), to_np(gate)
    # (i) the selection on the kernel's own FP32 logits is the oracle's, bit for bit
    o_idx, o_gate = O.route_topk(g_logits, w.k)
    np.testing.assert_array_equal(g_idx, o_idx)
    np.testing.assert_allclose(g_gate, o_gate, rtol=2e-6, atol=1e-7)
    # (ii) logits close to the FP64 oracle; indices equal away from near-ties
    ref = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    assert np.abs(g_logits - ref).max() < 1e-4 * max(1.0, np.abs(ref).max())
    r_idx, _ = O.route_topk(ref, w.k)
    assert check_routing(g_idx, r_idx, ref, O.topk_gap(ref, w.k)) > 0.98


@pytest.mark.parametrize("N,H,E,k", [(640, 512, 256, 8), (200, 1024, 32, 4), (8192, 7168, 256, 8),
                                     (257, 512, 96, 6)])
def test_route_topk_fused_x_quantisation_bit_exact(M, N, H, E, k):
    """The MXFP8 copy of x written by the router pass equals the oracle's quantiser."""
    w = synth.Workload("route_xq", N=N, H=H, I=128, E=E, k=k, S=N // 8 if N % 8 == 0 else 1,
                       dtype="mxfp8")
    inp = synth.make_inputs(w, device="cpu", with_weights=False)
    shape = M.Shape.of(w)
    idx = torch.empty((N, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((N, k), dtype=torch.float32, device="cuda")
    xq = torch.empty((N, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((N, H // 32), dtype=torch.uint8, device="cuda")
    M.moe_route_topk(inp["x"].cuda(), inp["w_router"].cuda(), None, shape, idx, gate, None, xq, xs)
    oc, os_ = O.quantize_mxfp8(O._f64(inp["x"]))
    np.testing.assert_array_equal(to_np(xs), os_)
    np.testing.assert_array_equal(to_np(xq), oc)
    # Repeated under concurrent HBM traffic from another stream, which reorders the
    # completion of the kernel's stage loads: the codes never change.
    x_d, wr_d = inp["x"].cuda(), inp["w_router"].cuda()
    noise = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    first_q, first_s = xq.clone(), xs.clone()
    for rep in range(12):
        with torch.cuda.stream(side):
            noise.fill_(rep)
        xq.zero_()
        xs.zero_()
        M.moe_route_topk(x_d, wr_d, None, shape, idx, gate, None, xq, xs)
        torch.cuda.synchronize()
        assert torch.equal(xq, first_q) and torch.equal(xs, first_s), rep


# -------------------------------------------------------------------------- layout
def _layout_case(M, idx_np, E, S):
    N, k = idx_np.shape
    w = synth.Workload("layout", N=N, H=256, I=128, E=E, k=k, S=S, dtype="bf16")
    shape = M.Shape.of(w)
    ws = _ws(M, shape)
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sched = torch.empty((N * k, 2), dtype=torch.int32, device="cuda")
    inv = torch.empty((N, k), dtype=torch.int32, device="cuda")
    M.moe_layout(idx, shape, counts, offsets, sched, inv, ws)
    assert M.moe_last_device_status(ws) == 0
    oc, oo, osch, oinv = O.layout(idx_np.astype(np.int32), E, S)
    np.testing.assert_array_equal(to_np(counts), oc)
    np.testing.assert_array_equal(to_np(offsets), oo)
    np.testing.assert_array_equal(to_np(sched), osch)
    np.testing.assert_array_equal(to_np(inv), oinv)


@pytest.mark.parametrize("N,E,k,S", [(64, 8, 2, 2), (4096, 64, 6, 8), (8192, 256, 8, 64),
                                     (1000, 33, 5, 10), (37, 4, 4, 1), (300, 1, 1, 3)])
def test_layout_bit_exact_random(M, N, E, k, S):
    rng = np.random.default_rng(N + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)])
    _layout_case(M, idx, E, S)


def test_layout_bit_exact_hot_and_empty_experts(M):
    rng = np.random.default_rng(5)
    N, E, k = 3000, 128, 4
    idx = np.empty((N, k), dtype=np.int64)
    for n in range(N):
        idx[n] = np.concatenate([[7, 100], rng.choice([1, 2, 3, 120], size=2, replace=False)])
    _layout_case(M, idx, E, 6)


def test_layout_reports_out_of_range_expert(M):
    w = synth.Workload("bad", N=64, H=256, I=128, E=8, k=2, S=2, dtype="bf16")
    shape = M.Shape.of(w)
    ws = _ws(M, shape)
    idx = torch.zeros((64, 2), dtype=torch.int32, device="cuda")
    idx[:, 1] = 1
    idx[10, 1] = 8             # out of range: recorded, skipped, nothing written for it
    counts = torch.empty(8, dtype=torch.int32, device="cuda")
    offsets = torch.empty(9, dtype=torch.int32, device="cuda")
    sched = torch.zeros((128, 2), dtype=torch.int32, device="cuda")
    inv = torch.zeros((64, 2), dtype=torch.int32, device="cuda")
    M.moe_layout(idx, shape, counts, offsets, sched, inv, ws)
    assert M.moe_last_device_status(ws) == M.MOE_ERR_DEVICE_CHECK
    assert int(counts.sum()) == 127
    assert M.moe_last_device_status(ws) == 0        # reading resets it


# ------------------------------------------------------------------------ dispatch
# Rows of 16-byte multiples go through the bulk-copy kernel (slot order, or token
# order through inv); MXFP8 at H=256 has 8-byte scale rows and takes the
# vector-load kernel.
@pytest.mark.parametrize("token_order", [False, True], ids=["slot_order", "token_order"])
@pytest.mark.parametrize("dtype,H", [("f32", 128), ("bf16", 1024), ("mxfp8", 1024), ("mxfp8", 256)])
def test_dispatch_pull_rows_by_schedule(M, dtype, H, token_order):
    rng = np.random.default_rng(3)
    N, E, k, S = 512, 16, 4, 8
    w = synth.Workload("pull", N=N, H=H, I=128, E=E, k=k, S=S, dtype=dtype)
    shape = M.Shape.of(w)
    ws = _ws(M, shape)
    rows = N // S
    elem = {"f32": 4, "bf16": 2, "mxfp8": 1}[dtype]
    shards = [torch.randint(0, 256, (rows, H * elem), dtype=torch.uint8, device="cuda") for _ in range(S)]
    sc = [torch.randint(0, 256, (rows, H // 32), dtype=torch.uint8, device="cuda") for _ in range(S)]
    tab = torch.tensor([t.data_ptr() for t in shards], dtype=torch.int64, device="cuda")
    tab_sf = torch.tensor([t.data_ptr() for t in sc], dtype=torch.int64, device="cuda")
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    _, _, sched_np, inv_np = O.layout(idx, E, S)
    sched = torch.from_numpy(sched_np).cuda()
    inv = torch.from_numpy(inv_np).cuda() if token_order else None
    T = N * k
    R = 640                                  # ring smaller than T: slots wrap
    ring = torch.zeros((R, H * elem), dtype=torch.uint8, device="cuda")
    ring_sf = torch.zeros((R, H // 32), dtype=torch.uint8, device="cuda")
    mx = dtype == "mxfp8"
    begin, count = 1400, 600              # rows 1400..1999 wrap past R
    M.moe_dispatch_pull(tab, tab_sf if mx else None, shape, sched, inv, begin, count, ring,
                        ring_sf if mx else None, R, ws)
    assert M.moe_last_device_status(ws) == 0
    allrows = torch.cat(shards).cpu()
    allsf = torch.cat(sc).cpu()
    got, got_sf = ring.cpu(), ring_sf.cpu()
    written = set()
    for t in range(begin, begin + count):
        src = sched_np[t, 0] * rows + sched_np[t, 1]
        assert torch.equal(got[t % R], allrows[src])
        if mx:
            assert torch.equal(got_sf[t % R], allsf[src])
        written.add(t % R)
    untouched = [r for r in range(R) if r not in written]
    assert not got[untouched].any()                 # nothing outside the slot range


def test_dispatch_token_broadcast_checks_schedule_entries(M):
    """With inv, a token's row is read once for its k slots; a slot whose schedule
    entry names another row is skipped and reported, and every slot written gets
    exactly the row its own schedule entry names."""
    rng = np.random.default_rng(4)
    N, E, k, S, H = 256, 16, 4, 4, 1024
    w = synth.Workload("pullchk", N=N, H=H, I=128, E=E, k=k, S=S, dtype="bf16")
    shape = M.Shape.of(w)
    ws = _ws(M, shape)
    rows = N // S
    shards = [torch.randint(0, 256, (rows, 2 * H), dtype=torch.uint8, device="cuda") for _ in range(S)]
    tab = torch.tensor([t.data_ptr() for t in shards], dtype=torch.int64, device="cuda")
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    _, _, sched_np, inv_np = O.layout(idx, E, S)
    n_bad = 37
    t_bad = int(inv_np[n_bad, 2])                 # the token's third slot names another row
    sched_np = sched_np.copy()
    other = (n_bad + 100) % N
    sched_np[t_bad] = [other // rows, other % rows]
    T = N * k
    ring = torch.zeros((T, 2 * H), dtype=torch.uint8, device="cuda")
    M.moe_dispatch_pull(tab, None, shape, torch.from_numpy(sched_np).cuda(), torch.from_numpy(inv_np).cuda(),
                        0, T, ring, None, T, ws)
    assert M.moe_last_device_status(ws) == M.MOE_ERR_DEVICE_CHECK
    allrows = torch.cat(shards).cpu()
    got = ring.cpu()
    for t in range(T):
        if t == t_bad:
            assert not got[t].any()
        else:
            src = sched_np[t, 0] * rows + sched_np[t, 1]
            assert torch.equal(got[t], allrows[src])


# ------------------------------------------------------------------------- combine
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_combine_matches_oracle(M, dtype):
    rng = np.random.default_rng(4)
    N, H, k = 300, 512, 6
    w = synth.Workload("comb", N=N, H=H, I=128, E=16, k=k, S=3, dtype=dtype)
    shape = M.Shape.of(w)
    ws = _ws(M, shape)
    T = N * k
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    y = torch.randn((T, H), dtype=torch.float32).to(tdt)
    inv = torch.from_numpy(rng.permutation(T).reshape(N, k).astype(np.int32))
    g = rng.random((N, k)).astype(np.float32)
    g /= g.sum(1, keepdims=True)
    gate = torch.from_numpy(g)
    out = torch.empty((N, H), dtype=tdt, device="cuda")
    M.moe_combine(y.cuda(), inv.cuda(), gate.cuda(), shape, out, ws)
    ref = O.combine(to_np(y).astype(np.float64), inv.numpy(), g.astype(np.float64))
    ref = O.round_to(ref, dtype)
    err = row_rel_err(to_np(out), ref)
    assert err.max() < (2e-6 if dtype == "f32" else 8e-3)


# -------------------------------------------------------------------- weight packing
def _expected_pack(w, rows_fn, NT, KB):
    """Tile images by definition: tile (e, n, kb) row r = weight row rows_fn(n, r),
    K bytes [128 kb, 128 kb + 128); chunk c of row r stored at chunk c ^ (r % 8)."""
    E = w.shape[0]
    out = np.empty((E, NT, KB, 256, 8, 16), dtype=np.uint8)
    for n in range(NT):
        src_rows = np.array([rows_fn(n, r) for r in range(256)])
        blk = w[:, src_rows, :].reshape(E, 256, KB, 8, 16)          # [E][r][kb][c][16]
        for r in range(256):
            perm = np.arange(8) ^ (r & 7)                               # position p holds chunk p ^ (r%8)
            out[:, n, :, r, :, :] = blk[:, r][:, :, perm, :]
    return out.reshape(-1)


def _expected_pack_sf(sf, rows_fn, NT, KB):
    E = sf.shape[0]
    out = np.empty((E, NT, KB, 2, 32, 4, 4), dtype=np.uint8)         # [..][half][lane][j][q]
    for n in range(NT):
        for half in range(2):
            for j in range(4):
                src_rows = np.array([rows_fn(n, 128 * half + 32 * j + lane) for lane in range(32)])
                v = sf[:, src_rows, :].reshape(E, 32, KB, 4)             # [E][lane][kb][q]
                out[:, n, :, half, :, j, :] = v.transpose(0, 2, 1, 3)
    return out.reshape(-1)


@pytest.mark.parametrize("dtype", ["mxfp8", "bf16"])
def test_pack_expert_weights_layout(M, dtype):
    from token_dispatch_expert_top_gb300.layer import pack_expert_weights
    E, H, I = 2, 512, 256
    w = synth.Workload("pack", N=8, H=H, I=I, E=E, k=1, S=1, dtype=dtype)
    shape = M.Shape.of(w)
    esz = 1 if dtype == "mxfp8" else 2
    g = torch.Generator().manual_seed(3)
    wgu = torch.randint(0, 256, (E, 2 * I, H * esz), generator=g, dtype=torch.uint8)
    wd = torch.randint(0, 256, (E, H, I * esz), generator=g, dtype=torch.uint8)
    sgu = torch.randint(0, 256, (E, 2 * I, H // 32), generator=g, dtype=torch.uint8) if esz == 1 else None
    sd = torch.randint(0, 256, (E, H, I // 32), generator=g, dtype=torch.uint8) if esz == 1 else None
    dev = lambda t: None if t is None else t.cuda()
    p_gu, p_gu_sf, p_d, p_d_sf = pack_expert_weights(shape, dev(wgu), dev(sgu), dev(wd), dev(sd))
    rows1 = lambda n, r: n * 128 + r if r < 128 else I + n * 128 + (r - 128)
    rows2 = lambda n, r: n * 256 + r
    np.testing.assert_array_equal(to_np(p_gu).reshape(-1),
                                  _expected_pack(wgu.numpy(), rows1, I // 128, H * esz // 128))
    np.testing.assert_array_equal(to_np(p_d).reshape(-1),
                                  _expected_pack(wd.numpy(), rows2, H // 256, I * esz // 128))
    if esz == 1:
        np.testing.assert_array_equal(to_np(p_gu_sf).reshape(-1),
                                      _expected_pack_sf(sgu.numpy(), rows1, I // 128, H // 128))
        np.testing.assert_array_equal(to_np(p_d_sf).reshape(-1),
                                      _expected_pack_sf(sd.numpy(), rows2, H // 256, I // 128))


# ---------------------------------------------------------------------- expert FFN
FFN_CASES = [
    ("f32", 128, 256, [0, 3, 40, 85]),
    ("bf16", 512, 256, [0, 1, 130, 255, 300]),
    ("mxfp8", 512, 256, [0, 1, 130, 255, 300]),
    ("bf16", 2048, 1408, [200, 0, 383, 129, 257, 1, 640, 128]),
    ("mxfp8", 2048, 1408, [200, 0, 383, 129, 257, 1, 640, 128]),
    ("mxfp8", 7168, 2048, [37, 0, 256, 129]),
    # ragged last m-tiles of every size class: 1, 31, 32 (a 32-row A box), 33 and more
    # (the 128-row box), full tiles, empty experts
    ("mxfp8", 512, 256, [160, 161, 288, 289, 129, 32, 31, 0, 1, 401, 128, 256]),
    ("bf16", 512, 256, [160, 161, 288, 289, 129, 32, 31, 0, 1, 401, 128, 256]),
    ("mxfp8", 7168, 2048, [160, 272, 257, 33]),
]


@pytest.mark.parametrize("dtype,H,I,counts", FFN_CASES,
                         ids=[f"{c[0]}-H{c[1]}-I{c[2]}-E{len(c[3])}" for c in FFN_CASES])
def test_expert_ffn_matches_oracle(M, dtype, H, I, counts):
    E = len(counts)
    T = sum(counts)
    # a shape whose T = N*k equals the slot count: k = 1, N = T
    w = synth.Workload("ffn", N=T, H=H, I=I, E=E, k=1, S=1, dtype=dtype)
    shape = M.Shape.of(w)
    ws = _ws(M, shape)
    g = torch.Generator().manual_seed(7)
    master = torch.float32 if dtype == "f32" else torch.bfloat16
    a = torch.randn((T, H), generator=g).to(master)
    wgu = (torch.randn((E, 2 * I, H), generator=g) / H ** 0.5).to(master)
    wd = (torch.randn((E, H, I), generator=g) / I ** 0.5).to(master)
    offsets_np = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    offsets = torch.from_numpy(offsets_np).cuda()
    y = torch.empty((T, H), dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device="cuda")
    from token_dispatch_expert_top_gb300.layer import pack_expert_weights, quantize_mxfp8
    if dtype == "mxfp8":
        a_c, a_s = quantize_mxfp8(a.cuda())
        packed = pack_expert_weights(shape, *quantize_mxfp8(wgu.cuda()), *quantize_mxfp8(wd.cuda()))
        M.moe_expert_ffn(a_c, a_s, offsets, *packed[:2], *packed[2:], shape, y, ws)
    else:
        packed = pack_expert_weights(shape, wgu.cuda(), None, wd.cuda(), None)
        M.moe_expert_ffn(a.cuda(), None, offsets, packed[0], None, packed[2], None, shape, y, ws)
    assert M.moe_last_device_status(ws) == 0
    got = to_np(y)
    a64 = O._f64(a)
    if dtype == "mxfp8":
        a64 = O.mxfp8_values(a64)
    for e in range(E):
        lo, hi = offsets_np[e], offsets_np[e + 1]
        if lo == hi:
            continue
        wg, wu, wdd = O.expert_operands(wgu[e], wd[e], dtype)
        ref = O.expert_ffn(a64[lo:hi], wg, wu, wdd, dtype)
        err = row_rel_err(got[lo:hi], ref)
        assert err.max() < TOL[dtype], (e, err.max())

