"""Device-side plumbing around the C ABI: holds a layer's device tensors (weights
quantised once by libmoe for the MXFP8 dtype), its workspace, and calls
moe_forward / moe_forward_fused.  PyTorch only allocates memory and supplies the
stream here; every step of the layer runs in libmoe's kernels."""
from __future__ import annotations

import torch

from . import moe as M
from .synth import Workload, master_dtype


def pack_expert_weights(shape, wgu, wgu_sf, wd, wd_sf):
    """Tile-packed copies of the expert weights (and scales), made by libmoe."""
    p_gu = torch.empty_like(wgu)
    p_d = torch.empty_like(wd)
    p_gu_sf = None if wgu_sf is None else torch.empty_like(wgu_sf)
    p_d_sf = None if wd_sf is None else torch.empty_like(wd_sf)
    M.moe_pack_expert_weights(shape, wgu, wgu_sf, wd, wd_sf, p_gu, p_gu_sf, p_d, p_d_sf)
    return p_gu, p_gu_sf, p_d, p_d_sf


def quantize_mxfp8(t: torch.Tensor):
    """MXFP8 codes and scales of t along its last axis, made by libmoe."""
    K = t.shape[-1]
    codes = torch.empty(t.shape, dtype=torch.uint8, device=t.device)
    scales = torch.empty(t.shape[:-1] + (K // 32,), dtype=torch.uint8, device=t.device)
    M.moe_quantize_mxfp8(t.contiguous(), codes, scales)
    return codes, scales


def pack_expert_weights_dgrad(shape, wgu: torch.Tensor, wd: torch.Tensor):
    """Transposed tile-packed copies of the BF16 master weights for the backward's
    dgrad GEMMs (MXFP8-quantised along their new K for the MXFP8 dtype), made by
    libmoe.  Returns (gate_up_t, gate_up_t_scales, down_t, down_t_scales)."""
    mx = shape.dtype == M.MOE_MXFP8
    E, H, I = shape.E, shape.H, shape.I
    Ip = (I + 255) // 256 * 256
    esz = 1 if mx else 2
    dev = wgu.device
    p_gu = torch.empty(E * H * 2 * I * esz, dtype=torch.uint8, device=dev)
    p_d = torch.empty(E * Ip * H * esz, dtype=torch.uint8, device=dev)
    p_gu_sf = torch.empty(E * H * 2 * I // 32, dtype=torch.uint8, device=dev) if mx else None
    p_d_sf = torch.empty(E * Ip * H // 32, dtype=torch.uint8, device=dev) if mx else None
    M.moe_pack_expert_weights_dgrad(shape, wgu.contiguous(), wd.contiguous(), p_gu, p_gu_sf, p_d,
                                    p_d_sf)
    return p_gu, p_gu_sf, p_d, p_d_sf


class MoeLayer:
    def __init__(self, w: Workload, inputs: dict, params: M.Params | None = None,
                 device: str = "cuda", keep_master: bool = False, train: bool = False):
        self.w = w
        self.shape = M.Shape.of(w)
        self.params = params
        dev = torch.device(device)
        self.x = inputs["x"].to(dev).contiguous()
        self.w_router = inputs["w_router"].to(dev).contiguous()
        self.bias = None if inputs.get("bias") is None else inputs["bias"].to(dev).float().contiguous()
        wgu = inputs["w_gate_up"].to(dev).contiguous()
        wd = inputs["w_down"].to(dev).contiguous()
        if w.dtype == "mxfp8":
            q_gu, q_gu_sf = quantize_mxfp8(wgu)
            q_d, q_d_sf = quantize_mxfp8(wd)
        else:
            q_gu, q_gu_sf, q_d, q_d_sf = wgu, None, wd, None
        self.wgu, self.wgu_sf, self.wd, self.wd_sf = pack_expert_weights(
            self.shape, q_gu, q_gu_sf, q_d, q_d_sf)
        del q_gu, q_gu_sf, q_d, q_d_sf
        self.train = train
        if train:
            self.wgu_t, self.wgu_t_sf, self.wd_t, self.wd_t_sf = pack_expert_weights_dgrad(
                self.shape, wgu, wd)
            T = w.T
            i32 = torch.int32
            self.saved = {
                "idx": torch.empty((w.N, w.k), dtype=i32, device=dev),
                "gate": torch.empty((w.N, w.k), dtype=torch.float32, device=dev),
                "inv": torch.empty((w.N, w.k), dtype=i32, device=dev),
                "offsets": torch.empty(w.E + 1, dtype=i32, device=dev),
                "sched": torch.empty((T, 2), dtype=i32, device=dev),
                "y": torch.empty((T, w.H), dtype=torch.bfloat16, device=dev),
                "uv": torch.empty((T, 2 * w.I), dtype=torch.bfloat16, device=dev),
            }
            self.saved_c = M.Saved.of(self.saved)
            self.bws = torch.empty(M.moe_backward_workspace_bytes(self.shape), dtype=torch.uint8,
                                   device=dev)
            M.moe_workspace_init(self.bws)
            self.dx = torch.empty((w.N, w.H), dtype=torch.bfloat16, device=dev)
            self.dw_router = torch.empty((w.E, w.H), dtype=torch.float32, device=dev)
            self.dbias = torch.empty(w.E, dtype=torch.float32, device=dev)
            self.dw_gate_up = torch.empty((w.E, 2 * w.I, w.H), dtype=torch.bfloat16, device=dev)
            self.dw_down = torch.empty((w.E, w.H, w.I), dtype=torch.bfloat16, device=dev)
        if keep_master:
            self.master = (wgu, wd)
        else:
            del wgu, wd
        nbytes = M.moe_workspace_bytes(self.shape, params)
        if nbytes == 0:
            raise M.MoeError("moe_workspace_bytes", M.MOE_ERR_INVALID_ARG)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        M.moe_workspace_init(self.ws)
        out_dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.out = torch.empty((w.N, w.H), dtype=out_dt, device=dev)
        self.idx = torch.empty((w.N, w.k), dtype=torch.int32, device=dev)
        self.gate = torch.empty((w.N, w.k), dtype=torch.float32, device=dev)

    def forward(self, x: torch.Tensor | None = None, fused: bool = False, params=None,
                out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None):
        """One forward layer, enqueued on `stream` (default: torch's current stream)."""
        fn = M.moe_forward_fused if fused else M.moe_forward
        fn(self.x if x is None else x, self.w_router, self.bias, self.wgu, self.wgu_sf, self.wd,
           self.wd_sf, self.shape, params if params is not None else self.params,
           self.out if out is None else out, self.idx, self.gate, self.ws, stream)
        return self.out if out is None else out

    def forward_macrobatched(self, macrobatches: int, x: torch.Tensor | None = None,
                             out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None):
        """The forward in `macrobatches` macrobatches (moe_forward_macrobatched), on a
        workspace of one slice per macrobatch, kept between calls."""
        if getattr(self, "macro_n", None) != macrobatches:
            nbytes = M.moe_macro_workspace_bytes(self.shape, self.params, macrobatches)
            if nbytes == 0:
                raise M.MoeError("moe_macro_workspace_bytes", M.MOE_ERR_INVALID_ARG)
            self.macro_ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.out.device)
            off = (-self.macro_ws.data_ptr()) % 256            # 256-byte aligned slices
            self.macro_ws = self.macro_ws[off:off + nbytes]
            self.macro_slice = nbytes // macrobatches
            for m in range(macrobatches):
                M.moe_workspace_init(self.macro_ws[m * self.macro_slice:(m + 1) * self.macro_slice])
            self.macro_n = macrobatches
        M.moe_forward_macrobatched(self.x if x is None else x, self.w_router, self.bias, self.wgu,
                                   self.wgu_sf, self.wd, self.wd_sf, self.shape, self.params, macrobatches,
                                   self.out if out is None else out, self.macro_ws, stream)
        return self.out if out is None else out

    def device_status(self) -> int:
        status = M.moe_last_device_status(self.ws)
        for m in range(getattr(self, "macro_n", 0) or 0):
            s = M.moe_last_device_status(self.macro_ws[m * self.macro_slice:(m + 1) * self.macro_slice])
            status = status or s
        return status

    def forward_train(self, x: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      stream: torch.cuda.Stream | None = None):
        """The staged forward, keeping the activations the backward needs."""
        M.moe_forward_train(self.x if x is None else x, self.w_router, self.bias, self.wgu,
                            self.wgu_sf, self.wd, self.wd_sf, self.shape, self.params,
                            self.out if out is None else out, self.saved_c, self.ws, stream)
        return self.out if out is None else out

    def backward(self, dout: torch.Tensor, x: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None, weights: bool = True):
        """Gradients of the last forward_train: (dx, dW_router, dbias, dW_gate_up,
        dW_down); the expert weight gradients are skipped (None) when not `weights`."""
        M.moe_backward(dout, self.x if x is None else x, self.w_router, self.saved_c, self.wgu_t,
                       self.wgu_t_sf, self.wd_t, self.wd_t_sf, self.shape, self.params, self.dx,
                       self.dw_router, self.dbias, self.dw_gate_up if weights else None,
                       self.dw_down if weights else None, self.bws, stream)
        if not weights:
            return self.dx, self.dw_router, self.dbias, None, None
        return self.dx, self.dw_router, self.dbias, self.dw_gate_up, self.dw_down

    def backward_status(self) -> int:
        return M.moe_last_device_status(self.bws)
