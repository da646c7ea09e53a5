// api.cu -- the extern "C" entry points declared in include/moe.h: argument
// checks, the workspace plan, and the launch sequences.  No function here
// allocates device memory or synchronises the host (except
// moe_last_device_status, whose job is to).
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

int num_sms_current() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

size_t act_elem(int dtype) { return dtype == MOE_F32 ? 4 : 2; }      // x, y, out
size_t op_elem(int dtype) { return dtype == MOE_F32 ? 4 : (dtype == MOE_BF16 ? 2 : 1); }  // GEMM operands

// Ring and minibatch geometry of the fused forward (moe_params_t resolved).
struct FusedGeom {
    int G, C;       // gather CTAs, compute CTAs
    int MB, R;      // slots per minibatch, ring slots (a multiple of MB)
    int nmb;        // bound on the minibatch count (every minibatch but the last holds >= MB/2 slots)
    int status;     // MOE_OK, or why these params cannot run
};

int num_sms_current();

FusedGeom resolve_fused(const moe_shape_t& s, const moe_params_t* p, int max_ctas) {
    FusedGeom g{};
    const int T = s.N * s.k;
    const int sms = num_sms_current();
    if (max_ctas <= 0) max_ctas = sms;
    // gather CTAs copy with the bulk-copy engine: ~1/25 of the SMs keeps up with the
    // expert FFN's consumption of slots (6 of 152 on a GB300)
    g.G = (p && p->gather_ctas > 0) ? p->gather_ctas : (sms >= 50 ? sms / 25 : 2);
    g.C = (p && p->compute_ctas > 0) ? p->compute_ctas : max_ctas - g.G;
    if (g.G < 1 || g.C < 1 || g.G + g.C > max_ctas) g.status = MOE_ERR_INVALID_ARG;
    const int Tp = T > 0 ? T : 1;
    if (p && p->minibatch > 0) {
        g.MB = p->minibatch;
    } else if (p && p->ring_slots > 0) {
        g.MB = p->ring_slots >= 64 ? p->ring_slots / 2 : p->ring_slots;
    } else {
        // four full waves of GEMM1 tiles over the compute SMs (the pages ask for at
        // least two; four measured faster), in whole 32-slot units
        const int waves = moe_min_minibatch(4, g.C > 0 ? g.C : 1, 128, 256, s.I);
        g.MB = ((waves + 31) / 32) * 32;
    }
    if (g.MB > Tp) g.MB = Tp;
    if (g.MB < 1) g.MB = 1;
    g.R = (p && p->ring_slots > 0) ? p->ring_slots : (4 * g.MB < Tp ? 4 * g.MB : ((Tp + g.MB - 1) / g.MB) * g.MB);
    if (g.R < g.MB || g.R % g.MB != 0) g.status = MOE_ERR_INVALID_ARG;
    g.nmb = T > 0 ? 2 * ((T + g.MB - 1) / g.MB) + 1 : 0;
    return g;
}

// Workspace regions, in order.  Every size depends only on the shape and params;
// one workspace serves both moe_forward and moe_forward_fused.
struct Plan {
    size_t header, cnt, base;               // layout scratch
    size_t idx, gate, counts, offsets, sched, inv;
    size_t xq, xq_sf, shard_tab, shard_sf_tab;
    size_t ring, ring_sf, h, h_sf, y, fused_ints;
    size_t total;
    int ring_slots;                         // rows of ring / h (>= T and >= the fused ring)
    FusedGeom fg;
};

Plan make_plan(const moe_shape_t& s, const moe_params_t* p) {
    const int64_t T = (int64_t)s.N * s.k;
    const int nch = layout_chunks((int)T);
    const bool mx = s.dtype == MOE_MXFP8;
    const FusedGeom fg = resolve_fused(s, p, 0);
    int R = (int)T > fg.R ? (int)T : fg.R;
    if (R < 1) R = 1;
    Plan pl{};
    pl.fg = fg;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align256(bytes);
        return o;
    };
    pl.header = take(sizeof(WsHeader));
    pl.cnt = take(sizeof(int32_t) * (size_t)nch * s.E);
    pl.base = take(sizeof(int32_t) * (size_t)nch * s.E);
    pl.idx = take(sizeof(int32_t) * (size_t)T);
    pl.gate = take(sizeof(float) * (size_t)T);
    pl.counts = take(sizeof(int32_t) * (size_t)s.E);
    pl.offsets = take(sizeof(int32_t) * (size_t)(s.E + 1));
    pl.sched = take(sizeof(int32_t) * 2 * (size_t)T);
    pl.inv = take(sizeof(int32_t) * (size_t)T);
    pl.xq = take(mx ? (size_t)s.N * s.H : 0);
    pl.xq_sf = take(mx ? (size_t)s.N * (s.H / 32) : 0);
    pl.shard_tab = take(sizeof(void*) * (size_t)s.S);
    pl.shard_sf_tab = take(sizeof(void*) * (size_t)s.S);
    pl.ring = take((size_t)R * s.H * op_elem(s.dtype));
    pl.ring_sf = take(mx ? (size_t)R * (s.H / 32) : 0);
    pl.h = take((size_t)R * s.I * op_elem(s.dtype));
    pl.h_sf = take(mx ? (size_t)R * (s.I / 32) : 0);
    pl.y = take((size_t)T * s.H * act_elem(s.dtype));
    pl.fused_ints = take(sizeof(int32_t) * fused_plan_ints((int)T, s.E, fg.nmb > 0 ? fg.nmb : 1));
    pl.total = off;
    pl.ring_slots = R;
    return pl;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// Workspace regions of the backward entry points, in order.
struct BwdPlan {
    size_t header, dy, dy_sf, dh, duv, duv_q, duv_sf, da, dgate, dlogit, slot_gate, slot_dlogit;
    size_t part, part_b, ppre;
    size_t pstage, blk_e, img_duv, sf_duv, img_x, sf_x, img_dy, sf_dy, img_h, sf_h;
    size_t total;
};

BwdPlan make_bwd_plan(const moe_shape_t& s) {
    const size_t T = (size_t)s.N * s.k;
    const bool mx = s.dtype == MOE_MXFP8;
    BwdPlan pl{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += align256(bytes);
        return o;
    };
    const size_t pmax = (size_t)router_max_pieces((int)T, s.E);
    pl.header = take(sizeof(WsHeader));
    pl.dy = take(T * s.H * (mx ? 1 : 2));
    pl.dy_sf = take(mx ? T * (s.H / 32) : 0);
    pl.dh = take(T * s.I * 2);
    pl.duv = take(T * 2 * s.I * 2);
    pl.duv_q = take(mx ? T * 2 * s.I : 0);
    pl.duv_sf = take(mx ? T * (2 * s.I / 32) : 0);
    pl.da = take(T * s.H * 2);
    pl.dgate = take(sizeof(float) * T);
    pl.dlogit = take(sizeof(float) * T);
    pl.slot_gate = take(sizeof(float) * T);
    pl.slot_dlogit = take(sizeof(float) * T);
    pl.part = take(sizeof(float) * pmax * s.H);
    pl.part_b = take(sizeof(float) * pmax);
    pl.ppre = take(sizeof(int32_t) * (s.E + 1));
    // wgrad operand images over the padded slot axis
    const size_t tp = (size_t)wgrad_max_padded_slots((int)T, s.E);
    const size_t esz = mx ? 1 : 2;
    const size_t Ip = (size_t)(s.I + 255) / 256 * 256;
    pl.pstage = take(sizeof(int32_t) * (s.E + 1));
    pl.blk_e = take(sizeof(int32_t) * (tp / 32));
    pl.img_duv = take(tp * 2 * s.I * esz);
    pl.sf_duv = take(mx ? tp * 2 * s.I / 32 : 0);
    pl.img_x = take(tp * s.H * esz);
    pl.sf_x = take(mx ? tp * s.H / 32 : 0);
    pl.img_dy = take(tp * s.H * esz);
    pl.sf_dy = take(mx ? tp * s.H / 32 : 0);
    pl.img_h = take(tp * Ip * esz);
    pl.sf_h = take(mx ? tp * Ip / 32 : 0);
    pl.total = off;
    return pl;
}

int check_shape(const moe_shape_t* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->N < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->k <= 0 || s->S <= 0)
        return MOE_ERR_INVALID_ARG;
    if (s->k > s->E || s->N % s->S != 0) return MOE_ERR_INVALID_ARG;
    if (s->dtype < MOE_F32 || s->dtype > MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    if (s->k > 32 || s->E > 1024) return MOE_ERR_UNSUPPORTED;
    if (s->H % 32 != 0 || s->I % 32 != 0) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)s->N * s->k > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
    if (s->dtype != MOE_F32 && (s->H % 256 != 0 || s->I % 128 != 0)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_ws(const moe_shape_t* s, const moe_params_t* p, void* ws, size_t bytes) {
    if (!ws || ((uintptr_t)ws & 31)) return MOE_ERR_WORKSPACE;
    if (bytes < make_plan(*s, p).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Shapes the backward supports: the tensor-core layers (BF16, MXFP8).
int check_bwd_shape(const moe_shape_t* s) {
    int rc = check_shape(s);
    if (rc) return rc;
    return s->dtype == MOE_F32 ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

int check_bwd_ws(const moe_shape_t* s, void* ws, size_t bytes) {
    if (!ws || ((uintptr_t)ws & 31)) return MOE_ERR_WORKSPACE;
    return bytes < make_bwd_plan(*s).total ? MOE_ERR_WORKSPACE : MOE_OK;
}

bool aligned32(const void* p) { return ((uintptr_t)p & 31) == 0; }

unsigned long long timeout_of(const moe_params_t* p) {
    return (p && p->timeout_ns > 0) ? (unsigned long long)p->timeout_ns : kDefaultTimeoutNs;
}

__global__ void fill_shard_table_kernel(const uint8_t** tab, const uint8_t* base, int64_t stride, int S) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s < S) tab[s] = base + stride * s;
}

int expert_ffn_impl(const void* a, const void* a_scales, int a_rows, const int32_t* offsets,
                    const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                    const void* w_d_scales, const moe_shape_t& s, void* y, void* ws,
                    unsigned long long timeout, cudaStream_t st, void* uv = nullptr) {
    const Plan pl = make_plan(s, nullptr);
    const int T = s.N * s.k;
    if (s.dtype == MOE_F32)
        return cuda_status(launch_ffn_f32((const float*)a, offsets, (const float*)w_gate_up,
                                          (const float*)w_down, T, s.H, s.I, s.E,
                                          at<float>(ws, pl.h), (float*)y, num_sms_current(), st));
    TcFfnCall c{};
    c.mx = s.dtype == MOE_MXFP8;
    c.T = T;
    c.H = s.H;
    c.I = s.I;
    c.E = s.E;
    c.a_rows = a_rows;
    c.a = a;
    c.a_sf = a_scales;
    c.offsets = offsets;
    c.w_gate_up = w_gate_up;
    c.w_gu_sf = w_gu_scales;
    c.w_down = w_down;
    c.w_d_sf = w_d_scales;
    c.h = at<void>(ws, pl.h);
    c.h_sf = at<void>(ws, pl.h_sf);
    c.y = y;
    c.uv = uv;
    c.ws = at<WsHeader>(ws, pl.header);
    c.timeout_ns = timeout;
    c.grid = num_sms_current();
    return cuda_status(launch_expert_ffn_tc(c, st));
}

}  // namespace

// The shape checks every entry point runs first (the no-allocation layout's too).
int validate_shape(const moe_shape_t* s) { return check_shape(s); }

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_shape_t* shape, const moe_params_t* params) {
    if (check_shape(shape) != MOE_OK) return 0;
    return make_plan(*shape, params).total;
}

int moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), (cudaStream_t)stream));
}

int moe_last_device_status(void* workspace, void* stream) {
    if (!workspace) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int status = 0;
    if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    return status;
}

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
        default: return "MOE_ERR_UNKNOWN";
    }
}

int moe_quantize_mxfp8(const void* in, int in_dtype, int64_t rows, int64_t K, uint8_t* codes,
                       uint8_t* scales, void* stream) {
    if (rows < 0 || K <= 0 || K % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (in_dtype != MOE_F32 && in_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!in || !codes || !scales || !aligned16(in) || !aligned16(codes)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_mxfp8(in, in_dtype, rows, K, codes, scales,
                                             num_sms_current(), (cudaStream_t)stream));
}

int moe_quantize_nvfp4(const void* in, int in_dtype, int64_t rows, int64_t K, uint8_t* codes,
                       uint8_t* scales, float* tensor_scale, void* stream) {
    if (rows < 0 || K <= 0 || K % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (in_dtype != MOE_F32 && in_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (!tensor_scale || ((uintptr_t)tensor_scale & 7)) return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!in || !codes || !scales || !aligned16(in) || ((uintptr_t)codes & 7)))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_nvfp4(in, in_dtype, rows, K, codes, scales, tensor_scale,
                                             num_sms_current(), (cudaStream_t)stream));
}

int moe_pack_expert_weights(const moe_shape_t* shape, const void* w_gate_up,
                            const uint8_t* w_gu_scales, const void* w_down,
                            const uint8_t* w_d_scales, void* packed_gate_up,
                            uint8_t* packed_gu_scales, void* packed_down, uint8_t* packed_d_scales,
                            void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!w_gate_up || !w_down || !packed_gate_up || !packed_down) return MOE_ERR_INVALID_ARG;
    if (mx && (!w_gu_scales || !w_d_scales || !packed_gu_scales || !packed_d_scales))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(packed_gate_up) ||
        !aligned16(packed_down))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t esz = op_elem(s.dtype);
    if (s.dtype == MOE_F32) {   // the SIMT path reads the natural layout
        const size_t b1 = (size_t)s.E * 2 * s.I * s.H * esz, b2 = (size_t)s.E * s.H * s.I * esz;
        if (cudaMemcpyAsync(packed_gate_up, w_gate_up, b1, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(packed_down, w_down, b2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (mx && (((uintptr_t)w_gu_scales & 3) || ((uintptr_t)w_d_scales & 3) ||
               ((uintptr_t)packed_gu_scales & 3) || ((uintptr_t)packed_d_scales & 3)))
        return MOE_ERR_INVALID_ARG;
    PackCall c{};
    c.mx = mx;
    c.E = s.E;
    c.H = s.H;
    c.I = s.I;
    c.w_gate_up = w_gate_up;
    c.w_gu_sf = w_gu_scales;
    c.w_down = w_down;
    c.w_d_sf = w_d_scales;
    c.p_gate_up = packed_gate_up;
    c.p_gu_sf = packed_gu_scales;
    c.p_down = packed_down;
    c.p_d_sf = packed_d_scales;
    c.num_sms = num_sms_current();
    return cuda_status(launch_pack_weights(c, st));
}

int moe_route_topk(const void* x, const void* w_router, const float* bias, const moe_shape_t* shape,
                   int32_t* idx, float* gate, float* logits_out, uint8_t* xq_codes,
                   uint8_t* xq_scales, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    if (!x || !w_router || !idx || !gate) return MOE_ERR_INVALID_ARG;
    if ((xq_codes != nullptr) != (xq_scales != nullptr)) return MOE_ERR_INVALID_ARG;
    if (xq_codes && (s.dtype != MOE_MXFP8 || !aligned16(xq_codes))) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    WsHeader* hdr = (workspace && workspace_bytes >= sizeof(WsHeader)) ? at<WsHeader>(workspace, 0)
                                                                         : nullptr;
    if (route_tc_supported(s.dtype, s.H, s.E, s.k))
        return cuda_status(launch_route_topk_tc(x, w_router, bias, s.N, s.H, s.E, s.k, idx, gate,
                                                logits_out, xq_codes, xq_scales, hdr,
                                                kDefaultTimeoutNs, st));
    rc = cuda_status(launch_route_topk_simt(x, w_router, bias, s.N, s.H, s.E, s.k, s.dtype, idx,
                                            gate, logits_out, st));
    if (rc || !xq_codes) return rc;
    return cuda_status(launch_quantize_mxfp8(x, MOE_BF16, s.N, s.H, xq_codes, xq_scales,
                                             num_sms_current(), st));
}

int moe_layout(const int32_t* idx, const moe_shape_t* shape, int32_t* counts, int32_t* offsets,
               int32_t* sched, int32_t* inv, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    rc = check_ws(shape, nullptr, workspace, workspace_bytes);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (!counts || !offsets || (s.N > 0 && (!idx || !sched || !inv))) return MOE_ERR_INVALID_ARG;
    const Plan pl = make_plan(s, nullptr);
    return cuda_status(launch_layout(idx, s.N, s.k, s.E, s.S, counts, offsets, sched, inv,
                                     at<int32_t>(workspace, pl.cnt), at<int32_t>(workspace, pl.base),
                                     at<WsHeader>(workspace, pl.header), (cudaStream_t)stream));
}

int moe_dispatch_pull(const void* const* shard_rows, const void* const* shard_scales,
                      const moe_shape_t* shape, const int32_t* sched, const int32_t* inv,
                      int slot_begin, int slot_count, void* ring, void* ring_scales, int ring_slots,
                      void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    const int T = s.N * s.k;
    if (slot_begin < 0 || slot_count < 0 || slot_begin + slot_count > T || ring_slots <= 0)
        return MOE_ERR_INVALID_ARG;
    if (slot_count == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!shard_rows || !sched || !ring || !aligned16(ring)) return MOE_ERR_INVALID_ARG;
    if (mx && (!shard_scales || !ring_scales)) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    const int row_bytes = s.H * (int)op_elem(s.dtype);
    const int scale_bytes = mx ? s.H / 32 : 0;
    return cuda_status(launch_dispatch_pull(shard_rows, shard_scales, sched, inv, T, s.k, slot_begin,
                                            slot_count, s.S, s.N / s.S, row_bytes, scale_bytes, ring,
                                            ring_scales, ring_slots, num_sms_current(),
                                            at<WsHeader>(workspace, 0), kDefaultTimeoutNs,
                                            (cudaStream_t)stream));
}

int moe_expert_ffn(const void* a, const void* a_scales, const int32_t* offsets,
                   const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                   const void* w_d_scales, const moe_shape_t* shape, void* y, void* workspace,
                   size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    rc = check_ws(shape, nullptr, workspace, workspace_bytes);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!a || !offsets || !w_gate_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (mx && (!a_scales || !w_gu_scales || !w_d_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w_gate_up) || !aligned16(w_down) || ((uintptr_t)y & 31))
        return MOE_ERR_INVALID_ARG;
    if (mx && (((uintptr_t)a_scales & 3) || ((uintptr_t)w_gu_scales & 3) || ((uintptr_t)w_d_scales & 3)))
        return MOE_ERR_INVALID_ARG;
    return expert_ffn_impl(a, a_scales, s.N * s.k, offsets, w_gate_up, w_gu_scales, w_down,
                           w_d_scales, s, y, workspace, kDefaultTimeoutNs, (cudaStream_t)stream);
}

int moe_combine(const void* y, const int32_t* inv, const float* gate, const moe_shape_t* shape,
                void* out, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    if (!y || !inv || !gate || !out || !aligned16(y) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_combine(y, inv, gate, s.N, s.H, s.k, s.N * s.k, s.dtype, out,
                                      num_sms_current(), at<WsHeader>(workspace, 0),
                                      (cudaStream_t)stream));
}

// The staged forward; with `sv`, the routing, layout, y and u|v go to the
// caller's saved-activation buffers (training).  With `combine_stream`, the
// combine runs there after `ffn_done` (recorded on `stream` once the FFN is
// issued), so the caller's stream can go on to the next macrobatch.
static int forward_staged(const void* x, const void* w_router, const float* bias,
                          const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                          const void* w_d_scales, const moe_shape_t* shape,
                          const moe_params_t* params, void* out, int32_t* idx_out, float* gate_out,
                          const moe_saved_t* sv, void* workspace, size_t workspace_bytes,
                          void* stream, cudaStream_t combine_stream = nullptr,
                          cudaEvent_t ffn_done = nullptr) {
    int rc = check_shape(shape);
    if (rc) return rc;
    rc = check_ws(shape, params, workspace, workspace_bytes);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!x || !w_router || !w_gate_up || !w_down || !out) return MOE_ERR_INVALID_ARG;
    if (mx && (!w_gu_scales || !w_d_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(w_gate_up) || !aligned16(w_down))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const Plan pl = make_plan(s, params);
    void* ws = workspace;
    WsHeader* hdr = at<WsHeader>(ws, pl.header);
    const int T = s.N * s.k;
    const int rows = s.N / s.S;
    int32_t* idx = sv ? sv->idx : (idx_out ? idx_out : at<int32_t>(ws, pl.idx));
    float* gate = sv ? sv->gate : (gate_out ? gate_out : at<float>(ws, pl.gate));
    int32_t* counts = at<int32_t>(ws, pl.counts);
    int32_t* offsets = sv ? sv->offsets : at<int32_t>(ws, pl.offsets);
    int32_t* sched = sv ? sv->sched : at<int32_t>(ws, pl.sched);
    int32_t* inv = sv ? sv->inv : at<int32_t>(ws, pl.inv);

    // 1. router + top-k (+ the MXFP8 copy of x each source shard serves)
    uint8_t* xq = mx ? at<uint8_t>(ws, pl.xq) : nullptr;
    uint8_t* xq_sf = mx ? at<uint8_t>(ws, pl.xq_sf) : nullptr;
    rc = moe_route_topk(x, w_router, bias, shape, idx, gate, nullptr, xq, xq_sf, ws,
                        workspace_bytes, stream);
    if (rc) return rc;
    // 2. layout
    rc = cuda_status(launch_layout(idx, s.N, s.k, s.E, s.S, counts, offsets, sched, inv,
                                   at<int32_t>(ws, pl.cnt), at<int32_t>(ws, pl.base), hdr, st));
    if (rc) return rc;
    // 3. pull dispatch through the table of S source-shard pointers
    const uint8_t** tab = at<const uint8_t*>(ws, pl.shard_tab);
    const uint8_t** tab_sf = at<const uint8_t*>(ws, pl.shard_sf_tab);
    const int row_bytes = s.H * (int)op_elem(s.dtype);
    const int tb = (s.S + 127) / 128;
    fill_shard_table_kernel<<<tb, 128, 0, st>>>(tab, mx ? xq : (const uint8_t*)x,
                                                (int64_t)rows * row_bytes, s.S);
    if (mx)
        fill_shard_table_kernel<<<tb, 128, 0, st>>>(tab_sf, xq_sf, (int64_t)rows * (s.H / 32), s.S);
    rc = cuda_status(cudaGetLastError());
    if (rc) return rc;
    void* ring = at<void>(ws, pl.ring);
    void* ring_sf = mx ? at<void>(ws, pl.ring_sf) : nullptr;
    rc = cuda_status(launch_dispatch_pull((const void* const*)tab, (const void* const*)tab_sf, sched,
                                          inv, T, s.k, 0, T, s.S, rows, row_bytes, mx ? s.H / 32 : 0, ring,
                                          ring_sf, pl.ring_slots, num_sms_current(), hdr,
                                          timeout_of(params), st));
    if (rc) return rc;
    // 4. grouped SwiGLU expert FFN
    void* y = sv ? sv->y : at<void>(ws, pl.y);
    rc = expert_ffn_impl(ring, ring_sf, pl.ring_slots, offsets, w_gate_up, w_gu_scales, w_down,
                         w_d_scales, s, y, ws, timeout_of(params), st, sv ? sv->uv : nullptr);
    if (rc) return rc;
    // 5. combine + weighted merge
    if (combine_stream) {
        rc = cuda_status(cudaEventRecord(ffn_done, st));
        if (rc) return rc;
        rc = cuda_status(cudaStreamWaitEvent(combine_stream, ffn_done, 0));
        if (rc) return rc;
        st = combine_stream;
    }
    rc = cuda_status(launch_combine(y, inv, gate, s.N, s.H, s.k, T, s.dtype, out,
                                    num_sms_current(), hdr, st));
    return rc;
}

int moe_forward(const void* x, const void* w_router, const float* bias, const void* w_gate_up,
                const void* w_gu_scales, const void* w_down, const void* w_d_scales,
                const moe_shape_t* shape, const moe_params_t* params, void* out, int32_t* idx_out,
                float* gate_out, void* workspace, size_t workspace_bytes, void* stream) {
    return forward_staged(x, w_router, bias, w_gate_up, w_gu_scales, w_down, w_d_scales, shape,
                          params, out, idx_out, gate_out, nullptr, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- macrobatches
// Workspace slice of one macrobatch (the shape with N / macrobatches tokens),
// rounded up to 256 bytes; 0 if the split is not allowed.
static size_t macro_slice_bytes(const moe_shape_t* shape, const moe_params_t* params, int macrobatches) {
    if (check_shape(shape) != MOE_OK || macrobatches < 1) return 0;
    if (shape->N % (macrobatches * shape->S) != 0) return 0;
    moe_shape_t sm = *shape;
    sm.N = shape->N / macrobatches;
    if (sm.N == 0) return 0;
    return (make_plan(sm, params).total + 255) / 256 * 256;
}

size_t moe_macro_workspace_bytes(const moe_shape_t* shape, const moe_params_t* params, int macrobatches) {
    return macro_slice_bytes(shape, params, macrobatches) * (size_t)(macrobatches > 0 ? macrobatches : 0);
}

// A second stream per device for the macrobatches' combines, created on first use.
static cudaStream_t macro_side_stream() {
    static cudaStream_t side[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!side[dev] && cudaStreamCreateWithFlags(&side[dev], cudaStreamNonBlocking) != cudaSuccess)
        side[dev] = nullptr;
    return side[dev];
}

int moe_forward_macrobatched(const void* x, const void* w_router, const float* bias, const void* w_gate_up,
                             const void* w_gu_scales, const void* w_down, const void* w_d_scales,
                             const moe_shape_t* shape, const moe_params_t* params, int macrobatches,
                             void* out, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (macrobatches < 1) return MOE_ERR_INVALID_ARG;
    if (s.N == 0) return MOE_OK;
    const size_t slice = macro_slice_bytes(shape, params, macrobatches);
    if (slice == 0) return MOE_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255)) return MOE_ERR_WORKSPACE;
    if (workspace_bytes < slice * (size_t)macrobatches) return MOE_ERR_WORKSPACE;
    if (!x || !out) return MOE_ERR_INVALID_ARG;
    moe_shape_t sm = s;
    sm.N = s.N / macrobatches;
    const size_t x_rows = (size_t)sm.N * s.H * op_elem(s.dtype == MOE_F32 ? MOE_F32 : MOE_BF16);
    const size_t o_rows = (size_t)sm.N * s.H * (s.dtype == MOE_F32 ? 4 : 2);
    cudaStream_t st = (cudaStream_t)stream;
    cudaStream_t side = macrobatches > 1 ? macro_side_stream() : nullptr;
    if (macrobatches > 1 && !side) return MOE_ERR_CUDA;
    // events: one per macrobatch (its FFN issued), one to join the side stream
    cudaEvent_t ev[65] = {};
    const int nev = macrobatches > 1 ? macrobatches + 1 : 0;
    if (nev > 65) return MOE_ERR_UNSUPPORTED;
    for (int i = 0; i < nev; ++i)
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return MOE_ERR_CUDA;
        }
    if (side) {   // the side stream starts after what the caller already queued
        rc = cuda_status(cudaEventRecord(ev[macrobatches], st));
        if (!rc) rc = cuda_status(cudaStreamWaitEvent(side, ev[macrobatches], 0));
    }
    for (int m = 0; !rc && m < macrobatches; ++m) {
        rc = forward_staged((const uint8_t*)x + m * x_rows, w_router, bias, w_gate_up, w_gu_scales, w_down,
                            w_d_scales, &sm, params, (uint8_t*)out + m * o_rows, nullptr, nullptr, nullptr,
                            (uint8_t*)workspace + m * slice, slice, stream, side, side ? ev[m] : nullptr);
    }
    if (side) {   // the caller's stream resumes after every combine
        const int rj = cuda_status(cudaEventRecord(ev[macrobatches], side));
        const int rw = rj ? rj : cuda_status(cudaStreamWaitEvent(st, ev[macrobatches], 0));
        if (!rc) rc = rw;
    }
    for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);   // released once their work completes
    return rc;
}

int moe_forward_fused(const void* x, const void* w_router, const float* bias,
                      const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                      const void* w_d_scales, const moe_shape_t* shape, const moe_params_t* params,
                      void* out, int32_t* idx_out, float* gate_out, void* workspace,
                      size_t workspace_bytes, void* stream) {
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.dtype == MOE_F32) return MOE_ERR_UNSUPPORTED;   // no tensor-core pipeline for FP32
    rc = check_ws(shape, params, workspace, workspace_bytes);
    if (rc) return rc;
    if (s.N == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!x || !w_router || !w_gate_up || !w_down || !out) return MOE_ERR_INVALID_ARG;
    if (mx && (!w_gu_scales || !w_d_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(w_gate_up) || !aligned16(w_down))
        return MOE_ERR_INVALID_ARG;
    const Plan pl = make_plan(s, params);
    const FusedGeom fg = resolve_fused(s, params, fused_max_ctas());
    if (fg.status) return fg.status;
    if (fg.R > pl.ring_slots || fg.nmb > pl.fg.nmb) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    void* ws = workspace;
    WsHeader* hdr = at<WsHeader>(ws, pl.header);
    const int T = s.N * s.k;
    const int rows = s.N / s.S;
    int32_t* idx = idx_out ? idx_out : at<int32_t>(ws, pl.idx);
    float* gate = gate_out ? gate_out : at<float>(ws, pl.gate);
    int32_t* counts = at<int32_t>(ws, pl.counts);
    int32_t* offsets = at<int32_t>(ws, pl.offsets);
    int32_t* sched = at<int32_t>(ws, pl.sched);
    int32_t* inv = at<int32_t>(ws, pl.inv);
    uint8_t* xq = mx ? at<uint8_t>(ws, pl.xq) : nullptr;
    uint8_t* xq_sf = mx ? at<uint8_t>(ws, pl.xq_sf) : nullptr;

    // routing and layout run first as their own kernels
    rc = moe_route_topk(x, w_router, bias, shape, idx, gate, nullptr, xq, xq_sf, ws, workspace_bytes,
                        stream);
    if (rc) return rc;
    rc = cuda_status(launch_layout(idx, s.N, s.k, s.E, s.S, counts, offsets, sched, inv,
                                   at<int32_t>(ws, pl.cnt), at<int32_t>(ws, pl.base), hdr, st));
    if (rc) return rc;
    const uint8_t** tab = at<const uint8_t*>(ws, pl.shard_tab);
    const uint8_t** tab_sf = at<const uint8_t*>(ws, pl.shard_sf_tab);
    const int row_bytes = s.H * (int)op_elem(s.dtype);
    const int tb = (s.S + 127) / 128;
    fill_shard_table_kernel<<<tb, 128, 0, st>>>(tab, mx ? xq : (const uint8_t*)x,
                                                (int64_t)rows * row_bytes, s.S);
    if (mx)
        fill_shard_table_kernel<<<tb, 128, 0, st>>>(tab_sf, xq_sf, (int64_t)rows * (s.H / 32), s.S);
    rc = cuda_status(cudaGetLastError());
    if (rc) return rc;

    FusedCall c{};
    c.ffn.mx = mx;
    c.ffn.T = T;
    c.ffn.H = s.H;
    c.ffn.I = s.I;
    c.ffn.E = s.E;
    c.ffn.a_rows = fg.R;
    c.ffn.a = at<void>(ws, pl.ring);
    c.ffn.a_sf = mx ? at<void>(ws, pl.ring_sf) : nullptr;
    c.ffn.offsets = offsets;
    c.ffn.w_gate_up = w_gate_up;
    c.ffn.w_gu_sf = w_gu_scales;
    c.ffn.w_down = w_down;
    c.ffn.w_d_sf = w_d_scales;
    c.ffn.h = at<void>(ws, pl.h);
    c.ffn.h_sf = mx ? at<void>(ws, pl.h_sf) : nullptr;
    c.ffn.y = at<void>(ws, pl.y);
    c.ffn.ws = hdr;
    c.ffn.timeout_ns = timeout_of(params);
    c.ffn.grid = fg.G + fg.C;
    c.N = s.N;
    c.H = s.H;
    c.E = s.E;
    c.k = s.k;
    c.S = s.S;
    c.T = T;
    c.MB = fg.MB;
    c.R = fg.R;
    c.nmb = fg.nmb;
    c.G = fg.G;
    c.C = fg.C;
    c.row_bytes = row_bytes;
    c.sf_bytes = mx ? s.H / 32 : 0;
    c.skip_ready = (params && params->test_skip_ready > 0) ? params->test_skip_ready - 1 : -1;
    c.reverse = (params && params->reverse_ring) ? 1 : 0;
    c.sched = sched;
    c.inv = inv;
    c.gate = gate;
    c.shard_rows = (const void* const*)tab;
    c.shard_sf = (const void* const*)tab_sf;
    c.out = out;
    c.plan_ints = at<int>(ws, pl.fused_ints);
    return cuda_status(launch_fused_forward(c, st));
}

int moe_min_minibatch(int waves, int compute_sms, int tile_m, int tile_n, int I) {
    if (waves <= 0 || compute_sms <= 0 || tile_m <= 0 || tile_n <= 0 || I <= 0) return 0;
    const long long num = (long long)waves * compute_sms * tile_m * tile_n;
    const long long den = 2LL * I;
    return (int)((num + den - 1) / den);
}

// ------------------------------------------------------------------ backward
size_t moe_backward_workspace_bytes(const moe_shape_t* shape) {
    if (check_bwd_shape(shape) != MOE_OK) return 0;
    return make_bwd_plan(*shape).total;
}

int moe_pack_expert_weights_dgrad(const moe_shape_t* shape, const void* w_gate_up,
                                  const void* w_down, void* packed_gate_up_t,
                                  uint8_t* packed_gu_t_scales, void* packed_down_t,
                                  uint8_t* packed_d_t_scales, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!w_gate_up || !w_down || !packed_gate_up_t || !packed_down_t) return MOE_ERR_INVALID_ARG;
    if (mx && (!packed_gu_t_scales || !packed_d_t_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(packed_gate_up_t) || !aligned16(packed_down_t)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    rc = cuda_status(launch_pack_transposed(mx, w_gate_up, s.E, 2 * s.I, s.H, packed_gate_up_t,
                                            packed_gu_t_scales, num_sms_current(), st));
    if (rc) return rc;
    return cuda_status(launch_pack_transposed(mx, w_down, s.E, s.H, s.I, packed_down_t,
                                              packed_d_t_scales, num_sms_current(), st));
}

int moe_expert_ffn_train(const void* a, const void* a_scales, const int32_t* offsets,
                         const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                         const void* w_d_scales, const moe_shape_t* shape, void* y, void* uv,
                         void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    if (!uv || !aligned32(uv)) return MOE_ERR_INVALID_ARG;
    rc = check_ws(shape, nullptr, workspace, workspace_bytes);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!a || !offsets || !w_gate_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (mx && (!a_scales || !w_gu_scales || !w_d_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned32(y))
        return MOE_ERR_INVALID_ARG;
    return expert_ffn_impl(a, a_scales, s.N * s.k, offsets, w_gate_up, w_gu_scales, w_down,
                           w_d_scales, s, y, workspace, kDefaultTimeoutNs, (cudaStream_t)stream, uv);
}

int moe_forward_train(const void* x, const void* w_router, const float* bias,
                      const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                      const void* w_d_scales, const moe_shape_t* shape, const moe_params_t* params,
                      void* out, const moe_saved_t* saved, void* workspace,
                      size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    if (!saved || !saved->idx || !saved->gate || !saved->inv || !saved->offsets || !saved->sched ||
        !saved->y || !saved->uv)
        return MOE_ERR_INVALID_ARG;
    if (!aligned32(saved->y) || !aligned32(saved->uv)) return MOE_ERR_INVALID_ARG;
    return forward_staged(x, w_router, bias, w_gate_up, w_gu_scales, w_down, w_d_scales, shape,
                          params, out, nullptr, nullptr, saved, workspace, workspace_bytes, stream);
}

int moe_reverse_combine(const void* dout, const void* y, const int32_t* inv, const float* gate,
                        const moe_shape_t* shape, void* dy, uint8_t* dy_scales, float* dgate,
                        float* dlogit, float* slot_gate, float* slot_dlogit, void* workspace,
                        size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!dout || !y || !inv || !gate || !dy || !dgate || !dlogit || !slot_gate || !slot_dlogit)
        return MOE_ERR_INVALID_ARG;
    if (mx != (dy_scales != nullptr)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dout) || !aligned16(y) || !aligned16(dy)) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_reverse_combine(mx, dout, y, inv, gate, s.N, s.H, s.k, s.N * s.k, dy,
                                              dy_scales, dgate, dlogit, slot_gate, slot_dlogit,
                                              num_sms_current(), at<WsHeader>(workspace, 0),
                                              (cudaStream_t)stream));
}

int moe_expert_ffn_dgrad(const void* dy, const uint8_t* dy_scales, const void* uv,
                         const int32_t* offsets, const void* wt_gate_up,
                         const uint8_t* wt_gu_scales, const void* wt_down,
                         const uint8_t* wt_d_scales, const moe_shape_t* shape, void* duv,
                         uint8_t* duv_codes, uint8_t* duv_scales, void* da, void* workspace,
                         size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    const bool mx = s.dtype == MOE_MXFP8;
    if (!dy || !uv || !offsets || !wt_gate_up || !wt_down || !duv || !da) return MOE_ERR_INVALID_ARG;
    if (mx && (!dy_scales || !wt_gu_scales || !wt_d_scales || !duv_codes || !duv_scales))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned32(uv) || !aligned16(wt_gate_up) || !aligned16(wt_down) ||
        !aligned32(duv) || !aligned32(da) || (mx && !aligned32(duv_codes)))
        return MOE_ERR_INVALID_ARG;
    if (mx && (((uintptr_t)dy_scales & 15) || ((uintptr_t)duv_scales & 15)))
        return MOE_ERR_INVALID_ARG;
    rc = check_bwd_ws(shape, workspace, workspace_bytes);
    if (rc) return rc;
    const BwdPlan pl = make_bwd_plan(s);
    TcDgradCall c{};
    c.mx = mx;
    c.T = s.N * s.k;
    c.H = s.H;
    c.I = s.I;
    c.E = s.E;
    c.a_rows = c.T;
    c.dy = dy;
    c.dy_sf = dy_scales;
    c.uv = uv;
    c.offsets = offsets;
    c.wt_down = wt_down;
    c.wt_d_sf = wt_d_scales;
    c.wt_gate_up = wt_gate_up;
    c.wt_gu_sf = wt_gu_scales;
    c.dh = at<void>(workspace, pl.dh);
    c.duv = duv;
    c.duv_q = duv_codes;
    c.duv_sf = duv_scales;
    c.da = da;
    c.ws = at<WsHeader>(workspace, pl.header);
    c.timeout_ns = kDefaultTimeoutNs;
    c.grid = num_sms_current();
    c.num_sms = num_sms_current();
    return cuda_status(launch_ffn_dgrad_tc(c, (cudaStream_t)stream));
}

int moe_reverse_dispatch(const void* da, const int32_t* inv, const int32_t* idx,
                         const float* dlogit, const void* w_router, const moe_shape_t* shape,
                         void* dx, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (s.N == 0) return MOE_OK;
    if (!da || !inv || !idx || !dlogit || !w_router || !dx) return MOE_ERR_INVALID_ARG;
    if (!aligned16(da) || !aligned16(w_router) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_reverse_dispatch(da, inv, idx, dlogit, w_router, s.N, s.H, s.k,
                                               s.N * s.k, s.E, dx, num_sms_current(),
                                               at<WsHeader>(workspace, 0), (cudaStream_t)stream));
}

int moe_router_wgrad(const void* x, const int32_t* sched, const int32_t* offsets,
                     const float* slot_dlogit, const moe_shape_t* shape, float* dw_router,
                     float* dbias, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    rc = check_bwd_ws(shape, workspace, workspace_bytes);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (!offsets || !dw_router || (s.N > 0 && (!x || !sched || !slot_dlogit))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dw_router) || ((uintptr_t)x & 7)) return MOE_ERR_INVALID_ARG;
    const BwdPlan pl = make_bwd_plan(s);
    return cuda_status(launch_router_wgrad(x, sched, offsets, slot_dlogit, s.N, s.H, s.E, s.N * s.k,
                                           s.N / s.S, dw_router, dbias, at<float>(workspace, pl.part),
                                           at<float>(workspace, pl.part_b),
                                           at<int32_t>(workspace, pl.ppre),
                                           at<WsHeader>(workspace, pl.header), (cudaStream_t)stream));
}

int moe_expert_wgrad(const void* duv, const void* x, const void* dout, const void* uv,
                     const int32_t* sched, const float* slot_gate, const int32_t* offsets,
                     const moe_shape_t* shape, void* dw_gate_up, void* dw_down, void* workspace,
                     size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    rc = check_bwd_ws(shape, workspace, workspace_bytes);
    if (rc) return rc;
    const moe_shape_t& s = *shape;
    if (!offsets || !dw_gate_up || !dw_down) return MOE_ERR_INVALID_ARG;
    if (s.N > 0 && (!duv || !x || !dout || !uv || !sched || !slot_gate)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(duv) || !aligned16(x) || !aligned16(dout) || !aligned16(uv) ||
        !aligned32(dw_gate_up) || !aligned32(dw_down))
        return MOE_ERR_INVALID_ARG;
    const BwdPlan pl = make_bwd_plan(s);
    void* ws = workspace;
    const bool mx = s.dtype == MOE_MXFP8;
    WgradCall c{};
    c.mx = mx;
    c.N = s.N;
    c.H = s.H;
    c.I = s.I;
    c.E = s.E;
    c.T = s.N * s.k;
    c.rows_per_shard = s.N / s.S;
    c.duv = duv;
    c.x = x;
    c.dout = dout;
    c.uv = uv;
    c.sched = sched;
    c.slot_gate = slot_gate;
    c.offsets = offsets;
    c.dw_gate_up = dw_gate_up;
    c.dw_down = dw_down;
    c.pstage = at<int32_t>(ws, pl.pstage);
    c.blk_e = at<int32_t>(ws, pl.blk_e);
    c.img_duv = at<uint8_t>(ws, pl.img_duv);
    c.sf_duv = mx ? at<uint8_t>(ws, pl.sf_duv) : nullptr;
    c.img_x = at<uint8_t>(ws, pl.img_x);
    c.sf_x = mx ? at<uint8_t>(ws, pl.sf_x) : nullptr;
    c.img_dy = at<uint8_t>(ws, pl.img_dy);
    c.sf_dy = mx ? at<uint8_t>(ws, pl.sf_dy) : nullptr;
    c.img_h = at<uint8_t>(ws, pl.img_h);
    c.sf_h = mx ? at<uint8_t>(ws, pl.sf_h) : nullptr;
    c.ws = at<WsHeader>(ws, pl.header);
    c.timeout_ns = kDefaultTimeoutNs;
    c.grid = num_sms_current();
    return cuda_status(launch_wgrad(c, (cudaStream_t)stream));
}

int moe_backward(const void* dout, const void* x, const void* w_router, const moe_saved_t* saved,
                 const void* wt_gate_up, const uint8_t* wt_gu_scales, const void* wt_down,
                 const uint8_t* wt_d_scales, const moe_shape_t* shape, const moe_params_t* params,
                 void* dx, float* dw_router, float* dbias, void* dw_gate_up, void* dw_down,
                 void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_bwd_shape(shape);
    if (rc) return rc;
    rc = check_bwd_ws(shape, workspace, workspace_bytes);
    if (rc) return rc;
    (void)params;
    const moe_shape_t& s = *shape;
    if (!saved) return MOE_ERR_INVALID_ARG;
    if (s.N == 0) {
        // an empty batch: no expert has slots, so every weight gradient is zero (dx has
        // no rows)
        cudaStream_t st = (cudaStream_t)stream;
        cudaError_t e = cudaSuccess;
        if (dw_router) e = cudaMemsetAsync(dw_router, 0, (size_t)s.E * s.H * sizeof(float), st);
        if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, (size_t)s.E * sizeof(float), st);
        if (e == cudaSuccess && dw_gate_up)
            e = cudaMemsetAsync(dw_gate_up, 0, (size_t)s.E * 2 * s.I * s.H * 2, st);
        if (e == cudaSuccess && dw_down) e = cudaMemsetAsync(dw_down, 0, (size_t)s.E * s.H * s.I * 2, st);
        return cuda_status(e);
    }
    const bool mx = s.dtype == MOE_MXFP8;
    const BwdPlan pl = make_bwd_plan(s);
    void* ws = workspace;
    uint8_t* dy_sf = mx ? at<uint8_t>(ws, pl.dy_sf) : nullptr;
    rc = moe_reverse_combine(dout, saved->y, saved->inv, saved->gate, shape, at<void>(ws, pl.dy),
                             dy_sf, at<float>(ws, pl.dgate), at<float>(ws, pl.dlogit),
                             at<float>(ws, pl.slot_gate), at<float>(ws, pl.slot_dlogit), ws,
                             workspace_bytes, stream);
    if (rc) return rc;
    rc = moe_expert_ffn_dgrad(at<void>(ws, pl.dy), dy_sf, saved->uv, saved->offsets, wt_gate_up,
                              wt_gu_scales, wt_down, wt_d_scales, shape, at<void>(ws, pl.duv),
                              mx ? at<uint8_t>(ws, pl.duv_q) : nullptr,
                              mx ? at<uint8_t>(ws, pl.duv_sf) : nullptr, at<void>(ws, pl.da), ws,
                              workspace_bytes, stream);
    if (rc) return rc;
    rc = moe_reverse_dispatch(at<void>(ws, pl.da), saved->inv, saved->idx, at<float>(ws, pl.dlogit),
                              w_router, shape, dx, ws, workspace_bytes, stream);
    if (rc) return rc;
    rc = moe_router_wgrad(x, saved->sched, saved->offsets, at<float>(ws, pl.slot_dlogit), shape,
                          dw_router, dbias, ws, workspace_bytes, stream);
    if (rc || (!dw_gate_up && !dw_down)) return rc;
    if (!dw_gate_up || !dw_down) return MOE_ERR_INVALID_ARG;
    return moe_expert_wgrad(at<void>(ws, pl.duv), x, dout, saved->uv, saved->sched,
                            at<float>(ws, pl.slot_gate), saved->offsets, shape, dw_gate_up, dw_down,
                            ws, workspace_bytes, stream);
}

}  // extern "C"
