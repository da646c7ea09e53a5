// route.cu -- router logits, softmax top-k and renormalised gates, one warp per
// token with warp-shuffle reductions.  Every token picks a few experts out of
// many each step ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost
// on NVIDIA GB300 NVL72", section 01); the gate is a softmax over the router
// logits, the k largest are kept and renormalised to sum 1.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kRouteWarps = 8;

template <typename In>
__device__ __forceinline__ float load_elem(const In* p, int64_t i) {
    if constexpr (sizeof(In) == 2)
        return bf16_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
    else
        return reinterpret_cast<const float*>(p)[i];
}

// Better candidate in the top-k order: larger logit, then lower expert index.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
    return v > bv || (v == bv && e >= 0 && (be < 0 || e < be));
}

// logits[n][e] = sum_h x[n][h] w[e][h] (+ bias[e]) accumulated in FP32 by a warp
// (lanes split h, shuffle tree per expert); then k rounds of warp arg-max over
// the logits not yet chosen; gates g_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0).
template <typename In>
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_simt_kernel(
    const In* __restrict__ x, const In* __restrict__ w, const float* __restrict__ bias, int N,
    int H, int E, int k, int32_t* __restrict__ idx, float* __restrict__ gate,
    float* __restrict__ logits_out) {
    extern __shared__ float sh_logits[];  // [kRouteWarps][E] logits, then chosen flags
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float* lg = sh_logits + warp * E;
    const int n = blockIdx.x * kRouteWarps + warp;
    if (n >= N) return;
    const In* xr = x + (int64_t)n * H;
    for (int e = 0; e < E; ++e) {
        const In* wr = w + (int64_t)e * H;
        float acc = 0.f;
        for (int h = lane; h < H; h += 32) acc = fmaf(load_elem(xr, h), load_elem(wr, h), acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) lg[e] = acc + (bias ? bias[e] : 0.f);
    }
    __syncwarp();
    if (logits_out)
        for (int e = lane; e < E; e += 32) logits_out[(int64_t)n * E + e] = lg[e];
    // chosen flags live in the sign of a shadow copy: keep a per-lane bitmask of
    // the experts this lane owns (e = lane + 32*i); E <= 1024 -> 32 bits per lane
    uint32_t taken = 0;
    float top_v0 = 0.f, my_sel_v = 0.f;
    int my_sel_e = -1;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = -1;
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
            if (taken & (1u << i)) continue;
            if (better(lg[e], e, bv, be)) {
                bv = lg[e];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (better(ov, oe, bv, be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be >= 0 && (be % 32) == lane) taken |= 1u << (be / 32);
        if (j == 0) top_v0 = bv;
        if (lane == j) {
            my_sel_v = bv;
            my_sel_e = be;
        }
    }
    // gates: softmax over the k selected logits (max = the first one)
    float p = (lane < k) ? expf(my_sel_v - top_v0) : 0.f;
    float z = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) {
        idx[(int64_t)n * k + lane] = my_sel_e;
        gate[(int64_t)n * k + lane] = p / z;
    }
}

cudaError_t launch_route_topk_simt(const void* x, const void* w, const float* bias, int N, int H,
                                   int E, int k, int dtype, int32_t* idx, float* gate,
                                   float* logits_out, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int blocks = (N + kRouteWarps - 1) / kRouteWarps;
    const size_t smem = sizeof(float) * kRouteWarps * E;
    if (dtype == MOE_F32)
        route_topk_simt_kernel<float><<<blocks, kRouteWarps * 32, smem, stream>>>(
            (const float*)x, (const float*)w, bias, N, H, E, k, idx, gate, logits_out);
    else
        route_topk_simt_kernel<uint16_t><<<blocks, kRouteWarps * 32, smem, stream>>>(
            (const uint16_t*)x, (const uint16_t*)w, bias, N, H, E, k, idx, gate, logits_out);
    return cudaGetLastError();
}

}  // namespace moe
