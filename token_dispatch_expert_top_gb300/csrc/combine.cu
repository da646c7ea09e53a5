// combine.cu -- every expert result returns to its token and is merged with the
// token's gate weights: out[n] = sum_j g[n][j] * y[inv[n][j]], FP32 accumulation
// in fixed j order (so the output is bitwise reproducible), one rounding at the
// end.  ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA
// GB300 NVL72", section 02 (push combine: the destination of each result is
// known) and section 03 (the final weighted merge is part of the layer).)
// On one GPU the push and the merge collapse into one pass that reads each y row
// once, by token, with no atomics.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kCombineWarps = 8;

// Work item = (token n, 32*VEC-column chunk); one warp per item, VEC columns per
// lane loaded as one 16-byte vector from each of the token's k slot rows.
template <bool BF16>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(
    const uint8_t* __restrict__ y, const int32_t* __restrict__ inv, const float* __restrict__ gate,
    int N, int H, int k, int T, uint8_t* __restrict__ out, WsHeader* ws) {
    constexpr int VEC = BF16 ? 8 : 4;
    constexpr int ESZ = BF16 ? 2 : 4;
    const int lane = threadIdx.x % 32;
    const int chunks = (H + 32 * VEC - 1) / (32 * VEC);
    const int64_t items = (int64_t)N * chunks;
    const int64_t gw = (int64_t)blockIdx.x * kCombineWarps + threadIdx.x / 32;
    const int64_t nw = (int64_t)gridDim.x * kCombineWarps;
    for (int64_t it = gw; it < items; it += nw) {
        const int n = (int)(it / chunks);
        const int col = (int)(it % chunks) * 32 * VEC + lane * VEC;
        const int my_slot = lane < k ? inv[(int64_t)n * k + lane] : 0;
        const float my_g = lane < k ? gate[(int64_t)n * k + lane] : 0.f;
        float acc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
        // the k slot rows in groups of KB: every load of a group is issued before
        // the group is summed, still in j order
        constexpr int KB = 8;
        for (int j0 = 0; j0 < k; j0 += KB) {
            uint4 q[KB];
            float gj[KB];
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
                const int j = j0 + jj;
                const int slot = __shfl_sync(0xffffffffu, my_slot, j & 31);
                gj[jj] = __shfl_sync(0xffffffffu, my_g, j & 31);
                q[jj] = make_uint4(0u, 0u, 0u, 0u);
                if (j < k) {
                    if (slot < 0 || slot >= T) {
                        if (lane == 0) set_status(ws, MOE_ERR_DEVICE_CHECK);
                        gj[jj] = 0.f;     // skipped, as an out-of-range slot always was
                    } else if (col < H) {
                        q[jj] = ld_nc_v4(y + ((int64_t)slot * H + col) * ESZ);
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
                if (j0 + jj >= k) break;
                const uint32_t w[4] = {q[jj].x, q[jj].y, q[jj].z, q[jj].w};
                const float g = gj[jj];
                if constexpr (BF16) {
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        acc[2 * p] = fmaf(g, bf16_to_f32((uint16_t)(w[p] & 0xFFFF)), acc[2 * p]);
                        acc[2 * p + 1] = fmaf(g, bf16_to_f32((uint16_t)(w[p] >> 16)), acc[2 * p + 1]);
                    }
                } else {
#pragma unroll
                    for (int p = 0; p < 4; ++p) acc[p] = fmaf(g, __uint_as_float(w[p]), acc[p]);
                }
            }
        }
        if (col < H) {
            uint4 o;
            if constexpr (BF16)
                o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            else
                o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                               __float_as_uint(acc[2]), __float_as_uint(acc[3]));
            st_v4(out + ((int64_t)n * H + col) * ESZ, o);
        }
    }
}

cudaError_t launch_combine(const void* y, const int32_t* inv, const float* gate, int N, int H,
                           int k, int T, int dtype, void* out, int num_sms, WsHeader* ws,
                           cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const bool bf16 = dtype != MOE_F32;
    const int vec = bf16 ? 8 : 4;
    const int64_t items = (int64_t)N * ((H + 32 * vec - 1) / (32 * vec));
    int64_t blocks = (items + kCombineWarps - 1) / kCombineWarps;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (bf16)
        combine_kernel<true><<<(unsigned)blocks, kCombineWarps * 32, 0, stream>>>(
            (const uint8_t*)y, inv, gate, N, H, k, T, (uint8_t*)out, ws);
    else
        combine_kernel<false><<<(unsigned)blocks, kCombineWarps * 32, 0, stream>>>(
            (const uint8_t*)y, inv, gate, N, H, k, T, (uint8_t*)out, ws);
    return cudaGetLastError();
}

}  // namespace moe
