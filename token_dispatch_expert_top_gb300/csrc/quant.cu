// quant.cu -- stand-alone MXFP8 quantisation along K (OCP MX v1.0 block rule).
// The layer's activations are quantised inside other kernels' data paths; this
// kernel prepares expert weights once and quantises x for the dispatch.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// One thread per 32-element block.  Consecutive threads take consecutive blocks
// of a row, so a warp reads 2 KB (BF16) or 4 KB (FP32) of contiguous input.
template <typename In>
__global__ void __launch_bounds__(256) quantize_mxfp8_kernel(const In* __restrict__ in,
                                                             int64_t rows, int64_t K,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
    const int64_t nb = K / 32;
    const int64_t total = rows * nb;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total;
         b += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = b / nb, c = b % nb;
        float v[32];
        const In* src = in + r * K + c * 32;
        if constexpr (sizeof(In) == 2) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 q = ld_nc_v4(src + 8 * i);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    v[8 * i + 2 * p] = bf16_to_f32((uint16_t)(w[p] & 0xFFFF));
                    v[8 * i + 2 * p + 1] = bf16_to_f32((uint16_t)(w[p] >> 16));
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint4 q = ld_nc_v4(src + 4 * i);
                v[4 * i + 0] = __uint_as_float(q.x);
                v[4 * i + 1] = __uint_as_float(q.y);
                v[4 * i + 2] = __uint_as_float(q.z);
                v[4 * i + 3] = __uint_as_float(q.w);
            }
        }
        uint32_t out[8];
        uint8_t s = mx_quantize32(v, out);
        uint8_t* dst = codes + r * K + c * 32;
        st_v4(dst, make_uint4(out[0], out[1], out[2], out[3]));
        st_v4(dst + 16, make_uint4(out[4], out[5], out[6], out[7]));
        scales[r * nb + c] = s;
    }
}

cudaError_t launch_quantize_mxfp8(const void* in, int in_dtype, int64_t rows, int64_t K,
                                  uint8_t* codes, uint8_t* scales, int num_sms,
                                  cudaStream_t stream) {
    const int64_t total = rows * (K / 32);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 16;
    if (blocks > cap) blocks = cap;
    if (in_dtype == MOE_BF16)
        quantize_mxfp8_kernel<uint16_t><<<(unsigned)blocks, 256, 0, stream>>>(
            (const uint16_t*)in, rows, K, codes, scales);
    else
        quantize_mxfp8_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(
            (const float*)in, rows, K, codes, scales);
    return cudaGetLastError();
}

}  // namespace moe
