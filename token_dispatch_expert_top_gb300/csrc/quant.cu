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

// ---------------------------------------------------------------------------------
// NVFP4: E2M1 elements, an E4M3 scale per 16 elements along K and one FP32 scale per
// tensor (s_t = amax / (6 * 448), so the largest block scale lands at E4M3's top).
// The tensor scale needs the tensor amax before any block can be scaled, so the
// quantisation is two passes over the input: an amax reduction, then the blocks.

// Eight E2M1 codes from eight FP32 values, round-to-nearest-even with saturation;
// value 2i lands in the low nibble of byte i/2 (the instruction puts its first
// source in the upper nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* q) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return r;
}

// Value of a non-negative E4M3 code (bias 7, 3 mantissa bits), exact in FP32.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 15, m = c & 7;
    return e ? __uint_as_float(((e + 120) << 23) | (m << 20)) : (float)m * 0x1p-9f;
}

template <typename In>
__device__ __forceinline__ void load16(const In* src, float* v) {
    if constexpr (sizeof(In) == 2) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
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
        for (int i = 0; i < 4; ++i) {
            uint4 q = ld_nc_v4(src + 4 * i);
            v[4 * i + 0] = __uint_as_float(q.x);
            v[4 * i + 1] = __uint_as_float(q.y);
            v[4 * i + 2] = __uint_as_float(q.z);
            v[4 * i + 3] = __uint_as_float(q.w);
        }
    }
}

// Pass 1: amax over the whole tensor.  Non-negative FP32 values order like their bit
// patterns, so the block maxima meet in one atomicMax on the bits.  Each thread
// takes four blocks of 16 a round, their loads issued before any is used.
template <typename In>
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const In* __restrict__ in, int64_t blocks16,
                                                         uint32_t* __restrict__ amax_bits) {
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; b + 3 * stride < blocks16; b += 4 * stride) {
        float v[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u) load16(in + (b + u * stride) * 16, v[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < 16; ++i) m = max(m, __float_as_uint(fabsf(v[u][i])));
    }
    for (; b < blocks16; b += stride) {
        float v[16];
        load16(in + b * 16, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) m = max(m, __float_as_uint(fabsf(v[i])));
    }
    m = __reduce_max_sync(0xffffffffu, m);
    __shared__ uint32_t part[8];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0u;
        m = __reduce_max_sync(0xffffffffu, m);
        if (threadIdx.x == 0 && m) atomicMax(amax_bits, m);
    }
}

// Pass 2: one thread per block of 16 (consecutive threads take consecutive blocks of
// a row).  Every FP32 step is one correctly rounded operation:
//   st = amax / 2688 (1 for an all-zero tensor),  sb = e4m3(amax_b / 6 / st),
//   d = value(sb) * st,  code_i = e2m1(x_i / d)  (all codes 0 when d is 0).
template <typename In>
__device__ __forceinline__ void nvfp4_block(float* v, float st, uint8_t* __restrict__ codes,
                                            uint8_t* __restrict__ scales, int64_t b) {
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[i]));
    const float t = __fdiv_rn(__fdiv_rn(am, 6.0f), st);
    const uint32_t sb = cvt_e4m3x2(t, 0.0f) & 0xFFu;
    const float d = __fmul_rn(e4m3_value(sb), st);
    uint2 out = make_uint2(0u, 0u);
    if (d != 0.0f) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __fdiv_rn(v[i], d);
        out.x = cvt_e2m1x8(v);
        out.y = cvt_e2m1x8(v + 8);
    }
    *reinterpret_cast<uint2*>(codes + b * 8) = out;
    scales[b] = (uint8_t)sb;
}

// Pass 2: blocks of 16 dealt over the threads (consecutive threads take consecutive
// blocks of a row), two a round with both loads issued first.  Every FP32 step is
// one correctly rounded operation:
//   st = amax / 2688 (1 for an all-zero tensor),  sb = e4m3(amax_b / 6 / st),
//   d = value(sb) * st,  code_i = e2m1(x_i / d)  (all codes 0 when d is 0).
template <typename In>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const In* __restrict__ in, int64_t rows,
                                                             int64_t K, float* __restrict__ st_amax,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
    const float amax = st_amax[1];
    const float st = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    const int64_t total = rows * (K / 16);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; b + stride < total; b += 2 * stride) {
        float v0[16], v1[16];
        load16(in + b * 16, v0);
        load16(in + (b + stride) * 16, v1);
        nvfp4_block<In>(v0, st, codes, scales, b);
        nvfp4_block<In>(v1, st, codes, scales, b + stride);
    }
    if (b < total) {
        float v[16];
        load16(in + b * 16, v);
        nvfp4_block<In>(v, st, codes, scales, b);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) st_amax[0] = st;
}

cudaError_t launch_quantize_nvfp4(const void* in, int in_dtype, int64_t rows, int64_t K,
                                  uint8_t* codes, uint8_t* scales, float* st_amax, int num_sms,
                                  cudaStream_t stream) {
    const int64_t total = rows * (K / 16);
    cudaError_t err = cudaMemsetAsync(st_amax + 1, 0, sizeof(float), stream);
    if (err != cudaSuccess) return err;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    if (in_dtype == MOE_BF16) {
        const uint16_t* src = (const uint16_t*)in;
        nvfp4_amax_kernel<uint16_t><<<(unsigned)blocks, 256, 0, stream>>>(src, total, (uint32_t*)(st_amax + 1));
        quantize_nvfp4_kernel<uint16_t><<<(unsigned)blocks, 256, 0, stream>>>(src, rows, K, st_amax, codes,
                                                                              scales);
    } else {
        const float* src = (const float*)in;
        nvfp4_amax_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(src, total, (uint32_t*)(st_amax + 1));
        quantize_nvfp4_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(src, rows, K, st_amax, codes,
                                                                           scales);
    }
    return cudaGetLastError();
}

}  // namespace moe
