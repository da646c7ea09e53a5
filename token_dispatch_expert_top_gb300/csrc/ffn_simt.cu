// ffn_simt.cu -- FP32 grouped SwiGLU expert FFN on the SIMT cores (the FP32
// layer keeps full FP32 products, which the tensor cores do not offer).  Slot
// rows of expert e are [offsets[e], offsets[e+1]); each thread computes one
// output element with a sequential FP32 dot product over K.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// Expert owning slot row t: the e with offsets[e] <= t < offsets[e+1].
__device__ __forceinline__ int expert_of_row(const int32_t* off, int E, int t) {
    int lo = 0, hi = E;  // find the last e with off[e] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ float dot_f32(const float* __restrict__ a, const float* __restrict__ b,
                                         int K) {
    float acc = 0.f;
    if ((K & 3) == 0) {
        const float4* a4 = reinterpret_cast<const float4*>(a);
        const float4* b4 = reinterpret_cast<const float4*>(b);
        for (int i = 0; i < K / 4; ++i) {
            const float4 x = a4[i], w = b4[i];
            acc = fmaf(x.x, w.x, acc);
            acc = fmaf(x.y, w.y, acc);
            acc = fmaf(x.z, w.z, acc);
            acc = fmaf(x.w, w.w, acc);
        }
    } else {
        for (int i = 0; i < K; ++i) acc = fmaf(a[i], b[i], acc);
    }
    return acc;
}

// h[t][i] = silu(a_t . Wg_e[i]) * (a_t . Wu_e[i])
__global__ void __launch_bounds__(256) ffn1_f32_kernel(const float* __restrict__ a,
                                                       const int32_t* __restrict__ offsets, int E,
                                                       const float* __restrict__ wgu, int T, int H,
                                                       int I, float* __restrict__ h) {
    extern __shared__ int32_t off[];
    for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = offsets[e];
    __syncthreads();
    const int64_t total = (int64_t)T * I;
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total;
         id += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(id / I), i = (int)(id % I);
        const int e = expert_of_row(off, E, t);
        const float* ar = a + (int64_t)t * H;
        const float* wg = wgu + ((int64_t)e * 2 * I + i) * H;
        const float* wu = wgu + ((int64_t)e * 2 * I + I + i) * H;
        const float u = dot_f32(ar, wg, H);
        const float v = dot_f32(ar, wu, H);
        h[id] = silu_f32(u) * v;
    }
}

// y[t][c] = h_t . Wd_e[c]
__global__ void __launch_bounds__(256) ffn2_f32_kernel(const float* __restrict__ h,
                                                       const int32_t* __restrict__ offsets, int E,
                                                       const float* __restrict__ wd, int T, int H,
                                                       int I, float* __restrict__ y) {
    extern __shared__ int32_t off[];
    for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = offsets[e];
    __syncthreads();
    const int64_t total = (int64_t)T * H;
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total;
         id += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(id / H), c = (int)(id % H);
        const int e = expert_of_row(off, E, t);
        y[id] = dot_f32(h + (int64_t)t * I, wd + ((int64_t)e * H + c) * I, I);
    }
}

cudaError_t launch_ffn_f32(const float* a, const int32_t* offsets, const float* wgu,
                           const float* wd, int T, int H, int I, int E, float* h_scratch, float* y,
                           int num_sms, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const size_t smem = sizeof(int32_t) * (E + 1);
    int64_t b1 = ((int64_t)T * I + 255) / 256, b2 = ((int64_t)T * H + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    ffn1_f32_kernel<<<(unsigned)(b1 < cap ? b1 : cap), 256, smem, stream>>>(a, offsets, E, wgu, T,
                                                                           H, I, h_scratch);
    ffn2_f32_kernel<<<(unsigned)(b2 < cap ? b2 : cap), 256, smem, stream>>>(h_scratch, offsets, E,
                                                                           wd, T, H, I, y);
    return cudaGetLastError();
}

}  // namespace moe
