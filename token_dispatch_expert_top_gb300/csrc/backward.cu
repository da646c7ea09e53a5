// backward.cu -- the memory-bound steps of the layer's backward pass, and the
// one-time packing of the expert weights for its dgrad GEMMs.
//
// [MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72": section 01 (training adds two exchanges in the direction opposite to
// dispatch and combine), section 02 (the backward pulls in the reverse combine and
// pushes in the reverse dispatch).  On one GPU:
//   reverse combine : every slot pulls its token's output gradient, scaled by the
//                     slot's gate (the dgrad GEMM operand, MXFP8-quantised along H
//                     or BF16), and the gate gradient dgate = <dout, y> of every
//                     (token, choice); the renormalised-gate Jacobian turns those
//                     into the selected logits' gradient in the same pass
//   reverse dispatch: every token adds its k slots' input gradients back, in j
//                     order through the inverse map (deterministic, no atomics),
//                     plus the router's input gradient sum_j dlogit_j W_r[e_j]
//   router wgrad    : dW_r[e] = sum over e's slots of dlogit * x[token], in slot
//                     order, as fixed pieces of 256 slots reduced in piece order
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// ------------------------------------------------------------- dgrad weight pack
// W natural [E][R][C] BF16 (the forward's K-major weight: R output rows, K = C).
// The dgrad GEMM needs W^T as its B operand: rows c (N), reduction over r (K).
// Packed like the forward's tiles: [E][ceil(C/256)][K-stages][32 KB], 16-byte
// chunk q of tile row t at chunk q ^ (t % 8); MXFP8 quantises along r (one scale
// per 32 consecutive r) and packs the scales as [..][K-stages][1 KB] images (word
// j of entry `lane` of half b holds the 4 K-step scales of tile row 128b+32j+lane).
// Tile rows past C are zero.  One thread per (e, c, 32-element block of r).
template <bool MX>
__global__ void __launch_bounds__(256) pack_transposed_kernel(const uint16_t* __restrict__ w, int E,
                                                              int R, int C, uint8_t* __restrict__ dst,
                                                              uint8_t* __restrict__ dst_sf) {
    const int Cp = (C + 255) / 256 * 256;
    const int nb = R / 32;
    const int KB = MX ? R / 128 : R / 64;
    const int NT = Cp / 256;
    const int64_t total = (int64_t)E * nb * Cp;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % Cp);                   // consecutive threads: consecutive c
        const int b = (int)((i / Cp) % nb);            // 32-row block of r
        const int e = (int)(i / ((int64_t)Cp * nb));
        float v[32];
        if (c < C) {
            const uint16_t* src = w + ((int64_t)e * R + (int64_t)b * 32) * C + c;
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = bf16_to_f32(src[(int64_t)q * C]);
        } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = 0.f;
        }
        const int n = c / 256, t = c % 256;
        if constexpr (MX) {
            uint32_t codes[8];
            const uint8_t s = mx_quantize32(v, codes);
            const int ks = b / 4, sub = b % 4;         // K-stage, 32-element step inside it
            uint8_t* tile = dst + (((int64_t)e * NT + n) * KB + ks) * 32768 + t * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int q = sub * 2 + h;
                st_v4(tile + ((q ^ (t & 7)) * 16),
                      make_uint4(codes[4 * h], codes[4 * h + 1], codes[4 * h + 2], codes[4 * h + 3]));
            }
            uint8_t* simg = dst_sf + (((int64_t)e * NT + n) * KB + ks) * 1024;
            const int half = t / 128, j = (t % 128) / 32, lane = t % 32;
            simg[(half * 128 + lane * 4 + j) * 4 + sub] = s;
        } else {
            uint32_t pk[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) pk[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
            const int ks = b / 2, sub = b % 2;         // 64 BF16 per K-stage
            uint8_t* tile = dst + (((int64_t)e * NT + n) * KB + ks) * 32768 + t * 128;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int q = sub * 4 + h;
                st_v4(tile + ((q ^ (t & 7)) * 16),
                      make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]));
            }
        }
    }
}

cudaError_t launch_pack_transposed(bool mx, const void* w, int E, int R, int C, void* dst,
                                   uint8_t* dst_sf, int num_sms, cudaStream_t stream) {
    const int Cp = (C + 255) / 256 * 256;
    const int64_t total = (int64_t)E * (R / 32) * Cp;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (mx)
        pack_transposed_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(
            (const uint16_t*)w, E, R, C, (uint8_t*)dst, dst_sf);
    else
        pack_transposed_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(
            (const uint16_t*)w, E, R, C, (uint8_t*)dst, nullptr);
    return cudaGetLastError();
}

// ------------------------------------------------------------- reverse combine
__device__ __forceinline__ void unpack_bf16x8(const uint4& q, float* f) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        f[2 * p] = bf16_to_f32((uint16_t)(w[p] & 0xFFFF));
        f[2 * p + 1] = bf16_to_f32((uint16_t)(w[p] >> 16));
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kBwdWarps = 8;

// One warp per token n.  Lane l covers columns 256c + 8l .. +7 of every 256-column
// chunk c, so four consecutive lanes hold one 32-element MX block.  For each of
// the token's k slots s_j (gate g_j):
//   dy[s_j]   = g_j * dout[n]  (FP32 product; MXFP8: the block amax is combined
//               over the four lanes and the codes follow the row quantiser's rule
//               exactly; BF16: rounded to nearest even)
//   dgate_j   = <dout[n], y[s_j]>  (per-lane FP32 partial sums, then a fixed
//               butterfly over the warp)
// then dlogit_j = g_j (dgate_j - sum_i g_i dgate_i), written per (token, choice)
// and per slot (with the slot's gate) for the router and expert weight gradients.
// A slot index outside [0, T) skips the token and records MOE_ERR_DEVICE_CHECK.
template <bool MX, int KMAX>
__global__ void __launch_bounds__(kBwdWarps * 32) reverse_combine_kernel(
    const uint16_t* __restrict__ dout, const uint16_t* __restrict__ y, const int32_t* __restrict__ inv,
    const float* __restrict__ gate, int N, int H, int k, int T, uint8_t* __restrict__ dy,
    uint8_t* __restrict__ dy_sf, float* __restrict__ dgate, float* __restrict__ dlogit,
    float* __restrict__ slot_gate, float* __restrict__ slot_dlogit, WsHeader* ws) {
    const int lane = threadIdx.x % 32;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + threadIdx.x / 32;
    const int64_t nw = (int64_t)gridDim.x * kBwdWarps;
    for (int64_t n = gw; n < N; n += nw) {
        const int my_slot = lane < k ? inv[n * k + lane] : 0;
        const float my_g = lane < k ? gate[n * k + lane] : 0.f;
        if (__any_sync(0xffffffffu, my_slot < 0 || my_slot >= T)) {
            if (lane == 0) set_status(ws, MOE_ERR_DEVICE_CHECK);
            continue;
        }
        int slot[KMAX];
        float g[KMAX], dot[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
            g[j] = __shfl_sync(0xffffffffu, my_g, j);
            dot[j] = 0.f;
        }
        for (int col = lane * 8; col < H; col += 256) {
            float d[8];
            unpack_bf16x8(ld_nc_v4(dout + n * H + col), d);
            uint4 yv[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < k) yv[j] = ld_nc_v4(y + (int64_t)slot[j] * H + col);
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j >= k) continue;
                float yy[8], s[8];
                unpack_bf16x8(yv[j], yy);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    dot[j] = fmaf(d[q], yy[q], dot[j]);
                    s[q] = g[j] * d[q];
                }
                const int64_t row = slot[j];
                if constexpr (MX) {
                    float amax = 0.f;
#pragma unroll
                    for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(s[q]));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                    const int se = mx_scale_exponent(amax);
                    const float is = mx_inv_scale(se);
                    const uint32_t lo = (uint32_t)cvt_e4m3x2(s[0] * is, s[1] * is) |
                                        ((uint32_t)cvt_e4m3x2(s[2] * is, s[3] * is) << 16);
                    const uint32_t hi = (uint32_t)cvt_e4m3x2(s[4] * is, s[5] * is) |
                                        ((uint32_t)cvt_e4m3x2(s[6] * is, s[7] * is) << 16);
                    *reinterpret_cast<uint2*>(dy + row * H + col) = make_uint2(lo, hi);
                    if ((lane & 3) == 0) dy_sf[row * (H / 32) + col / 32] = (uint8_t)(se + 127);
                } else {
                    st_v4(dy + (row * H + col) * 2,
                          make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]),
                                     pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7])));
                }
            }
        }
        float mean = 0.f, mine_dot = 0.f, mine_g = 0.f;
        int mine_slot = 0;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j >= k) continue;
            const float t = warp_sum(dot[j]);
            mean = fmaf(g[j], t, mean);
            if (lane == j) {
                mine_dot = t;
                mine_g = g[j];
                mine_slot = slot[j];
            }
        }
        if (lane < k) {
            const float dl = mine_g * (mine_dot - mean);
            dgate[n * k + lane] = mine_dot;
            dlogit[n * k + lane] = dl;
            slot_gate[mine_slot] = mine_g;
            slot_dlogit[mine_slot] = dl;
        }
    }
}

cudaError_t launch_reverse_combine(bool mx, const void* dout, const void* y, const int32_t* inv,
                                   const float* gate, int N, int H, int k, int T, void* dy,
                                   uint8_t* dy_sf, float* dgate, float* dlogit, float* slot_gate,
                                   float* slot_dlogit, int num_sms, WsHeader* ws, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    int64_t blocks = ((int64_t)N + kBwdWarps - 1) / kBwdWarps;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
#define MOE_RC_LAUNCH(MXV, KM)                                                                   \
    reverse_combine_kernel<MXV, KM><<<(unsigned)blocks, kBwdWarps * 32, 0, stream>>>(            \
        (const uint16_t*)dout, (const uint16_t*)y, inv, gate, N, H, k, T, (uint8_t*)dy, dy_sf,   \
        dgate, dlogit, slot_gate, slot_dlogit, ws)
    if (mx) {
        if (k <= 8) MOE_RC_LAUNCH(true, 8);
        else if (k <= 16) MOE_RC_LAUNCH(true, 16);
        else MOE_RC_LAUNCH(true, 32);
    } else {
        if (k <= 8) MOE_RC_LAUNCH(false, 8);
        else if (k <= 16) MOE_RC_LAUNCH(false, 16);
        else MOE_RC_LAUNCH(false, 32);
    }
#undef MOE_RC_LAUNCH
    return cudaGetLastError();
}

// ------------------------------------------------------------- SwiGLU backward
// One thread per (slot row t, 8 consecutive columns of I); four consecutive lanes
// hold one 32-column MX block (I/8 is a multiple of 4, so blocks never straddle a
// row).  With s = sigma(u):
//   du = dh * v * (s + u s (1 - s)),   dv = dh * u * s
// from BF16 dh and the kept BF16 u|v, in FP32; du|dv stored as BF16 (du in
// columns 0..I-1, dv in I..2I-1) and, MXFP8, quantised along I per 32-block (the
// block amax combined over the four lanes, then the row quantiser's rule).
template <bool MX>
__global__ void __launch_bounds__(256) swiglu_backward_kernel(const uint16_t* __restrict__ dh,
                                                              const uint16_t* __restrict__ uv, int T, int I,
                                                              uint16_t* __restrict__ duv,
                                                              uint8_t* __restrict__ duv_q,
                                                              uint8_t* __restrict__ duv_sf) {
    const int ng = I / 8;
    const int64_t total = (int64_t)T * ng;
    const int lane = threadIdx.x % 32;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // every lane of a warp runs the same number of iterations (the shuffles need all 32)
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x - lane); base < total; base += stride) {
        const int64_t b = base + lane;
        const bool ok = b < total;
        const int64_t r = ok ? b / ng : 0;
        const int col = ok ? (int)(b % ng) * 8 : 0;
        float d[8], u[8], v[8];
        if (ok) {
            unpack_bf16x8(ld_nc_v4(dh + r * I + col), d);
            unpack_bf16x8(ld_nc_v4(uv + r * 2 * I + col), u);
            unpack_bf16x8(ld_nc_v4(uv + r * 2 * I + I + col), v);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) d[q] = u[q] = v[q] = 0.f;
        }
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float s = 1.0f / (1.0f + expf(-u[q]));
                o[q] = part == 0 ? d[q] * v[q] * (s + u[q] * s * (1.0f - s)) : d[q] * u[q] * s;
            }
            const int64_t c = col + (part ? I : 0);
            if (ok)
                st_v4(duv + r * 2 * I + c, make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                                      pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7])));
            if constexpr (MX) {
                float amax = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(o[q]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const int se = mx_scale_exponent(amax);
                const float is = mx_inv_scale(se);
                const uint32_t lo = (uint32_t)cvt_e4m3x2(o[0] * is, o[1] * is) |
                                    ((uint32_t)cvt_e4m3x2(o[2] * is, o[3] * is) << 16);
                const uint32_t hi = (uint32_t)cvt_e4m3x2(o[4] * is, o[5] * is) |
                                    ((uint32_t)cvt_e4m3x2(o[6] * is, o[7] * is) << 16);
                if (ok) {
                    *reinterpret_cast<uint2*>(duv_q + r * 2 * I + c) = make_uint2(lo, hi);
                    if ((lane & 3) == 0) duv_sf[r * (2 * I / 32) + c / 32] = (uint8_t)(se + 127);
                }
            }
        }
    }
}

cudaError_t launch_swiglu_backward(bool mx, const void* dh, const void* uv, int T, int I, void* duv,
                                   uint8_t* duv_q, uint8_t* duv_sf, int num_sms, cudaStream_t stream) {
    const int64_t total = (int64_t)T * (I / 8);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (mx)
        swiglu_backward_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(
            (const uint16_t*)dh, (const uint16_t*)uv, T, I, (uint16_t*)duv, duv_q, duv_sf);
    else
        swiglu_backward_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(
            (const uint16_t*)dh, (const uint16_t*)uv, T, I, (uint16_t*)duv, nullptr, nullptr);
    return cudaGetLastError();
}

// ------------------------------------------------------------- reverse dispatch
// Work item = (token n, 256-column chunk); one warp per item, 8 columns per lane.
//   dx[n] = sum_j da[inv[n][j]]  +  sum_j dlogit[n][j] * W_r[idx[n][j]]
// both sums in j order in FP32 (the slot part first), rounded once to BF16.  Few
// registers per thread, so many warps per SM keep the row loads in flight (the
// forward combine's pattern).  A slot or expert index out of range skips that
// term and records MOE_ERR_DEVICE_CHECK.
__global__ void __launch_bounds__(kBwdWarps * 32) reverse_dispatch_kernel(
    const uint16_t* __restrict__ da, const int32_t* __restrict__ inv, const int32_t* __restrict__ idx,
    const float* __restrict__ dlogit, const uint16_t* __restrict__ w_router, int N, int H, int k,
    int T, int E, uint16_t* __restrict__ dx, WsHeader* ws) {
    const int lane = threadIdx.x % 32;
    const int chunks = H / 256;
    const int64_t items = (int64_t)N * chunks;
    const int64_t gw = (int64_t)blockIdx.x * kBwdWarps + threadIdx.x / 32;
    const int64_t nw = (int64_t)gridDim.x * kBwdWarps;
    for (int64_t it = gw; it < items; it += nw) {
        const int64_t n = it / chunks;
        const int col = (int)(it % chunks) * 256 + lane * 8;
        int my_slot = lane < k ? inv[n * k + lane] : 0;
        const int my_e = lane < k ? idx[n * k + lane] : 0;
        const float my_dl = lane < k ? dlogit[n * k + lane] : 0.f;
        if (lane < k && (my_slot < 0 || my_slot >= T || my_e < 0 || my_e >= E)) {
            set_status(ws, MOE_ERR_DEVICE_CHECK);
            my_slot = -1;
        }
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, j);
            if (slot < 0) continue;
            float f[8];
            unpack_bf16x8(ld_nc_v4(da + (int64_t)slot * H + col), f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
        for (int j = 0; j < k; ++j) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, j);
            const int e = __shfl_sync(0xffffffffu, my_e, j);
            const float dl = __shfl_sync(0xffffffffu, my_dl, j);
            if (slot < 0) continue;
            float f[8];
            unpack_bf16x8(ld_nc_v4(w_router + (int64_t)e * H + col), f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(dl, f[q], acc[q]);
        }
        st_v4(dx + n * H + col, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                           pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
    }
}

cudaError_t launch_reverse_dispatch(const void* da, const int32_t* inv, const int32_t* idx,
                                    const float* dlogit, const void* w_router, int N, int H, int k,
                                    int T, int E, void* dx, int num_sms, WsHeader* ws,
                                    cudaStream_t stream) {
    const int64_t items = (int64_t)N * (H / 256);
    if (items == 0) return cudaSuccess;
    int64_t blocks = (items + kBwdWarps - 1) / kBwdWarps;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    reverse_dispatch_kernel<<<(unsigned)blocks, kBwdWarps * 32, 0, stream>>>(
        (const uint16_t*)da, inv, idx, dlogit, (const uint16_t*)w_router, N, H, k, T, E, (uint16_t*)dx, ws);
    return cudaGetLastError();
}

// ----------------------------------------------------------------- router wgrad
// Pieces: expert e's slots [offsets[e], offsets[e+1]) cut into ceil(count/256)
// pieces of 256 (the last shorter); piece p of the whole layer is the p-th in
// expert order.  ppre[e] = pieces before expert e (ppre[E] = all pieces).
__device__ void piece_prefix(const int32_t* offsets, int E, int32_t* ppre) {
    const int lane = threadIdx.x % 32;
    const int per = (E + 31) / 32;
    const int lo = min(lane * per, E), hi = min(lo + per, E);
    int s = 0;
    for (int e = lo; e < hi; ++e) s += (offsets[e + 1] - offsets[e] + kRouterPiece - 1) / kRouterPiece;
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - s;
    for (int e = lo; e < hi; ++e) {
        ppre[e] = run;
        run += (offsets[e + 1] - offsets[e] + kRouterPiece - 1) / kRouterPiece;
    }
    if (lane == 31) ppre[E] = incl;
}

// CTA (piece p, 1024-column chunk): part[p][h] = sum over the piece's slots s, in
// slot order, of slot_dlogit[s] * x[token(s)][h], FP32; part_b[p] = sum of the
// piece's slot_dlogit.  Each thread owns 4 columns (8-byte loads of x rows).
__global__ void __launch_bounds__(256) router_wgrad_partial_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ sched, const int32_t* __restrict__ offsets,
    const float* __restrict__ slot_dlogit, int E, int H, int N, int rows_per_shard,
    float* __restrict__ part, float* __restrict__ part_b, int32_t* __restrict__ ppre_out, WsHeader* ws) {
    extern __shared__ int32_t ppre[];
    if (threadIdx.x < 32) piece_prefix(offsets, E, ppre);
    __syncthreads();
    const int p = blockIdx.x;
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) ppre_out[e] = ppre[e];
    if (p >= ppre[E]) return;
    int lo = 0, hi = E;   // last e with ppre[e] <= p
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ppre[mid] <= p) lo = mid; else hi = mid;
    }
    const int s0 = offsets[lo] + (p - ppre[lo]) * kRouterPiece;
    const int s1 = min(s0 + kRouterPiece, offsets[lo + 1]);
    const int h = blockIdx.y * 1024 + threadIdx.x * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float accb = 0.f;
    for (int s = s0; s < s1; ++s) {
        const int64_t tok = (int64_t)sched[2 * s] * rows_per_shard + sched[2 * s + 1];
        const float d = slot_dlogit[s];
        accb += d;
        if (tok < 0 || tok >= N) {
            if (threadIdx.x == 0) set_status(ws, MOE_ERR_DEVICE_CHECK);
            continue;
        }
        if (h < H) {
            const uint2 q = *reinterpret_cast<const uint2*>(x + tok * H + h);
            acc[0] = fmaf(d, bf16_to_f32((uint16_t)(q.x & 0xFFFF)), acc[0]);
            acc[1] = fmaf(d, bf16_to_f32((uint16_t)(q.x >> 16)), acc[1]);
            acc[2] = fmaf(d, bf16_to_f32((uint16_t)(q.y & 0xFFFF)), acc[2]);
            acc[3] = fmaf(d, bf16_to_f32((uint16_t)(q.y >> 16)), acc[3]);
        }
    }
    if (h < H)
        *reinterpret_cast<float4*>(part + (int64_t)p * H + h) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (blockIdx.y == 0 && threadIdx.x == 0) part_b[p] = accb;
}

// CTA (expert e, 1024-column chunk): dW_r[e][h] = sum of e's pieces in piece
// order; dbias[e] likewise.  An expert without slots gets zeros.
__global__ void __launch_bounds__(256) router_wgrad_reduce_kernel(
    const float* __restrict__ part, const float* __restrict__ part_b, const int32_t* __restrict__ ppre,
    int E, int H, float* __restrict__ dw, float* __restrict__ db) {
    const int e = blockIdx.x;
    const int h = blockIdx.y * 1024 + threadIdx.x * 4;
    const int p0 = ppre[e], p1 = ppre[e + 1];
    if (h < H) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = p0; p < p1; ++p) {
            const float4 v = *reinterpret_cast<const float4*>(part + (int64_t)p * H + h);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        *reinterpret_cast<float4*>(dw + (int64_t)e * H + h) = acc;
    }
    if (blockIdx.y == 0 && threadIdx.x == 0 && db) {
        float b = 0.f;
        for (int p = p0; p < p1; ++p) b += part_b[p];
        db[e] = b;
    }
}

cudaError_t launch_router_wgrad(const void* x, const int32_t* sched, const int32_t* offsets,
                                const float* slot_dlogit, int N, int H, int E, int T,
                                int rows_per_shard, float* dw, float* db, float* part, float* part_b,
                                int32_t* ppre, WsHeader* ws, cudaStream_t stream) {
    const int pmax = router_max_pieces(T, E);
    const dim3 g1((unsigned)pmax, (unsigned)((H + 1023) / 1024));
    router_wgrad_partial_kernel<<<g1, 256, sizeof(int32_t) * (E + 1), stream>>>(
        (const uint16_t*)x, sched, offsets, slot_dlogit, E, H, N, rows_per_shard, part, part_b, ppre, ws);
    const dim3 g2((unsigned)E, (unsigned)((H + 1023) / 1024));
    router_wgrad_reduce_kernel<<<g2, 256, 0, stream>>>(part, part_b, ppre, E, H, dw, db);
    return cudaGetLastError();
}

}  // namespace moe
