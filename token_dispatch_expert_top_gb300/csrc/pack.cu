// pack.cu -- one-time repacking of the expert weights into the tile images the
// grouped GEMMs load with single bulk copies.
//
// The GEMMs consume B in tiles of 256 output rows x 128 bytes of K per K-stage
// (GEMM1: 128 W_gate rows then the matching 128 W_up rows; GEMM2: 256 W_down
// rows).  In the natural K-major layout such a tile is 256 separate 128-byte
// segments, i.e. 256 TMA row requests per stage.  Packed, each tile is the exact
// 32 KB shared-memory image the MMA reads (K-major, 128-byte swizzle: 16-byte
// chunk c of tile row r stored at chunk c ^ (r % 8) of that row), stored
// contiguously as [E][n-tile][k-stage][32 KB], so one bulk copy moves it.  The
// MXFP8 scales of a tile are packed the same way as the 1 KB image tcgen05.cp
// moves into tensor memory: two [32 lanes][4 words] blocks, word j of lane r of
// block c holding the four K-step scale bytes of tile row 128c + 32j + r.
// Packed and natural layouts have the same size.  FP32 weights are used by the
// SIMT path in their natural layout and are copied unchanged.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// Weight row of tile row r (0..255) of N tile n.
__device__ __forceinline__ int tile_row_src(bool gemm1, int n, int r, int I) {
    if (gemm1) return r < 128 ? n * 128 + r : I + n * 128 + (r - 128);
    return n * 256 + r;
}

// One thread per 16-byte chunk of the packed codes.
__global__ void __launch_bounds__(256) pack_tiles_kernel(const uint8_t* __restrict__ src, int E,
                                                         int rows, int kbytes, int I, bool gemm1,
                                                         uint8_t* __restrict__ dst) {
    const int KB = kbytes / 128;                   // K-stages of 128 bytes
    const int NT = gemm1 ? I / 128 : rows / 256;   // N tiles
    const int64_t total = (int64_t)E * NT * KB * 2048;   // 16-byte chunks (32 KB per tile)
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int pos = (int)(i & 2047);           // chunk position in the tile image
        const int64_t tile = i >> 11;
        const int kb = (int)(tile % KB);
        const int n = (int)((tile / KB) % NT);
        const int e = (int)(tile / ((int64_t)KB * NT));
        const int r = pos >> 3;                    // tile row
        const int c = (pos & 7) ^ (r & 7);         // K chunk held at this position
        const int srow = tile_row_src(gemm1, n, r, I);
        const uint8_t* s = src + ((int64_t)e * rows + srow) * kbytes + kb * 128 + c * 16;
        st_v4(dst + i * 16, ld_nc_v4(s));
    }
}

// One thread per 4-byte word of the packed scales (1 KB = 256 words per tile).
__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ src, int E,
                                                          int rows, int kbytes, int I, bool gemm1,
                                                          uint8_t* __restrict__ dst) {
    const int KB = kbytes / 128;
    const int NT = gemm1 ? I / 128 : rows / 256;
    const int ksf = kbytes / 32;                   // scale bytes per weight row
    const int64_t total = (int64_t)E * NT * KB * 256;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int w = (int)(i & 255);              // word in the 1 KB image
        const int64_t tile = i >> 8;
        const int kb = (int)(tile % KB);
        const int n = (int)((tile / KB) % NT);
        const int e = (int)(tile / ((int64_t)KB * NT));
        const int blk = w >> 7;                    // 128-row half of the tile
        const int lane = (w >> 2) & 31;
        const int j = w & 3;
        const int r = blk * 128 + 32 * j + lane;   // tile row
        const int srow = tile_row_src(gemm1, n, r, I);
        const uint8_t* s = src + ((int64_t)e * rows + srow) * ksf + kb * 4;
        reinterpret_cast<uint32_t*>(dst)[i] = *reinterpret_cast<const uint32_t*>(s);
    }
}

cudaError_t launch_pack_weights(const PackCall& c, cudaStream_t stream) {
    const int elem = c.mx ? 1 : 2;
    const int64_t cap = (int64_t)c.num_sms * 16;
    auto blocks = [&](int64_t n) { return (unsigned)((n + 255) / 256 < cap ? (n + 255) / 256 : cap); };
    // GEMM1: [E][2I][H] ; GEMM2: [E][H][I]
    const int kb1 = c.H * elem, kb2 = c.I * elem;
    pack_tiles_kernel<<<blocks((int64_t)c.E * 2 * c.I * c.H * elem / 16), 256, 0, stream>>>(
        (const uint8_t*)c.w_gate_up, c.E, 2 * c.I, kb1, c.I, true, (uint8_t*)c.p_gate_up);
    pack_tiles_kernel<<<blocks((int64_t)c.E * c.H * c.I * elem / 16), 256, 0, stream>>>(
        (const uint8_t*)c.w_down, c.E, c.H, kb2, c.I, false, (uint8_t*)c.p_down);
    if (c.mx) {
        pack_scales_kernel<<<blocks((int64_t)c.E * 2 * c.I * c.H / 128), 256, 0, stream>>>(
            c.w_gu_sf, c.E, 2 * c.I, kb1, c.I, true, c.p_gu_sf);
        pack_scales_kernel<<<blocks((int64_t)c.E * c.H * c.I / 128), 256, 0, stream>>>(
            c.w_d_sf, c.E, c.H, kb2, c.I, false, c.p_d_sf);
    }
    return cudaGetLastError();
}

}  // namespace moe
