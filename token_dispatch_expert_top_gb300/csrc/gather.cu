// gather.cu -- pull dispatch: the expert side reads the token rows it needs from
// the source shards, knowing only (source shard, row), and writes them into its
// own ring of token slots in expert-contiguous order.  ([MoK-2.37x] = "Cursor's
// MoK achieves 2.37x performance boost on NVIDIA GB300 NVL72", section 02: pull
// replaces push for the forward dispatch; the receiver arranges local placement.)
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kGatherWarps = 8;

// Copy a row of n16 16-byte units (plus an optional second row of m16 units, the
// scales) with every load of a batch issued before any store: up to 16 + 1
// 16-byte loads in flight per lane.
__device__ __forceinline__ void copy_rows_v4(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                             int n16, uint8_t* __restrict__ dst2,
                                             const uint8_t* __restrict__ src2, int m16, int lane) {
    constexpr int U = 16;
    for (int b = 0; b < n16 || b < m16; b += 32 * U) {
        uint4 v[U], w;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = b + lane + 32 * u;
            if (j < n16) v[u] = ld_nc_v4(src + 16 * (int64_t)j);
        }
        const int j2 = b + lane;
        if (j2 < m16) w = ld_nc_v4(src2 + 16 * (int64_t)j2);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = b + lane + 32 * u;
            if (j < n16) st_v4(dst + 16 * (int64_t)j, v[u]);
        }
        if (j2 < m16) st_v4(dst2 + 16 * (int64_t)j2, w);
    }
}

// Bytes not a multiple of 16 (small rows): 4-byte units.
__device__ __forceinline__ void copy_u32(uint8_t* dst, const uint8_t* src, int n4, int lane) {
    for (int j = lane; j < n4; j += 32)
        reinterpret_cast<uint32_t*>(dst)[j] = reinterpret_cast<const uint32_t*>(src)[j];
}

// One warp per slot, grid-stride.  Slot t goes to ring row t % ring_slots.
__global__ void __launch_bounds__(kGatherWarps * 32) dispatch_pull_kernel(
    const uint8_t* const* __restrict__ shard_rows, const uint8_t* const* __restrict__ shard_scales,
    const int32_t* __restrict__ sched, int slot_begin, int slot_count, int S, int rows_per_shard,
    int row_bytes, int scale_bytes, uint8_t* __restrict__ ring, uint8_t* __restrict__ ring_scales,
    int ring_slots, WsHeader* ws) {
    const int lane = threadIdx.x % 32;
    const int gw = blockIdx.x * kGatherWarps + threadIdx.x / 32;
    const int nw = gridDim.x * kGatherWarps;
    for (int i = gw; i < slot_count; i += nw) {
        const int t = slot_begin + i;
        const int s = sched[2 * (int64_t)t];
        const int r = sched[2 * (int64_t)t + 1];
        if (s < 0 || s >= S || r < 0 || r >= rows_per_shard) {
            if (lane == 0) set_status(ws, MOE_ERR_DEVICE_CHECK);
            continue;
        }
        const int64_t dst_row = t % ring_slots;
        uint8_t* drow = ring + dst_row * row_bytes;
        const uint8_t* srow = shard_rows[s] + (int64_t)r * row_bytes;
        uint8_t* dsc = scale_bytes ? ring_scales + dst_row * scale_bytes : nullptr;
        const uint8_t* ssc = scale_bytes ? shard_scales[s] + (int64_t)r * scale_bytes : nullptr;
        if ((row_bytes & 15) == 0 && (scale_bytes & 15) == 0) {
            copy_rows_v4(drow, srow, row_bytes >> 4, dsc, ssc, scale_bytes >> 4, lane);
        } else {
            if ((row_bytes & 15) == 0)
                copy_rows_v4(drow, srow, row_bytes >> 4, nullptr, nullptr, 0, lane);
            else
                copy_u32(drow, srow, row_bytes >> 2, lane);
            if (scale_bytes) copy_u32(dsc, ssc, scale_bytes >> 2, lane);
        }
    }
}

cudaError_t launch_dispatch_pull(const void* const* shard_rows, const void* const* shard_scales,
                                 const int32_t* sched, int slot_begin, int slot_count, int S,
                                 int rows_per_shard, int row_bytes, int scale_bytes, void* ring,
                                 void* ring_scales, int ring_slots, int num_sms, WsHeader* ws,
                                 cudaStream_t stream) {
    if (slot_count <= 0) return cudaSuccess;
    int blocks = (slot_count + kGatherWarps - 1) / kGatherWarps;
    if (blocks > num_sms * 8) blocks = num_sms * 8;
    dispatch_pull_kernel<<<blocks, kGatherWarps * 32, 0, stream>>>(
        (const uint8_t* const*)shard_rows, (const uint8_t* const*)shard_scales, sched, slot_begin,
        slot_count, S, rows_per_shard, row_bytes, scale_bytes, (uint8_t*)ring,
        (uint8_t*)ring_scales, ring_slots, ws);
    return cudaGetLastError();
}

}  // namespace moe
