// gather.cu -- pull dispatch: the expert side reads the token rows it needs from
// the source shards, knowing only (source shard, row), and writes them into its
// own ring of token slots in expert-contiguous order.  ([MoK-2.37x] = "Cursor's
// MoK achieves 2.37x performance boost on NVIDIA GB300 NVL72", section 02: pull
// replaces push for the forward dispatch; the receiver arranges local placement.)
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kGatherWarps = 8;

// Copy n16 16-byte units, lanes interleaved, U loads in flight per lane.
template <int U>
__device__ __forceinline__ void copy_v4(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                        int n16, int lane) {
    int j = lane;
    for (; j + 32 * (U - 1) < n16; j += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = ld_nc_v4(src + 16 * (int64_t)(j + 32 * u));
#pragma unroll
        for (int u = 0; u < U; ++u) st_v4(dst + 16 * (int64_t)(j + 32 * u), v[u]);
    }
    for (; j < n16; j += 32) st_v4(dst + 16 * (int64_t)j, ld_nc_v4(src + 16 * (int64_t)j));
}

// Bytes not a multiple of 16 (small rows): 4-byte units.
__device__ __forceinline__ void copy_u32(uint8_t* dst, const uint8_t* src, int n4, int lane) {
    for (int j = lane; j < n4; j += 32)
        reinterpret_cast<uint32_t*>(dst)[j] = reinterpret_cast<const uint32_t*>(src)[j];
}

__device__ __forceinline__ void copy_row(uint8_t* dst, const uint8_t* src, int bytes, int lane) {
    if ((bytes & 15) == 0)
        copy_v4<8>(dst, src, bytes >> 4, lane);
    else
        copy_u32(dst, src, bytes >> 2, lane);
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
        copy_row(ring + dst_row * row_bytes, shard_rows[s] + (int64_t)r * row_bytes, row_bytes,
                 lane);
        if (scale_bytes)
            copy_row(ring_scales + dst_row * scale_bytes,
                     shard_scales[s] + (int64_t)r * scale_bytes, scale_bytes, lane);
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
