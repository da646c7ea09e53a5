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
// scales) with every load of a batch issued before any store: up to 8 + 1
// 16-byte loads in flight per lane (a shallow batch keeps registers low, so many
// warps per SM keep enough bytes in flight).  Sources are read k times over the
// dispatch, so their lines are kept in L2; ring rows are streamed out.
__device__ __forceinline__ void copy_rows_v4(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                             int n16, uint8_t* __restrict__ dst2,
                                             const uint8_t* __restrict__ src2, int m16, int lane) {
    constexpr int U = 8;
    const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
    for (int b = 0; b < n16 || b < m16; b += 32 * U) {
        uint4 v[U], w;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = b + lane + 32 * u;
            if (j < n16) v[u] = ld_nc_v4_hint(src + 16 * (int64_t)j, keep);
        }
        const int j2 = b + lane;
        if (j2 < m16) w = ld_nc_v4_hint(src2 + 16 * (int64_t)j2, keep);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = b + lane + 32 * u;
            if (j < n16) st_v4_hint(dst + 16 * (int64_t)j, v[u], stream);
        }
        if (j2 < m16) st_v4_hint(dst2 + 16 * (int64_t)j2, w, stream);
    }
}

// Bytes not a multiple of 16 (small rows): 4-byte units.
__device__ __forceinline__ void copy_u32(uint8_t* dst, const uint8_t* src, int n4, int lane) {
    for (int j = lane; j < n4; j += 32)
        reinterpret_cast<uint32_t*>(dst)[j] = reinterpret_cast<const uint32_t*>(src)[j];
}

// One warp per slot, grid-stride.  Slot t goes to ring row t % ring_slots.
__global__ void __launch_bounds__(kGatherWarps * 32, 2) dispatch_pull_kernel(
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

// ----------------------------------------------------------- bulk-copy variant
// Rows whose code and scale lengths are multiples of 16 bytes move through the
// bulk-copy engine: in each warp one lane streams its slots through a ring of
// row buffers in shared memory -- a bulk load (source row kept in L2: it is read
// k times over the dispatch) then a bulk store of the same buffer (ring rows
// streamed out) -- so a few threads per SM keep ~100 KB+ in flight without
// holding the data in registers.  A buffer is refilled once the bulk store that
// read it is LAG stores old and has finished reading (bulk-group accounting).
// This kernel visits the slots in slot order (no inverse map given); with the
// inverse map the token-broadcast kernel below is used.
// Sizing (both kernels), measured on the DeepSeek-V3 layer's dispatch (545 MB,
// L2 flushed): a store lag of 1 and two CTAs of 4 warps per SM (about 100 KB of
// buffers each).
constexpr int kBulkWarps = 4;
constexpr int kBulkLag = 1;
constexpr int kBulkMaxBuf = 16;

__global__ void __launch_bounds__(kBulkWarps * 32, 1) dispatch_bulk_kernel(
    const uint8_t* const* __restrict__ shard_rows, const uint8_t* const* __restrict__ shard_scales,
    const int32_t* __restrict__ sched, int slot_begin, int slot_count, int S, int rows_per_shard,
    int row_bytes, int scale_bytes, uint8_t* __restrict__ ring, uint8_t* __restrict__ ring_scales,
    int ring_slots, int nbuf, WsHeader* ws, unsigned long long timeout_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort[kBulkWarps];
    __shared__ int s_slot[kBulkWarps][kBulkMaxBuf];   // destination slot of each row buffer
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int unit = row_bytes + scale_bytes;
    uint8_t* buf = smem + (size_t)warp * nbuf * unit;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kBulkWarps * nbuf * unit) + warp * kBulkMaxBuf;
    if (lane == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(&bars[b], 1);
        s_abort[warp] = 0;
        fence_mbar_init();
    }
    __syncwarp();

    // This warp's positions (slot_begin + position): chunks of 32 consecutive
    // positions, chunk c = gw + i * nw.
    const int npos = slot_count;
    const int gw = blockIdx.x * kBulkWarps + warp, nw = gridDim.x * kBulkWarps;
    const int nchunks = (npos + 31) / 32;
    if (gw >= nchunks) return;
    const int my_chunks = (nchunks - gw + nw - 1) / nw;
    const int last = gw + (my_chunks - 1) * nw;
    const int total = (my_chunks - 1) * 32 + min(32, npos - last * 32);
    auto pos_of = [&](int q) { return (gw + (q >> 5) * nw) * 32 + (q & 31); };

    const unsigned long long deadline = globaltimer_ns() + timeout_ns;
    const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
    volatile int* abort_flag = &s_abort[warp];
    uint32_t bad = 0;          // bit b: buffer b holds nothing to store (skipped or invalid)
    int chunk_sched_q = -1;    // first q of the chunk whose schedule entries the lanes hold
    int my_s = 0, my_r = 0, my_t = -1;

    // Issue the bulk load of the q-th slot into buffer q % nbuf (all lanes call;
    // lane 0 issues).
    auto load = [&](int q) {
        const int c0 = q & ~31;
        if (c0 != chunk_sched_q) {
            chunk_sched_q = c0;
            const int i = pos_of(c0) + lane;
            my_t = -1;
            if (i < npos) {
                const int t = slot_begin + i;
                my_t = t;
                my_s = sched[2 * (int64_t)t];
                my_r = sched[2 * (int64_t)t + 1];
            }
        }
        const int sidx = __shfl_sync(0xffffffffu, my_s, q & 31);
        const int ridx = __shfl_sync(0xffffffffu, my_r, q & 31);
        const int tq = __shfl_sync(0xffffffffu, my_t, q & 31);
        if (lane == 0) {
            const int b = q % nbuf;
            uint8_t* dst = buf + (size_t)b * unit;
            s_slot[warp][b] = tq;
            if (tq < 0) {                  // not this call's slot
                bad |= 1u << b;
                mbar_arrive(&bars[b]);
                return;
            }
            bool ok = sidx >= 0 && sidx < S && ridx >= 0 && ridx < rows_per_shard;
            const uint8_t* src = ok ? shard_rows[sidx] + (int64_t)ridx * row_bytes : nullptr;
            const uint8_t* ssrc = (ok && scale_bytes) ? shard_scales[sidx] + (int64_t)ridx * scale_bytes : nullptr;
            if (ok && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(ssrc)) & 15)) ok = false;
            if (ok) {
                bad &= ~(1u << b);
                mbar_arrive_expect_tx(&bars[b], (uint32_t)unit);
                bulk_load_hint(dst, src, (uint32_t)row_bytes, &bars[b], keep);
                if (scale_bytes) bulk_load_hint(dst + row_bytes, ssrc, (uint32_t)scale_bytes, &bars[b], keep);
            } else {
                set_status(ws, MOE_ERR_DEVICE_CHECK);
                bad |= 1u << b;
                mbar_arrive(&bars[b]);
            }
        }
    };

    const int pre = min(nbuf, total);
    for (int q = 0; q < pre; ++q) load(q);
    int q = 0;
    for (; q < total; ++q) {
        if (lane == 0) {
            const int b = q % nbuf;
            if (!mbar_wait_bounded(&bars[b], (uint32_t)((q / nbuf) & 1), abort_flag, ws, deadline)) {
                // give up: nothing more is issued; drain what is in flight below
            } else if (!(bad & (1u << b))) {
                fence_proxy_async_smem();
                const int64_t dr = s_slot[warp][b] % ring_slots;
                const uint8_t* src = buf + (size_t)b * unit;
                bulk_store_hint(ring + dr * row_bytes, src, (uint32_t)row_bytes, stream);
                if (scale_bytes)
                    bulk_store_hint(ring_scales + dr * scale_bytes, src + row_bytes, (uint32_t)scale_bytes, stream);
            }
            bulk_commit_group();
            bulk_wait_group_read<kBulkLag>();
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int qn = q - kBulkLag + nbuf;     // refill the buffer whose store is now LAG old
        if (q >= kBulkLag && qn < total) load(qn);
    }
    if (lane == 0) {
        if (*abort_flag) {
            // let loads already issued land before the block's shared memory goes away
            const unsigned long long d2 = globaltimer_ns() + 1000000ull;
            while (globaltimer_ns() < d2) {
            }
        }
        bulk_wait_group_all();
    }
}

// ------------------------------------------------------ token-broadcast variant
// With the inverse map, the k slots of token n all pull the same source row: the
// warp reads each slot's schedule entry, fetches the row named by the first slot
// in range once (one bulk load into a shared-memory buffer) and writes it to every
// slot in range with k bulk stores from that buffer.  A slot whose schedule entry
// names another row is skipped and recorded as MOE_ERR_DEVICE_CHECK (inv and
// sched come from one moe_layout call, where this cannot happen).  One HBM read
// per token feeds k ring rows, so few loads in flight keep the stores busy and
// the kernel runs at the HBM write rate.  Warp w takes tokens w, w + nw, ...; a
// buffer is refilled once its store group is LAG groups old and has finished
// reading it.
constexpr int kBcastMaxBuf = 8;

__global__ void __launch_bounds__(kBulkWarps * 32, 1) dispatch_bcast_kernel(
    const uint8_t* const* __restrict__ shard_rows, const uint8_t* const* __restrict__ shard_scales,
    const int32_t* __restrict__ sched, const int32_t* __restrict__ inv, int N, int k, int slot_begin,
    int slot_count, int S, int rows_per_shard, int row_bytes, int scale_bytes, uint8_t* __restrict__ ring,
    uint8_t* __restrict__ ring_scales, int ring_slots, int nbuf, WsHeader* ws, unsigned long long timeout_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort[kBulkWarps];
    __shared__ int s_dst[kBulkWarps][kBcastMaxBuf][32];   // ring row per slot of the buffer's token (-1: none)
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int unit = row_bytes + scale_bytes;
    const int64_t T = (int64_t)N * k;
    uint8_t* buf = smem + (size_t)warp * nbuf * unit;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kBulkWarps * nbuf * unit) + warp * kBcastMaxBuf;
    if (lane == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(&bars[b], 1);
        s_abort[warp] = 0;
        fence_mbar_init();
    }
    __syncwarp();

    const int gw = blockIdx.x * kBulkWarps + warp, nw = gridDim.x * kBulkWarps;
    if (gw >= N) return;
    const int total = (N - gw + nw - 1) / nw;     // tokens of this warp
    const unsigned long long deadline = globaltimer_ns() + timeout_ns;
    const uint64_t stream = l2_policy_evict_first();
    volatile int* abort_flag = &s_abort[warp];
    uint32_t bad = 0;          // bit b: buffer b holds nothing to store

    // Read the schedule entries of the q-th token's slots (lane j: slot j) and
    // issue the bulk load of its row into buffer q % nbuf (lane 0).
    auto load = [&](int q) {
        const int64_t n = gw + (int64_t)q * nw;
        const int b = q % nbuf;
        int t = -1, s = -1, r = -1;
        if (lane < k) {
            t = inv[n * k + lane];
            if (t >= 0 && t < T) {
                s = sched[2 * (int64_t)t];
                r = sched[2 * (int64_t)t + 1];
            } else {
                set_status(ws, MOE_ERR_DEVICE_CHECK);
                t = -1;
            }
        }
        const bool in_range = t >= slot_begin && t < slot_begin + slot_count;
        const uint32_t m = __ballot_sync(0xffffffffu, in_range);
        const int first = m ? __ffs(m) - 1 : 0;
        const int s0 = __shfl_sync(0xffffffffu, s, first);
        const int r0 = __shfl_sync(0xffffffffu, r, first);
        bool ok = m != 0 && s0 >= 0 && s0 < S && r0 >= 0 && r0 < rows_per_shard;
        const uint8_t* src = ok ? shard_rows[s0] + (int64_t)r0 * row_bytes : nullptr;
        const uint8_t* ssrc = (ok && scale_bytes) ? shard_scales[s0] + (int64_t)r0 * scale_bytes : nullptr;
        if (ok && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(ssrc)) & 15)) ok = false;
        const bool mine = ok && in_range && s == s0 && r == r0;
        if (in_range && !mine) set_status(ws, MOE_ERR_DEVICE_CHECK);
        s_dst[warp][b][lane] = mine ? (int)(t % ring_slots) : -1;
        const bool any = __any_sync(0xffffffffu, mine);
        __syncwarp();
        if (lane == 0) {
            if (any) {
                bad &= ~(1u << b);
                mbar_arrive_expect_tx(&bars[b], (uint32_t)unit);
                uint8_t* dst = buf + (size_t)b * unit;
                bulk_load(dst, src, (uint32_t)row_bytes, &bars[b]);
                if (scale_bytes) bulk_load(dst + row_bytes, ssrc, (uint32_t)scale_bytes, &bars[b]);
            } else {
                bad |= 1u << b;
                mbar_arrive(&bars[b]);
            }
        }
    };

    const int pre = min(nbuf, total);
    for (int q = 0; q < pre; ++q) load(q);
    for (int q = 0; q < total; ++q) {
        if (lane == 0) {
            const int b = q % nbuf;
            if (!mbar_wait_bounded(&bars[b], (uint32_t)((q / nbuf) & 1), abort_flag, ws, deadline)) {
                // give up: nothing more is issued; drain what is in flight below
            } else if (!(bad & (1u << b))) {
                fence_proxy_async_smem();
                const uint8_t* src = buf + (size_t)b * unit;
                for (int j = 0; j < k; ++j) {
                    const int dr = s_dst[warp][b][j];
                    if (dr < 0) continue;
                    bulk_store_hint(ring + (int64_t)dr * row_bytes, src, (uint32_t)row_bytes, stream);
                    if (scale_bytes)
                        bulk_store_hint(ring_scales + (int64_t)dr * scale_bytes, src + row_bytes,
                                        (uint32_t)scale_bytes, stream);
                }
            }
            bulk_commit_group();
            bulk_wait_group_read<kBulkLag>();
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int qn = q - kBulkLag + nbuf;     // refill the buffer whose stores are now LAG groups old
        if (q >= kBulkLag && qn < total) load(qn);
    }
    if (lane == 0) {
        if (*abort_flag) {
            const unsigned long long d2 = globaltimer_ns() + 1000000ull;
            while (globaltimer_ns() < d2) {
            }
        }
        bulk_wait_group_all();
    }
}

cudaError_t launch_dispatch_pull(const void* const* shard_rows, const void* const* shard_scales,
                                 const int32_t* sched, const int32_t* order, int order_len, int order_k,
                                 int slot_begin, int slot_count, int S, int rows_per_shard,
                                 int row_bytes, int scale_bytes, void* ring, void* ring_scales,
                                 int ring_slots, int num_sms, WsHeader* ws,
                                 unsigned long long timeout_ns, cudaStream_t stream) {
    if (slot_count <= 0) return cudaSuccess;
    const int unit = row_bytes + scale_bytes;
    const int bars_bytes = kBulkWarps * kBulkMaxBuf * 8;
    auto buffers = [&](int budget) {
        const int n = unit > 0 ? (budget - bars_bytes) / (kBulkWarps * unit) : 0;
        return n > kBulkMaxBuf ? kBulkMaxBuf : n;
    };
    // two CTAs per SM when half the shared memory still holds a full pipeline of
    // row buffers (LAG + 2), one CTA with the whole budget for wider rows
    int nbuf = buffers(100 * 1024);
    if (nbuf < kBulkLag + 2) nbuf = buffers(200 * 1024);
    const bool bulk = row_bytes % 16 == 0 && scale_bytes % 16 == 0 && nbuf >= kBulkLag + 2 &&
                      (reinterpret_cast<uintptr_t>(ring) & 15) == 0 &&
                      (scale_bytes == 0 || (reinterpret_cast<uintptr_t>(ring_scales) & 15) == 0);
    if (bulk && order && order_k > 0 && order_k <= 32 && order_len % order_k == 0) {
        const int nb = nbuf > kBcastMaxBuf ? kBcastMaxBuf : nbuf;
        const size_t smem = (size_t)kBulkWarps * nb * unit + (size_t)kBulkWarps * kBcastMaxBuf * 8;
        cudaError_t e = cudaFuncSetAttribute(dispatch_bcast_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const int static_smem = kBulkWarps * (kBcastMaxBuf * 32 + 1) * 4;
        int per_sm = (int)((227 * 1024) / (smem + static_smem + 1024));
        if (per_sm < 1) per_sm = 1;
        const int N = order_len / order_k;
        int blocks = (N + kBulkWarps - 1) / kBulkWarps;
        if (blocks > num_sms * per_sm) blocks = num_sms * per_sm;
        dispatch_bcast_kernel<<<blocks, kBulkWarps * 32, smem, stream>>>(
            (const uint8_t* const*)shard_rows, (const uint8_t* const*)shard_scales, sched, order, N, order_k,
            slot_begin, slot_count, S, rows_per_shard, row_bytes, scale_bytes, (uint8_t*)ring,
            (uint8_t*)ring_scales, ring_slots, nb, ws, timeout_ns);
        return cudaGetLastError();
    }
    if (bulk) {
        const size_t smem = (size_t)kBulkWarps * nbuf * unit + bars_bytes;
        cudaError_t e = cudaFuncSetAttribute(dispatch_bulk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int per_sm = (int)((227 * 1024) / (smem + 1024));
        if (per_sm < 1) per_sm = 1;
        const int nchunks = (slot_count + 31) / 32;
        int blocks = (nchunks + kBulkWarps - 1) / kBulkWarps;
        if (blocks > num_sms * per_sm) blocks = num_sms * per_sm;
        dispatch_bulk_kernel<<<blocks, kBulkWarps * 32, smem, stream>>>(
            (const uint8_t* const*)shard_rows, (const uint8_t* const*)shard_scales, sched, slot_begin,
            slot_count, S, rows_per_shard, row_bytes, scale_bytes, (uint8_t*)ring, (uint8_t*)ring_scales,
            ring_slots, nbuf, ws, timeout_ns);
        return cudaGetLastError();
    }
    int blocks = (slot_count + kGatherWarps - 1) / kGatherWarps;
    if (blocks > num_sms * 8) blocks = num_sms * 8;
    dispatch_pull_kernel<<<blocks, kGatherWarps * 32, 0, stream>>>(
        (const uint8_t* const*)shard_rows, (const uint8_t* const*)shard_scales, sched, slot_begin,
        slot_count, S, rows_per_shard, row_bytes, scale_bytes, (uint8_t*)ring,
        (uint8_t*)ring_scales, ring_slots, ws);
    return cudaGetLastError();
}

}  // namespace moe
