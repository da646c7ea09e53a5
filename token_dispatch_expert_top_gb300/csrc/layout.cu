// layout.cu -- sort-free token layout ("schedule").  The flat list of choices
// (n, j) -> expert is placed expert-contiguously with a stable counting placement,
// in three short kernels: per-chunk expert counts (warp match + shared-memory
// atomics), a per-expert exclusive scan over chunks (one warp per expert), and a warp-ballot rank that
// writes each choice's slot, the two-column (source shard, row) pull schedule and
// the inverse map.  ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost
// on NVIDIA GB300 NVL72", section 01: count per expert, decide placement, keep an
// expert's tokens together for the grouped GEMM; [Kittens] = "Смесь котят…",
// pull paragraph: a two-column schedule built without sorting.)
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int kLayoutWarps = 8;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

constexpr int kLayoutIters = kLayoutChunk / 32;

// A warp's expert ids of one chunk, all loads issued before any is used (lane l
// holds choice begin + 32*i + l in v[i]; -1 past the end), so a chunk costs one
// load latency rather than one per 32 choices.
__device__ __forceinline__ void load_chunk(const int32_t* __restrict__ idx, int begin, int end, int lane,
                                           int (&v)[kLayoutIters]) {
#pragma unroll
    for (int i = 0; i < kLayoutIters; ++i) {
        const int t = begin + 32 * i + lane;
        v[i] = (t < end) ? idx[t] : -1;
    }
}

// Chunk c covers flat choices [c*kLayoutChunk, min((c+1)*kLayoutChunk, T)).
// One warp per chunk; counts go to cnt[e][c] (expert-major, so that each
// expert's per-chunk counts are contiguous for the scan).
__global__ void __launch_bounds__(kLayoutWarps * 32) layout_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int nchunks, int32_t* __restrict__ cnt,
    WsHeader* ws) {
    extern __shared__ int32_t sh[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int32_t* hist = sh + warp * E;
    const int c = blockIdx.x * kLayoutWarps + warp;
    if (c >= nchunks) return;
    const int begin = c * kLayoutChunk;
    const int end = min(begin + kLayoutChunk, T);
    int ev[kLayoutIters];
    load_chunk(idx, begin, end, lane, ev);
    for (int e = lane; e < E; e += 32) hist[e] = 0;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kLayoutIters; ++i) {
        const int t = begin + 32 * i + lane;
        int e = ev[i];
        if (t < end && (e < 0 || e >= E)) {
            set_status(ws, MOE_ERR_DEVICE_CHECK);
            e = -1;
        }
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (same & lanemask_lt()) == 0) atomicAdd(&hist[e], __popc(same));
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) cnt[(int64_t)e * nchunks + c] = hist[e];
}

// Exclusive scan over an int array of length n by one warp: each lane takes a
// contiguous run, the run totals are scanned with shuffles.  Writes out[i] =
// base + sum_{i' < i} in[i'] and returns the total (in every lane).
// Runs of up to 8 values are held in registers, their loads issued together.
__device__ __forceinline__ int warp_inclusive_sum(int s, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
    }
    return s;
}

__device__ __forceinline__ int warp_exclusive_scan(const int32_t* in, int32_t* out, int n, int base,
                                                   int lane) {
    const int per = (n + 31) / 32;
    const int lo = min(lane * per, n), hi = min(lo + per, n);
    if (per <= 8) {
        int v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (lo + j < hi) ? in[lo + j] : 0;
        int s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) s += v[j];
        const int incl = warp_inclusive_sum(s, lane);
        int run = base + incl - s;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (lo + j < hi) {
                out[lo + j] = run;
                run += v[j];
            }
        return __shfl_sync(0xffffffffu, incl, 31);
    }
    int s = 0;
    for (int i = lo; i < hi; ++i) s += in[i];
    const int incl = warp_inclusive_sum(s, lane);
    int run = base + incl - s;
    for (int i = lo; i < hi; ++i) {
        const int c = in[i];
        out[i] = run;
        run += c;
    }
    return __shfl_sync(0xffffffffu, incl, 31);
}

// One warp per expert: base[e][c] = sum_{c' < c} cnt[e][c'];  counts[e] = total.
__global__ void __launch_bounds__(kLayoutWarps * 32) layout_scan_kernel(
    const int32_t* __restrict__ cnt, int nchunks, int E, int32_t* __restrict__ base,
    int32_t* __restrict__ counts) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int e = blockIdx.x * kLayoutWarps + warp;
    if (e >= E) return;
    const int total = warp_exclusive_scan(cnt + (int64_t)e * nchunks, base + (int64_t)e * nchunks,
                                          nchunks, 0, lane);
    if (lane == 0) counts[e] = total;
}

// Every block first scans counts into the expert offsets (block 0 also writes
// them out); then one warp per chunk walks its choices in flat order 32 at a
// time: lanes holding the same expert find each other with a match, rank
// themselves by lane order, and the group's first lane advances the cursor.
__global__ void __launch_bounds__(kLayoutWarps * 32) layout_place_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int nchunks,
    const int32_t* __restrict__ base, const int32_t* __restrict__ counts, int rows_per_shard,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sched, int32_t* __restrict__ inv) {
    extern __shared__ int32_t sh[];
    int32_t* off = sh;                         // [E+1]
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int32_t* cursor = sh + (E + 1) + warp * E;
    const int c = blockIdx.x * kLayoutWarps + warp;
    const int begin = c * kLayoutChunk;
    const int end = min(begin + kLayoutChunk, T);
    int ev[kLayoutIters];
    load_chunk(idx, begin, end, lane, ev);   // in flight while the offsets are scanned
    if (warp == 0) {
        const int total = warp_exclusive_scan(counts, off, E, 0, lane);
        if (lane == 0) off[E] = total;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off[e];
    if (c >= nchunks) return;
    for (int e = lane; e < E; e += 32) cursor[e] = off[e] + base[(int64_t)e * nchunks + c];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kLayoutIters; ++i) {
        const int t = begin + 32 * i + lane;
        int e = ev[i];
        if (e >= E) e = -1;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lanemask_lt());
        const int cur = (e >= 0) ? cursor[e] : 0;
        __syncwarp();
        if (e >= 0) {
            const int slot = cur + rank;
            const int n = t / k;
            sched[2 * (int64_t)slot] = n / rows_per_shard;
            sched[2 * (int64_t)slot + 1] = n % rows_per_shard;
            inv[t] = slot;
            if (rank == 0) cursor[e] = cur + __popc(same);
        }
        __syncwarp();
    }
}

cudaError_t launch_layout(const int32_t* idx, int N, int k, int E, int S, int32_t* counts,
                          int32_t* offsets, int32_t* sched, int32_t* inv, int32_t* cnt_scratch,
                          int32_t* base_scratch, WsHeader* ws, cudaStream_t stream) {
    const int T = N * k;
    const int nchunks = layout_chunks(T);
    const int blocks = (nchunks + kLayoutWarps - 1) / kLayoutWarps;
    if (nchunks > 0)
        layout_count_kernel<<<blocks, kLayoutWarps * 32, sizeof(int32_t) * kLayoutWarps * E,
                              stream>>>(idx, T, E, nchunks, cnt_scratch, ws);
    layout_scan_kernel<<<(E + kLayoutWarps - 1) / kLayoutWarps, kLayoutWarps * 32, 0, stream>>>(
        cnt_scratch, nchunks, E, base_scratch, counts);
    layout_place_kernel<<<blocks > 0 ? blocks : 1, kLayoutWarps * 32,
                          sizeof(int32_t) * ((E + 1) + kLayoutWarps * E), stream>>>(
        idx, T, k, E, nchunks, base_scratch, counts, N / S, offsets, sched, inv);
    return cudaGetLastError();
}

}  // namespace moe
