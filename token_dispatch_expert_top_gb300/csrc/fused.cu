// fused.cu -- the persistent forward kernel: gather, expert FFN and combine as
// roles of ONE launch, handing minibatches of token slots between SM groups
// through GPU-local counters, with a fixed-size ring of slots that is refilled
// as soon as the slots it holds have been consumed.
// ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72", section 02: one megakernel; some SMs do dispatch/combine/state, the
// rest only the expert FFN; a GPU-local counter tells the compute side when a
// full batch of tokens has arrived and the comm side when results are ready; the
// minibatch should give at least two full waves of GEMM tiles; a fixed-size ring
// token buffer absorbs the rate difference, no worst-case buffer, no CPU in the
// loop, no dropped tokens.  [Kittens], megakernel paragraph: bitwise determinism.)
//
// Slots [0, T) in expert-sorted order are cut into minibatches of MB slots.
// Minibatch b lives in ring buffer b mod NR (NR = R / MB buffers of MB slots).
//   gather CTAs   copy the rows of minibatch b into its ring buffer once the
//                 GEMM2 tiles of minibatch b - NR (the buffer's previous tenant)
//                 are done, then bump gather_done[b];
//   compute CTAs  run the tcgen05 pipeline over the tile sequence
//                 [GEMM1 tiles of 0][GEMM2 tiles of 0][GEMM1 tiles of 1]...
//                 (round-robin over compute CTAs); a GEMM1 tile waits for
//                 gather_done[b], a GEMM2 tile for its m-tile's GEMM1 counter;
//                 h lives in a ring too, y in a [T][H] buffer;
//   every CTA     combines tokens once all GEMM2 tiles are done.
// Every dependency points backwards in that order, so the schedule cannot
// deadlock; every wait is bounded by timeout_ns from kernel start, after which
// the kernel records MOE_ERR_TIMEOUT, raises a global abort flag and returns.
#include "common.cuh"
#include "gemm_roles.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

// ------------------------------------------------------------ global counters
__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}


// Spin until *ctr >= target.  Gives up (false) when the global abort flag is
// raised or the deadline passes (then it raises the flag and records a timeout).
__device__ bool wait_counter(const int* ctr, int target, int* abort_g, WsHeader* ws,
                             unsigned long long deadline) {
    uint32_t n = 0;
    while (ld_acquire(ctr) < target) {
        if (ld_acquire(abort_g)) return false;
        if ((++n & 63u) == 0) {
            if (globaltimer_ns() > deadline) {
                atomicExch(abort_g, 1);
                set_status(ws, MOE_ERR_TIMEOUT);
                return false;
            }
        }
        __nanosleep(64);
    }
    return true;
}

// Make this thread's global stores visible to other CTAs and to the TMA (async
// proxy) of other CTAs before a counter is bumped.
__device__ __forceinline__ void publish_fence() {
    fence_proxy_async_global();
    __threadfence();
}

}  // namespace

// The compute schedule is a list of 2*nmb segments, each all GEMM1 or all GEMM2
// tiles of one minibatch.  With two or more ring buffers it is software-pipelined,
//   G1(0) G1(1) G2(0) G1(2) G2(1) ... G1(nmb-1) G2(nmb-2) G2(nmb-1),
// so a GEMM2 tile's inputs were finished a whole minibatch earlier; with a single
// ring buffer it is G1(0) G2(0) G1(1) G2(1) ... (the gather of b needs G2(b-1)).
struct Segment {
    int kind, b;
};

__host__ __device__ __forceinline__ Segment segment_of(int j, int nmb, bool interleave) {
    if (!interleave) return Segment{j & 1, j >> 1};
    if (j == 0) return Segment{0, 0};
    if (j == 2 * nmb - 1) return Segment{1, nmb - 1};
    return (j & 1) ? Segment{0, (j + 1) >> 1} : Segment{1, (j >> 1) - 1};
}

// Counters and plan arrays in the workspace (int32).  nmb is the number of
// minibatches the plan kernel cut (at most the host's bound nmb_max).
struct FusedPlan {
    int* tbase;        // [2*nmb+1] tile prefix over the segments of the schedule
    int* pbase;        // [nmb+1] m-tile prefix over minibatches (P_b each)
    int* elo;          // [nmb] first expert overlapping minibatch b
    int* cut;          // [nmb+1] first slot of minibatch b; cut[nmb] = T
    int* nmb;          // [1] minibatches
    int* gather_done;  // [nmb] gather CTAs done with minibatch b
    int* g1_done;      // [pbase[nmb]] epilogue-warp reports of GEMM1 tiles per m-tile
    int* g2_done;      // [nmb] epilogue-warp reports of GEMM2 tiles per minibatch
    int* g2_all;       // [1]  epilogue-warp reports of all GEMM2 tiles
    int* abort_g;      // [1]  set when any wait gave up
};

struct FusedArgs {
    FusedPlan plan;
    const int32_t* offsets;   // [E+1]
    const int32_t* sched;     // [T][2]
    const int32_t* inv;       // [N][k]
    const float* gate;        // [N][k]
    const uint8_t* const* shard_rows;
    const uint8_t* const* shard_sf;
    uint8_t* ring;            // [R][H] (codes or BF16)
    uint8_t* ring_sf;         // [R][H/32]
    uint8_t* y;               // [T][H] BF16
    uint8_t* out;             // [N][H] BF16
    int N, H, E, k, S, T;
    int MB, NR, nmb_max;      // minibatch capacity, ring buffers, bound on the minibatch count
    int G;                    // gather CTAs (blockIdx.x < G)
    int row_bytes, sf_bytes;  // gathered row and its scales
    int skip_ready;           // test hook: minibatch whose gather_done is never bumped (-1: none)
    int plan_smem;            // compute CTAs keep tbase / pbase / elo in shared memory
    WsHeader* ws;
    unsigned long long timeout_ns;
};

// End of the minibatch that starts at slot lo (slots in expert order, at most MB
// of them).  It ends on an expert boundary when one falls in the second half of
// the minibatch, else inside the expert that crosses lo + MB at a whole number of
// 128-row m-tiles from that expert's start, so minibatch edges cut as few experts
// (extra ragged m-tiles, a second pass over their weights) as possible.  Every
// minibatch but the last holds at least max(1, MB/2) slots.
__device__ int minibatch_cut(const int32_t* off, int E, int T, int MB, int lo) {
    const int target = lo + MB;
    if (target >= T) return T;
    const int half = MB / 2 > 1 ? MB / 2 : 1;
    int a = 0, z = E - 1;                 // expert e with off[e] < target <= off[e+1]
    while (a < z) {
        const int mid = (a + z) >> 1;
        if (off[mid + 1] >= target) z = mid; else a = mid + 1;
    }
    if (off[a + 1] == target) return target;
    if (off[a] - lo >= half) return off[a];
    const int c2 = off[a] + ((target - off[a]) / tc::BM) * tc::BM;
    if (c2 - lo >= half) return c2;
    return target;
}

// Start of the minibatch that ends at slot hi when the slots are cut from the
// last one down (reverse traversal): the mirror of minibatch_cut.  It starts on
// an expert boundary when one falls in the minibatch's upper half of slots, else
// inside the expert that crosses hi - MB at a whole number of 128-row m-tiles from
// that expert's start (rounded up, so the minibatch holds at most MB slots).
__device__ int minibatch_cut_rev(const int32_t* off, int E, int MB, int hi) {
    const int target = hi - MB;
    if (target <= 0) return 0;
    const int half = MB / 2 > 1 ? MB / 2 : 1;
    int a = 0, z = E - 1;                 // expert e with off[e] <= target < off[e+1]
    while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (off[mid] <= target) a = mid; else z = mid - 1;
    }
    if (off[a] == target) return target;
    if (hi - off[a + 1] >= half) return off[a + 1];
    const int c2 = off[a] + ((target - off[a] + tc::BM - 1) / tc::BM) * tc::BM;
    if (c2 < hi && hi - c2 >= half) return c2;
    return target;
}

// Minibatch b is the slots between cut[b] and cut[b+1] (ascending cuts in slot
// order, descending in reverse traversal).
__device__ __forceinline__ void minibatch_range(const int32_t* cut, int b, int& lo, int& hi) {
    lo = min(cut[b], cut[b + 1]);
    hi = max(cut[b], cut[b + 1]);
}

// One block: cuts the slots into minibatches, then per-minibatch m-tile counts,
// prefixes and first experts; zeroes the counters.
__global__ void __launch_bounds__(1024) fused_plan_kernel(const int32_t* __restrict__ offsets, int E,
                                                          int T, int MB, int nmb_max, int nt1, int nt2,
                                                          int interleave, int reverse, FusedPlan plan,
                                                          int counters_len, int* counters, WsHeader* ws) {
    extern __shared__ int32_t off[];
    __shared__ int s_nmb;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = offsets[e];
    for (int i = threadIdx.x; i < counters_len; i += blockDim.x) counters[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        int b = 0;
        if (!reverse) {
            int lo = 0;
            while (lo < T && b < nmb_max) {
                plan.cut[b++] = lo;
                lo = minibatch_cut(off, E, T, MB, lo);
            }
            if (lo < T) set_status(ws, MOE_ERR_DEVICE_CHECK);   // cannot happen: the bound holds
            plan.cut[b] = T;
        } else {
            int hi = T;
            while (hi > 0 && b < nmb_max) {
                plan.cut[b++] = hi;
                hi = minibatch_cut_rev(off, E, MB, hi);
            }
            if (hi > 0) set_status(ws, MOE_ERR_DEVICE_CHECK);   // cannot happen: the bound holds
            plan.cut[b] = 0;
        }
        *plan.nmb = b;
        s_nmb = b;
    }
    __syncthreads();
    const int nmb = s_nmb;
    for (int b = threadIdx.x; b < nmb; b += blockDim.x) {
        int lo, hi;
        minibatch_range(plan.cut, b, lo, hi);
        int a = 0, z = E;  // first e with off[e+1] > lo
        while (a < z) {
            const int mid = (a + z) >> 1;
            if (off[mid + 1] > lo) z = mid; else a = mid + 1;
        }
        plan.elo[b] = a;
        int P = 0;
        for (int e = a; e < E && off[e] < hi; ++e) {
            const int len = min(off[e + 1], hi) - max(off[e], lo);
            if (len > 0) P += (len + tc::BM - 1) / tc::BM;
        }
        plan.pbase[b] = P;   // the count for now; the scan below turns it into prefixes
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // m-tile prefix over minibatches (each lane touches only its own b's)
        const int lane = threadIdx.x;
        const int per = (nmb + 31) / 32;
        const int lo = min(lane * per, nmb), hi = min(lo + per, nmb);
        int s = 0;
        for (int b = lo; b < hi; ++b) s += plan.pbase[b];
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - s;
        for (int b = lo; b < hi; ++b) {
            const int P = plan.pbase[b];
            plan.pbase[b] = run;
            run += P;
        }
        __syncwarp();
        if (lane == 31) plan.pbase[nmb] = incl;
        __syncwarp();
        // tile prefix over the 2*nmb segments of the schedule
        const int nseg = 2 * nmb;
        const int pers = (nseg + 31) / 32;
        const int slo = min(lane * pers, nseg), shi = min(slo + pers, nseg);
        auto seg_tiles = [&](int j) {
            const Segment sg = segment_of(j, nmb, interleave != 0);
            return (plan.pbase[sg.b + 1] - plan.pbase[sg.b]) * (sg.kind == 0 ? nt1 : nt2);
        };
        int ss = 0;
        for (int j = slo; j < shi; ++j) ss += seg_tiles(j);
        int sincl = ss;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, sincl, o);
            if (lane >= o) sincl += v;
        }
        int srun = sincl - ss;
        for (int j = slo; j < shi; ++j) {
            plan.tbase[j] = srun;
            srun += seg_tiles(j);
        }
        if (lane == 31) plan.tbase[nseg] = sincl;
    }
}

// Tiles of the fused schedule: per minibatch, its GEMM1 tiles then its GEMM2
// tiles, each ordered expert-major, then N tile, then m-tile (as in the staged
// kernel), so compute CTAs working at the same time share both the weight tile
// (same expert and N tile) and the token rows (same expert and m-tile) in L2.
// (With the N tile outermost, the reuses of an A tile are a whole wave apart and
// the weight stream evicts it from L2 in between.)
struct MinibatchTiles {
    static constexpr bool kDeps = true;         // tiles wait for other CTAs (a dependency thread checks)
    static constexpr bool kSaveUV = false;
    const FusedArgs* a;
    const int32_t* off;       // offsets in shared memory
    const int32_t *tb, *pb, *el, *ct;   // the plan's tbase / pbase / elo / cut (shared memory when they fit)
    int nmb;                  // minibatches
    int nt1, nt2, c0, C;      // N tiles of GEMM1 / GEMM2, this CTA's index among C
    __device__ int first() const { return c0; }
    __device__ int next(int t) const { return t + C; }
    __device__ int count() const { return tb[2 * nmb]; }
    __device__ int kind_of(int t) const {
        int lo = 0, hi = 2 * nmb;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tb[mid] <= t) lo = mid; else hi = mid;
        }
        return segment_of(lo, nmb, a->NR >= 2).kind;
    }
    __device__ TileInfo tile(int t) const {
        int lo = 0, hi = 2 * nmb;   // last segment j with tbase[j] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tb[mid] <= t) lo = mid; else hi = mid;
        }
        const Segment sg = segment_of(lo, nmb, a->NR >= 2);
        const int b = sg.b;
        const int nt = sg.kind == 0 ? nt1 : nt2;
        int r = t - tb[lo];              // tile within the segment
        TileInfo tl;
        tl.kind = sg.kind;
        int s_lo, s_hi;
        minibatch_range(ct, b, s_lo, s_hi);
        int e = el[b], mbase = 0, mt = 0;   // expert piece, its first m-tile index, its m-tiles
        for (; e < a->E; ++e) {
            const int len = min(off[e + 1], s_hi) - max(off[e], s_lo);
            mt = len > 0 ? (len + tc::BM - 1) / tc::BM : 0;
            if (r < mt * nt) break;
            r -= mt * nt;
            mbase += mt;
        }
        const int m = e < a->E ? r % mt : 0;
        tl.n = e < a->E ? r / mt : 0;
        const int mi = mbase + m;
        int piece0, piece_end;
        if (e < a->E) {
            piece0 = max(off[e], s_lo) + m * tc::BM;   // first slot of the m-tile
            piece_end = min(off[e + 1], s_hi);
        } else {                                       // plan and decode disagree: store nothing
            set_status(a->ws, MOE_ERR_DEVICE_CHECK);
            e = a->E - 1;
            piece0 = piece_end = s_lo;
        }
        const int ring_row = (b % a->NR) * a->MB + (piece0 - s_lo);
        tl.e = e;
        tl.a_row0 = ring_row;
        tl.out_row0 = tl.kind == 0 ? ring_row : piece0;
        tl.nrows = min(piece_end - piece0, tc::BM);
        tl.mb = b;
        tl.midx = pb[b] + mi;
        return tl;
    }
    // What a tile's A operand waits for: its minibatch's gather (every CTA takes
    // part in minibatch 0, the gather CTAs alone in the others), or all GEMM1
    // N tiles of its m-tile.
    __device__ const int* dep_counter(const TileInfo& tl, int* target) const {
        const FusedPlan& pl = a->plan;
        if (tl.kind == 0) {
            *target = tl.mb == 0 ? (int)gridDim.x : a->G;
            return pl.gather_done + tl.mb;
        }
        *target = nt1 * tc::EPI_WARPS;
        return pl.g1_done + tl.midx;
    }
    __device__ bool wait_inputs(const TileInfo& tl, const Pipe& p) const {
        const FusedPlan& pl = a->plan;
        int target;
        const int* ctr = dep_counter(tl, &target);
        if (!wait_counter(ctr, target, pl.abort_g, a->ws, p.deadline)) {
            *p.abort_flag = 1;
            return false;
        }
        fence_proxy_async_global();   // the rows another CTA stored may now be read by TMA
        return true;
    }
    __device__ void tile_stored(const TileInfo& tl, const Pipe&) const {
        publish_fence();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            if (tl.kind == 0) {
                atomicAdd(a->plan.g1_done + tl.midx, 1);
            } else {
                atomicAdd(a->plan.g2_done + tl.mb, 1);
                atomicAdd(a->plan.g2_all, 1);
            }
        }
    }
};

// One slot's row (n16 16-byte words) and its MXFP8 scales (m8 8-byte words: a
// scale row is H/32 bytes, a multiple of 8 but not always of 16), by one warp.
__device__ __forceinline__ void copy_slot_row(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                              int n16, uint8_t* __restrict__ dst2,
                                              const uint8_t* __restrict__ src2, int m8, int lane) {
    constexpr int U = 16;
    for (int b = 0; b < n16; b += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = b + lane + 32 * u;
            if (j < n16) v[u] = ld_nc_v4(src + 16 * (int64_t)j);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = b + lane + 32 * u;
            if (j < n16) st_v4(dst + 16 * (int64_t)j, v[u]);
        }
    }
    for (int j = lane; j < m8; j += 32)
        reinterpret_cast<uint2*>(dst2)[j] = reinterpret_cast<const uint2*>(src2)[j];
}

// Copy the rows of minibatch b into its ring buffer, warp gw of nw, then make
// them visible to other CTAs' TMA and count this CTA in gather_done[b].
__device__ void gather_minibatch(const FusedArgs& a, int b, int gw, int nw) {
    const int lane = threadIdx.x & 31;
    const FusedPlan& pl = a.plan;
    int lo, hi;
    minibatch_range(pl.cut, b, lo, hi);
    const int base = (b % a.NR) * a.MB;
    for (int t = lo + gw; t < hi; t += nw) {
        const int s = a.sched[2 * (int64_t)t];
        const int r = a.sched[2 * (int64_t)t + 1];
        if (s < 0 || s >= a.S || r < 0 || r >= a.N / a.S) {
            if (lane == 0) set_status(a.ws, MOE_ERR_DEVICE_CHECK);
            continue;
        }
        const int64_t dr = base + (t - lo);
        const bool has_sf = a.sf_bytes > 0;
        copy_slot_row(a.ring + dr * a.row_bytes, a.shard_rows[s] + (int64_t)r * a.row_bytes,
                      a.row_bytes >> 4, has_sf ? a.ring_sf + dr * a.sf_bytes : nullptr,
                      has_sf ? a.shard_sf[s] + (int64_t)r * a.sf_bytes : nullptr,
                      has_sf ? a.sf_bytes >> 3 : 0, lane);
    }
    publish_fence();
    __syncthreads();
    if (threadIdx.x == 0 && b != a.skip_ready) atomicAdd(pl.gather_done + b, 1);
}

// Bulk-copy gather of one minibatch by one stream (lane 0 of a warp issues, all
// lanes call): the stream's share of the slots moves through its ring of
// shared-memory row buffers, a bulk load then a bulk store per slot, with up to
// nbuf - LAG loads in flight.  q0 counts the positions this stream handled in
// earlier minibatches, so each buffer's barrier phase carries on across
// minibatches.  Returns the positions handled (every one arrives once on its
// buffer's barrier, copied or not), or -1 when a wait gave up.
constexpr int kGatherLag = 2;
constexpr int kGatherMaxBuf = 16;
constexpr int kGatherMaxStreams = 6;

__device__ int gather_stream_bulk(const FusedArgs& a, int b, int gs, int ns, uint8_t* buf, uint64_t* bars,
                                  int nbuf, int q0, volatile int* abort_flag, unsigned long long deadline) {
    const int lane = threadIdx.x & 31;
    const FusedPlan& pl = a.plan;
    int lo, hi;
    minibatch_range(pl.cut, b, lo, hi);
    const int base = (b % a.NR) * a.MB;
    const int unit = a.row_bytes + a.sf_bytes;
    const int nslots = hi - lo;
    const int nchunks = (nslots + 31) / 32;
    if (gs >= nchunks) return 0;
    const int my_chunks = (nchunks - gs + ns - 1) / ns;
    const int last = gs + (my_chunks - 1) * ns;
    const int total = (my_chunks - 1) * 32 + min(32, nslots - last * 32);
    auto slot_of = [&](int q) { return lo + (gs + (q >> 5) * ns) * 32 + (q & 31); };
    uint32_t bad = 0;
    int chunk_q = -1, my_s = 0, my_r = 0;
    auto load = [&](int q) {
        const int c0 = q & ~31;
        if (c0 != chunk_q) {
            chunk_q = c0;
            const int t = slot_of(c0) + lane;
            if (t < hi) {
                my_s = a.sched[2 * (int64_t)t];
                my_r = a.sched[2 * (int64_t)t + 1];
            }
        }
        const int sidx = __shfl_sync(0xffffffffu, my_s, q & 31);
        const int ridx = __shfl_sync(0xffffffffu, my_r, q & 31);
        if (lane == 0) {
            const int bi = (q0 + q) % nbuf;
            uint8_t* dst = buf + (size_t)bi * unit;
            bool ok = sidx >= 0 && sidx < a.S && ridx >= 0 && ridx < a.N / a.S;
            const uint8_t* src = ok ? a.shard_rows[sidx] + (int64_t)ridx * a.row_bytes : nullptr;
            const uint8_t* ssrc = (ok && a.sf_bytes) ? a.shard_sf[sidx] + (int64_t)ridx * a.sf_bytes : nullptr;
            if (ok && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(ssrc)) & 15)) ok = false;
            if (ok) {
                bad &= ~(1u << bi);
                mbar_arrive_expect_tx(&bars[bi], (uint32_t)unit);
                bulk_load(dst, src, (uint32_t)a.row_bytes, &bars[bi]);
                if (a.sf_bytes) bulk_load(dst + a.row_bytes, ssrc, (uint32_t)a.sf_bytes, &bars[bi]);
            } else {
                set_status(a.ws, MOE_ERR_DEVICE_CHECK);
                bad |= 1u << bi;
                mbar_arrive(&bars[bi]);
            }
        }
    };
    const int pre = min(nbuf, total);
    for (int q = 0; q < pre; ++q) load(q);
    int q = 0;
    for (; q < total; ++q) {
        if (lane == 0) {
            const int gq = q0 + q, bi = gq % nbuf;
            if (mbar_wait_bounded(&bars[bi], (uint32_t)((gq / nbuf) & 1), abort_flag, a.ws, deadline) &&
                !(bad & (1u << bi))) {
                const int64_t dr = base + (slot_of(q) - lo);
                const uint8_t* src = buf + (size_t)bi * unit;
                bulk_store(a.ring + dr * a.row_bytes, src, (uint32_t)a.row_bytes);
                if (a.sf_bytes) bulk_store(a.ring_sf + dr * a.sf_bytes, src + a.row_bytes, (uint32_t)a.sf_bytes);
            }
            bulk_commit_group();
            bulk_wait_group_read<kGatherLag>();
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const int qn = q - kGatherLag + nbuf;
        if (q >= kGatherLag && qn < total) load(qn);
    }
    if (lane == 0) {
        bulk_wait_group_all();         // the stores are complete: the rows are in global memory
        fence_proxy_async_global();    // ... and ordered before this thread's later generic accesses
    }
    __syncwarp();
    return *abort_flag ? -1 : total;
}

// Gather role: minibatch by minibatch (from 1: every CTA of the launch gathers
// minibatch 0 first), wait for the ring buffer, copy, publish.  Rows of 16-byte
// multiples go through the bulk-copy engine (up to six warps as streams, each
// with its own row buffers in this CTA's shared memory); others are copied with
// vector loads by every warp.
__device__ void gather_role(const FusedArgs& a, int nmb, unsigned long long deadline, int nt2, uint8_t* smem) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x / 32) + warp;
    const int nw = a.G * (blockDim.x / 32);
    const FusedPlan& pl = a.plan;
    __shared__ int s_ok;
    __shared__ int s_abort[kGatherMaxStreams];
    const int unit = a.row_bytes + a.sf_bytes;
    const int budget = tc::OFF_TAIL - kGatherMaxStreams * kGatherMaxBuf * 8;
    int nstreams = unit > 0 ? budget / (4 * unit) : 0;
    if (nstreams > kGatherMaxStreams) nstreams = kGatherMaxStreams;
    const bool bulk = a.row_bytes % 16 == 0 && a.sf_bytes % 16 == 0 && nstreams >= 1;
    int nbuf = bulk ? budget / (nstreams * unit) : 0;
    if (nbuf > kGatherMaxBuf) nbuf = kGatherMaxBuf;
    uint8_t* buf = smem + (size_t)warp * nbuf * unit;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nstreams * nbuf * unit) + warp * kGatherMaxBuf;
    if (bulk && warp < nstreams && lane == 0) {
        for (int i = 0; i < nbuf; ++i) mbar_init(&bars[i], 1);
        s_abort[warp] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    int q0 = 0;
    for (int b = 1; b < nmb; ++b) {
        if (threadIdx.x == 0) {
            bool ok = true;
            if (b >= a.NR) {
                const int prev = b - a.NR;
                const int target = (pl.pbase[prev + 1] - pl.pbase[prev]) * nt2 * tc::EPI_WARPS;
                ok = wait_counter(pl.g2_done + prev, target, pl.abort_g, a.ws, deadline);
            }
            s_ok = ok && !ld_acquire(pl.abort_g);
        }
        __syncthreads();
        if (!s_ok) return;
        if (bulk) {
            if (warp < nstreams) {
                const int n = gather_stream_bulk(a, b, blockIdx.x * nstreams + warp, a.G * nstreams, buf, bars,
                                                 nbuf, q0, &s_abort[warp], deadline);
                if (n < 0) {
                    if (lane == 0) {
                        atomicExch(pl.abort_g, 1);
                        // let loads already issued land before this CTA's shared memory goes away
                        const unsigned long long d2 = globaltimer_ns() + 1000000ull;
                        while (globaltimer_ns() < d2) {
                        }
                    }
                } else {
                    q0 += n;
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                if (b != a.skip_ready) atomicAdd(pl.gather_done + b, 1);
            }
        } else {
            gather_minibatch(a, b, gw, nw);
        }
    }
}

// Combine role (every CTA, after all GEMM2 tiles): out[n] = sum_j g[n][j] y[inv[n][j]]
// in FP32, fixed j order, one warp per (token, 256-column chunk).  Only one CTA of
// 12 warps fits on an SM here, so each warp takes two items at a time and issues
// the loads of up to eight slot rows of both before it accumulates (same order
// of additions as the stand-alone combine kernel).
__device__ void combine_role(const FusedArgs& a) {
    constexpr int IW = 2, JB = 8;
    const int lane = threadIdx.x & 31;
    const int chunks = (a.H + 255) / 256;
    const int64_t items = (int64_t)a.N * chunks;
    const int64_t gw = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t it0 = gw * IW; it0 < items; it0 += nw * IW) {
        int n[IW], col[IW], my_slot[IW];
        float my_g[IW], acc[IW][8];
        bool live[IW];
#pragma unroll
        for (int i = 0; i < IW; ++i) {
            const int64_t it = it0 + i;
            live[i] = it < items;
            n[i] = live[i] ? (int)(it / chunks) : 0;
            col[i] = live[i] ? (int)(it % chunks) * 256 + lane * 8 : a.H;
            my_slot[i] = (live[i] && lane < a.k) ? a.inv[(int64_t)n[i] * a.k + lane] : 0;
            my_g[i] = (live[i] && lane < a.k) ? a.gate[(int64_t)n[i] * a.k + lane] : 0.f;
#pragma unroll
            for (int v = 0; v < 8; ++v) acc[i][v] = 0.f;
        }
        for (int j0 = 0; j0 < a.k; j0 += JB) {
            uint4 q[IW][JB];
            float g[IW][JB];
            uint32_t use[IW] = {0u, 0u};
#pragma unroll
            for (int u = 0; u < JB; ++u) {
                const int j = j0 + u;
#pragma unroll
                for (int i = 0; i < IW; ++i) {
                    const int slot = __shfl_sync(0xffffffffu, my_slot[i], j & 31);
                    g[i][u] = __shfl_sync(0xffffffffu, my_g[i], j & 31);
                    if (!live[i] || j >= a.k) continue;
                    if (slot < 0 || slot >= a.T) {
                        if (lane == 0) set_status(a.ws, MOE_ERR_DEVICE_CHECK);
                        continue;
                    }
                    if (col[i] < a.H) {
                        // y was stored by other CTAs of this launch: read it through L2
                        q[i][u] = ld_cg_v4(a.y + ((int64_t)slot * a.H + col[i]) * 2);
                        use[i] |= 1u << u;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < JB; ++u) {
#pragma unroll
                for (int i = 0; i < IW; ++i) {
                    if (!(use[i] & (1u << u))) continue;
                    const uint32_t w[4] = {q[i][u].x, q[i][u].y, q[i][u].z, q[i][u].w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        acc[i][2 * p] = fmaf(g[i][u], bf16_to_f32((uint16_t)(w[p] & 0xFFFF)), acc[i][2 * p]);
                        acc[i][2 * p + 1] = fmaf(g[i][u], bf16_to_f32((uint16_t)(w[p] >> 16)), acc[i][2 * p + 1]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < IW; ++i)
            if (live[i] && col[i] < a.H)
                st_v4(a.out + ((int64_t)n[i] * a.H + col[i]) * 2,
                      make_uint4(pack_bf16x2(acc[i][0], acc[i][1]), pack_bf16x2(acc[i][2], acc[i][3]),
                                 pack_bf16x2(acc[i][4], acc[i][5]), pack_bf16x2(acc[i][6], acc[i][7])));
    }
}

template <bool MX>
__global__ void __launch_bounds__(tc::THREADS, 1)
    fused_forward_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA2,
                         const __grid_constant__ CUtensorMap tmS1a, const __grid_constant__ CUtensorMap tmS2a,
                         const __grid_constant__ CUtensorMap tmT1, const __grid_constant__ CUtensorMap tmT2,
                         const __grid_constant__ GemmSide s1, const __grid_constant__ GemmSide s2,
                         const __grid_constant__ FusedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const unsigned long long deadline = globaltimer_ns() + a.timeout_ns;
    const FusedPlan& pl = a.plan;
    __shared__ int s_nmb;
    if (threadIdx.x == 0) s_nmb = *pl.nmb;   // written by the plan launch before this one
    __syncthreads();
    const int nmb = s_nmb;
    const int warps = blockDim.x / 32;

    // the pipeline fills faster when every CTA gathers the first minibatch
    if (nmb > 0) gather_minibatch(a, 0, blockIdx.x * warps + threadIdx.x / 32, gridDim.x * warps);

    if ((int)blockIdx.x < a.G) {
        gather_role(a, nmb, deadline, s2.n_tiles, smem);
    } else {
        // the tile decode runs at every tile boundary in four roles: keep what it
        // reads in shared memory (the plan was written by the previous launch)
        int32_t* off = reinterpret_cast<int32_t*>(smem + tc::OFF_TAIL);
        for (int e = threadIdx.x; e <= a.E; e += blockDim.x) off[e] = a.offsets[e];
        const int32_t *tb = pl.tbase, *pb = pl.pbase, *el = pl.elo, *ct = pl.cut;
        if (a.plan_smem) {
            int32_t* stb = off + (a.E + 1);
            int32_t* spb = stb + (2 * a.nmb_max + 1);
            int32_t* sel = spb + (a.nmb_max + 1);
            int32_t* sct = sel + a.nmb_max;
            for (int i = threadIdx.x; i <= 2 * nmb; i += blockDim.x) stb[i] = pl.tbase[i];
            for (int i = threadIdx.x; i <= nmb; i += blockDim.x) spb[i] = pl.pbase[i];
            for (int i = threadIdx.x; i < nmb; i += blockDim.x) sel[i] = pl.elo[i];
            for (int i = threadIdx.x; i <= nmb; i += blockDim.x) sct[i] = pl.cut[i];
            tb = stb;
            pb = spb;
            el = sel;
            ct = sct;
        }
        __syncthreads();
        MinibatchTiles src{&a, off, tb, pb, el, ct, nmb, s1.n_tiles, s2.n_tiles, (int)blockIdx.x - a.G,
                           (int)gridDim.x - a.G};
        const GemmMaps maps{&tmA1, &tmA2, &tmS1a, &tmS2a, &tmT1, &tmT2};
        const GemmSides sides{&s1, &s2};
        run_gemm_pipeline<MX>(smem, maps, sides, src, a.ws, a.timeout_ns);
    }

    // combine once every GEMM2 tile has been stored
    __shared__ int s_go;
    if (threadIdx.x == 0) {
        const int target = pl.pbase[nmb] * s2.n_tiles * tc::EPI_WARPS;
        s_go = wait_counter(pl.g2_all, target, pl.abort_g, a.ws, deadline) ? 1 : 0;
    }
    __syncthreads();
    if (s_go) combine_role(a);
}

// ------------------------------------------------------------------ host side
cudaError_t launch_fused_forward(const FusedCall& c, cudaStream_t stream) {
    if (c.T == 0) return cudaSuccess;
    // plan arrays and counters live in one int region of the workspace
    int* w = c.plan_ints;
    // (c.nmb is the bound on the minibatch count; the plan kernel cuts the actual ones)
    FusedPlan pl;
    pl.tbase = w;
    pl.pbase = w + (2 * c.nmb + 2);
    pl.elo = pl.pbase + (c.nmb + 1);
    pl.cut = pl.elo + (c.nmb + 1);
    int* counters = pl.cut + (c.nmb + 2);
    const int max_m = fused_max_mtiles(c.T, c.E, c.nmb);
    pl.gather_done = counters;
    pl.g2_done = counters + c.nmb;
    pl.g2_all = counters + 2 * c.nmb;
    pl.abort_g = counters + 2 * c.nmb + 1;
    pl.nmb = counters + 2 * c.nmb + 2;
    pl.g1_done = counters + 2 * c.nmb + 8;
    const int counters_len = 2 * c.nmb + 8 + max_m;

    FfnMaps m;
    GemmSide s1, s2;
    if (!encode_ffn_maps(c.ffn, &m, &s1, &s2)) return cudaErrorInvalidValue;
    fused_plan_kernel<<<1, 1024, sizeof(int32_t) * (c.E + 1), stream>>>(
        c.ffn.offsets, c.E, c.T, c.MB, c.nmb, s1.n_tiles, s2.n_tiles, (c.R / c.MB) >= 2 ? 1 : 0, c.reverse, pl,
        counters_len, counters, c.ffn.ws);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    FusedArgs a{};
    a.plan = pl;
    a.offsets = c.ffn.offsets;
    a.sched = c.sched;
    a.inv = c.inv;
    a.gate = c.gate;
    a.shard_rows = (const uint8_t* const*)c.shard_rows;
    a.shard_sf = (const uint8_t* const*)c.shard_sf;
    a.ring = (uint8_t*)c.ffn.a;
    a.ring_sf = (uint8_t*)c.ffn.a_sf;
    a.y = (uint8_t*)c.ffn.y;
    a.out = (uint8_t*)c.out;
    a.N = c.N;
    a.H = c.H;
    a.E = c.E;
    a.k = c.k;
    a.S = c.S;
    a.T = c.T;
    a.MB = c.MB;
    a.NR = c.R / c.MB;
    a.nmb_max = c.nmb;
    a.G = c.G;
    a.row_bytes = c.row_bytes;
    a.sf_bytes = c.sf_bytes;
    a.skip_ready = c.skip_ready;
    a.ws = c.ffn.ws;
    a.timeout_ns = c.ffn.timeout_ns;

    size_t smem = 1024 + tc::OFF_TAIL + sizeof(int32_t) * (c.E + 1);
    const size_t plan_bytes = sizeof(int32_t) * ((size_t)5 * c.nmb + 3);
    a.plan_smem = smem + plan_bytes <= (size_t)227 * 1024 ? 1 : 0;
    if (a.plan_smem) smem += plan_bytes;
    void* kern = c.ffn.mx ? (void*)fused_forward_kernel<true> : (void*)fused_forward_kernel<false>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    void* args[] = {&m.a1, &m.a2, &m.s1a, &m.s2a, &m.t1, &m.t2, &s1, &s2, &a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.G + c.C);
    cfg.blockDim = dim3(tc::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: they wait on each other
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

int fused_max_ctas() {
    int dev = 0, sms = 0, per = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const size_t smem = 1024 + tc::OFF_TAIL + sizeof(int32_t) * 1025;
    if (cudaFuncSetAttribute(fused_forward_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fused_forward_kernel<true>, tc::THREADS,
                                                      smem) != cudaSuccess)
        return 0;
    return per * sms;
}

}  // namespace moe
