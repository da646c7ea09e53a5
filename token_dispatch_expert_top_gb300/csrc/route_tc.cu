// route_tc.cu -- router on the tensor cores: logits = x . W_r (BF16 products,
// FP32 accumulation in tensor memory) for a 128-token tile per CTA, then softmax
// top-k and renormalised gates in the epilogue, one token per thread.  When the
// layer is MXFP8 the same pass quantises x for the dispatch: eight warps read each
// K-stage of x from shared memory (where TMA put it for the MMA) and write its E4M3
// codes and UE8M0 scales, so x is read from HBM once.
// ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72": section 01, each token picks a few experts per step; section 02, MXFP8
// activation quantisation folded into the data path.)
//
// CTA = 16 warps:  w0 TMA producer (4-stage ring), w1 MMA issuer + TMEM owner,
//                  w2-3 idle,
//                  w4-11 x quantisers (MXFP8 only; every K-stage, one 32-element
//                  block of one token row per thread),
//                  then all 16 warps: the top-k epilogue.  Warp w reads the logits of
//                  token rows 32(w%4)..+31 (its tensor-memory lane quarter) over one
//                  of up to four column ranges (w/4), keeps their top-k, and the
//                  first warp of each quarter merges the four sorted lists.
// Split mode (E >= 64, E % 32 == 0, H >= 128): a cluster of two CTAs shares a
// 128-token tile, each taking half of K for every expert (twice the CTAs; each x
// byte crosses from L2 once) and quantising its half of x.  The partial logits
// then cross through distributed shared memory, into the partner's drained x
// ring: each CTA completes the logits of half of the experts and takes their
// top-k, and the second CTA hands its per-token candidates to the first, which
// merges the two sorted lists and writes idx and gates.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace moe {

namespace rt {
constexpr int BM = 128;
constexpr int A_BYTES = BM * 128;            // 128 tokens x 64 BF16
constexpr int B_BYTES = 256 * 128;           // up to 256 experts x 64 BF16
constexpr int THREADS = 512;
constexpr int QUANT_WARPS = 8;
constexpr int STAGES = 4;                    // even: a stage's index has the parity of its K-stages
// Shared-memory layout: a ring of x tiles and weight tiles.  In split mode the x
// part of the ring (64 KB) afterwards receives the partner CTA's partial logits.
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;     // full, empty, tfull, cand, qdone, pfree, xdata
constexpr int WARPS = THREADS / 32;
constexpr int MAX_SUB = 4;                   // column ranges of the epilogue's top-k
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem base, abort flag
constexpr int OFF_BIAS = OFF_MISC + 16;
constexpr int OFF_CAND = OFF_BIAS + 256 * 4;       // split mode: partner's candidates
inline size_t smem_bytes(int kmax) { return 1024 + OFF_CAND + (size_t)kmax * BM * 8; }
static_assert(STAGES * A_BYTES >= BM * 128 * 4, "the x ring holds 128 partial logits per token");
static_assert(STAGES * B_BYTES >= BM * MAX_SUB * 32 * 8, "the weight ring holds every sub-list (k <= 32)");
static_assert(BM * 8 * 8 >= QUANT_WARPS * 32 * 4, "the candidate area holds the quantisers' scratch words");
}  // namespace rt

struct RouteArgs {
    int N, H, E, k;
    const float* bias;
    int32_t* idx;
    float* gate;
    float* logits_out;
    uint8_t* xq;          // [N][H] codes, or null
    uint8_t* xq_sf;       // [N][H/32]
    WsHeader* ws;
    unsigned long long timeout_ns;
    uint32_t tmem_cols;
};

// Keep the KMAX largest (value, index) pairs, sorted by descending value; equal
// values keep the earlier (lower) index first because a newcomer only moves up
// past strictly smaller values.  The comparisons against the old list are
// independent of each other: entries from the newcomer's position on shift down
// by one in a single pass of selects, with no chain of compare-and-swap steps.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], float v, int e) {
    bool gt[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) gt[i] = v > tv[i];      // true from the insertion point on
#pragma unroll
    for (int i = KMAX - 1; i > 0; --i) {
        const float nv = gt[i - 1] ? tv[i - 1] : v;
        const int ni = gt[i - 1] ? ti[i - 1] : e;
        tv[i] = gt[i] ? nv : tv[i];
        ti[i] = gt[i] ? ni : ti[i];
    }
    if (gt[0]) {
        tv[0] = v;
        ti[0] = e;
    }
}

template <int KMAX, bool QUANT, bool SPLIT>
__global__ void __launch_bounds__(rt::THREADS, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    RouteArgs args) {
    using namespace rt;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = full + 2 * STAGES;
    uint64_t* cand_bar = tfull + 1;     // split: the partner's top-k candidates are here
    uint64_t* qdone = tfull + 2;        // split: this CTA's quantisers are past their last stage
    uint64_t* pfree = tfull + 3;        // split: the partner's x ring may be overwritten
    uint64_t* xdata = tfull + 4;        // split: the partner's partial logits are here
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    float* cand_v = reinterpret_cast<float*>(smem + OFF_CAND);                 // [BM][KMAX]
    int* cand_i = reinterpret_cast<int*>(smem + OFF_CAND + BM * KMAX * 4);     // [BM][KMAX]
    // split: the partner's partial logits of this CTA's experts, [EH/4][BM][4] FP32,
    // written over the x part of the ring once neither CTA reads it any more
    float* xpart = reinterpret_cast<float*>(smem + OFF_A);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    float* sbias = reinterpret_cast<float*>(smem + OFF_BIAS);
    // the quantisers' scratch words: the candidate area, which the partner fills
    // only after every warp of this CTA has left its main-loop role
    volatile uint32_t* sdep = reinterpret_cast<volatile uint32_t*>(smem + OFF_CAND);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = SPLIT ? (int)cluster_ctarank() : 0;      // which half of K, and of the experts' top-k
    const uint32_t peer = (uint32_t)half ^ 1u;
    const int row0 = (SPLIT ? blockIdx.x / 2 : blockIdx.x) * BM;
    const int KB = args.H / 64;
    const int kb_lo = SPLIT ? half * ((KB + 1) / 2) : 0;     // first K-stage of this CTA
    const int nkb = SPLIT ? (half ? KB / 2 : (KB + 1) / 2) : KB;
    const int E = args.E;                                     // MMA width: every expert
    const int EH = SPLIT ? E / 2 : E;                         // experts whose top-k this CTA takes
    const int e0 = half * EH;                                 // first of them
    const uint32_t b_bytes = (uint32_t)E * 128;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            // MMA + every quantiser warp
            mbar_init(&empty[s], QUANT ? 1 + QUANT_WARPS : 1);
        }
        mbar_init(tfull, 1);
        mbar_init(cand_bar, 4);                               // the partner's four merging warps
        mbar_init(qdone, QUANT_WARPS);
        mbar_init(pfree, WARPS);                              // every warp of the partner
        mbar_init(xdata, WARPS);                              // every warp of the partner
        *abort_flag = 0;
        if (SPLIT)
            fence_mbar_init_cluster();
        else
            fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, args.tmem_cols);
        tmem_relinquish();
    }
    for (int e = threadIdx.x; e < EH; e += THREADS) sbias[e] = args.bias ? args.bias[e0 + e] : 0.f;
    tc_fence_before();
    __syncthreads();
    if constexpr (SPLIT) cluster_sync();   // the partner's barriers exist before any arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const unsigned long long deadline = globaltimer_ns() + args.timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int j = 0; j < nkb; ++j) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.ws, deadline)) break;
                mbar_arrive_expect_tx(&full[stage], A_BYTES + b_bytes);
                tma_load_2d(smem + OFF_A + stage * A_BYTES, &tmX, &full[stage], (kb_lo + j) * 64, row0);
                tma_load_2d(smem + OFF_B + stage * B_BYTES, &tmW, &full[stage], (kb_lo + j) * 64, 0);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16(BM, E);
            for (int j = 0; j < nkb; ++j) {
                if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.ws, deadline)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + OFF_A + stage * A_BYTES);
                const uint32_t sb = smem_u32(smem + OFF_B + stage * B_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem_base, sdesc_kmajor_sw128(sa + 32 * k), sdesc_kmajor_sw128(sb + 32 * k),
                             idesc, (j | k) != 0);
                mma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (ok) mma_commit(tfull);
        }
    } else if (warp >= 4 && warp < 12) {
        if constexpr (QUANT) {
            // Thread = (token row r, 32-element block b of the stage's 64).  Every
            // quantiser warp takes every K-stage in order, so the stage is released
            // once each thread has converted one block.
            const int tq = (warp - 4) * 32 + lane;
            const int r = tq & (BM - 1);
            const int b = tq >> 7;
            const int row = row0 + r;
            int stage = 0;
            uint32_t phase = 0;
            for (int j = 0; j < nkb; ++j) {
                if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.ws, deadline)) break;
                const int kb = kb_lo + j;
                const uint8_t* tile = smem + OFF_A + stage * A_BYTES + r * 128;
                uint4 qv[4];
                uint32_t dep = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // 128-byte swizzle: 16-byte chunk cc of row r sits at chunk cc ^ (r % 8)
                    const int cc = 4 * b + c;
                    qv[c] = *reinterpret_cast<const uint4*>(tile + ((cc ^ (r & 7)) << 4));
                    dep ^= qv[c].x ^ qv[c].y ^ qv[c].z ^ qv[c].w;
                }
                // Release the stage as soon as every lane holds its words: a store of
                // `dep` (which needs every loaded word) into this thread's scratch word
                // cannot be performed before the reads have returned, and the proxy
                // fence orders it, and the reads, before the next TMA (async-proxy)
                // refill.  The conversion and the global stores then run off the
                // ring's path.
                sdep[tq] = dep;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                float v[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        v[8 * c + 2 * p] = bf16_to_f32((uint16_t)(w[p] & 0xFFFF));
                        v[8 * c + 2 * p + 1] = bf16_to_f32((uint16_t)(w[p] >> 16));
                    }
                }
                uint32_t cb[8];
                const uint8_t sc = mx_quantize32(v, cb);
                if (row < args.N) {   // one full 32-byte sector of codes and the block's scale
                    st_v8(args.xq + (int64_t)row * args.H + kb * 64 + b * 32, cb);
                    args.xq_sf[(int64_t)row * (args.H / 32) + kb * 2 + b] = sc;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if constexpr (SPLIT) {
                __syncwarp();
                if (lane == 0) mbar_arrive(qdone);
            }
        }
    }

    // ------------------------------------------------------------ epilogue (all warps)
    __syncwarp();
    {
        const int q = warp & 3;
        const int sub = warp >> 2;
        const int rl = 32 * q + lane;             // token row within the tile
        const int row = row0 + rl;
        const int nsub = EH % 64 == 0 ? 4 : (EH % 32 == 0 ? 2 : 1);   // column ranges, 16-column multiples
        const int per = EH / nsub;
        const bool active = sub < nsub;
        float tv[KMAX];
        int ti[KMAX];
#pragma unroll
        for (int i = 0; i < KMAX; ++i) {
            tv[i] = -INFINITY;
            ti[i] = -1;
        }
        bool got = mbar_wait_bounded(tfull, 0, abort_flag, args.ws, deadline);
        if (got) tc_fence_after();
        const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
        if constexpr (SPLIT) {
            // Each CTA holds partial logits over its half of K for every expert.
            // Once this CTA's ring is idle (MMAs and quantisers done), the partner
            // may write into it; every warp then sends its rows' partials of its
            // column range of the partner's experts into the partner's ring and
            // waits for the reverse.
            if (got && QUANT) got = mbar_wait_bounded(qdone, 0, abort_flag, args.ws, deadline);
            __syncwarp();
            if (got && lane == 0) mbar_arrive_remote(pfree, peer);
            if (got) got = mbar_wait_bounded_cluster(pfree, 0, abort_flag, args.ws, deadline);
            if (got && active) {
                for (int c = 0; c < per / 16; ++c) {
                    const int col = sub * per + 16 * c;
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tq + peer * EH + col, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_cluster_v4(mapa_shared(smem_u32(xpart + ((col / 4 + i) * BM + rl) * 4), peer),
                                      r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
                }
            }
            __syncwarp();
            if (got && lane == 0) mbar_arrive_remote(xdata, peer);
            if (got) got = mbar_wait_bounded_cluster(xdata, 0, abort_flag, args.ws, deadline);
        }
        if (got && active) {
            for (int c = 0; c < per / 16; ++c) {
                const int col = sub * per + 16 * c;
                uint32_t r[16];
                tmem_ld_32x32b_x16(tq + e0 + col, r);
                tmem_ld_wait();
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
                if constexpr (SPLIT) {
                    // the two K halves add in the same order on both CTAs (FP32
                    // addition commutes), so a logit does not depend on its owner
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 pp = *reinterpret_cast<const float4*>(xpart + ((col / 4 + i) * BM + rl) * 4);
                        v[4 * i] += pp.x;
                        v[4 * i + 1] += pp.y;
                        v[4 * i + 2] += pp.z;
                        v[4 * i + 3] += pp.w;
                    }
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] += sbias[col + i];
                if (args.logits_out && row < args.N) {
                    float* dst = args.logits_out + (int64_t)row * args.E + e0 + col;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_v4(dst + 4 * i, make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                                      __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])));
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) topk_insert<KMAX>(tv, ti, v[i], e0 + col + i);
            }
        }
        // Publish each column range's sorted list in the idle weight ring, then the
        // quarter's first warp merges them: repeatedly the largest head, the lower
        // expert index first on equal logits -- the order topk_insert keeps -- so
        // the result is the top-k of all this CTA's experts.
        float* lv = reinterpret_cast<float*>(smem + OFF_B);                       // [BM][MAX_SUB][KMAX]
        int* li = reinterpret_cast<int*>(smem + OFF_B + BM * MAX_SUB * KMAX * 4);
        if (got && active) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                lv[(rl * MAX_SUB + sub) * KMAX + j] = tv[j];
                li[(rl * MAX_SUB + sub) * KMAX + j] = ti[j];
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(1 + q), "r"(128) : "memory");    // the 4 warps of quarter q
        if (sub == 0) {
            if (got) {
                int head[MAX_SUB] = {0, 0, 0, 0};
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    int best = -1, bi = 0;
                    float bv = 0.f;
#pragma unroll
                    for (int u = 0; u < MAX_SUB; ++u) {
                        if (u >= nsub || head[u] >= KMAX) continue;
                        const float v = lv[(rl * MAX_SUB + u) * KMAX + head[u]];
                        const int i = li[(rl * MAX_SUB + u) * KMAX + head[u]];
                        if (best < 0 || v > bv || (v == bv && i < bi)) {
                            best = u;
                            bv = v;
                            bi = i;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < MAX_SUB; ++u) head[u] += best == u ? 1 : 0;
                    tv[j] = bv;
                    ti[j] = bi;
                }
            }
            bool write = row < args.N;
            if constexpr (SPLIT) {
                if (half == 1) {
                    // hand this half's candidates to the first CTA of the pair (its
                    // shared memory, through the cluster), then tell it they are there
                    if (got) {
#pragma unroll
                        for (int j = 0; j < KMAX; ++j) {
                            const uint32_t av = mapa_shared(smem_u32(cand_v + rl * KMAX + j), 0);
                            const uint32_t ai = mapa_shared(smem_u32(cand_i + rl * KMAX + j), 0);
                            asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(av), "r"(__float_as_uint(tv[j]))
                                         : "memory");
                            asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(ai), "r"(ti[j]) : "memory");
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(cand_bar, 0);
                    }
                    write = false;
                } else {
                    // the other half's top-k joins after this half's: its experts have
                    // higher indices, so equal logits keep the lower index first
                    if (got && mbar_wait_bounded_cluster(cand_bar, 0, abort_flag, args.ws, deadline)) {
#pragma unroll
                        for (int j = 0; j < KMAX; ++j)
                            topk_insert<KMAX>(tv, ti, cand_v[rl * KMAX + j], cand_i[rl * KMAX + j]);
                    } else {
                        write = false;
                    }
                }
            }
            if (got && write) {
                float z = 0.f;
                float p[KMAX];
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    p[j] = (j < args.k) ? expf(tv[j] - tv[0]) : 0.f;
                    z += p[j];
                }
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < args.k) {
                        args.idx[(int64_t)row * args.k + j] = ti[j];
                        args.gate[(int64_t)row * args.k + j] = p[j] / z;
                    }
                }
            }
        }
    }

    if (*abort_flag) {
        const unsigned long long d2 = globaltimer_ns() + 1000000ull;
        while (globaltimer_ns() < d2) {
        }
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA of a pair leaves while the other may still write to its memory
    if constexpr (SPLIT) cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, args.tmem_cols);
}

bool route_tc_supported(int dtype, int H, int E, int k) {
    return dtype != MOE_F32 && E % 16 == 0 && E <= 256 && H % 64 == 0 && k <= 32;
}

template <int KMAX, bool QUANT>
static cudaError_t launch_route(const CUtensorMap& tx, const CUtensorMap& tw, const RouteArgs& a,
                                int tiles, bool split, cudaStream_t st) {
    const size_t smem = rt::smem_bytes(KMAX);
    if (!split) {
        auto kern = route_tc_kernel<KMAX, QUANT, false>;
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<tiles, rt::THREADS, smem, st>>>(tx, tw, a);
        return cudaGetLastError();
    }
    auto kern = route_tc_kernel<KMAX, QUANT, true>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * tiles);
    cfg.blockDim = dim3(rt::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tx, tw, a);
}

cudaError_t launch_route_topk_tc(const void* x, const void* w, const float* bias, int N, int H,
                                 int E, int k, int32_t* idx, float* gate, float* logits_out,
                                 uint8_t* xq, uint8_t* xq_sf, WsHeader* ws,
                                 unsigned long long timeout_ns, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    // two CTAs per token tile, each with half of K, when there are two K-stages
    // and the experts' halves (whose top-k each CTA takes) are whole 16-column
    // tensor-memory loads of at least 32
    const bool split = E >= 64 && E % 32 == 0 && H >= 128;
    CUtensorMap tx, tw;
    {
        uint64_t dims[2] = {(uint64_t)H, (uint64_t)N};
        uint64_t str[1] = {(uint64_t)H * 2};
        uint32_t box[2] = {64, (uint32_t)rt::BM};
        if (!encode_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, str, box))
            return cudaErrorInvalidValue;
        uint64_t dw[2] = {(uint64_t)H, (uint64_t)E};
        uint32_t bw[2] = {64, (uint32_t)E};
        if (!encode_tmap(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, dw, str, bw))
            return cudaErrorInvalidValue;
    }
    RouteArgs a{};
    a.N = N;
    a.H = H;
    a.E = E;
    a.k = k;
    a.bias = bias;
    a.idx = idx;
    a.gate = gate;
    a.logits_out = logits_out;
    a.xq = xq;
    a.xq_sf = xq_sf;
    a.ws = ws;
    a.timeout_ns = timeout_ns;
    uint32_t cols = 32;
    while (cols < (uint32_t)E) cols <<= 1;
    a.tmem_cols = cols;
    const int tiles = (N + rt::BM - 1) / rt::BM;
    const bool quant = xq != nullptr;
    if (k <= 8)
        return quant ? launch_route<8, true>(tx, tw, a, tiles, split, stream)
                     : launch_route<8, false>(tx, tw, a, tiles, split, stream);
    if (k <= 16)
        return quant ? launch_route<16, true>(tx, tw, a, tiles, split, stream)
                     : launch_route<16, false>(tx, tw, a, tiles, split, stream);
    return quant ? launch_route<32, true>(tx, tw, a, tiles, split, stream)
                 : launch_route<32, false>(tx, tw, a, tiles, split, stream);
}

}  // namespace moe
