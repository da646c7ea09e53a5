// gemm_roles.cuh -- the warp roles of libmoe's tcgen05 grouped-GEMM pipeline,
// shared by the stand-alone expert-FFN kernels (gemm_tc.cu) and the persistent
// fused forward kernel (fused.cu).
//
// One CTA of 12 warps per SM runs a software pipeline over a sequence of output
// tiles handed out by a tile source:
//   warp 0      producer: per K-stage, the A tile (128 rows x 128 B) by a TMA
//               tensor load and the B tile (256 rows x 128 B) plus, for MXFP8,
//               its 1 KB scale image by two bulk copies from the tile-packed
//               weights, into a 4-stage shared-memory ring; for MXFP8 with
//               K % 512 == 0 also the A scale bytes of four K-stages at a time
//   warp 1      TMEM owner and MMA issuer (one thread): tcgen05.mma 128x256,
//               kind::f16 (BF16) or kind::mxf8f6f4 with UE8M0 block scales
//   warp 2      A scale-factor transposer (MXFP8): builds the [32 lanes][4 words]
//               block of the A rows that tcgen05.cp moves into tensor memory (the
//               B scales arrive already in that form)
//   warp 3      dependency thread (tile sources whose tiles wait for other CTAs):
//               runs ahead over the tile sequence, waits for each tile's inputs
//               and raises a shared-memory counter that the producer checks, so
//               the producer never stalls on a round trip to global memory
//   warps 4-11  epilogue: two warps per tensor-memory lane quarter, each taking
//               half the columns, drain the FP32 accumulator into registers,
//               release it, then apply SwiGLU (+ MXFP8 quantisation of h along I)
//               or BF16 conversion and store.
// A tile is GEMM1 (+SwiGLU; kind 0) or GEMM2 (kind 1; also the form of the
// backward's two dgrad GEMMs).  The source (first / next
// / count / kind_of / tile / wait_inputs / tile_stored) decides the
// order, where each tile's A rows come from, where its output goes, and what a
// tile waits for before its A operand (or its A scales) may be loaded -- nothing
// for the stand-alone kernels; the gather or GEMM1 counters in the fused kernel,
// waited on by whichever thread loads them -- and what each
// epilogue warp signals once its share of a tile is stored.
#pragma once

#include "common.cuh"

namespace moe {

namespace tc {
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int SFG = 2;                                     // scale staging groups (4 K-stages each)
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = BN * 128;
constexpr int SFA_BYTES = 512;                             // [32 lanes][4 words]: 128 rows x 4 K-steps
constexpr int SFB_BYTES = 1024;                            // two such blocks (256 rows)
constexpr int SFSA_BYTES = BM * 16;                        // staged A scales: 128 rows x 16 B (4 stages)
constexpr int B_TILE = B_BYTES;                            // packed B tile image
constexpr int SFB_TILE = SFB_BYTES;                        // packed B scale image
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_SFSA = OFF_SFB + STAGES * SFB_BYTES;
constexpr int OFF_BAR = OFF_SFSA + SFG * SFSA_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 3 + 2 * SFG;        // full, empty, tfull, tempty, drain, sfull, sempty
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;           // tmem base, abort flag, ready count
constexpr int OFF_TAIL = OFF_MISC + 16;                    // kernel-specific tail
constexpr int TMEM_COLS = 512;
constexpr int TCOL_SFA = 256;                              // + stage*4
constexpr int TCOL_SFB = 256 + 4 * STAGES;                 // + stage*8
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (4 + EPI_WARPS) * 32;
}  // namespace tc

// One of the two GEMMs of the expert FFN.
struct GemmSide {
    int K;                    // reduction length (H for GEMM1, I for GEMM2)
    int n_tiles;              // N tiles per expert
    int up_off;               // GEMM1: first up row inside w_gate_up (= I)
    int b_rows;               // rows of one expert's weight matrix (2I or H)
    int sf_tma;               // MXFP8 A scales staged by TMA (K % 512 == 0)
    int a_rows;               // rows of the A tensor (scale loads stay inside)
    const uint8_t* a_sf;      // MXFP8: [a_rows][K/32]
    const uint8_t* b_pk;      // tile-packed weights [E][n_tiles][K-stages][32 KB]
    const uint8_t* sfb_pk;    // MXFP8: tile-packed scales [E][n_tiles][K-stages][1 KB]
    uint8_t* out;             // GEMM1: h [rows][I] (codes or BF16); GEMM2: y BF16 [rows][H]
                              // (the backward's dgrad GEMMs: dh [rows][I], da [rows][H])
    uint8_t* out_sf;          // GEMM1 MXFP8: h scales [rows][I/32]
    int out_ld;               // row length of out in elements
    uint8_t* aux;             // GEMM1 in training: where to save u|v (BF16 [rows][2I])
    int n_valid;              // GEMM2 form: output columns (tile columns past it are padding)
};

// The tensor maps of both GEMMs, picked by tile kind with a select (no indexed
// array, which would live in local memory).
struct GemmMaps {
    const CUtensorMap *a0, *a1;       // A operand of GEMM1 / GEMM2
    const CUtensorMap *sfa0, *sfa1;   // A scales (TMA-staged) of GEMM1 / GEMM2
    const CUtensorMap *t0, *t1;       // A operand with 32-row boxes, for tiles of <= 32 rows
                                      // (an expert's ragged last m-tile); null: not used
    __device__ const CUtensorMap* a(int kind) const { return kind ? a1 : a0; }
    __device__ const CUtensorMap* sfa(int kind) const { return kind ? sfa1 : sfa0; }
    __device__ const CUtensorMap* tail(int kind) const { return kind ? t1 : t0; }
};
constexpr int kTailRows = 32;

// The two GEMM descriptions, picked the same way.  They point at kernel
// parameters declared __grid_constant__, so nothing is copied to local memory.
struct GemmSides {
    const GemmSide *s0, *s1;
    __device__ const GemmSide& operator[](int kind) const { return kind ? *s1 : *s0; }
};

struct TileInfo {
    int kind;                 // 0: GEMM1 + SwiGLU, 1: GEMM2 (or either dgrad GEMM of the
                              // backward, which have the same form)
    int e, n;                 // expert, N tile
    int a_row0;               // first row of the A tile in its tensor
    int out_row0;             // first output row
    int nrows;                // valid rows of the tile (<= 128)
    int mb, midx;             // fused kernel: minibatch, m-tile counter index
};

struct Pipe {
    uint8_t* smem;
    uint64_t *full, *empty, *tfull, *tempty, *drain, *sfull, *sempty;
    uint32_t tmem_base;
    volatile int* abort_flag;
    volatile int* ready;      // tiles whose inputs the dependency thread has seen complete
    WsHeader* ws;
    unsigned long long deadline;
};

__device__ __forceinline__ uint32_t word_of(const uint4& v, int q) {
    return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// Barrier initialisation (one thread) and tensor-memory allocation (warp 1).
template <bool MX>
__device__ __forceinline__ void pipe_init(Pipe& p, uint8_t* smem, WsHeader* ws) {
    using namespace tc;
    p.smem = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    p.full = bars;
    p.empty = bars + STAGES;
    p.tfull = bars + 2 * STAGES;
    p.tempty = p.tfull + 1;
    p.drain = p.tfull + 2;
    p.sfull = p.tfull + 3;
    p.sempty = p.sfull + SFG;
    p.abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    p.ready = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
    p.ws = ws;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&p.full[s], MX ? 2 : 1);
            mbar_init(&p.empty[s], 1);
        }
        mbar_init(p.tfull, 1);
        mbar_init(p.tempty, EPI_WARPS);
        mbar_init(p.drain, 1);
        for (int g = 0; g < SFG; ++g) {
            mbar_init(&p.sfull[g], 1);
            mbar_init(&p.sempty[g], 1);
        }
        *p.abort_flag = 0;
        *p.ready = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(reinterpret_cast<uint32_t*>(smem + OFF_MISC), TMEM_COLS);
        tmem_relinquish();
    }
}

// ------------------------------------------------------------------ TMA producer
template <bool MX, class Src>
__device__ void producer_role(const Pipe& p, const GemmMaps& maps, const GemmSides& sides, Src& src) {
    using namespace tc;
    int stage = 0, g = 0;
    uint32_t phase = 0, gphase = 0;
    int ordinal = 0;          // tiles of this CTA so far
    for (int t = src.first(); t < src.count(); t = src.next(t)) {
        const TileInfo tl = src.tile(t);
        const GemmSide& sd = sides[tl.kind];
        if constexpr (Src::kDeps) {
            // the dependency thread has acquired this tile's inputs (bounded wait)
            ++ordinal;
            uint32_t n = 0;
            while (ld_acquire_cta(p.ready) < ordinal) {
                if (*p.abort_flag) return;
                if ((++n & 255u) == 0 && globaltimer_ns() > p.deadline) {
                    *p.abort_flag = 1;
                    set_status(p.ws, MOE_ERR_TIMEOUT);
                    return;
                }
            }
            fence_proxy_async_global();   // rows other CTAs stored may now be read by TMA
        }
        const bool sf_tma = MX && sd.sf_tma;
        const int KB = sd.K / (MX ? 128 : 64);
        const int64_t tile0 = ((int64_t)tl.e * sd.n_tiles + tl.n) * KB;   // first packed K-stage
        for (int kb = 0; kb < KB; ++kb) {
            if (sf_tma && (kb & 3) == 0) {
                if (!mbar_wait_bounded(&p.sempty[g], gphase ^ 1, p.abort_flag, p.ws, p.deadline)) return;
                mbar_arrive_expect_tx(&p.sfull[g], SFSA_BYTES);
                tma_load_2d(p.smem + OFF_SFSA + g * SFSA_BYTES, maps.sfa(tl.kind), &p.sfull[g], kb * 4,
                            tl.a_row0);
                if (++g == SFG) {
                    g = 0;
                    gphase ^= 1;
                }
            }
            if (!mbar_wait_bounded(&p.empty[stage], phase ^ 1, p.abort_flag, p.ws, p.deadline)) return;
            uint8_t* sa = p.smem + OFF_A + stage * A_BYTES;
            uint8_t* sb = p.smem + OFF_B + stage * B_BYTES;
            // A tile of a few rows: load only its first kTailRows rows; the MMA still
            // runs all 128, and the rows past the tile are never stored
            const CUtensorMap* ta = maps.a(tl.kind);
            int a_bytes = A_BYTES;
            if (tl.nrows <= kTailRows && maps.tail(tl.kind) != nullptr) {
                ta = maps.tail(tl.kind);
                a_bytes = kTailRows * 128;
            }
            // the weight tile first: for the first CTA on an (expert, N tile) it comes
            // from DRAM, the longer wait (measured 0.8% faster than A first)
            mbar_arrive_expect_tx(&p.full[stage], a_bytes + B_BYTES + (MX ? SFB_BYTES : 0));
            bulk_load(sb, sd.b_pk + (tile0 + kb) * B_TILE, B_TILE, &p.full[stage]);
            if (MX)
                bulk_load(p.smem + OFF_SFB + stage * SFB_BYTES, sd.sfb_pk + (tile0 + kb) * SFB_TILE,
                          SFB_TILE, &p.full[stage]);
            tma_load_2d(sa, ta, &p.full[stage], kb * (MX ? 128 : 64), tl.a_row0);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
}

// ----------------------------------------------------- dependency thread (warp 3)
// Walks the same tile sequence as the producer, waits (bounded) for each tile's
// inputs and publishes the count of ready tiles in shared memory.
template <class Src>
__device__ void deps_role(const Pipe& p, Src& src) {
    int n = 0;
    for (int t = src.first(); t < src.count(); t = src.next(t)) {
        const TileInfo tl = src.tile(t);
        if (!src.wait_inputs(tl, p)) return;
        st_release_cta(p.ready, ++n);
    }
}

// ------------------------------------------------------------------- MMA issuer
template <bool MX, class Src>
__device__ void mma_role(const Pipe& p, const GemmSides& sides, Src& src) {
    using namespace tc;
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    const uint32_t d_tmem = p.tmem_base;
    bool ok = true;
    for (int t = src.first(); ok && t < src.count(); t = src.next(t)) {
        const int KB = sides[src.kind_of(t)].K / (MX ? 128 : 64);   // the issuer needs only the tile's K
        if (!mbar_wait_bounded(p.tempty, acc_phase ^ 1, p.abort_flag, p.ws, p.deadline)) break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait_bounded(&p.full[stage], phase, p.abort_flag, p.ws, p.deadline)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(p.smem + OFF_A + stage * A_BYTES);
            const uint32_t sb = smem_u32(p.smem + OFF_B + stage * B_BYTES);
            if constexpr (MX) {
                const uint32_t sfa_t = p.tmem_base + TCOL_SFA + stage * 4;
                const uint32_t sfb_t = p.tmem_base + TCOL_SFB + stage * 8;
                tmem_cp_32x128b_x4(sfa_t, sdesc_sf_block(smem_u32(p.smem + OFF_SFA + stage * SFA_BYTES)));
                tmem_cp_32x128b_x4(sfb_t, sdesc_sf_block(smem_u32(p.smem + OFF_SFB + stage * SFB_BYTES)));
                tmem_cp_32x128b_x4(sfb_t + 4, sdesc_sf_block(smem_u32(p.smem + OFF_SFB + stage * SFB_BYTES + 512)));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_mxf8(d_tmem, sdesc_kmajor_sw128(sa + 32 * k), sdesc_kmajor_sw128(sb + 32 * k),
                             idesc_mxf8(BM, BN, k, k), sfa_t, sfb_t, (kb | k) != 0);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(d_tmem, sdesc_kmajor_sw128(sa + 32 * k), sdesc_kmajor_sw128(sb + 32 * k),
                             idesc_bf16(BM, BN), (kb | k) != 0);
            }
            mma_commit(&p.empty[stage]);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (ok) mma_commit(p.tfull);
        acc_phase ^= 1;
    }
    // wait until every tensor-core operation issued here has finished
    mma_commit(p.drain);
    const unsigned long long d2 = globaltimer_ns() + 1000000ull;
    while (!mbar_try_wait(p.drain, 0) && globaltimer_ns() < d2) {
    }
}

// ----------------------------------------- A scale factors (MXFP8, whole warp 2)
// Each K-stage needs a [32 lanes][4 words] block for the A rows: word j of lane r
// holds the four K-step scales of row 32j + r.  tcgen05.cp moves that block into
// tensor memory; the B scales arrive already packed this way.
template <class Src>
__device__ void sf_role(const Pipe& p, const GemmSides& sides, Src& src) {
    using namespace tc;
    const int lane = threadIdx.x % 32;
    int stage = 0, g = 0;
    uint32_t phase = 0, gphase = 0;
    for (int t = src.first(); t < src.count(); t = src.next(t)) {
        const TileInfo tl = src.tile(t);
        const GemmSide& sd = sides[tl.kind];
        const int KB = sd.K / 128;
        const int ksf = sd.K / 32;                  // scale bytes per row
        if (sd.sf_tma) {
            for (int kb = 0; kb < KB; ++kb) {
                if ((kb & 3) == 0 && !mbar_wait_bounded(&p.sfull[g], gphase, p.abort_flag, p.ws, p.deadline))
                    return;
                if (!mbar_wait_bounded(&p.empty[stage], phase ^ 1, p.abort_flag, p.ws, p.deadline)) return;
                const int q = kb & 3;
                const uint8_t* sa = p.smem + OFF_SFSA + g * SFSA_BYTES + 4 * q;
                uint32_t a[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) a[j] = *reinterpret_cast<const uint32_t*>(sa + (32 * j + lane) * 16);
                reinterpret_cast<uint4*>(p.smem + OFF_SFA + stage * SFA_BYTES)[lane] =
                    make_uint4(a[0], a[1], a[2], a[3]);
                // every lane's reads are consumed by its own store before the fence,
                // so the releases below cannot overtake them
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&p.full[stage]);
                    if (q == 3) mbar_arrive(&p.sempty[g]);
                }
                if (q == 3 && ++g == SFG) {
                    g = 0;
                    gphase ^= 1;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        } else {
            // Scale rows that are not 16-byte multiples: direct 4-byte loads.  The A
            // scales may have been written earlier in this launch by other CTAs
            // (fused kernel), so every lane first waits for the tile's inputs
            // itself (its own acquire) and the loads bypass L1.
            if (!src.wait_inputs(tl, p)) return;
            for (int kb4 = 0; kb4 < KB; kb4 += 4) {
                uint4 va[4];
                const int nq = min(4, KB - kb4);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = tl.a_row0 + 32 * j + lane;
                    uint32_t w[4] = {0, 0, 0, 0};
                    for (int q = 0; q < nq; ++q)
                        if (row < sd.a_rows) w[q] = ld_cg_u32(sd.a_sf + (int64_t)row * ksf + (kb4 + q) * 4);
                    va[j] = make_uint4(w[0], w[1], w[2], w[3]);
                }
                for (int q = 0; q < nq; ++q) {
                    if (!mbar_wait_bounded(&p.empty[stage], phase ^ 1, p.abort_flag, p.ws, p.deadline)) return;
                    reinterpret_cast<uint4*>(p.smem + OFF_SFA + stage * SFA_BYTES)[lane] =
                        make_uint4(word_of(va[0], q), word_of(va[1], q), word_of(va[2], q), word_of(va[3], q));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p.full[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    }
}

// --------------------------------------------------------- epilogue (warps 4-11)
template <bool MX, class Src>
__device__ void epilogue_role(const Pipe& p, const GemmSides& sides, Src& src) {
    using namespace tc;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    uint32_t acc_phase = 0;
    for (int t = src.first(); t < src.count(); t = src.next(t)) {
        const TileInfo tl = src.tile(t);
        const GemmSide& sd = sides[tl.kind];
        if (!mbar_wait_bounded(p.tfull, acc_phase, p.abort_flag, p.ws, p.deadline)) return;
        tc_fence_after();
        const int r = 32 * q + lane;
        const bool valid = r < tl.nrows;
        const int64_t row = tl.out_row0 + r;
        const uint32_t tq = p.tmem_base + ((uint32_t)(32 * q) << 16);
        if (tl.kind == 0) {
            // GEMM1: h = silu(gate) * up over this warp's 64 of the 128 h columns.
            // All four accumulator chunks are read with one wait and the
            // accumulator is released before any arithmetic.
            uint32_t g0[32], u0[32], g1[32], u1[32];
            tmem_ld_32x32b_x32(tq + 32 * (half * 2), g0);
            tmem_ld_32x32b_x32(tq + 128 + 32 * (half * 2), u0);
            tmem_ld_32x32b_x32(tq + 32 * (half * 2 + 1), g1);
            tmem_ld_32x32b_x32(tq + 128 + 32 * (half * 2 + 1), u1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p.tempty);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint32_t* g = c2 ? g1 : g0;
                const uint32_t* u = c2 ? u1 : u0;
                float hv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) hv[i] = silu_f32(__uint_as_float(g[i])) * __uint_as_float(u[i]);
                const int col = tl.n * 128 + 32 * (half * 2 + c2);
                uint32_t pk[16];
                if constexpr (Src::kSaveUV) if (valid) {
                    // training: keep the pre-activations for the SwiGLU backward
                    uint8_t* dst = sd.aux + (row * 2 * sd.out_ld + col) * 2;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
                    st_v8(dst, pk);
                    st_v8(dst + 32, pk + 8);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
                    dst += (int64_t)sd.out_ld * 2;
                    st_v8(dst, pk);
                    st_v8(dst + 32, pk + 8);
                }
                if constexpr (MX) {
                    const uint8_t sc = mx_quantize32(hv, pk);
                    if (valid) {
                        st_v8(sd.out + row * sd.out_ld + col, pk);
                        sd.out_sf[row * (sd.out_ld / 32) + col / 32] = sc;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
                    if (valid) {
                        uint8_t* dst = sd.out + (row * sd.out_ld + col) * 2;
                        st_v8(dst, pk);
                        st_v8(dst + 32, pk + 8);
                    }
                }
            }
        } else {
            // GEMM2: y tile in BF16, this warp's 128 of the 256 columns (one wait,
            // release, then convert and store)
            uint32_t v[4][32];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_ld_32x32b_x32(tq + 32 * (half * 4 + c4), v[c4]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p.tempty);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(v[c4][2 * i]), __uint_as_float(v[c4][2 * i + 1]));
                const int col = tl.n * BN + 32 * (half * 4 + c4);
                if (valid && col < sd.n_valid) {
                    uint8_t* dst = sd.out + (row * sd.out_ld + col) * 2;
                    st_v8(dst, pk);
                    st_v8(dst + 32, pk + 8);
                }
            }
        }
        // each epilogue warp reports its own part of the tile (no barrier between
        // the warps, so a warp that gave up cannot stall the others)
        src.tile_stored(tl, p);
        acc_phase ^= 1;
    }
}

// Runs the four roles of the pipeline over src on this CTA (all 12 warps), then
// releases tensor memory.  smem must be 1024-byte aligned.
template <bool MX, class Src>
__device__ void run_gemm_pipeline(uint8_t* smem, const GemmMaps& maps, const GemmSides& sides, Src& src,
                                  WsHeader* ws, unsigned long long timeout_ns) {
    using namespace tc;
    Pipe p;
    pipe_init<MX>(p, smem, ws);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0 && lane == 0) {
        prefetch_tmap(maps.a0);
        prefetch_tmap(maps.a1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    p.tmem_base = *reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    p.deadline = globaltimer_ns() + timeout_ns;

    if (warp == 0) {
        if (lane == 0) producer_role<MX>(p, maps, sides, src);
    } else if (warp == 1) {
        if (lane == 0) mma_role<MX>(p, sides, src);
    } else if (warp == 2) {
        if constexpr (MX) sf_role(p, sides, src);
    } else if (warp == 3) {
        if constexpr (Src::kDeps)
            if (lane == 0) deps_role(p, src);
    } else {
        epilogue_role<MX>(p, sides, src);
    }

    if (*p.abort_flag) {
        // let any copy still in flight land before the CTA's memory is released
        const unsigned long long d2 = globaltimer_ns() + 1000000ull;
        while (globaltimer_ns() < d2) {
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(p.tmem_base, TMEM_COLS);
}

}  // namespace moe
