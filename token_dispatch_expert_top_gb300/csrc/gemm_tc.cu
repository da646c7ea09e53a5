// gemm_tc.cu -- grouped expert GEMMs on the sm_103a tensor cores (tcgen05).
//
// One persistent kernel template covers both expert GEMMs of the SwiGLU FFN, in
// BF16 (kind::f16) and block-scaled MXFP8 (kind::mxf8f6f4, one UE8M0 scale per 32
// K-elements):
//   GEMM1 + SwiGLU: [u v] = a . [Wg Wu]  ->  h = silu(u) * v  (BF16, or MXFP8
//                   quantised along I in the epilogue: each epilogue thread owns
//                   one row and 32 consecutive columns, i.e. whole scale blocks)
//   GEMM2        : y = h . Wd  ->  BF16
// Expert segments of rows are [offsets[e], offsets[e+1]) of the A operand; the
// kernel reads the offsets on device and enumerates (expert, m-tile, n-tile)
// tiles itself, m-tiles innermost so consecutive CTAs share weight tiles in L2.
// ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72": section 01, the grouped GEMM fed expert-contiguous input on Blackwell
// tensor cores; section 02, SwiGLU and MXFP8 activation quantisation inside the
// GEMM data path rather than a separate quantise kernel.)
//
// CTA = 8 warps, one CTA per SM:
//   warp 0      TMA producer (A tile 128 x 128 B, B tile 256 x 128 B per stage)
//   warp 1      TMEM allocator + MMA issuer (one thread)
//   warp 2      scale-factor loader (MXFP8): reads the [rows][K/32] scale bytes,
//               transposes them into the [32 lanes][4 words] blocks tcgen05.cp
//               moves to tensor memory
//   warp 3      idle after the prologue
//   warps 4-7   epilogue: tensor memory -> registers -> SwiGLU / convert -> global
// Tile 128 x 256 (M x N), K-stage 128 bytes, 4-stage smem ring, FP32 accumulator
// in 256 tensor-memory columns.  Every wait is bounded (a deadline on the GPU
// clock); when one runs out the CTA records MOE_ERR_TIMEOUT and winds down.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

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
constexpr int SFSA_BYTES = BM * 16;                        // staged scales: 128 rows x 16 B (4 stages)
constexpr int SFSB_BYTES = BN * 16;
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_SFSA = OFF_SFB + STAGES * SFB_BYTES;
constexpr int OFF_SFSB = OFF_SFSA + SFG * SFSA_BYTES;
constexpr int OFF_BAR = OFF_SFSB + SFG * SFSB_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 3 + 2 * SFG;        // full, empty, tfull, tempty, drain, sfull, sempty
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;           // tmem base, abort flag
constexpr int OFF_MPRE = OFF_MISC + 16;                    // int32 mpre[E+1]
constexpr int TMEM_COLS = 512;
constexpr int TCOL_SFA = 256;                              // + stage*4
constexpr int TCOL_SFB = 256 + 4 * STAGES;                 // + stage*8
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (4 + EPI_WARPS) * 32;
inline size_t smem_bytes(int E) { return 1024 + OFF_MPRE + sizeof(int32_t) * (E + 1); }
}  // namespace tc

struct TcArgs {
    const int32_t* offsets;   // [E+1] row segments of A per expert
    int E;
    int K;                    // reduction length (H for GEMM1, I for GEMM2)
    int n_tiles;              // N tiles per expert
    int I;                    // GEMM1: offset of the up rows inside w_gate_up
    int a_rows;               // rows of the A tensor (scale loads stay inside)
    int b_rows;               // rows of one expert's weight matrix (2I or H)
    int sf_tma;               // MXFP8 with K % 512 == 0: scales staged by TMA
    const uint8_t* a_sf;      // MXFP8: [a_rows][K/32]
    const uint8_t* b_sf;      // MXFP8: [E][b_rows][K/32]
    uint8_t* out;             // GEMM1: h codes/BF16 [a_rows][I]; GEMM2: y BF16 [a_rows][H]
    uint8_t* out_sf;          // GEMM1 MXFP8: h scales [a_rows][I/32]
    int out_ld;               // row length of out in elements
    WsHeader* ws;
    unsigned long long timeout_ns;
};

// (expert, m-tile, n-tile) of linear tile t; tiles are expert-major, then n, then m.
struct Tile {
    int e, m, n, row0, row_end;
};

__device__ __forceinline__ Tile tile_at(int t, const int32_t* mpre, const int32_t* offsets, int E,
                                        int n_tiles) {
    const int q = t / n_tiles;
    int lo = 0, hi = E;  // last e with mpre[e] <= q (upper bound - 1)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (mpre[mid] <= q) lo = mid; else hi = mid;
    }
    Tile tl;
    tl.e = lo;
    const int mt = mpre[lo + 1] - mpre[lo];
    const int local = t - mpre[lo] * n_tiles;
    tl.n = local / mt;
    tl.m = local % mt;
    tl.row0 = offsets[lo] + tl.m * tc::BM;
    tl.row_end = min(offsets[lo + 1], tl.row0 + tc::BM);
    return tl;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int q) {
    return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

template <bool MX, bool SWIGLU>
__global__ void __launch_bounds__(tc::THREADS, 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmSFA,
                           const __grid_constant__ CUtensorMap tmSFB, TcArgs args) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tfull + 2;
    uint64_t* sfull = tfull + 3;
    uint64_t* sempty = sfull + SFG;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    int32_t* mpre = reinterpret_cast<int32_t*>(smem + OFF_MPRE);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int E = args.E;
    const int KB = args.K / (MX ? 128 : 64);   // K stages (128 bytes each)
    const bool sf_tma = MX && args.sf_tma;

    // ---------------------------------------------------------------- prologue
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], MX ? 2 : 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, EPI_WARPS);
        mbar_init(drain, 1);
        for (int g = 0; g < SFG; ++g) {
            mbar_init(&sfull[g], 1);
            mbar_init(&sempty[g], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (sf_tma) {
            prefetch_tmap(&tmSFA);
            prefetch_tmap(&tmSFB);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 3) {
        // m-tile prefix over experts: mpre[e+1] = mpre[e] + ceil(count_e / BM)
        const int per = (E + 31) / 32;
        const int lo = min(lane * per, E), hi = min(lo + per, E);
        int s = 0;
        for (int e = lo; e < hi; ++e) s += (args.offsets[e + 1] - args.offsets[e] + BM - 1) / BM;
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - s;
        for (int e = lo; e < hi; ++e) {
            mpre[e] = run;
            run += (args.offsets[e + 1] - args.offsets[e] + BM - 1) / BM;
        }
        if (lane == 31) mpre[E] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total_tiles = mpre[E] * args.n_tiles;
    const unsigned long long deadline = globaltimer_ns() + args.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0, g = 0;
            uint32_t phase = 0, gphase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const Tile tl = tile_at(t, mpre, args.offsets, E, args.n_tiles);
                const int brow0 = SWIGLU ? tl.n * 128 : tl.n * BN;
                const int brow1 = SWIGLU ? args.I + tl.n * 128 : tl.n * BN + 128;
                for (int kb = 0; kb < KB; ++kb) {
                    if (sf_tma && (kb & 3) == 0) {
                        if (!mbar_wait_bounded(&sempty[g], gphase ^ 1, abort_flag, args.ws, deadline)) {
                            ok = false;
                            break;
                        }
                        uint8_t* sa = smem + OFF_SFSA + g * SFSA_BYTES;
                        uint8_t* sb = smem + OFF_SFSB + g * SFSB_BYTES;
                        mbar_arrive_expect_tx(&sfull[g], SFSA_BYTES + SFSB_BYTES);
                        tma_load_2d(sa, &tmSFA, &sfull[g], kb * 4, tl.row0);
                        tma_load_3d(sb, &tmSFB, &sfull[g], kb * 4, brow0, tl.e);
                        tma_load_3d(sb + SFSB_BYTES / 2, &tmSFB, &sfull[g], kb * 4, brow1, tl.e);
                        if (++g == SFG) {
                            g = 0;
                            gphase ^= 1;
                        }
                    }
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.ws, deadline)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + OFF_A + stage * A_BYTES;
                    uint8_t* sb = smem + OFF_B + stage * B_BYTES;
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
                    const int kx = kb * (MX ? 128 : 64);
                    tma_load_2d(sa, &tmA, &full[stage], kx, tl.row0);
                    if (SWIGLU) {
                        tma_load_3d(sb, &tmB, &full[stage], kx, brow0, tl.e);
                        tma_load_3d(sb + B_BYTES / 2, &tmB, &full[stage], kx, brow1, tl.e);
                    } else {
                        tma_load_3d(sb, &tmB, &full[stage], kx, brow0, tl.e);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t d_tmem = tmem_base;
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                if (!mbar_wait_bounded(tempty, acc_phase ^ 1, abort_flag, args.ws, deadline)) break;
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.ws, deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + OFF_A + stage * A_BYTES);
                    const uint32_t sb = smem_u32(smem + OFF_B + stage * B_BYTES);
                    if constexpr (MX) {
                        const uint32_t sfa_t = tmem_base + TCOL_SFA + stage * 4;
                        const uint32_t sfb_t = tmem_base + TCOL_SFB + stage * 8;
                        tmem_cp_32x128b_x4(sfa_t, sdesc_sf_block(smem_u32(smem + OFF_SFA + stage * SFA_BYTES)));
                        tmem_cp_32x128b_x4(sfb_t, sdesc_sf_block(smem_u32(smem + OFF_SFB + stage * SFB_BYTES)));
                        tmem_cp_32x128b_x4(sfb_t + 4, sdesc_sf_block(smem_u32(smem + OFF_SFB + stage * SFB_BYTES + 512)));
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
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) mma_commit(tfull);
                acc_phase ^= 1;
            }
            // wait until every tensor-core operation issued here has finished
            mma_commit(drain);
            const unsigned long long d2 = globaltimer_ns() + 1000000ull;
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() < d2) {
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------ scale factors (MXFP8 only)
        // Each K-stage needs, for the A rows and for both 128-row halves of B, a
        // [32 lanes][4 words] block: word j of lane r holds the four K-step scales of
        // row 32j + r.  tcgen05.cp moves that block into tensor memory.
        if constexpr (MX) {
            int stage = 0, g = 0;
            uint32_t phase = 0, gphase = 0;
            bool ok = true;
            const int ksf = args.K / 32;                // scale bytes per row
            for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
                const Tile tl = tile_at(t, mpre, args.offsets, E, args.n_tiles);
                if (sf_tma) {
                    for (int kb = 0; kb < KB; ++kb) {
                        if ((kb & 3) == 0 &&
                            !mbar_wait_bounded(&sfull[g], gphase, abort_flag, args.ws, deadline)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.ws, deadline)) {
                            ok = false;
                            break;
                        }
                        const int q = kb & 3;
                        const uint8_t* sa = smem + OFF_SFSA + g * SFSA_BYTES + 4 * q;
                        const uint8_t* sb = smem + OFF_SFSB + g * SFSB_BYTES + 4 * q;
                        uint32_t a[4], b[8];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            a[j] = *reinterpret_cast<const uint32_t*>(sa + (32 * j + lane) * 16);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            b[i] = *reinterpret_cast<const uint32_t*>(sb + (32 * i + lane) * 16);
                        uint4* sfa = reinterpret_cast<uint4*>(smem + OFF_SFA + stage * SFA_BYTES);
                        uint4* sfb = reinterpret_cast<uint4*>(smem + OFF_SFB + stage * SFB_BYTES);
                        sfa[lane] = make_uint4(a[0], a[1], a[2], a[3]);
                        sfb[lane] = make_uint4(b[0], b[1], b[2], b[3]);
                        sfb[32 + lane] = make_uint4(b[4], b[5], b[6], b[7]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&full[stage]);
                            if (q == 3) mbar_arrive(&sempty[g]);
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
                    // scales whose rows are not 16-byte multiples: direct loads
                    const uint8_t* bsf = args.b_sf + (int64_t)tl.e * args.b_rows * ksf;
                    int brow[8];
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            brow[c * 4 + j] = SWIGLU ? (c * args.I + tl.n * 128 + 32 * j + lane)
                                                     : (tl.n * BN + c * 128 + 32 * j + lane);
                    for (int kb4 = 0; ok && kb4 < KB; kb4 += 4) {
                        uint4 va[4], vb[8];
                        const int nq = min(4, KB - kb4);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int row = tl.row0 + 32 * j + lane;
                            uint32_t w[4] = {0, 0, 0, 0};
                            for (int q = 0; q < nq; ++q)
                                if (row < args.a_rows)
                                    w[q] = *reinterpret_cast<const uint32_t*>(args.a_sf + (int64_t)row * ksf + (kb4 + q) * 4);
                            va[j] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            uint32_t w[4] = {0, 0, 0, 0};
                            for (int q = 0; q < nq; ++q)
                                w[q] = *reinterpret_cast<const uint32_t*>(bsf + (int64_t)brow[i] * ksf + (kb4 + q) * 4);
                            vb[i] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        for (int q = 0; q < nq; ++q) {
                            if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.ws, deadline)) {
                                ok = false;
                                break;
                            }
                            uint4* sfa = reinterpret_cast<uint4*>(smem + OFF_SFA + stage * SFA_BYTES);
                            uint4* sfb = reinterpret_cast<uint4*>(smem + OFF_SFB + stage * SFB_BYTES);
                            sfa[lane] = make_uint4(word_of(va[0], q), word_of(va[1], q), word_of(va[2], q), word_of(va[3], q));
                            sfb[lane] = make_uint4(word_of(vb[0], q), word_of(vb[1], q), word_of(vb[2], q), word_of(vb[3], q));
                            sfb[32 + lane] = make_uint4(word_of(vb[4], q), word_of(vb[5], q), word_of(vb[6], q), word_of(vb[7], q));
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&full[stage]);
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1;
                            }
                        }
                    }
                }
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------------ epilogue
        // Two warps per tensor-memory lane quarter, each taking half of the tile's
        // columns.  A warp first moves its whole share of the accumulator into
        // registers (converted), releases the accumulator to the MMA issuer, and
        // only then writes to global memory, so the next tile's MMAs overlap it.
        const int q = warp & 3;
        const int half = (warp - 4) >> 2;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const Tile tl = tile_at(t, mpre, args.offsets, E, args.n_tiles);
            if (!mbar_wait_bounded(tfull, acc_phase, abort_flag, args.ws, deadline)) break;
            tc_fence_after();
            const int row = tl.row0 + 32 * q + lane;
            const bool valid = row < tl.row_end;
            const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
            if constexpr (SWIGLU) {
                uint32_t pk[2][16];
                uint8_t sc[2];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int c = half * 2 + c2;
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(tq + 32 * c, g);
                    tmem_ld_32x32b_x32(tq + 128 + 32 * c, u);
                    tmem_ld_wait();
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        hv[i] = silu_f32(__uint_as_float(g[i])) * __uint_as_float(u[i]);
                    if constexpr (MX) {
                        sc[c2] = mx_quantize32(hv, pk[c2]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[c2][i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
                if (valid) {
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int col = tl.n * 128 + 32 * (half * 2 + c2);
                        if constexpr (MX) {
                            uint8_t* dst = args.out + (int64_t)row * args.out_ld + col;
                            st_v4(dst, make_uint4(pk[c2][0], pk[c2][1], pk[c2][2], pk[c2][3]));
                            st_v4(dst + 16, make_uint4(pk[c2][4], pk[c2][5], pk[c2][6], pk[c2][7]));
                            args.out_sf[(int64_t)row * (args.out_ld / 32) + col / 32] = sc[c2];
                        } else {
                            uint8_t* dst = args.out + ((int64_t)row * args.out_ld + col) * 2;
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                st_v4(dst + 16 * p, make_uint4(pk[c2][4 * p], pk[c2][4 * p + 1],
                                                               pk[c2][4 * p + 2], pk[c2][4 * p + 3]));
                        }
                    }
                }
            } else {
                uint32_t pk[4][16];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tq + 32 * (half * 4 + c4), v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[c4][i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
                if (valid) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint8_t* dst = args.out +
                                       ((int64_t)row * args.out_ld + tl.n * BN + 32 * (half * 4 + c4)) * 2;
#pragma unroll
                        for (int p = 0; p < 4; ++p)
                            st_v4(dst + 16 * p, make_uint4(pk[c4][4 * p], pk[c4][4 * p + 1],
                                                           pk[c4][4 * p + 2], pk[c4][4 * p + 3]));
                    }
                }
            }
            acc_phase ^= 1;
        }
    }

    // ---------------------------------------------------------------- teardown
    if (*abort_flag) {
        // let any copy still in flight land before the CTA's memory is released
        const unsigned long long d2 = globaltimer_ns() + 1000000ull;
        while (globaltimer_ns() < d2) {
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------ host side
template <bool MX, bool SWIGLU>
static cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                              const CUtensorMap& tsb, const TcArgs& args, int grid,
                              cudaStream_t stream) {
    auto kern = tc_grouped_gemm_kernel<MX, SWIGLU>;
    const size_t smem = tc::smem_bytes(args.E);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, tc::THREADS, smem, stream>>>(ta, tb, tsa, tsb, args);
    return cudaGetLastError();
}

// Scale tensors as 16-byte-wide TMA boxes of 128 rows (four K-stages of scales).
static bool encode_sf_maps(CUtensorMap* tsa, CUtensorMap* tsb, const void* a_sf, int a_rows,
                           const void* b_sf, int b_rows, int E, int K) {
    const uint64_t ksf = (uint64_t)K / 32;
    uint64_t da[2] = {ksf, (uint64_t)a_rows};
    uint64_t sa[1] = {ksf};
    uint32_t ba[2] = {16, 128};
    if (!encode_tmap(tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a_sf, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    uint64_t db[3] = {ksf, (uint64_t)b_rows, (uint64_t)E};
    uint64_t sb[2] = {ksf, (uint64_t)b_rows * ksf};
    uint32_t bb[3] = {16, 128, 1};
    return encode_tmap(tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, b_sf, db, sb, bb, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// a: [a_rows][K] (codes or BF16); weights as documented in moe.h.
cudaError_t launch_expert_ffn_tc(const TcFfnCall& c, cudaStream_t stream) {
    const bool mx = c.mx;
    const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t esz = mx ? 1 : 2;
    const uint32_t bk = mx ? 128 : 64;
    if (c.T == 0) return cudaSuccess;
    // GEMM1: A = a [T][H], B = w_gate_up [E][2I][H] (two 128-row boxes per stage)
    CUtensorMap ta1, tb1, ta2, tb2;
    {
        uint64_t dims[2] = {(uint64_t)c.H, (uint64_t)c.a_rows};
        uint64_t str[1] = {(uint64_t)c.H * esz};
        uint32_t box[2] = {bk, 128};
        if (!encode_tmap(&ta1, dt, 2, c.a, dims, str, box)) return cudaErrorInvalidValue;
        uint64_t dimsb[3] = {(uint64_t)c.H, (uint64_t)2 * c.I, (uint64_t)c.E};
        uint64_t strb[2] = {(uint64_t)c.H * esz, (uint64_t)2 * c.I * c.H * esz};
        uint32_t boxb[3] = {bk, 128, 1};
        if (!encode_tmap(&tb1, dt, 3, c.w_gate_up, dimsb, strb, boxb)) return cudaErrorInvalidValue;
    }
    // GEMM2: A = h [T][I], B = w_down [E][H][I] (one 256-row box per stage)
    {
        uint64_t dims[2] = {(uint64_t)c.I, (uint64_t)c.a_rows};
        uint64_t str[1] = {(uint64_t)c.I * esz};
        uint32_t box[2] = {bk, 128};
        if (!encode_tmap(&ta2, dt, 2, c.h, dims, str, box)) return cudaErrorInvalidValue;
        uint64_t dimsb[3] = {(uint64_t)c.I, (uint64_t)c.H, (uint64_t)c.E};
        uint64_t strb[2] = {(uint64_t)c.I * esz, (uint64_t)c.H * c.I * esz};
        uint32_t boxb[3] = {bk, 256, 1};
        if (!encode_tmap(&tb2, dt, 3, c.w_down, dimsb, strb, boxb)) return cudaErrorInvalidValue;
    }
    TcArgs a1{};
    a1.offsets = c.offsets;
    a1.E = c.E;
    a1.K = c.H;
    a1.n_tiles = c.I / 128;
    a1.I = c.I;
    a1.a_rows = c.a_rows;
    a1.b_rows = 2 * c.I;
    a1.a_sf = (const uint8_t*)c.a_sf;
    a1.b_sf = (const uint8_t*)c.w_gu_sf;
    a1.out = (uint8_t*)c.h;
    a1.out_sf = (uint8_t*)c.h_sf;
    a1.out_ld = c.I;
    a1.ws = c.ws;
    a1.timeout_ns = c.timeout_ns;
    TcArgs a2 = a1;
    a2.K = c.I;
    a2.n_tiles = c.H / tc::BN;
    a2.b_rows = c.H;
    a2.a_sf = (const uint8_t*)c.h_sf;
    a2.b_sf = (const uint8_t*)c.w_d_sf;
    a2.out = (uint8_t*)c.y;
    a2.out_sf = nullptr;
    a2.out_ld = c.H;
    CUtensorMap ts1a{}, ts1b{}, ts2a{}, ts2b{};
    if (mx) {
        a1.sf_tma = (c.H % 512) == 0;
        a2.sf_tma = (c.I % 512) == 0;
        if (a1.sf_tma && !encode_sf_maps(&ts1a, &ts1b, c.a_sf, c.a_rows, c.w_gu_sf, 2 * c.I, c.E, c.H))
            return cudaErrorInvalidValue;
        if (a2.sf_tma && !encode_sf_maps(&ts2a, &ts2b, c.h_sf, c.a_rows, c.w_d_sf, c.H, c.E, c.I))
            return cudaErrorInvalidValue;
    }
    cudaError_t err;
    if (mx) {
        err = launch_one<true, true>(ta1, tb1, ts1a, ts1b, a1, c.grid, stream);
        if (err != cudaSuccess) return err;
        err = launch_one<true, false>(ta2, tb2, ts2a, ts2b, a2, c.grid, stream);
    } else {
        err = launch_one<false, true>(ta1, tb1, ts1a, ts1b, a1, c.grid, stream);
        if (err != cudaSuccess) return err;
        err = launch_one<false, false>(ta2, tb2, ts2a, ts2b, a2, c.grid, stream);
    }
    return err;
}

}  // namespace moe
