// wgrad.cu -- the expert weight gradients of the backward pass: grouped GEMMs
// whose reduction runs over each expert's slots, on the sm_103a tensor cores.
//
// For expert e with slots [offsets[e], offsets[e+1]):
//   dW_gate_up[e] = [du dv]^T . a      ([2I x H]; a = the master x rows)
//   dW_down[e]    = dy^T . h           ([H x I]; h = silu(u) v from the kept u|v)
// written as BF16 master gradients (zeros for an expert without slots).
// ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72", section 01: the backward's expert computation on Blackwell tensor
// cores, grouped per expert like the forward's.)
//
// Operands.  A tcgen05 operand is K-major, so the slot-major rows (du|dv, x,
// g*dout, u|v) are first transposed by `wgrad_pack_kernel` into tile images:
// per operand matrix of R rows (R padded to 256) and the padded slot axis (each
// expert's slots padded to a multiple of 128, expert e starting at 128 *
// pstage[e]), image (kb, rb) = rows 128 rb .. +127 x one K-stage (128 MXFP8 or
// 64 BF16 slots) as the 16 KB shared-memory image the MMA reads (128-byte rows,
// 16-byte chunk q of row r at chunk q ^ (r % 8)), stored [kb][rb].  MXFP8
// quantises along the slots (blocks of 32 from the expert's first slot) and packs
// the scales as the 512-byte [32 lanes][4 words] image tcgen05.cp moves to tensor
// memory.  A B tile (256 rows) is two adjacent images: one bulk copy.
//
// GEMM.  One persistent CTA of 12 warps per SM over tiles (expert, GEMM, n, m):
//   warp 0   producer: bulk copies of the A and B images (and scale images) into
//            a 3-stage ring
//   warp 1   TMEM owner + MMA issuer; the last K-stage of an expert issues only
//            the 32-slot (MXFP8) or 16-slot (BF16) steps that hold slots
//   warps 2-3 zero the gradients of the experts without slots with streaming
//            vector stores, alongside the MMA-bound tiles (warp 3 first lists
//            the experts with and without slots)
//   warps 4-11 epilogue: accumulator -> BF16 -> a 64 KB staging tile in shared
//            memory -> TMA tensor stores into dW; the stores run asynchronously
//            while the next tile computes
// Every wait is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT and stops.
#include "common.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace moe {

namespace wg {
constexpr int STAGES = 3;
constexpr int IMG = 16384;                     // one 128-row x 128-byte image
constexpr int A_BYTES = IMG, B_BYTES = 2 * IMG;
constexpr int SFA_BYTES = 512, SFB_BYTES = 1024;
constexpr int C_BYTES = 128 * 256 * 2;         // output tile staging (BF16)
constexpr int BOX = 32 * 128;                  // one TMA store box: 32 rows x 64 BF16
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_C = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SFA = OFF_C + C_BYTES;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 3;       // full, empty, tfull, tempty, drain
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_LIST = OFF_MISC + 16;        // experts with / without slots (2 x 1024 ints)
constexpr int MAX_E = 1024;
constexpr int OFF_PROG = OFF_LIST + 2 * MAX_E * 4;   // K-stages whose tiles are stored
constexpr int SMEM = OFF_PROG + 16;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (4 + EPI_WARPS) * 32;
constexpr int TMEM_COLS = 512;
constexpr int TCOL_SFA = 256;
constexpr int TCOL_SFB = 256 + 4 * STAGES;
}  // namespace wg

// ------------------------------------------------------------- slot padding
// pstage[e] = sum over e' < e of ceil(count_e' / 128): expert e's first padded
// slot is 128 * pstage[e]; pstage[E] covers all experts.  blk_e[b] = the expert
// of 32-slot block b of the padded slot axis.  One warp.
__global__ void wgrad_pstage_kernel(const int32_t* __restrict__ offsets, int E, int32_t* __restrict__ pstage,
                                    int32_t* __restrict__ blk_e) {
    const int lane = threadIdx.x % 32;
    const int per = (E + 31) / 32;
    const int lo = min(lane * per, E), hi = min(lo + per, E);
    int s = 0;
    for (int e = lo; e < hi; ++e) s += (offsets[e + 1] - offsets[e] + 127) / 128;
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - s;
    for (int e = lo; e < hi; ++e) {
        pstage[e] = run;
        const int n = (offsets[e + 1] - offsets[e] + 127) / 128;
        for (int b = 4 * run; b < 4 * (run + n); ++b) blk_e[b] = e;
        run += n;
    }
    if (lane == 31) pstage[E] = incl;
}

// ------------------------------------------------------------- operand packing
enum { WG_DUV = 0, WG_X = 1, WG_DY = 2, WG_H = 3 };

__device__ __forceinline__ void unpack_bf16x8_w(const uint4& q, float* f) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        f[2 * p] = bf16_to_f32((uint16_t)(w[p] & 0xFFFF));
        f[2 * p + 1] = bf16_to_f32((uint16_t)(w[p] >> 16));
    }
}

struct WgPackArgs {
    const uint16_t* src;      // DUV: du|dv [T][2I]; X: x [N][H]; DY: dout [N][H]; H: u|v [T][2I]
    const int32_t* sched;     // [T][2] (X, DY)
    const float* slot_gate;   // [T] (DY)
    const int32_t* offsets;   // [E+1]
    const int32_t* pstage;    // [E+1]
    const int32_t* blk_e;     // [padded slots / 32]
    int E, C, Cp, ld, I, rows_per_shard, N;
    uint8_t* img;             // [Tp/KS][RB][16 KB]
    uint8_t* sf;              // MXFP8: [Tp/128][RB][512]
    int RB;                   // row blocks of 128 (R padded to 256)
};

// CTA = (32-slot block of the padded slot axis, 512 operand rows).  Phase 1: the
// 32 slot rows' 512 values are read as contiguous 16-byte vectors into shared
// memory (zeros past the expert's slots or past C).  Phase 2: thread t takes
// operand rows c0 + t and c0 + 256 + t and quantises / rounds their 32 slots into
// the images.
constexpr int kPackCols = 512;
constexpr int kPackPitch = kPackCols + 4;       // floats per shared row (16-byte stores spread)
constexpr int kPackPitch16 = kPackCols + 8;     // BF16 elements per shared row

template <int SRC, bool MX>
__global__ void __launch_bounds__(256) wgrad_pack_kernel(const __grid_constant__ WgPackArgs a, WsHeader* ws) {
    // BF16 sources (du|dv, x, dY) are staged as their raw BF16 bits, which is exact
    // and halves the shared memory (more CTAs per SM); g*dY takes its slot's gate
    // when it is quantised (the same FP32 product), and h, computed from u|v, is
    // staged as FP32.
    constexpr bool RAW = SRC == WG_DUV || SRC == WG_X || SRC == WG_DY;
    extern __shared__ uint4 smem_pack[];
    __shared__ float sgate[32];
    float* tile = reinterpret_cast<float*>(smem_pack);        // [32][kPackPitch] FP32
    uint16_t* tile16 = reinterpret_cast<uint16_t*>(smem_pack); // [32][kPackPitch16] BF16
    const int P0 = blockIdx.x * 32;
    if (P0 >= a.pstage[a.E] * 128) return;
    const int e = a.blk_e[blockIdx.x];
    const int local0 = P0 - a.pstage[e] * 128;
    const int cnt = a.offsets[e + 1] - a.offsets[e];
    const int s0 = a.offsets[e] + local0;
    const int c0 = blockIdx.y * kPackCols;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // Each warp takes slot rows warp, warp+8, warp+16, warp+24: their indices
    // first, then all their row loads, so the dependent chain (schedule entry,
    // token, row) is waited on once per warp, not once per row.
    bool live[4];
    int64_t src_row[4];
    float gs[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = warp + 8 * j;
        const int64_t sl = s0 + i;
        live[j] = local0 + i < cnt;
        src_row[j] = sl;
        gs[j] = 1.0f;
        if constexpr (SRC == WG_X || SRC == WG_DY) {
            if (live[j]) {
                const int64_t tok = (int64_t)a.sched[2 * sl] * a.rows_per_shard + a.sched[2 * sl + 1];
                if (SRC == WG_DY) gs[j] = a.slot_gate[sl];
                if (tok < 0 || tok >= a.N) {
                    if (lane == 0) set_status(ws, MOE_ERR_DEVICE_CHECK);
                    live[j] = false;
                }
                src_row[j] = tok;
            }
        }
    }
    constexpr int NV = SRC == WG_H ? 2 : 1;     // vectors per column group (u and v for h)
    uint4 raw[4][2][NV];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
            const int col = c0 + hv * 256 + lane * 8;
            const bool ok = live[j] && col < a.C;
#pragma unroll
            for (int t = 0; t < NV; ++t)
                raw[j][hv][t] = ok ? ld_nc_v4(a.src + src_row[j] * a.ld + (t ? a.I : 0) + col)
                                   : make_uint4(0, 0, 0, 0);
        }
    if constexpr (SRC == WG_DY) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (lane == 0) sgate[warp + 8 * j] = gs[j];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
            if constexpr (RAW) {
                *reinterpret_cast<uint4*>(tile16 + (warp + 8 * j) * kPackPitch16 + hv * 256 + lane * 8) =
                    raw[j][hv][0];
                continue;
            }
            float v[8];
            unpack_bf16x8_w(raw[j][hv][0], v);
            if constexpr (SRC == WG_H) {   // h = silu(u) * v from the kept u|v
                float w2[8];
                unpack_bf16x8_w(raw[j][hv][1], w2);
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = silu_f32(v[q]) * w2[q];
            }
            float4* dst = reinterpret_cast<float4*>(tile + (warp + 8 * j) * kPackPitch + hv * 256 + lane * 8);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    __syncthreads();
#pragma unroll 1
    for (int hv = 0; hv < 2; ++hv) {
        const int c = c0 + hv * 256 + threadIdx.x;
        if (c >= a.Cp) break;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] = RAW ? bf16_to_f32(tile16[i * kPackPitch16 + hv * 256 + threadIdx.x])
                       : tile[i * kPackPitch + hv * 256 + threadIdx.x];
            if constexpr (SRC == WG_DY) v[i] = sgate[i] * v[i];
        }
        const int rb = c / 128, r = c % 128;
        if constexpr (MX) {
            uint32_t codes[8];
            const uint8_t sc = mx_quantize32(v, codes);
            const int kb = P0 / 128, sub = (P0 % 128) / 32;
            uint8_t* row = a.img + ((int64_t)kb * a.RB + rb) * wg::IMG + r * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int q = sub * 2 + h;
                st_v4(row + ((q ^ (r & 7)) * 16),
                      make_uint4(codes[4 * h], codes[4 * h + 1], codes[4 * h + 2], codes[4 * h + 3]));
            }
            a.sf[((int64_t)kb * a.RB + rb) * 512 + ((r % 32) * 4 + r / 32) * 4 + sub] = sc;
        } else {
            uint32_t pk[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) pk[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
            const int kb = P0 / 64, sub = (P0 % 64) / 32;
            uint8_t* row = a.img + ((int64_t)kb * a.RB + rb) * wg::IMG + r * 128;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int q = sub * 4 + h;
                st_v4(row + ((q ^ (r & 7)) * 16), make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]));
            }
        }
    }
}

// ------------------------------------------------------------------ the GEMMs
struct WgTile {
    int e, g, m, n;           // expert, GEMM (0: dW_gate_up, 1: dW_down), M tile, N tile
    int KB;                   // K-stages holding slots (0: the expert has none)
    int last_steps;           // MMA K-steps in the last stage
    int kbase;                // first K-stage of the expert in the images
};

// The tile order of one CTA: the tiles of the experts with slots, expert-major
// then N tile then M tile, dealt round-robin over the CTAs, so CTAs at the same
// step work on the same expert and share its operands through L2.  Experts
// without slots get no tiles (their gradients are zero-filled separately).
struct WgSchedule {
    const int32_t* work;      // experts with slots, in order (shared memory)
    int per, n;               // tiles per expert; this CTA's tile count

    __device__ void init(const int32_t* w_list, int nw, int per_) {
        work = w_list;
        per = per_;
        const int G = gridDim.x, c = blockIdx.x;
        const long long W = (long long)nw * per;
        n = W > c ? (int)((W - c - 1) / G + 1) : 0;
    }
    // (expert, tile within the expert) of step s of this CTA
    __device__ void at(int s, int& e, int& l) const {
        const long long t = blockIdx.x + (long long)s * gridDim.x;
        e = work[t / per];
        l = (int)(t % per);
    }
};

template <bool MX>
__device__ __forceinline__ WgTile wg_tile(const WgSchedule& sc, int s, const WgGemm& g0, const WgGemm& g1,
                                          const int32_t* offsets, const int32_t* pstage) {
    constexpr int KS = MX ? 128 : 64, KSTEP = MX ? 32 : 16;
    const int t0 = g0.m_tiles * g0.n_tiles;
    WgTile w;
    int l;
    sc.at(s, w.e, l);
    w.g = l >= t0;
    if (w.g) l -= t0;
    const int mt = w.g ? g1.m_tiles : g0.m_tiles;
    w.n = l / mt;
    w.m = l % mt;
    const int cnt = offsets[w.e + 1] - offsets[w.e];
    w.KB = (cnt + KS - 1) / KS;
    w.kbase = pstage[w.e] * (128 / KS);
    w.last_steps = w.KB > 0 ? (cnt - (w.KB - 1) * KS + KSTEP - 1) / KSTEP : 0;
    return w;
}

template <bool MX>
__global__ void __launch_bounds__(wg::THREADS, 1)
    wgrad_gemm_kernel(const __grid_constant__ WgGemm g0, const __grid_constant__ WgGemm g1,
                      const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                      const int32_t* __restrict__ offsets, const int32_t* __restrict__ pstage, int E,
                      WsHeader* ws, unsigned long long timeout_ns) {
    using namespace wg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tfull + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    int32_t* w_list = reinterpret_cast<int32_t*>(smem + OFF_LIST);
    int32_t* z_list = w_list + MAX_E;
    int32_t* n_lists = reinterpret_cast<int32_t*>(smem + OFF_MISC + 8);
    volatile int* progress = reinterpret_cast<volatile int*>(smem + OFF_PROG);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, EPI_WARPS);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *progress = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(reinterpret_cast<uint32_t*>(smem + OFF_MISC), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 3) {   // the two expert lists, in expert order
        int nw = 0, nz = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const bool has = e < E && offsets[e + 1] > offsets[e];
            const bool none = e < E && !has;
            const unsigned bw = __ballot_sync(0xffffffffu, has), bz = __ballot_sync(0xffffffffu, none);
            const unsigned below = (1u << lane) - 1u;
            if (has) w_list[nw + __popc(bw & below)] = e;
            if (none) z_list[nz + __popc(bz & below)] = e;
            nw += __popc(bw);
            nz += __popc(bz);
        }
        if (lane == 0) {
            n_lists[0] = nw;
            n_lists[1] = nz;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    const unsigned long long deadline = globaltimer_ns() + timeout_ns;
    WgSchedule sc;
    sc.init(w_list, n_lists[0], g0.m_tiles * g0.n_tiles + g1.m_tiles * g1.n_tiles);

    if (warp == 0) {
        if (lane == 0) {   // producer
            int stage = 0;
            uint32_t phase = 0;
            for (int s = 0; s < sc.n; ++s) {
                const WgTile w = wg_tile<MX>(sc, s, g0, g1, offsets, pstage);
                const WgGemm& G = w.g ? g1 : g0;
                bool ok = true;
                for (int kb = 0; kb < w.KB; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, ws, deadline)) {
                        ok = false;
                        break;
                    }
                    const int64_t gk = w.kbase + kb;
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES + (MX ? SFA_BYTES + SFB_BYTES : 0));
                    bulk_load(smem + OFF_A + stage * A_BYTES, G.a_img + (gk * G.a_rb + w.m) * IMG, A_BYTES,
                              &full[stage]);
                    bulk_load(smem + OFF_B + stage * B_BYTES, G.b_img + (gk * G.b_rb + 2 * w.n) * IMG, B_BYTES,
                              &full[stage]);
                    if (MX) {
                        bulk_load(smem + OFF_SFA + stage * SFA_BYTES, G.a_sf + (gk * G.a_rb + w.m) * 512,
                                  SFA_BYTES, &full[stage]);
                        bulk_load(smem + OFF_SFB + stage * SFB_BYTES, G.b_sf + (gk * G.b_rb + 2 * w.n) * 512,
                                  SFB_BYTES, &full[stage]);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int s = 0; ok && s < sc.n; ++s) {
                const WgTile w = wg_tile<MX>(sc, s, g0, g1, offsets, pstage);
                if (!mbar_wait_bounded(tempty, acc_phase ^ 1, abort_flag, ws, deadline)) break;
                tc_fence_after();
                for (int kb = 0; kb < w.KB; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, ws, deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int steps = kb == w.KB - 1 ? w.last_steps : 4;
                    const uint32_t sa = smem_u32(smem + OFF_A + stage * A_BYTES);
                    const uint32_t sb = smem_u32(smem + OFF_B + stage * B_BYTES);
                    if constexpr (MX) {
                        const uint32_t sfa_t = tmem_base + TCOL_SFA + stage * 4;
                        const uint32_t sfb_t = tmem_base + TCOL_SFB + stage * 8;
                        tmem_cp_32x128b_x4(sfa_t, sdesc_sf_block(smem_u32(smem + OFF_SFA + stage * SFA_BYTES)));
                        tmem_cp_32x128b_x4(sfb_t, sdesc_sf_block(smem_u32(smem + OFF_SFB + stage * SFB_BYTES)));
                        tmem_cp_32x128b_x4(sfb_t + 4,
                                           sdesc_sf_block(smem_u32(smem + OFF_SFB + stage * SFB_BYTES + 512)));
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (k < steps)
                                mma_mxf8(tmem_base, sdesc_kmajor_sw128(sa + 32 * k), sdesc_kmajor_sw128(sb + 32 * k),
                                         idesc_mxf8(128, 256, k, k), sfa_t, sfb_t, (kb | k) != 0);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (k < steps)
                                mma_bf16(tmem_base, sdesc_kmajor_sw128(sa + 32 * k), sdesc_kmajor_sw128(sb + 32 * k),
                                         idesc_bf16(128, 256), (kb | k) != 0);
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
            mma_commit(drain);
            const unsigned long long d2 = globaltimer_ns() + 1000000ull;
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() < d2) {
            }
        }
    } else if (warp == 2 || warp == 3) {
        // Zero fill: dW_gate_up[e] and dW_down[e] of an expert without slots are
        // contiguous byte ranges (out_estride bytes each, a multiple of 16).  They
        // are cut into 64 KB chunks dealt over (CTA, warp); a warp's 32 lanes write
        // 512 contiguous bytes per store.  Streaming stores keep the zeros from
        // evicting the working tiles' operands from L2.  The stores are paced by
        // the CTA's own MMA work (K-stages of tiles already stored): written in one
        // burst they saturate HBM with writes and stall the operand loads of the
        // tiles, which then run after them instead of beside them.
        constexpr int64_t CH = 65536;
        const int64_t b0 = g0.out_estride, b1 = g1.out_estride;
        const int64_t c0 = (b0 + CH - 1) / CH, c1 = (b1 + CH - 1) / CH;
        const int64_t total = (int64_t)n_lists[1] * (c0 + c1);
        const int64_t first = 2 * (int64_t)blockIdx.x + (warp - 2), stride = 2 * (int64_t)gridDim.x;
        const int64_t mine = total > first ? (total - first - 1) / stride + 1 : 0;
        int64_t work = 0;
        if (mine > 0)
            for (int s = 0; s < sc.n; ++s) work += wg_tile<MX>(sc, s, g0, g1, offsets, pstage).KB;
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
        int64_t i = 0;
        for (int64_t t = first; t < total; t += stride, ++i) {
            // chunk i waits until i <= mine * (progress + 2 stages of lead) / work
            uint32_t n = 0;
            while (work > 0 && i * work > mine * ((int64_t)*progress + 2) && !*abort_flag) {
                __nanosleep(1000);
                if ((++n & 63u) == 0 && globaltimer_ns() > deadline) {
                    *abort_flag = 1;
                    set_status(ws, MOE_ERR_TIMEOUT);
                }
            }
            if (*abort_flag) break;
            const int e = z_list[t / (c0 + c1)];
            int64_t r = t % (c0 + c1);
            const bool second = r >= c0;
            if (second) r -= c0;
            const int64_t bytes = second ? b1 : b0;
            uint8_t* dst = (second ? g1.out : g0.out) + (int64_t)e * bytes + r * CH;
            const int64_t len = bytes - r * CH < CH ? bytes - r * CH : CH;
            for (int64_t off = (int64_t)lane * 16; off < len; off += 512)
                __stcs(reinterpret_cast<uint4*>(dst + off), zero4);
        }
    } else if (warp >= 4) {   // epilogue
        // Warp (q, half) owns rows 32q..32q+31 and columns 128 half..+127 of the
        // tile: two TMA store boxes of 32 rows x 64 BF16 (128-byte swizzle) in
        // shared memory, written from registers, then stored by lane 0.
        const int q = warp & 3;
        const int half = (warp - 4) >> 2;
        uint8_t* box0 = smem + OFF_C + (q * 2 + half) * 2 * BOX;
        uint32_t acc_phase = 0;
        for (int s = 0; s < sc.n; ++s) {
            const WgTile w = wg_tile<MX>(sc, s, g0, g1, offsets, pstage);
            uint32_t v[4][32];
            if (!mbar_wait_bounded(tfull, acc_phase, abort_flag, ws, deadline)) break;
            tc_fence_after();
            const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_ld_32x32b_x32(tq + 32 * (half * 4 + c4), v[c4]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
            acc_phase ^= 1;
            if (lane == 0) bulk_wait_group_read<0>();   // the previous tile's stores have left the boxes
            __syncwarp();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint8_t* rowp = box0 + (c4 >> 1) * BOX + lane * 128;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int qc = (c4 & 1) * 4 + h;   // 16-byte chunk of the 128-byte box row
                    const uint32_t* f = v[c4] + 8 * h;
                    *reinterpret_cast<uint4*>(rowp + ((qc ^ (lane & 7)) * 16)) =
                        make_uint4(pack_bf16x2(__uint_as_float(f[0]), __uint_as_float(f[1])),
                                   pack_bf16x2(__uint_as_float(f[2]), __uint_as_float(f[3])),
                                   pack_bf16x2(__uint_as_float(f[4]), __uint_as_float(f[5])),
                                   pack_bf16x2(__uint_as_float(f[6]), __uint_as_float(f[7])));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const CUtensorMap* tm = w.g ? &tm1 : &tm0;
                const int M = w.g ? g1.m_tiles * 128 : g0.m_tiles * 128;
                const int y = w.e * M + w.m * 128 + 32 * q;
                const int x = w.n * 256 + half * 128;
                const int nv = w.g ? g1.n_valid : g0.n_valid;   // boxes wholly past it are skipped
                if (x < nv) tma_store_2d(tm, box0, x, y);
                if (x + 64 < nv) tma_store_2d(tm, box0 + BOX, x + 64, y);
                bulk_commit_group();
                if (warp == 4) *progress = *progress + w.KB;
            }
        }
        if (lane == 0) bulk_wait_group_all();
    }

    if (*abort_flag) {
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
cudaError_t launch_wgrad(const WgradCall& c, cudaStream_t stream) {
    if (c.T == 0 && c.E == 0) return cudaSuccess;
    const bool mx = c.mx;
    const int Ip = (c.I + 255) / 256 * 256;
    const int tp = wgrad_max_padded_slots(c.T, c.E);
    wgrad_pstage_kernel<<<1, 32, 0, stream>>>(c.offsets, c.E, c.pstage, c.blk_e);
    WgPackArgs pa{};
    pa.sched = c.sched;
    pa.slot_gate = c.slot_gate;
    pa.offsets = c.offsets;
    pa.pstage = c.pstage;
    pa.blk_e = c.blk_e;
    pa.E = c.E;
    pa.I = c.I;
    pa.rows_per_shard = c.rows_per_shard;
    pa.N = c.N;
    auto pack = [&](int src, const void* p, int C, int Cp, int ld, uint8_t* img, uint8_t* sf) {
        WgPackArgs q = pa;
        q.src = (const uint16_t*)p;
        q.C = C;
        q.Cp = Cp;
        q.ld = ld;
        q.img = img;
        q.sf = sf;
        q.RB = Cp / 128;
        const dim3 grid((unsigned)(tp / 32), (unsigned)((Cp + kPackCols - 1) / kPackCols));
        const size_t sm = (src == WG_DUV || src == WG_X || src == WG_DY) ? sizeof(uint16_t) * 32 * kPackPitch16
                                                         : sizeof(float) * 32 * kPackPitch;
#define MOE_WG_PACK(S)                                                                                \
    if (mx) {                                                                                         \
        cudaFuncSetAttribute(wgrad_pack_kernel<S, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             (int)sm);                                                                \
        wgrad_pack_kernel<S, true><<<grid, 256, sm, stream>>>(q, c.ws);                               \
    } else {                                                                                          \
        cudaFuncSetAttribute(wgrad_pack_kernel<S, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,\
                             (int)sm);                                                                \
        wgrad_pack_kernel<S, false><<<grid, 256, sm, stream>>>(q, c.ws);                              \
    }
        switch (src) {
            case WG_DUV: MOE_WG_PACK(WG_DUV); break;
            case WG_X: MOE_WG_PACK(WG_X); break;
            case WG_DY: MOE_WG_PACK(WG_DY); break;
            default: MOE_WG_PACK(WG_H); break;
        }
#undef MOE_WG_PACK
    };
    pack(WG_DUV, c.duv, 2 * c.I, 2 * c.I, 2 * c.I, c.img_duv, c.sf_duv);
    pack(WG_X, c.x, c.H, c.H, c.H, c.img_x, c.sf_x);
    pack(WG_DY, c.dout, c.H, c.H, c.H, c.img_dy, c.sf_dy);
    pack(WG_H, c.uv, c.I, Ip, 2 * c.I, c.img_h, c.sf_h);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    WgGemm g0{};   // dW_gate_up[e] = [du dv]^T . x   (M = 2I, N = H)
    g0.a_img = c.img_duv;
    g0.a_sf = c.sf_duv;
    g0.a_rb = 2 * c.I / 128;
    g0.b_img = c.img_x;
    g0.b_sf = c.sf_x;
    g0.b_rb = c.H / 128;
    g0.m_tiles = 2 * c.I / 128;
    g0.n_tiles = c.H / 256;
    g0.n_valid = c.H;
    g0.out = (uint8_t*)c.dw_gate_up;
    g0.out_estride = (int64_t)2 * c.I * c.H * 2;
    g0.out_ld = c.H;
    WgGemm g1{};   // dW_down[e] = dy^T . h          (M = H, N = I padded to 256)
    g1.a_img = c.img_dy;
    g1.a_sf = c.sf_dy;
    g1.a_rb = c.H / 128;
    g1.b_img = c.img_h;
    g1.b_sf = c.sf_h;
    g1.b_rb = Ip / 128;
    g1.m_tiles = c.H / 128;
    g1.n_tiles = Ip / 256;
    g1.n_valid = c.I;
    g1.out = (uint8_t*)c.dw_down;
    g1.out_estride = (int64_t)c.H * c.I * 2;
    g1.out_ld = c.I;
    // TMA store maps over the two gradients: [E*2I][H] and [E*H][I] BF16, boxes of
    // 32 rows x 64 columns with 128-byte swizzle; columns past I are clipped.
    CUtensorMap tm0, tm1;
    {
        uint64_t dims[2] = {(uint64_t)c.H, (uint64_t)c.E * 2 * c.I};
        uint64_t str[1] = {(uint64_t)c.H * 2};
        uint32_t box[2] = {64, 32};
        if (!encode_tmap(&tm0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.dw_gate_up, dims, str, box))
            return cudaErrorInvalidValue;
    }
    {
        uint64_t dims[2] = {(uint64_t)c.I, (uint64_t)c.E * c.H};
        uint64_t str[1] = {(uint64_t)c.I * 2};
        uint32_t box[2] = {64, 32};
        if (!encode_tmap(&tm1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.dw_down, dims, str, box))
            return cudaErrorInvalidValue;
    }
    const size_t smem = 1024 + wg::SMEM;
    if (mx) {
        err = cudaFuncSetAttribute(wgrad_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        wgrad_gemm_kernel<true><<<c.grid, wg::THREADS, smem, stream>>>(g0, g1, tm0, tm1, c.offsets, c.pstage,
                                                                       c.E, c.ws, c.timeout_ns);
    } else {
        err = cudaFuncSetAttribute(wgrad_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        wgrad_gemm_kernel<false><<<c.grid, wg::THREADS, smem, stream>>>(g0, g1, tm0, tm1, c.offsets, c.pstage,
                                                                        c.E, c.ws, c.timeout_ns);
    }
    return cudaGetLastError();
}

}  // namespace moe
