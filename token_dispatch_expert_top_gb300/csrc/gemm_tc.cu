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
// The weights come tile-packed (pack.cu): one bulk copy per 32 KB B tile.
// ([MoK-2.37x] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72": section 01, the grouped GEMM fed expert-contiguous input on Blackwell
// tensor cores; section 02, SwiGLU and MXFP8 activation quantisation inside the
// GEMM data path rather than a separate quantise kernel.)
//
// CTA = 12 warps, one CTA per SM (the roles of gemm_roles.cuh):
//   warp 0      TMA producer (A tile 128 x 128 B, B tile 256 x 128 B per stage)
//   warp 1      TMEM allocator + MMA issuer (one thread)
//   warp 2      scale-factor loader (MXFP8): reads the [rows][K/32] scale bytes,
//               transposes them into the [32 lanes][4 words] blocks tcgen05.cp
//               moves to tensor memory
//   warp 3      the expert m-tile prefix in the prologue, then idle (the fused
//               kernel's dependency thread)
//   warps 4-11  epilogue: tensor memory -> registers -> SwiGLU / convert -> global
// Tile 128 x 256 (M x N), K-stage 128 bytes, 4-stage smem ring, FP32 accumulator
// in 256 tensor-memory columns.  Every wait is bounded (a deadline on the GPU
// clock); when one runs out the CTA records MOE_ERR_TIMEOUT and winds down.
#include "common.cuh"
#include "gemm_roles.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace moe {

// Tiles of one grouped GEMM over expert segments: expert-major, then N tile,
// then M tile, so CTAs working on consecutive tiles share a weight tile in L2.
template <int KIND, bool SAVE = false>
struct ExpertTiles {
    static constexpr bool kDeps = false;        // inputs are always ready
    static constexpr bool kSaveUV = SAVE;       // GEMM1 also stores u|v (training)
    static constexpr int kind = KIND;
    const int32_t* offsets;   // [E+1]
    const int32_t* mpre;      // [E+1] prefix of ceil(count_e / 128), in shared memory
    int E, n_tiles, total;
    __device__ int first() const { return blockIdx.x; }
    __device__ int next(int t) const { return t + gridDim.x; }
    __device__ int count() const { return total; }
    __device__ int kind_of(int) const { return kind; }
    __device__ TileInfo tile(int t) const {
        const int q = t / n_tiles;
        int lo = 0, hi = E;  // last e with mpre[e] <= q
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (mpre[mid] <= q) lo = mid; else hi = mid;
        }
        TileInfo tl;
        tl.kind = kind;
        tl.e = lo;
        const int mt = mpre[lo + 1] - mpre[lo];
        const int local = t - mpre[lo] * n_tiles;
        tl.n = local / mt;
        const int m = local % mt;
        tl.a_row0 = offsets[lo] + m * tc::BM;
        tl.out_row0 = tl.a_row0;
        tl.nrows = min(offsets[lo + 1] - tl.a_row0, tc::BM);
        tl.mb = 0;
        tl.midx = 0;
        return tl;
    }
    __device__ bool wait_inputs(const TileInfo&, const Pipe&) const { return true; }
    __device__ void tile_stored(const TileInfo&, const Pipe&) const {}
};

template <bool MX, int KIND, bool SAVE>
__global__ void __launch_bounds__(tc::THREADS, 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmT,
                           const __grid_constant__ CUtensorMap tmSFA,
                           const __grid_constant__ GemmSide side,
                           const int32_t* offsets, int E, WsHeader* ws,
                           unsigned long long timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    int32_t* mpre = reinterpret_cast<int32_t*>(smem + tc::OFF_TAIL);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 3) {
        // m-tile prefix over experts: mpre[e+1] = mpre[e] + ceil(count_e / BM)
        const int per = (E + 31) / 32;
        const int lo = min(lane * per, E), hi = min(lo + per, E);
        int s = 0;
        for (int e = lo; e < hi; ++e) s += (offsets[e + 1] - offsets[e] + tc::BM - 1) / tc::BM;
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - s;
        for (int e = lo; e < hi; ++e) {
            mpre[e] = run;
            run += (offsets[e + 1] - offsets[e] + tc::BM - 1) / tc::BM;
        }
        if (lane == 31) mpre[E] = incl;
    }
    __syncthreads();
    ExpertTiles<KIND, SAVE> src{offsets, mpre, E, side.n_tiles, mpre[E] * side.n_tiles};
    const GemmMaps maps{&tmA, &tmA, &tmSFA, &tmSFA, &tmT, &tmT};
    const GemmSides sides{&side, &side};
    run_gemm_pipeline<MX>(smem, maps, sides, src, ws, timeout_ns);
}

// ------------------------------------------------------------------ host side
inline size_t gemm_smem_bytes(int E) { return 1024 + tc::OFF_TAIL + sizeof(int32_t) * (E + 1); }

template <bool MX, int KIND, bool SAVE = false>
static cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tt, const CUtensorMap& tsa,
                              const GemmSide& side, const int32_t* offsets, int E, WsHeader* ws,
                              unsigned long long timeout_ns, int grid, cudaStream_t stream) {
    auto kern = tc_grouped_gemm_kernel<MX, KIND, SAVE>;
    const size_t smem = gemm_smem_bytes(E);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, tc::THREADS, smem, stream>>>(ta, tt, tsa, side, offsets, E, ws, timeout_ns);
    return cudaGetLastError();
}

// A scales as 16-byte-wide TMA boxes of 128 rows (four K-stages of scales).
static bool encode_sfa_map(CUtensorMap* tsa, const void* a_sf, int a_rows, int K) {
    const uint64_t ksf = (uint64_t)K / 32;
    uint64_t da[2] = {ksf, (uint64_t)a_rows};
    uint64_t sa[1] = {ksf};
    uint32_t ba[2] = {16, 128};
    return encode_tmap(tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a_sf, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// An A operand map: [rows][K] MXFP8 codes or BF16, boxes of `box_rows` rows x 128
// bytes, 128-byte swizzle.
static bool encode_a_map(CUtensorMap* m, bool mx, const void* base, int K, int rows, int box_rows) {
    const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t esz = mx ? 1 : 2;
    uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
    uint64_t str[1] = {(uint64_t)K * esz};
    uint32_t box[2] = {mx ? 128u : 64u, (uint32_t)box_rows};
    return encode_tmap(m, dt, 2, base, dims, str, box);
}

// A operand maps of both GEMMs (a [a_rows][H] and h [a_rows][I], 128-row boxes and
// kTailRows-row boxes for ragged tiles), the A scale maps when TMA-staged, and the
// two GemmSides over the tile-packed weights.
bool encode_ffn_maps(const TcFfnCall& c, FfnMaps* m, GemmSide* s1, GemmSide* s2) {
    const bool mx = c.mx;
    if (!encode_a_map(&m->a1, mx, c.a, c.H, c.a_rows, 128) ||
        !encode_a_map(&m->t1, mx, c.a, c.H, c.a_rows, kTailRows) ||
        !encode_a_map(&m->a2, mx, c.h, c.I, c.a_rows, 128) ||
        !encode_a_map(&m->t2, mx, c.h, c.I, c.a_rows, kTailRows))
        return false;
    *s1 = GemmSide{};
    s1->K = c.H;
    s1->n_tiles = c.I / 128;
    s1->up_off = c.I;
    s1->b_rows = 2 * c.I;
    s1->a_rows = c.a_rows;
    s1->a_sf = (const uint8_t*)c.a_sf;
    s1->b_pk = (const uint8_t*)c.w_gate_up;
    s1->sfb_pk = (const uint8_t*)c.w_gu_sf;
    s1->out = (uint8_t*)c.h;
    s1->out_sf = (uint8_t*)c.h_sf;
    s1->out_ld = c.I;
    s1->aux = (uint8_t*)c.uv;
    *s2 = *s1;
    s2->aux = nullptr;
    s2->K = c.I;
    s2->n_tiles = c.H / tc::BN;
    s2->up_off = 0;
    s2->b_rows = c.H;
    s2->a_sf = (const uint8_t*)c.h_sf;
    s2->b_pk = (const uint8_t*)c.w_down;
    s2->sfb_pk = (const uint8_t*)c.w_d_sf;
    s2->out = (uint8_t*)c.y;
    s2->out_sf = nullptr;
    s2->out_ld = c.H;
    s2->n_valid = c.H;
    m->s1a = CUtensorMap{};
    m->s2a = CUtensorMap{};
    if (mx) {
        s1->sf_tma = (c.H % 512) == 0;
        s2->sf_tma = (c.I % 512) == 0;
        if (s1->sf_tma && !encode_sfa_map(&m->s1a, c.a_sf, c.a_rows, c.H)) return false;
        if (s2->sf_tma && !encode_sfa_map(&m->s2a, c.h_sf, c.a_rows, c.I)) return false;
    }
    return true;
}

cudaError_t launch_expert_ffn_tc(const TcFfnCall& c, cudaStream_t stream) {
    if (c.T == 0) return cudaSuccess;
    FfnMaps m;
    GemmSide s1, s2;
    if (!encode_ffn_maps(c, &m, &s1, &s2)) return cudaErrorInvalidValue;
    cudaError_t err;
    if (c.mx) {
        err = c.uv ? launch_one<true, 0, true>(m.a1, m.t1, m.s1a, s1, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream)
                   : launch_one<true, 0>(m.a1, m.t1, m.s1a, s1, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream);
        if (err != cudaSuccess) return err;
        err = launch_one<true, 1>(m.a2, m.t2, m.s2a, s2, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream);
    } else {
        err = c.uv ? launch_one<false, 0, true>(m.a1, m.t1, m.s1a, s1, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream)
                   : launch_one<false, 0>(m.a1, m.t1, m.s1a, s1, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream);
        if (err != cudaSuccess) return err;
        err = launch_one<false, 1>(m.a2, m.t2, m.s2a, s2, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream);
    }
    return err;
}

// ------------------------------------------------------------- backward (dgrad)
// dgrad of GEMM2: dh = dy . W_down over A = dy [rows][H] (K = H) and the
// transposed-packed W_down (N = I, padded to 256-column tiles), stored as BF16;
// the SwiGLU derivative (backward.cu) then makes du|dv; dgrad of GEMM1:
// da = [du dv] . [W_gate; W_up] over A = du|dv [rows][2I] (K = 2I) and the
// transposed-packed W_gate_up (N = H).  Both run the GEMM2 form of the kernel.
cudaError_t launch_ffn_dgrad_tc(const TcDgradCall& c, cudaStream_t stream) {
    if (c.T == 0) return cudaSuccess;
    const bool mx = c.mx;
    const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t esz = mx ? 1 : 2;
    const uint32_t bk = mx ? 128 : 64;
    CUtensorMap m_dy, m_duv, t_dy, t_duv, s_dy = CUtensorMap{}, s_duv = CUtensorMap{};
    const void* a1 = mx ? c.duv_q : c.duv;
    if (!encode_a_map(&m_dy, mx, c.dy, c.H, c.a_rows, 128) ||
        !encode_a_map(&t_dy, mx, c.dy, c.H, c.a_rows, kTailRows) ||
        !encode_a_map(&m_duv, mx, a1, 2 * c.I, c.a_rows, 128) ||
        !encode_a_map(&t_duv, mx, a1, 2 * c.I, c.a_rows, kTailRows))
        return cudaErrorInvalidValue;
    GemmSide s2{};   // dgrad of GEMM2 -> dh
    s2.K = c.H;
    s2.n_tiles = (c.I + tc::BN - 1) / tc::BN;
    s2.a_rows = c.a_rows;
    s2.a_sf = (const uint8_t*)c.dy_sf;
    s2.b_pk = (const uint8_t*)c.wt_down;
    s2.sfb_pk = (const uint8_t*)c.wt_d_sf;
    s2.out = (uint8_t*)c.dh;
    s2.out_ld = c.I;
    s2.n_valid = c.I;
    GemmSide s1{};   // dgrad of GEMM1 -> da
    s1.K = 2 * c.I;
    s1.n_tiles = c.H / tc::BN;
    s1.a_rows = c.a_rows;
    s1.a_sf = (const uint8_t*)c.duv_sf;
    s1.b_pk = (const uint8_t*)c.wt_gate_up;
    s1.sfb_pk = (const uint8_t*)c.wt_gu_sf;
    s1.out = (uint8_t*)c.da;
    s1.out_ld = c.H;
    s1.n_valid = c.H;
    if (mx) {
        s2.sf_tma = (c.H % 512) == 0;
        s1.sf_tma = ((2 * c.I) % 512) == 0;
        if (s2.sf_tma && !encode_sfa_map(&s_dy, c.dy_sf, c.a_rows, c.H)) return cudaErrorInvalidValue;
        if (s1.sf_tma && !encode_sfa_map(&s_duv, c.duv_sf, c.a_rows, 2 * c.I)) return cudaErrorInvalidValue;
    }
    cudaError_t err = mx ? launch_one<true, 1>(m_dy, t_dy, s_dy, s2, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream)
                         : launch_one<false, 1>(m_dy, t_dy, s_dy, s2, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream);
    if (err != cudaSuccess) return err;
    err = launch_swiglu_backward(mx, c.dh, c.uv, c.T, c.I, c.duv, (uint8_t*)c.duv_q, (uint8_t*)c.duv_sf,
                                 c.num_sms, stream);
    if (err != cudaSuccess) return err;
    return mx ? launch_one<true, 1>(m_duv, t_duv, s_duv, s1, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream)
              : launch_one<false, 1>(m_duv, t_duv, s_duv, s1, c.offsets, c.E, c.ws, c.timeout_ns, c.grid, stream);
}

}  // namespace moe
