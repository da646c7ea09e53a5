// kernels.cuh -- launch functions of libmoe's kernels (host side), shared between
// the kernel sources and the C-ABI layer in api.cu.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kLayoutChunk = 256;  // flat (token, choice) entries per layout chunk
inline int layout_chunks(int T) { return (T + kLayoutChunk - 1) / kLayoutChunk; }

cudaError_t launch_quantize_mxfp8(const void* in, int in_dtype, int64_t rows, int64_t K,
                                  uint8_t* codes, uint8_t* scales, int num_sms,
                                  cudaStream_t stream);
cudaError_t launch_quantize_nvfp4(const void* in, int in_dtype, int64_t rows, int64_t K,
                                  uint8_t* codes, uint8_t* scales, float* st_amax, int num_sms,
                                  cudaStream_t stream);

cudaError_t launch_route_topk_simt(const void* x, const void* w, const float* bias, int N, int H,
                                   int E, int k, int dtype, int32_t* idx, float* gate,
                                   float* logits_out, cudaStream_t stream);

bool route_tc_supported(int dtype, int H, int E, int k);

cudaError_t launch_route_topk_tc(const void* x, const void* w, const float* bias, int N, int H,
                                 int E, int k, int32_t* idx, float* gate, float* logits_out,
                                 uint8_t* xq, uint8_t* xq_sf, WsHeader* ws,
                                 unsigned long long timeout_ns, cudaStream_t stream);

cudaError_t launch_layout(const int32_t* idx, int N, int k, int E, int S, int32_t* counts,
                          int32_t* offsets, int32_t* sched, int32_t* inv, int32_t* cnt_scratch,
                          int32_t* base_scratch, WsHeader* ws, cudaStream_t stream);

// order (nullable, order_len entries): the inverse map, flattened ([N][order_k]);
// each token's row is read once and written to its slots in range.
cudaError_t launch_dispatch_pull(const void* const* shard_rows, const void* const* shard_scales,
                                 const int32_t* sched, const int32_t* order, int order_len, int order_k,
                                 int slot_begin, int slot_count, int S, int rows_per_shard,
                                 int row_bytes, int scale_bytes, void* ring, void* ring_scales,
                                 int ring_slots, int num_sms, WsHeader* ws,
                                 unsigned long long timeout_ns, cudaStream_t stream);

cudaError_t launch_combine(const void* y, const int32_t* inv, const float* gate, int N, int H,
                           int k, int T, int dtype, void* out, int num_sms, WsHeader* ws,
                           cudaStream_t stream);

cudaError_t launch_ffn_f32(const float* a, const int32_t* offsets, const float* wgu,
                           const float* wd, int T, int H, int I, int E, float* h_scratch, float* y,
                           int num_sms, cudaStream_t stream);

// One call of the tensor-core expert FFN (GEMM1 + SwiGLU, then GEMM2).
struct TcFfnCall {
    bool mx;                  // MXFP8 operands (else BF16)
    int T, H, I, E;
    int a_rows;               // rows of a / h / y buffers (>= T)
    const void* a;            // [a_rows][H]
    const void* a_sf;         // [a_rows][H/32] (MXFP8)
    const int32_t* offsets;   // [E+1]
    const void* w_gate_up;    // tile-packed GEMM1 weights (pack.cu)
    const void* w_gu_sf;      // tile-packed GEMM1 scales (MXFP8)
    const void* w_down;       // tile-packed GEMM2 weights
    const void* w_d_sf;       // tile-packed GEMM2 scales (MXFP8)
    void* h;                  // [a_rows][I] scratch
    void* h_sf;               // [a_rows][I/32] scratch (MXFP8)
    void* y;                  // [a_rows][H] BF16
    void* uv;                 // training: u|v saved as BF16 [a_rows][2I], or null
    WsHeader* ws;
    unsigned long long timeout_ns;
    int grid;                 // persistent CTAs (one per SM)
};

cudaError_t launch_expert_ffn_tc(const TcFfnCall& c, cudaStream_t stream);

// Backward of the tensor-core expert FFN: the two dgrad GEMMs.
struct TcDgradCall {
    bool mx;
    int T, H, I, E;
    int a_rows;               // rows of dy / uv / duv / da (>= T)
    const void* dy;           // [a_rows][H] (codes or BF16)
    const void* dy_sf;        // [a_rows][H/32] (MXFP8)
    const void* uv;           // [a_rows][2I] BF16 saved by the forward
    const int32_t* offsets;   // [E+1]
    const void* wt_down;      // transposed-packed W_down (N = I padded to 256)
    const void* wt_d_sf;
    const void* wt_gate_up;   // transposed-packed W_gate_up (N = H, K = 2I)
    const void* wt_gu_sf;
    void* dh;                 // [a_rows][I] BF16 scratch
    void* duv;                // [a_rows][2I] BF16 (out)
    void* duv_q;              // [a_rows][2I] codes (MXFP8, out)
    void* duv_sf;             // [a_rows][2I/32] (MXFP8, out)
    void* da;                 // [a_rows][H] BF16 (out)
    WsHeader* ws;
    unsigned long long timeout_ns;
    int grid;
    int num_sms;
};
cudaError_t launch_ffn_dgrad_tc(const TcDgradCall& c, cudaStream_t stream);
// du = dh * v * silu'(u), dv = dh * silu(u) from BF16 dh [T][I] and u|v [T][2I] ->
// du|dv BF16 [T][2I] and, MXFP8, codes [T][2I] + scales [T][2I/32] along I.
cudaError_t launch_swiglu_backward(bool mx, const void* dh, const void* uv, int T, int I, void* duv,
                                   uint8_t* duv_q, uint8_t* duv_sf, int num_sms, cudaStream_t stream);

// Backward memory-bound steps (backward.cu).
constexpr int kRouterPiece = 256;   // slots per router-wgrad piece
inline int router_max_pieces(int T, int E) { return T / kRouterPiece + E; }
cudaError_t launch_pack_transposed(bool mx, const void* w, int E, int R, int C, void* dst,
                                   uint8_t* dst_sf, int num_sms, cudaStream_t stream);
cudaError_t launch_reverse_combine(bool mx, const void* dout, const void* y, const int32_t* inv,
                                   const float* gate, int N, int H, int k, int T, void* dy,
                                   uint8_t* dy_sf, float* dgate, float* dlogit, float* slot_gate,
                                   float* slot_dlogit, int num_sms, WsHeader* ws, cudaStream_t stream);
cudaError_t launch_reverse_dispatch(const void* da, const int32_t* inv, const int32_t* idx,
                                    const float* dlogit, const void* w_router, int N, int H, int k,
                                    int T, int E, void* dx, int num_sms, WsHeader* ws,
                                    cudaStream_t stream);
// Expert weight gradients (wgrad.cu).
inline int wgrad_max_padded_slots(int T, int E) { return 128 * (T / 128 + E); }
struct WgGemm {
    const uint8_t* a_img;     // A operand images [K-stages][a_rb][16 KB]
    const uint8_t* a_sf;      // MXFP8 scale images [K-stages of 128][a_rb][512]
    int a_rb;
    const uint8_t* b_img;
    const uint8_t* b_sf;
    int b_rb;
    int m_tiles, n_tiles, n_valid;
    uint8_t* out;             // BF16 [E][M][N]: out + e*out_estride + (row*out_ld + col)*2
    int64_t out_estride;      // bytes
    int out_ld;               // elements
};
struct WgradCall {
    bool mx;
    int N, H, I, E, T, rows_per_shard;
    const void* duv;          // [T][2I] BF16
    const void* x;            // [N][H] BF16
    const void* dout;         // [N][H] BF16
    const void* uv;           // [T][2I] BF16
    const int32_t* sched;
    const float* slot_gate;
    const int32_t* offsets;
    void* dw_gate_up;         // [E][2I][H] BF16 (out)
    void* dw_down;            // [E][H][I] BF16 (out)
    int32_t* pstage;          // [E+1] scratch
    int32_t* blk_e;           // [wgrad_max_padded_slots / 32] scratch
    uint8_t *img_duv, *sf_duv, *img_x, *sf_x, *img_dy, *sf_dy, *img_h, *sf_h;   // scratch
    WsHeader* ws;
    unsigned long long timeout_ns;
    int grid;
};
cudaError_t launch_wgrad(const WgradCall& c, cudaStream_t stream);

cudaError_t launch_router_wgrad(const void* x, const int32_t* sched, const int32_t* offsets,
                                const float* slot_dlogit, int N, int H, int E, int T,
                                int rows_per_shard, float* dw, float* db, float* part, float* part_b,
                                int32_t* ppre, WsHeader* ws, cudaStream_t stream);

// One-time repacking of natural K-major expert weights into tile images.
struct PackCall {
    bool mx;
    int E, H, I;
    const void* w_gate_up;    // [E][2I][H] codes or BF16
    const uint8_t* w_gu_sf;   // [E][2I][H/32]
    const void* w_down;       // [E][H][I]
    const uint8_t* w_d_sf;    // [E][H][I/32]
    void* p_gate_up;
    uint8_t* p_gu_sf;
    void* p_down;
    uint8_t* p_d_sf;
    int num_sms;
};
cudaError_t launch_pack_weights(const PackCall& c, cudaStream_t stream);

// Fused persistent forward (gather, expert FFN, combine in one launch).
// Upper bound on the m-tiles of all minibatches: each piece (expert x minibatch)
// of L slots takes ceil(L/128) <= L/128 + 1 tiles and there are at most E + nmb
// pieces.
inline int fused_max_mtiles(int T, int E, int nmb) { return T / 128 + E + 2 * nmb + 8; }
// int32 entries of the plan + counter region: tbase [2nmb+2], pbase [nmb+1],
// elo [nmb+1], cut [nmb+2], then the counters
inline size_t fused_plan_ints(int T, int E, int nmb) {
    return (size_t)(2 * nmb + 2) + 2 * (nmb + 1) + (nmb + 2) + 2 * nmb + 8 + fused_max_mtiles(T, E, nmb);
}
struct FusedCall {
    TcFfnCall ffn;            // a = ring [R][H], h = ring [R][I], y = [T][H]
    int N, H, E, k, S, T;
    int MB, R, nmb, G, C;
    int row_bytes, sf_bytes;
    int skip_ready;           // -1: none
    int reverse;              // minibatches cut from the last slot down
    const int32_t* sched;
    const int32_t* inv;
    const float* gate;
    const void* const* shard_rows;
    const void* const* shard_sf;
    void* out;
    int* plan_ints;
};
cudaError_t launch_fused_forward(const FusedCall& c, cudaStream_t stream);
int fused_max_ctas();

// TMA maps of both expert GEMMs (operands and, for MXFP8, staged scales).
struct FfnMaps {
    CUtensorMap a1, a2, s1a, s2a;
    CUtensorMap t1, t2;       // A operands with 32-row boxes (ragged last m-tiles)
};
struct GemmSide;
bool encode_ffn_maps(const TcFfnCall& c, FfnMaps* m, GemmSide* s1, GemmSide* s2);

// Shape validation shared by the entry points (api.cu): MOE_OK or the status to
// return before anything is launched.
int validate_shape(const moe_shape_t* s);

}  // namespace moe
