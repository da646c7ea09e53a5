/*
 * moe.h -- C ABI of libmoe, a single-GPU forward Mixture-of-Experts layer for
 * GB300 (sm_103a): top-k routing, sort-free token layout, pull-style gather from
 * virtual source shards into a ring of token slots, grouped SwiGLU expert FFN
 * (FP32, BF16 or block-scaled MXFP8 on tcgen05 tensor cores), and a gate-weighted
 * combine back to token order; plus one persistent kernel that runs gather,
 * expert FFN and combine as roles on separate SMs.
 *
 * The method is the one described on
 *   [MoK-2.37x] "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
 *               NVL72" (KuCoin news flash; Spanish, Vietnamese, Hindi and
 *               Traditional Chinese editions; sections 01, 02, 03)
 *   [Kittens]   "Смесь котят: как Cursor создал открытое ядро, ускоряющее обучение
 *               ИИ до 2.4 раз" (qubstore.ru; paragraphs on pull dispatch, the ring
 *               buffer and the megakernel)
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller (typically a
 *     PyTorch allocation).  The library never allocates device memory; scratch
 *     space comes from a caller-owned workspace sized by moe_workspace_bytes().
 *     One exception: moe_layout_noalloc's fixed 1 MiB scratch array, part of the
 *     library's device image on every GPU that loads it, held from the library's
 *     load until the process exits.
 *   - Shapes and parameters are passed in HOST structs and read during the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call only enqueues work and returns; none synchronises the
 *     host except moe_last_device_status().
 *   - Argument errors (null pointers, unsupported shapes, a workspace that is too
 *     small) are detected on the host before anything is launched and returned as
 *     a moe_status_t; nothing is enqueued in that case.  A failed launch returns
 *     MOE_ERR_CUDA.
 *   - Errors only the device can see (an expert index out of range, a schedule
 *     entry outside its shard, a bounded wait that ran out) are recorded in a
 *     status word at the start of the workspace (first error wins) and read with
 *     moe_last_device_status().  Kernels that detect one skip the offending work
 *     and return; they never trap.
 *   - The workspace must be 32-byte aligned (MOE_ERR_WORKSPACE otherwise); the
 *     library carves 256-byte-aligned regions out of it.
 *   - Row-major layouts throughout.  Expert weights are quantised (MXFP8) and
 *     repacked into GEMM tile images once, by moe_quantize_mxfp8 and
 *     moe_pack_expert_weights, before any forward call.
 *
 * Number formats (moe_shape_t.dtype)
 *   MOE_F32   : x, router weight, expert weights, y and out are FP32.
 *   MOE_BF16  : x, router weight, expert weights, h, y and out are BF16; every
 *               contraction accumulates in FP32.
 *   MOE_MXFP8 : x, router weight and out are BF16; the expert GEMM operands (the
 *               gathered token rows, W_gate/W_up, h, W_down) are MXFP8: E4M3 codes
 *               plus one UE8M0 scale byte per 32 consecutive elements along K
 *               (OCP MX v1.0; scale exponent floor(log2(amax)) - 8, saturating
 *               round-to-nearest-even codes).  Scales are stored row-major next to
 *               their codes: [rows][K/32] bytes.  y is BF16.  Accumulation FP32.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shape */
    MOE_ERR_UNSUPPORTED = 2,   /* a shape or dtype the library has no kernel for */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_bytes() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out (see moe_params_t.timeout_ns) */
    MOE_ERR_DEVICE_CHECK = 6   /* device: an index was out of range; the item was skipped */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_MXFP8 = 2 } moe_dtype_t;

/* Layer shape.  N tokens of hidden size H, E experts of intermediate size I,
 * k experts per token, S virtual source shards of N/S consecutive tokens each
 * (N must be a multiple of S).  T = N*k token slots. */
typedef struct {
    int N, H, I, E, k, S;
    int dtype; /* moe_dtype_t */
} moe_shape_t;

/* Tuning of the persistent forward kernel (moe_forward_fused); zero fields take
 * defaults.  The ring holds `ring_slots` token slots; slots are handed from the
 * gather role to the compute role in minibatches of `minibatch` slots
 * ([MoK-2.37x] section 02: SM split, GPU-local counters, minibatch of at least
 * two full GEMM waves, fixed-size ring token buffer reused as soon as a slot's
 * results have left).  timeout_ns bounds every device-side wait. */
typedef struct {
    int ring_slots;        /* ring capacity in token slots; 0 = 4 minibatches (<= T)  */
    int minibatch;         /* slots per handoff; 0 = four waves of GEMM1 tiles         */
    int gather_ctas;       /* CTAs in the gather + combine role; 0 = SMs / 25          */
    int compute_ctas;      /* CTAs in the expert-FFN role; 0 = all remaining SMs       */
    long long timeout_ns;  /* bound on each device-side wait; 0 = 2e9 (two seconds)    */
    int test_skip_ready;   /* test hook, 0 = off.  When m+1 > 0, the gather role never
                              publishes minibatch m, so the compute role's bounded
                              wait runs out and the call reports MOE_ERR_TIMEOUT.  */
    int reverse_ring;      /* fused forward: 0 = minibatches walk the slots in order; 1 =
                              in reverse, the last slots first ([Kittens], ring-buffer
                              paragraph: the forward walks the ring backwards so the
                              backward finds the last activations still resident).
                              The output is the same bit for bit.                    */
} moe_params_t;

/* Bytes of workspace every entry point below needs for this shape and these
 * params (params may be NULL: defaults).  Its first 256 bytes hold the device
 * status word and must be zeroed once with moe_workspace_init() before first use. */
size_t moe_workspace_bytes(const moe_shape_t* shape, const moe_params_t* params);

/* Zero the workspace header (status word and counters) on `stream`. */
int moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise `stream`, read the device status word of `workspace`, reset it to
 * MOE_OK and return what it held.  The only entry point that blocks the host. */
int moe_last_device_status(void* workspace, void* stream);

/* Human-readable name of a moe_status_t value (static string). */
const char* moe_status_string(int status);

/* MXFP8 quantisation along K of a row-major [rows][K] matrix (OCP MX v1.0 block
 * rule; the layer's configuration names it for GEMM operands; [MoK-2.37x]
 * section 02 fuses it into the data path for activations).  Used for the
 * expert weights (once, offline) and as a stand-alone test of the rule.
 *   in      : [rows][K], in_dtype MOE_F32 or MOE_BF16
 *   codes   : [rows][K] E4M3 bytes          (out)
 *   scales  : [rows][K/32] UE8M0 bytes      (out)
 * K must be a multiple of 32.  Bit-exact with the oracle on identical input. */
int moe_quantize_mxfp8(const void* in, int in_dtype, int64_t rows, int64_t K,
                       uint8_t* codes, uint8_t* scales, void* stream);

/* Macrobatched forward: the N tokens are cut into `macrobatches` equal, consecutive
 * macrobatches that run the staged path one after another on `stream`, while each
 * macrobatch's combine runs on a second stream of the library's, so it overlaps the
 * routing, layout and dispatch of the next macrobatch ([MoK-2.37x] section 02:
 * the previous macrobatch's combine overlaps the next one's dispatch; [Kittens],
 * ring-buffer paragraph).  Every step is per token or per slot, so `out` is
 * bitwise equal to moe_forward's.  On one GPU the expert weights are streamed once
 * per macrobatch, so more macrobatches are slower; the split serves the pipelined
 * exchange of a multi-GPU layer.
 *   N must be a multiple of macrobatches * S;  out : [N][H] (as moe_forward)
 *   workspace : moe_macro_workspace_bytes() bytes, 256-byte aligned: one slice per
 *               macrobatch of moe_workspace_bytes(shape with N / macrobatches)
 *               rounded up to 256 bytes; the status word of every slice must be
 *               zeroed with moe_workspace_init() before first use, and device errors
 *               are recorded in the slice of the macrobatch that met them.
 * The call returns after queueing; `stream` waits for every combine.  The second
 * stream is created on the first call on a device. */
size_t moe_macro_workspace_bytes(const moe_shape_t* shape, const moe_params_t* params, int macrobatches);
int moe_forward_macrobatched(const void* x, const void* w_router, const float* bias, const void* w_gate_up,
                             const void* w_gu_scales, const void* w_down, const void* w_d_scales,
                             const moe_shape_t* shape, const moe_params_t* params, int macrobatches,
                             void* out, void* workspace, size_t workspace_bytes, void* stream);

/* NVFP4 quantisation along K of a row-major [rows][K] matrix.  [Kittens] names
 * NVFP4, beside MXFP8, as a format of the team's earlier training kernels without
 * defining it (paragraph on the year of compute-only kernels); the format taken is the OCP MX v1.0 FP4 E2M1 element
 * with NVIDIA's published two-level scaling: one E4M3 scale per 16 consecutive
 * elements and one FP32 scale per tensor.  With every step one correctly rounded
 * FP32 operation:
 *   s_t  = amax / 2688 over the whole tensor (1 if it is all zero),
 *   s_b  = E4M3(amax_block / 6 / s_t)        (round to nearest even, saturating),
 *   d    = value(s_b) * s_t,
 *   code = E2M1(x / d) (nearest even, saturating at 6; 0 for every element if d = 0).
 *   in           : [rows][K], in_dtype MOE_F32 or MOE_BF16, finite, 16-byte aligned
 *   codes        : [rows][K/2] bytes, two E2M1 codes per byte, element 2i in the low
 *                  nibble of byte i (out; 8-byte aligned)
 *   scales       : [rows][K/16] E4M3 bytes (out)
 *   tensor_scale : device float[2] (out): [0] = s_t, [1] = the tensor amax
 * K must be a multiple of 16.  Two passes over the input (the amax, then the blocks)
 * on `stream`.  Bit-exact with the oracle on identical input.  The grouped GEMMs do
 * not take this format. */
int moe_quantize_nvfp4(const void* in, int in_dtype, int64_t rows, int64_t K,
                       uint8_t* codes, uint8_t* scales, float* tensor_scale, void* stream);

/* One-time repacking of the expert weights into the layout the grouped GEMMs
 * read (pull dispatch lets the receiver choose its own placement, [MoK-2.37x]
 * section 02; the same holds for the static weights).  Input is the natural
 * K-major layout; output has the same size and is what moe_expert_ffn,
 * moe_forward and moe_forward_fused take:
 *   w_gate_up [E][2I][H] (rows 0..I-1 W_gate^T, rows I..2I-1 W_up^T),
 *   w_down [E][H][I] (W_down^T); MXFP8: E4M3 codes plus [rows][K/32] scales.
 *   packed_gate_up : [E][I/128][K-stages][32 KB]: per N tile of 128 h columns and
 *                    K-stage of 128 bytes (128 E4M3 or 64 BF16 values), the 128
 *                    gate rows then the 128 up rows, 128 bytes each, 16-byte chunk
 *                    c of row r stored at chunk c ^ (r % 8) of that row
 *   packed_down    : [E][H/256][K-stages][32 KB], 256 down rows per tile, same form
 *   packed_*_scales: [..][K-stages][1 KB]: two 128-row halves of [32][4] words,
 *                    word j of entry r holding the 4 K-step scales of row 32j + r
 * FP32 weights are copied unchanged (the FP32 path reads them as they are). */
int moe_pack_expert_weights(const moe_shape_t* shape, const void* w_gate_up,
                            const uint8_t* w_gu_scales, const void* w_down,
                            const uint8_t* w_d_scales, void* packed_gate_up,
                            uint8_t* packed_gu_scales, void* packed_down, uint8_t* packed_d_scales,
                            void* stream);

/* Router + top-k ([MoK-2.37x] section 01: every token picks a few experts each
 * step; configuration: softmax over the router logits, top-k, gates renormalised
 * to sum 1).
 *   x          : [N][H]  FP32 (MOE_F32) or BF16 (otherwise)
 *   w_router   : [E][H]  same dtype as x (W_r transposed: expert-major)
 *   bias       : [E] FP32 added to the logits, or NULL
 *   idx        : [N][k] int32, the k experts by descending logit; equal logits
 *                keep the lower expert index first                   (out)
 *   gate       : [N][k] FP32, softmax of the selected logits (= the full
 *                softmax renormalised over the k choices)            (out)
 *   logits_out : [N][E] FP32 logits as the kernel computed them, or NULL
 *   xq_codes, xq_scales : for MOE_MXFP8, [N][H] and [N][H/32] MXFP8 copy of x
 *                (the dispatch operand), or NULL to skip
 * Logits accumulate in FP32 (BF16 products on tensor cores when E%16==0,
 * E<=256 and H%64==0; FP32 SIMT otherwise).  With E>=64 and E%32==0 the two
 * halves of H accumulate separately and their FP32 sums are added once, so a
 * logit may differ in its last bits from a single running sum; idx and gate are
 * always the selection on the returned logits. */
int moe_route_topk(const void* x, const void* w_router, const float* bias,
                   const moe_shape_t* shape, int32_t* idx, float* gate, float* logits_out,
                   uint8_t* xq_codes, uint8_t* xq_scales,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Sort-free layout ("schedule"; [MoK-2.37x] section 01 and [Kittens] pull
 * paragraph: count tokens per expert, place them expert-contiguously, a
 * two-column schedule built without sorting).
 *   idx     : [N][k] int32 expert choices
 *   counts  : [E] tokens per expert                                  (out)
 *   offsets : [E+1] exclusive scan of counts, offsets[E] = T, unpadded (out)
 *   sched   : [T][2] int32 (source shard, row within shard) per slot  (out)
 *   inv     : [N][k] int32 slot of choice (n, j)                      (out)
 * Inside an expert, slots follow ascending token index (a stable counting
 * placement: per-chunk expert counts via warp match + shared-memory atomics, an
 * exclusive scan, then a warp-ballot rank).  Bit-exact with the oracle. */
int moe_layout(const int32_t* idx, const moe_shape_t* shape, int32_t* counts, int32_t* offsets,
               int32_t* sched, int32_t* inv, void* workspace, size_t workspace_bytes,
               void* stream);

/* Pull dispatch ([MoK-2.37x] section 02: the expert side reads the rows it needs,
 * knowing only the source shard and the row; it picks the local placement).
 * Copies slots [slot_begin, slot_begin + slot_count) into the ring: slot t gets
 * row sched[t] = (shard, row) and goes to ring row t % ring_slots.
 *   shard_rows   : DEVICE array of S device pointers; shard s holds N/S rows of
 *                  H elements (FP32 / BF16) or H E4M3 codes (MXFP8)
 *   shard_scales : DEVICE array of S device pointers to [N/S][H/32] scales
 *                  (MXFP8 only; NULL otherwise)
 *   sched        : [T][2] from moe_layout
 *   inv          : [N][k] from the same moe_layout call as sched, or NULL.  Given,
 *                  the k slots of each token are handled together: every slot's
 *                  schedule entry is read, the row named by the token's first slot
 *                  in range is fetched from HBM once and written to each of its
 *                  slots in range; a slot whose entry names another row is skipped
 *                  and recorded as MOE_ERR_DEVICE_CHECK.  NULL: slot order, each
 *                  slot copying its own schedule entry
 *   ring, ring_scales : [ring_slots][row] destination (ring_scales MXFP8 only),
 *                  16-byte aligned
 * Shard row bases must be 16-byte aligned: a schedule entry whose source row is
 * not (or lies outside its shard) is skipped and recorded as
 * MOE_ERR_DEVICE_CHECK.  When both the row and its scale row are multiples of 16
 * bytes, rows move through the bulk-copy engine (per warp, one lane streams rows
 * through a ring of shared-memory row buffers: a bulk load, then one bulk store
 * per slot); otherwise one warp per slot row copies with 16- or 4-byte vector
 * loads and stores, in slot order. */
int moe_dispatch_pull(const void* const* shard_rows, const void* const* shard_scales,
                      const moe_shape_t* shape, const int32_t* sched, const int32_t* inv,
                      int slot_begin, int slot_count, void* ring, void* ring_scales, int ring_slots,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Grouped SwiGLU expert FFN over expert-contiguous slot rows ([MoK-2.37x]
 * sections 01-02: grouped GEMM fed expert-contiguous input; SwiGLU and MXFP8
 * quantisation of activations inside the GEMM data path).  For each expert e and
 * each row r in [offsets[e], offsets[e+1]):
 *   [u v] = a_r . [W_gate,e W_up,e];  h = silu(u) * v  (rounded to BF16, or
 *   MXFP8-quantised along I, or kept FP32);  y_r = h . W_down,e
 *   a, a_scales : [T][H] slot rows in slot order (+ [T][H/32] scales, MXFP8)
 *   offsets     : [E+1] DEVICE exclusive scan of expert counts (read on device;
 *                 the host never learns the counts)
 *   w_gate_up, w_gu_scales, w_down, w_d_scales : the expert weights in the
 *                 tile-packed layout written by moe_pack_expert_weights (W_gate /
 *                 W_up / W_down; scales NULL unless MXFP8)
 *   y           : [T][H] FP32 (MOE_F32) or BF16, 32-byte aligned       (out)
 * BF16 / MXFP8 run on tcgen05 tensor cores (128x256 tiles, A by TMA, B by bulk
 * copies of packed tiles, accumulators in tensor memory) and need H % 256 == 0 and
 * I % 128 == 0; MOE_F32 runs a SIMT kernel. */
int moe_expert_ffn(const void* a, const void* a_scales, const int32_t* offsets,
                   const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                   const void* w_d_scales, const moe_shape_t* shape, void* y,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Combine and final weighted merge ([MoK-2.37x] sections 02-03: every result
 * returns to its token; the gate-weighted merge is part of the layer).
 *   out[n] = sum_{j=0..k-1} gate[n][j] * y[inv[n][j]], FP32 accumulation in j
 *   order, rounded once to out's dtype (FP32 for MOE_F32, BF16 otherwise).
 *   y: [T][H] slot rows;  inv, gate: [N][k];  out: [N][H]. */
int moe_combine(const void* y, const int32_t* inv, const float* gate, const moe_shape_t* shape,
                void* out, void* workspace, size_t workspace_bytes, void* stream);

/* Whole forward layer, one kernel per step on `stream` (route, layout, pull,
 * expert FFN, combine) with every intermediate in the workspace.
 *   x, w_router, bias : as moe_route_topk
 *   w_* : tile-packed expert weights as moe_expert_ffn (moe_pack_expert_weights)
 *   out : [N][H]
 *   idx_out, gate_out : optional [N][k] copies of the routing (NULL to skip)
 * The MXFP8 copy of x is written once per source shard into the workspace and
 * pulled from there through a device table of S shard pointers. */
int moe_forward(const void* x, const void* w_router, const float* bias,
                const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                const void* w_d_scales, const moe_shape_t* shape, const moe_params_t* params,
                void* out, int32_t* idx_out, float* gate_out,
                void* workspace, size_t workspace_bytes, void* stream);

/* Same layer, with gather, expert FFN and combine in ONE persistent kernel whose
 * CTAs take the gather/combine role or the compute role ([MoK-2.37x] section 02:
 * megakernel with an explicit SM split; GPU-local counters hand each minibatch
 * from the gather side to the compute side and back; a fixed-size ring of token
 * slots is refilled as soon as its slots are consumed; no host round trip and no
 * dropped tokens).  Routing and layout run first as their own kernels.  Output is
 * bit-identical to moe_forward for every ring size, minibatch and SM split
 * ([Kittens], megakernel paragraph: bitwise determinism). */
int moe_forward_fused(const void* x, const void* w_router, const float* bias,
                      const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                      const void* w_d_scales, const moe_shape_t* shape,
                      const moe_params_t* params, void* out, int32_t* idx_out, float* gate_out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* moe_layout without a workspace, for callers that cannot allocate device memory at
 * call time: a serving process that reserves all its device memory at start-up and
 * allocates nothing afterwards, or a plug-in whose host owns the allocator.  The pages
 * describe no such entry point; it exists for those callers only.
 *   Same arguments, shape checks and results as moe_layout, minus the workspace
 *   (H, I and dtype are checked exactly as moe_layout checks them).  Its scratch
 *   (per-chunk expert counts and their scan) is a fixed 1 MiB __device__ array
 *   compiled into the library, resident on every GPU that loads it until the
 *   process exits.  Shapes with ceil(N*k/256) * E > 131072 are rejected with
 *   MOE_ERR_WORKSPACE before anything is launched.
 *   The first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress (that device must be current).  The address is cached
 *   with the id of the device's current context; after a device reset (or another
 *   teardown of the context) the next call looks it up again.
 *   Every call on a device uses that device's one copy of the array and leaves
 *   its contents behind: calls that overlap on the same GPU (for example on two
 *   streams) race.  Calls on different GPUs use different copies.
 *   Expert indices out of range are skipped but not reported (there is no status
 *   word without a workspace). */
int moe_layout_noalloc(const int32_t* idx, const moe_shape_t* shape, int32_t* counts,
                       int32_t* offsets, int32_t* sched, int32_t* inv, void* stream);

/* ------------------------------------------------------------------------- */
/* Backward pass ([MoK-2.37x] section 01: training adds two exchanges in the    */
/* direction opposite to dispatch and combine; section 02: the backward pulls   */
/* in the reverse combine and pushes in the reverse dispatch).  BF16 and MXFP8  */
/* layers only (MOE_ERR_UNSUPPORTED for MOE_F32).  The backward is the exact    */
/* derivative of the forward with every rounding point passed straight through */
/* and the top-k choice held fixed: only the k selected logits of a token get a */
/* gradient, through the renormalised gates.                                    */
/* ------------------------------------------------------------------------- */

/* Activations the forward keeps for the backward (all DEVICE, caller-owned,
 * written by moe_forward_train):
 *   idx, gate, inv : [N][k] int32 / FP32 / int32   (as moe_route_topk, moe_layout)
 *   offsets        : [E+1] int32, sched : [T][2] int32   (as moe_layout)
 *   y              : [T][H] BF16 expert outputs in slot order (32-byte aligned)
 *   uv             : [T][2I] BF16 pre-activations of every slot: u = a.W_gate in
 *                    columns 0..I-1, v = a.W_up in columns I..2I-1 (32-byte aligned) */
typedef struct {
    int32_t* idx;
    float* gate;
    int32_t* inv;
    int32_t* offsets;
    int32_t* sched;
    void* y;
    void* uv;
} moe_saved_t;

/* Bytes of workspace the backward entry points need (dy, du|dv, da, gate and
 * logit gradients, router-gradient partial sums, the weight-gradient operand
 * images).  0 for an invalid shape.  The
 * first 256 bytes are the status header, as for moe_workspace_bytes(). */
size_t moe_backward_workspace_bytes(const moe_shape_t* shape);

/* One-time packing of the expert weights for the dgrad GEMMs: the transposes of
 * the forward's weights, quantised (MXFP8) along the forward's OUTPUT dimension,
 * which is the dgrad GEMMs' reduction dimension, in the tile-image form of
 * moe_pack_expert_weights.
 *   w_gate_up : [E][2I][H] BF16 master weights (natural layout, not packed)
 *   w_down    : [E][H][I]  BF16 master weights
 *   packed_gate_up_t : [E][H/256][2I/KS][32 KB], tile row = h, K = the 2I rows of
 *                      w_gate_up (KS = 128 for MXFP8, 64 for BF16)         (out)
 *   packed_gu_t_scales : [E][H/256][2I/128][1 KB] (MXFP8; NULL for BF16)  (out)
 *   packed_down_t : [E][Ip/256][H/KS][32 KB], tile row = i, K = h, Ip = I
 *                   rounded up to a multiple of 256 (padding rows are zero) (out)
 *   packed_d_t_scales : [E][Ip/256][H/128][1 KB] (MXFP8; NULL for BF16)   (out)
 * All pointers 16-byte aligned. */
int moe_pack_expert_weights_dgrad(const moe_shape_t* shape, const void* w_gate_up,
                                  const void* w_down, void* packed_gate_up_t,
                                  uint8_t* packed_gu_t_scales, void* packed_down_t,
                                  uint8_t* packed_d_t_scales, void* stream);

/* moe_expert_ffn that also writes the pre-activations u|v of every slot row
 * ([T][2I] BF16, as moe_saved_t.uv) for the SwiGLU backward.  BF16/MXFP8 only. */
int moe_expert_ffn_train(const void* a, const void* a_scales, const int32_t* offsets,
                         const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                         const void* w_d_scales, const moe_shape_t* shape, void* y, void* uv,
                         void* workspace, size_t workspace_bytes, void* stream);

/* The staged forward (moe_forward) for training: same output, and every
 * activation the backward needs goes to `saved` (all fields required).  Takes
 * the forward's workspace (moe_workspace_bytes). */
int moe_forward_train(const void* x, const void* w_router, const float* bias,
                      const void* w_gate_up, const void* w_gu_scales, const void* w_down,
                      const void* w_d_scales, const moe_shape_t* shape, const moe_params_t* params,
                      void* out, const moe_saved_t* saved, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Reverse combine (pulled by slot, [MoK-2.37x] section 02).  For every token n
 * and choice j, slot s = inv[n][j], gate g = gate[n][j]:
 *   dy[s]          = g * dout[n]   (FP32 product, then MXFP8-quantised along H
 *                                    with the MX rule of moe_quantize_mxfp8, or
 *                                    rounded to BF16)
 *   dgate[n][j]    = <dout[n], y[s]>            (FP32 accumulation)
 *   dlogit[n][j]   = g * (dgate[n][j] - sum_i gate[n][i] * dgate[n][i])
 *   slot_gate[s] = g,  slot_dlogit[s] = dlogit[n][j]
 *   dout : [N][H] BF16;  y : [T][H] BF16 (moe_saved_t.y)
 *   dy, dy_scales : [T][H] codes + [T][H/32] scales (MXFP8), or [T][H] BF16 with
 *                   dy_scales NULL                                       (out)
 *   dgate, dlogit : [N][k] FP32 (out);  slot_gate, slot_dlogit : [T] FP32 (out)
 * An inverse-map entry outside [0, T) skips its token and records
 * MOE_ERR_DEVICE_CHECK.  Needs only the status header of the workspace. */
int moe_reverse_combine(const void* dout, const void* y, const int32_t* inv, const float* gate,
                        const moe_shape_t* shape, void* dy, uint8_t* dy_scales, float* dgate,
                        float* dlogit, float* slot_gate, float* slot_dlogit, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Expert dgrad: the two grouped dgrad GEMMs of the SwiGLU FFN on tcgen05, over
 * the expert segments [offsets[e], offsets[e+1]) of the slot rows:
 *   dh = dy . W_down,e ;  du = dh * v * silu'(u) ;  dv = dh * silu(u)
 *   da = du . W_gate,e + dv . W_up,e
 *   dy, dy_scales : moe_reverse_combine's dy
 *   uv            : moe_saved_t.uv
 *   wt_* : moe_pack_expert_weights_dgrad's output
 *   duv           : [T][2I] BF16, du in columns 0..I-1, dv in I..2I-1     (out)
 *   duv_codes, duv_scales : MXFP8 copy of duv quantised along 2I ([T][2I] +
 *                   [T][2I/32]; the operand of the second GEMM), NULL for BF16 (out)
 *   da            : [T][H] BF16 input gradient of every slot              (out)
 * FP32 accumulation; the derivative of silu is evaluated in FP32 from the saved
 * BF16 u and v.  All row buffers 32-byte aligned. */
int moe_expert_ffn_dgrad(const void* dy, const uint8_t* dy_scales, const void* uv,
                         const int32_t* offsets, const void* wt_gate_up,
                         const uint8_t* wt_gu_scales, const void* wt_down,
                         const uint8_t* wt_d_scales, const moe_shape_t* shape, void* duv,
                         uint8_t* duv_codes, uint8_t* duv_scales, void* da, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Reverse dispatch (pushed back to each token, [MoK-2.37x] section 02) plus the
 * router's input gradient:
 *   dx[n] = sum_j da[inv[n][j]] + sum_j dlogit[n][j] * w_router[idx[n][j]]
 * each sum in j order in FP32 (slots first), rounded once to BF16.  No atomics:
 * deterministic.
 *   da : [T][H] BF16;  inv, idx : [N][k];  dlogit : [N][k] FP32;
 *   w_router : [E][H] BF16;  dx : [N][H] BF16 (out)
 * An index out of range skips its terms and records MOE_ERR_DEVICE_CHECK. */
int moe_reverse_dispatch(const void* da, const int32_t* inv, const int32_t* idx,
                         const float* dlogit, const void* w_router, const moe_shape_t* shape,
                         void* dx, void* workspace, size_t workspace_bytes, void* stream);

/* Router weight gradient: dW_r[e] = sum over expert e's slots s (in slot order)
 * of slot_dlogit[s] * x[token(s)], dbias[e] = sum of slot_dlogit over them;
 * token(s) = shard * (N/S) + row from sched.  Pieces of 256 slots are summed in
 * FP32 and then reduced in piece order, so the result is deterministic.
 *   x : [N][H] BF16;  sched : [T][2];  offsets : [E+1];  slot_dlogit : [T] FP32
 *   dw_router : [E][H] FP32 (out);  dbias : [E] FP32 (out, may be NULL)
 * Needs moe_backward_workspace_bytes() of workspace. */
int moe_router_wgrad(const void* x, const int32_t* sched, const int32_t* offsets,
                     const float* slot_dlogit, const moe_shape_t* shape, float* dw_router,
                     float* dbias, void* workspace, size_t workspace_bytes, void* stream);

/* Expert weight gradients: for every expert e, GEMMs that reduce over its slots
 * [offsets[e], offsets[e+1]) on tcgen05,
 *   dW_gate_up[e] = [du dv]^T . x[token(s)]     dW_down[e] = (g * dout[token(s)])^T . h
 * with h = silu(u) * v recomputed from the kept u|v, FP32 accumulation, BF16
 * results; an expert without slots gets zeros.  Each operand is first transposed
 * into K-major tile images over the slot axis (each expert's slots padded to 128
 * with zeros); MXFP8 quantises it along the slots, in blocks of 32 from the
 * expert's first slot (the block-scaled MMA reduces along its K).
 *   duv : [T][2I] BF16 (moe_expert_ffn_dgrad);  x, dout : [N][H] BF16;
 *   uv : moe_saved_t.uv;  sched, offsets : moe_layout;  slot_gate : [T] FP32
 *   (moe_reverse_combine)
 *   dw_gate_up : [E][2I][H] BF16 (rows as w_gate_up), dw_down : [E][H][I] BF16,
 *   both 32-byte aligned                                                    (out)
 * Needs moe_backward_workspace_bytes() of workspace. */
int moe_expert_wgrad(const void* duv, const void* x, const void* dout, const void* uv,
                     const int32_t* sched, const float* slot_gate, const int32_t* offsets,
                     const moe_shape_t* shape, void* dw_gate_up, void* dw_down, void* workspace,
                     size_t workspace_bytes, void* stream);

/* The backward of the layer, one kernel per step on `stream`: reverse combine,
 * expert dgrad, reverse dispatch, router gradient, expert weight gradients.  With
 * N = 0 every weight gradient is zero (dx has no rows).
 *   dout : [N][H] BF16;  x, w_router : the forward's inputs;  saved : filled by
 *   moe_forward_train;  wt_* : moe_pack_expert_weights_dgrad's output
 *   dx : [N][H] BF16;  dw_router : [E][H] FP32;  dbias : [E] FP32 or NULL;
 *   dw_gate_up, dw_down : as moe_expert_wgrad, or both NULL to skip them  (out)
 * Needs moe_backward_workspace_bytes() of workspace. */
int moe_backward(const void* dout, const void* x, const void* w_router, const moe_saved_t* saved,
                 const void* wt_gate_up, const uint8_t* wt_gu_scales, const void* wt_down,
                 const uint8_t* wt_d_scales, const moe_shape_t* shape, const moe_params_t* params,
                 void* dx, float* dw_router, float* dbias, void* dw_gate_up, void* dw_down,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Smallest minibatch (in slots) that gives `waves` full waves of GEMM1 tiles of
 * tile_m x tile_n over `compute_sms` SMs when GEMM1 has 2*I output columns
 * ([MoK-2.37x] section 02: a minibatch should form at least two full waves; the
 * pages estimate about 2368 tokens for H=7168, I=2048).  Host-only arithmetic. */
int moe_min_minibatch(int waves, int compute_sms, int tile_m, int tile_n, int I);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
