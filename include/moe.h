/*
 * moe.h - C ABI of the GB300 (sm_103a) routed Mixture-of-Experts layer.
 *
 * The layer (one GPU) runs, in order:
 *   S1 router logits        logits = x . W_r (fp32)
 *   S2 top-k routing        k experts per token, softmax over the selected
 *                           logits, times routed_scale
 *   S3/S4 dispatch          per-expert counts, exclusive offsets and a stable
 *                           token-major permutation, all on the device; x is
 *                           quantised to MXFP8 once per token
 *   S5 grouped GEMM W1      h = a . W1_e, epilogue: SwiGLU, routing weight,
 *                           MXFP8 requantisation of the result y1
 *   S7 grouped GEMM W2      z = y1 . W2_e, bf16
 *   S8 combine              out[t] = sum over the token's k' rows of z
 *   S9 backward             dgrad with a fused dSwiGLU + quantise/transpose
 *                           epilogue, wgrads, router gradient
 * Sources: GC-MoE summary ("GC-MoE: Overlapping Expert-Parallel Token
 * Dispatch with FP8/FP4 Grouped GEMM via CUDA Green Contexts"), Approach:
 * role1 routing-count aggregation and token dispatch in BM blocks, role2
 * W1 with SwiGLU / routing weight / requantisation fused in the epilogue then
 * W2 emitting BF16 fragments, role3 combine; Developer notes: weights are
 * prepacked once by the caller, one workspace instance serialises its calls
 * (Limitations). NVIDIA blog "Boosting MoE training throughput with advanced
 * fusion kernels": SwiGLU formula and the gate/up column repack (section on
 * GLU epilogue fusion), per-group token counts kept in device memory so no
 * host sync is needed (section on removing host-device sync), MXFP8
 * quantisation with a transposed copy fused into the GEMM (section on
 * MXFP8/NVFP4 quantisation fusion), GroupGemm + dActivation +
 * Quantize/Transpose for the backward.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked "device" must point to device memory of the current
 *   device; "host" pointers to host memory. Every device buffer is allocated
 *   and owned by the caller. The library never allocates, frees or
 *   synchronises inside the compute calls below (moe_read_status excepted),
 *   so every compute call can be captured into a CUDA graph.
 * - `stream` is a cudaStream_t passed as void*. All device work is enqueued on
 *   it, in order; NULL means the legacy default stream.
 * - Device pointers must be 16-byte aligned.
 * - bf16 values are passed as their raw 16-bit patterns (uint16_t).
 * - Matrices are row-major. "[R, C]" means R rows of C contiguous elements.
 * - MXFP8 data: E4M3 element codes plus one E8M0 scale code per 32
 *   consecutive elements along the contiguous axis: a matrix [R, C] has scales
 *   [R, C/32]. The block exponent e is the smallest integer with
 *   max|v| <= 448 * 2^e (clamped to [-127, 127]); elements are
 *   round-to-nearest-even E4M3 of v / 2^e.
 * - Notation: T tokens, H hidden, I expert FFN width, E routed experts,
 *   k top-k, S = n_shared shared experts (width I, always on, weight 1),
 *   k' = k + S slots per token, G = E + S expert groups, R = T * k' rows.
 *   Row r of the grouped GEMMs belongs to group e when
 *   offsets[e] <= r < offsets[e+1]; within a group rows keep increasing flat
 *   assignment index a = t * k' + j (slot j < k: the j-th routed expert,
 *   slots k..k'-1: the shared experts).
 * - Errors found on the host (NULL pointers, bad shapes, T > T_max,
 *   misalignment, workspace too small) return a status and enqueue nothing.
 *   Errors only visible on the device (an expert id outside [0, E), a NaN
 *   logit) set bits of a sticky status word inside the workspace and skip the
 *   offending writes; read it with moe_read_status. No kernel traps.
 * - One workspace must not be used by two calls that may run concurrently.
 * - The forward chain's kernels are launched with programmatic dependent
 *   launch: each waits for the kernel before it on the stream to complete
 *   before touching memory, so the stream order the caller sees is the
 *   plain one (a kernel of the caller's enqueued before a call completes
 *   before the call's kernels read or write anything).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* NULL pointer, bad shape or alignment        */
    MOE_ERR_UNSUPPORTED = 2, /* valid request this build does not implement */
    MOE_ERR_WORKSPACE = 3,   /* workspace or output buffer too small         */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed                   */
    MOE_ERR_DEVICE = 5       /* the device status word reports an error      */
} moe_status_t;

/* bits of the device status word */
#define MOE_DEV_BAD_EXPERT_ID 0x1 /* routing id outside [0, E)              */
#define MOE_DEV_NAN_LOGIT 0x2     /* NaN among a token's logits (ranked as -inf) */
#define MOE_DEV_BAD_PACK 0x4      /* packed weight blob header mismatch      */
#define MOE_DEV_TIMEOUT 0x8       /* a kernel gave up waiting on itself      */

enum { MOE_ACT_SWIGLU = 0, MOE_ACT_SWIGLU_CLAMP = 1, MOE_ACT_GEGLU = 2, MOE_ACT_SRELU = 3 };
enum { MOE_WFMT_NVFP4 = 0, MOE_WFMT_MXFP8 = 1, MOE_WFMT_MXFP4 = 2 };
enum { MOE_PACK_FORWARD = 0, MOE_PACK_DGRAD = 1 };

/* Layer configuration (plain data, validated by moe_config_validate).
 * act = MOE_ACT_SWIGLU:        act(g, u) = g * sigmoid(g) * u
 * act = MOE_ACT_SWIGLU_CLAMP:  g' = clamp(g, -act_limit, act_limit),
 *                              u' = clamp(u, -act_limit, act_limit),
 *                              act = g' * sigmoid(act_alpha * g') * u'
 * act = MOE_ACT_GEGLU:         act(g, u) = GELU(g) * u, GELU(v) = v * Phi(v)
 *                              with Phi the standard normal CDF (exact erf
 *                              form). The gated activations are those the
 *                              NVIDIA blog's fused kernels list (kernel
 *                              families: SwiGLU, GeGLU, with clamping).
 * act = MOE_ACT_SRELU:         the non-gated squared ReLU the blog also lists
 *                              (sReLU): W1 has I outputs h (no up half) and
 *                              act = max(h, 0)^2; its backward (MXFP8) takes
 *                              dh = w_row * dY1 * 2 max(h, 0). Without
 *                              w1_bias, not in the fused W1 -> W2 layer.
 * weight_fmt = MOE_WFMT_NVFP4: E2M1 elements, E4M3 scale per 16 along K,
 *                              fp32 scale per (group, matrix)
 * weight_fmt = MOE_WFMT_MXFP8: E4M3 elements, E8M0 scale per 32 along K
 * weight_fmt = MOE_WFMT_MXFP4: E2M1 elements, E8M0 scale per 32 along K (the
 *                              GC-MoE summary's "(1,1,32)" recipe: Limitations;
 *                              the block-scaled FP8 x FP4 MMA: Key
 *                              contributions); forward only */
typedef struct moe_config {
    int32_t H, I, E, k;
    int32_t n_shared;     /* 0 or 1                                          */
    int32_t T_max;        /* largest T any call with this config may pass    */
    int32_t act;
    float act_alpha;
    float act_limit;
    float routed_scale;   /* multiplies the renormalised routing weights     */
    int32_t weight_fmt;
    int32_t max_sms;      /* 0: use every SM; else cap the GEMM grids        */
    int32_t w1_bias;      /* 1: W1 carries a per-group fp32 bias [2I] (gate b,
                           * up c) added before the activation; the
                           * backward returns its gradient db1
                           * (the NVIDIA blog's SwiGLU(xW + b, xV + c) and its
                           * fused bias-vector epilogue, kernel families) */
    int32_t dispatch_sms; /* 0..64. Where moe_layer_fused holds and > 0 (it
                           * must be below the kernel's CTA count), the
                           * layer runs partitioned: that many CTAs (one per
                           * SM) of the fused W1 -> W2 kernel fill the token
                           * ring (the gathered W1 operand rows) group by
                           * group and raise a per-group ring flag; the
                           * other CTAs run W1 -> W2, each waiting (bounded;
                           * MOE_DEV_TIMEOUT) for a group's flag before it
                           * reads the group's rows. 0: the rows are
                           * gathered by a launch of their own first.
                           * Results are the same bits either way. Source:
                           * GC-MoE summary, Approach (a small dispatch
                           * partition fills the token ring and publishes
                           * its counter, the compute partition acquires
                           * ring blocks) and Limitations (the partition
                           * size was not ablated). */
} moe_config_t;

/* Unpacked expert weights (device pointers), one entry per group e < G, in
 * the layout "one row per output feature, reduction axis contiguous":
 *   which = MOE_PACK_FORWARD: W1 rows n < 2I (gate features then up
 *     features; MOE_ACT_SRELU: rows n < I), K = H; W2 rows n < H, K = I.
 *   which = MOE_PACK_DGRAD (MXFP8 only, training): W1 copy with rows h < H,
 *     K = 2I (MOE_ACT_SRELU: K = I); W2 copy with rows i < I, K = H
 *     (quantised along that K).
 * NVFP4: w*_q [G, N, K/2] bytes, element 2i in the low nibble of byte i;
 *        w*_s [G, N, K/16] E4M3 codes; w*_gs [G] fp32.
 * MXFP8: w*_q [G, N, K] E4M3 codes; w*_s [G, N, K/32] E8M0 codes;
 *        w*_gs ignored (may be NULL).
 * MXFP4: w*_q [G, N, K/2] bytes, element 2i in the low nibble of byte i;
 *        w*_s [G, N, K/32] E8M0 codes; w*_gs ignored (may be NULL). */
typedef struct moe_weights_view {
    const uint8_t* w1_q;
    const uint8_t* w1_s;
    const float* w1_gs;
    const uint8_t* w2_q;
    const uint8_t* w2_s;
    const float* w2_gs;
    const float* b1;      /* [G, 2I] fp32 (gate then up); required when
                           * cfg->w1_bias, else ignored (may be NULL)        */
} moe_weights_view_t;

/* Dispatch results (device pointers, caller-owned; see moe_workspace_view
 * for a ready-made set inside a workspace). */
typedef struct moe_dispatch {
    int32_t* topk_ids;  /* [T, k]   expert ids, best first                    */
    float* topk_w;      /* [T, k]   routing weights                           */
    int32_t* counts;    /* [G]      rows per group                            */
    int32_t* offsets;   /* [G + 1]  exclusive prefix sum of counts            */
    int32_t* perm_src;  /* [R]      row r <- flat assignment t*k' + j         */
    int32_t* inv;       /* [R]      flat assignment -> row                    */
    float* w_row;       /* [R]      routing weight of row r (1 for shared)    */
    uint8_t* xq;        /* [T, H]   MXFP8 codes of x (one copy per token)     */
    uint8_t* xs;        /* [T, H/32] E8M0 scales of x                         */
} moe_dispatch_t;

/* Tensors the training forward saves for moe_layer_backward (device,
 * caller-owned; sizes from moe_train_sizes). Pad rows: every group's rows are
 * padded with zero rows to a multiple of 128; poff[e] is the padded offset. */
typedef struct moe_train_save {
    uint16_t* h;        /* [R, 2I] bf16 W1 output before the activation
                           ([R, I] for MOE_ACT_SRELU)                         */
    uint8_t* y1t_q;     /* [I, R_pad] MXFP8 of y (activation x routing weight)
                           quantised along the padded row axis               */
    uint8_t* y1t_s;     /* [R_pad/128, I] 32-bit words of its E8M0 scales:
                           byte j of word [w, i] is the scale of feature i,
                           padded rows 32(4w+j) .. 32(4w+j)+31                */
    uint8_t* at_q;      /* [H, R_pad] MXFP8 of the gathered x rows, quantised
                           along the padded row axis                          */
    uint8_t* at_s;      /* [R_pad/128, H] words of its scales, as y1t_s       */
    int32_t* poff;      /* [G + 1] padded row offsets                         */
    float* amax;        /* nullable [2]: the NVFP4 training recipe's amaxes of
                           y (activation x routing weight): [0] = max |y|,
                           [1] = max |(H16 / 4) . block| over the Hadamard
                           rotations of y's transpose, blocks of 16 rows of
                           one expert (zero-padded), H16 Sylvester's Hadamard
                           matrix. Source: NVIDIA blog, section on fusing
                           MXFP8/NVFP4 quantisation (per-tensor amax for the
                           forward, amax of the transposed Hadamard-rotated
                           output for the backward).                        */
} moe_train_save_t;

/* Pointers into a workspace (all device). */
typedef struct moe_ws_view {
    float* logits;      /* [T_max, E]                                         */
    moe_dispatch_t d;   /* dispatch results                                   */
    uint8_t* y1_q;      /* [R_max, I] MXFP8 codes of y1                       */
    uint8_t* y1_s;      /* [R_max, I/32]                                      */
    uint16_t* z;        /* [R_max, H] bf16 W2 output                          */
    int32_t* status;    /* sticky device status word                          */
} moe_ws_view_t;

/* ---- configuration, sizes ---------------------------------------------- */

/* Host only. MOE_OK if the config is supported: H, I multiples of 64,
 * 1 <= k <= E, k' <= 32, G <= 2048, n_shared in {0, 1}, T_max >= 0.
 * Source: GC-MoE summary, Limitations (the Appendix A shape constraints:
 * top-k plus the shared slot within 32, at most 2048 experts); the H / I
 * multiples here follow this library's 64-wide K chunks, not the pages. */
moe_status_t moe_config_validate(const moe_config_t* cfg);

/* Host only. Bytes of workspace for calls with T <= T_max (cfg->T_max).
 * Source: GC-MoE summary, Limitations (one workspace instance per operator;
 * calls that share it are serialised). */
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Host only. Carves the named buffers out of a workspace of at least
 * moe_workspace_size bytes at device address ws (no device access). The
 * pages have no counterpart: an inspection aid of this library. */
moe_status_t moe_workspace_view(const moe_config_t* cfg, void* ws, moe_ws_view_t* view);

/* Host only. Bytes of the packed weight blob for `which`. Source: GC-MoE
 * summary, Developer notes (weights converted once into the prepacked
 * form). */
moe_status_t moe_packed_weights_size(const moe_config_t* cfg, int which, size_t* bytes);

/* Host only. Sizes of the training save buffers for T tokens: R_pad upper
 * bound (rows of the padded transposed copies). Source: NVIDIA blog, section
 * on fusing MXFP8/NVFP4 quantisation (the transposed MXFP8 copies kept for
 * the backward). */
moe_status_t moe_train_sizes(const moe_config_t* cfg, int T, int64_t* r_pad_max);

/* ---- S0 weight prepack (once, at load time) ------------------------------ */

/* Rearranges the unpacked weights `src` into the opaque blob `dst` (device,
 * dst_bytes >= moe_packed_weights_size) used by the grouped GEMMs: per group,
 * tiles of 128 output features (W1 tiles hold 64 gate and the matching 64 up
 * features, so SwiGLU completes inside one tile), each tile stored as
 * contiguous 64-wide K chunks carrying their scales. Source: GC-MoE summary,
 * Developer notes (K128 prepacked FP4 weights, converted once by the caller)
 * and the NVIDIA blog's gate/up column repack done at checkpoint load. */
moe_status_t moe_prepack_weights(const moe_config_t* cfg, const moe_weights_view_t* src, int which,
                                 void* dst, size_t dst_bytes, void* stream);

/* Debug export of the packed layout (tests): writes matrix `mat` (1 = W1 or
 * its dgrad copy, 2 = W2 or its dgrad copy) of every group of the blob
 * `packed` (device, from moe_prepack_weights with the same cfg and `which`)
 * back to the plain layout of moe_weights_view_t: NVFP4 q [G, N, K/2],
 * s [G, N, K/16]; MXFP8 q [G, N, K], s [G, N, K/32] (device, caller-owned).
 * Prepacking followed by this export returns the source bytes exactly.
 * Not on the hot path; enqueued on stream like the compute calls. */
moe_status_t moe_debug_unpack_weights(const moe_config_t* cfg, const void* packed, int which, int mat,
                                      uint8_t* q, uint8_t* s, void* stream);

/* Runs, in one thread, the bounded wait the fused layer's W2 tiles use on
 * their group's ready flag (flag: device int32, waited on until non-zero),
 * giving up after limit_cycles SM clock cycles (> 0) and then setting
 * MOE_DEV_TIMEOUT in the workspace status word. For tests of the timeout
 * path: a flag that nothing sets must end in MOE_DEV_TIMEOUT with the
 * context still usable. The pages have no counterpart. */
moe_status_t moe_debug_flag_wait(const moe_config_t* cfg, const int32_t* flag, int64_t limit_cycles, void* ws,
                                 void* stream);

/* ---- forward steps ------------------------------------------------------ */

/* S1. logits [T, E] fp32 (device) = x [T, H] bf16 (device) . W_r [H, E] fp32
 * (device), fp32 accumulation. ws: the workspace (holds split partials).
 * Source: GC-MoE summary, Approach (role1 starts from the tokens' routing);
 * the pages take the logits as given, and the router product x . W_r is the
 * plainest step that produces them from the workloads' router weights. */
moe_status_t moe_router_logits(const moe_config_t* cfg, const uint16_t* x, const float* W_r, int T,
                               float* logits, void* ws, void* stream);

/* S1 without a workspace, for callers that cannot allocate device memory
 * where they need logits (an allocator-free region, a host that hands out no
 * device buffers, a path where cudaMalloc's implicit synchronisation is not
 * allowed). The pages have no counterpart: this is a convenience of this
 * library. Same result as moe_router_logits, bit for bit; the split partial
 * sums live in one static 4 MiB device array that every GPU loading the
 * library holds until process exit. A call whose partials would exceed it
 * (split count x T x E > 2^20 floats) returns MOE_ERR_WORKSPACE and enqueues
 * nothing. Nothing is allocated or freed. All calls on a device share the
 * array and leave their partials in it (each call overwrites what it reads,
 * so nothing needs clearing); calls whose kernels may overlap on the GPU race
 * on it and must be serialised. The array's device address is looked up
 * the first time a call is made in a given CUDA context (the primary
 * context, a context the caller created, or one converted from a green
 * context) and cached under that context's unique id, so each context, and
 * the context that replaces the primary one after cudaDeviceReset, gets its
 * own lookup; make the first call in each context before any stream capture
 * in it. x [T, H] bf16, W_r [H, E] fp32, logits [T, E]
 * fp32, all device. */
moe_status_t moe_router_logits_noalloc(const moe_config_t* cfg, const uint16_t* x, const float* W_r, int T,
                                       float* logits, void* stream);

/* S2-S4. From logits [T, E] fp32 (device): top-k ids and weights, counts,
 * offsets, permutation, inverse, row weights, and the MXFP8 copy of x
 * [T, H] bf16 (device). Outputs in *d (device buffers). Bit-exact and
 * deterministic: ties in the logits go to the lower expert id; rows of a
 * group keep increasing t*k' + j. T = 0 writes zero counts and offsets.
 * Source: GC-MoE summary, Approach (role1 aggregates the routing counts and
 * places the tokens into expert blocks); NVIDIA blog, section on removing
 * host-device sync (per-group counts stay in device memory). */
moe_status_t moe_route_dispatch(const moe_config_t* cfg, const float* logits, const uint16_t* x, int T,
                                const moe_dispatch_t* d, void* ws, void* stream);

/* S2 alone: top-k ids [T, k] and weights [T, k] from logits (device).
 * Source: GC-MoE summary, Approach (role1's top-k routing). */
moe_status_t moe_route_topk(const moe_config_t* cfg, const float* logits, int T, int32_t* topk_ids,
                            float* topk_w, void* ws, void* stream);

/* S3-S4 alone: dispatch from given top-k ids/weights (device) and x.
 * d->topk_ids / d->topk_w are read, the other fields of *d written.
 * Source: as moe_route_dispatch (device-side counts and token placement). */
moe_status_t moe_dispatch(const moe_config_t* cfg, const uint16_t* x, int T, const moe_dispatch_t* d,
                          void* ws, void* stream);

/* S5-S6. Grouped W1 over the dispatched rows with the fused epilogue
 * y1 = MXFP8(w_row * act(h[:, :I], h[:, I:])); y1_q [R, I], y1_s [R, I/32]
 * (device). save (nullable): training tensors h, y1t, at, poff.
 * Source: GC-MoE summary, Approach and Key contributions (W1's epilogue
 * applies SwiGLU, the routing weight and the FP8 requantisation); NVIDIA
 * blog, GLU epilogue section (gate and up columns of one tile meet in the
 * epilogue) and MXFP8 section (the transposed copy). */
moe_status_t moe_grouped_gemm_w1_swiglu_quant(const moe_config_t* cfg, const moe_dispatch_t* d, int T,
                                              const void* packed_w, uint8_t* y1_q, uint8_t* y1_s,
                                              const moe_train_save_t* save, void* ws, void* stream);

/* S7. Grouped W2: z [R, H] bf16 (device) = y1 . W2_e, fp32 accumulation.
 * Source: GC-MoE summary, Approach (role2's W2 writes BF16 fragments). */
moe_status_t moe_grouped_gemm_w2(const moe_config_t* cfg, const moe_dispatch_t* d, int T,
                                 const uint8_t* y1_q, const uint8_t* y1_s, const void* packed_w,
                                 uint16_t* z, void* ws, void* stream);

/* S8. out [T, H] bf16 (device): out[t] = bf16(sum_j c_j * z[inv[t*k'+j]])
 * summed in fp32 in slot order j = 0..k'-1, c_j = topk_w[t, j] for routed
 * slots and 1 for shared slots when topk_w is non-NULL, else c_j = 1 (the
 * routing weight was applied in the W1 epilogue). Source: GC-MoE summary,
 * Approach (role3 combines the BF16 fragments of each token). */
moe_status_t moe_combine(const moe_config_t* cfg, const uint16_t* z, const int32_t* inv, const float* topk_w,
                         int T, uint16_t* out, void* stream);

/* Whole forward. Exactly one of W_r (router weights [H, E] fp32) and
 * logits_in ([T, E] fp32) is non-NULL. out [T, H] bf16. save nullable
 * (training). Intermediates live in ws (see moe_workspace_view). Source:
 * GC-MoE summary, Approach (role1 dispatch, role2 W1 then W2, role3
 * combine); NVIDIA blog, section on removing host-device sync (the whole
 * layer captures into one CUDA graph). */
moe_status_t moe_layer_forward(const moe_config_t* cfg, const uint16_t* x, const float* W_r,
                               const float* logits_in, int T, const void* packed_w, uint16_t* out,
                               const moe_train_save_t* save, void* ws, void* stream);

/* *fused (host) = 1 when moe_layer_forward with this config and T (and no
 * training save) runs W1, its epilogue and W2 as one persistent kernel:
 * NVFP4 weights, I <= 2048, at most 2 token rows per group on average. The
 * last W1 tile of each group to finish converts the group's y1 rows into
 * W2's operand and sets a flag that the group's W2 tiles wait for (bounded:
 * MOE_DEV_TIMEOUT). Otherwise 0: W1, the epilogue kernel and W2 run as
 * separate launches. Both give the same bits; the step-wise calls split K
 * the same way at these sizes. Source: GC-MoE summary, Key contributions
 * (the per-block W1-completion tracking that lets W2 start without a
 * separate launch); FlashDMoE abstract (one persistent kernel for the
 * layer). */
moe_status_t moe_layer_fused(const moe_config_t* cfg, int T, int32_t* fused);

/* ---- backward (MXFP8 weights, n_shared = 0) ------------------------------ */

/* Gradients of L = sum(dout * out) for the forward that filled ws and save
 * with the same T: dx [T, H] bf16 (expert path only), dW1 [E, H, 2I] bf16 in
 * the logical W1 layout (gate columns then up columns; [E, H, I] for
 * MOE_ACT_SRELU), dW2 [E, I, H] bf16,
 * dlogits [T, E] fp32; with cfg->w1_bias, db1 [E, 2I] fp32 (gate b then up
 * c: the sum of dh over each group's rows; NULL otherwise, else
 * MOE_ERR_INVALID_ARG). packed_w_dgrad: moe_prepack_weights(..., DGRAD, ...).
 * The router's own dense GEMM gradients (dlogits . W_r^T, x^T . dlogits) are
 * left to the caller. Source: NVIDIA blog, kernel families (GroupGemm +
 * dActivation + Quantize/Transpose) and the MXFP8 section (weight gradients
 * from the transposed MXFP8 copies). */
moe_status_t moe_layer_backward(const moe_config_t* cfg, const uint16_t* dout, const uint16_t* x, int T,
                                const moe_train_save_t* save, const void* packed_w_dgrad, uint16_t* dx,
                                uint16_t* dW1, uint16_t* dW2, float* dlogits, float* db1, void* ws,
                                void* stream);

/* ---- status --------------------------------------------------------------- */

/* Synchronises `stream`, copies the workspace status word to *out (host) and
 * clears it. Not for use inside graph capture. The pages have no
 * counterpart: device-side error reporting of this library. */
moe_status_t moe_read_status(const moe_config_t* cfg, void* ws, int32_t* out, void* stream);

/* Clears the workspace status word (enqueued on stream; capturable). The
 * pages have no counterpart. */
moe_status_t moe_clear_status(const moe_config_t* cfg, void* ws, void* stream);

/* Static description of a status code. The pages have no counterpart. */
const char* moe_status_string(moe_status_t s);

/* Number of kernels the last host call enqueued (for launch accounting).
 * The pages have no counterpart. */
int moe_last_launch_count(void);

/* Optional phase timing for moe_layer_forward, per calling thread. With
 * `events` non-NULL (MOE_N_PHASE_EVENTS cudaEvent_t handles created by the
 * caller), each later moe_layer_forward on this thread records, on its
 * stream: [0] at entry, [1] after routing, dispatch and the gather of the
 * W1 operand rows, [2] after the W1 grouped-GEMM kernel, [3] after the W1
 * epilogue, [4] after the W2 grouped-GEMM kernel, [5] after the combine.
 * In the fused layer (moe_layer_fused) [2], [3] and [4] are recorded one
 * after the other behind the one W1 -> W2 kernel.
 * NULL switches it off. Host only; the events must outlive the calls that
 * record them. A call made while its stream is being captured into a CUDA
 * graph records them as event-record nodes, so every replay of that graph
 * records them again. The pages have no counterpart: a measurement aid. */
#define MOE_N_PHASE_EVENTS 6
moe_status_t moe_set_phase_events(void* const* events);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
