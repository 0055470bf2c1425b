/*
 * moe_gb300.h -- C ABI of a single-GPU (GB300, sm_103a) mixture-of-experts layer:
 * router GEMM -> top-k -> per-expert histogram / prefix sum / token<->slot permutation ->
 * permute -> grouped SwiGLU expert GEMMs -> weighted combine (+ optional shared expert),
 * and the backward pass of all of it.
 *
 * What the layer is.  "Megatron-Bridge 深度剖析：MoE 大模型训练加速的工程之道":
 *   §Motivation -- a DeepSeek-style layer: 128 SwiGLU experts (gate_proj, up_proj,
 *     down_proj), top-6 sigmoid routing;
 *   §Expert Parallel 基础, workflow figure -- Step 1 the router picks top-k experts per token;
 *     Step 2 tokens are regrouped by expert (an all-to-all across GPUs; on one GPU a local
 *     permutation); Step 3 the experts run and the results go back to token order;
 *   §计算融合 / Grouped GEMM -- all experts' GEMMs in one launch over ragged token counts,
 *     expert weights stored contiguously (weight0, weight1, ...);
 *   §Permute Fusion -- the permutation is a memory copy that groups each expert's tokens;
 *   §Shared Expert Overlap -- a shared expert every token goes through, added to the routed
 *     output;
 *   §权重映射策略 (GatedMLPMapping) -- fc1 = [gate_proj; up_proj], shape (2*ffn, hidden).
 * "Add Megatron-Core MTP training for Qwen3.5 MoE" (What's in it) -- the shared-expert gate.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller, unless a parameter says otherwise.
 *     The library allocates no device memory in any call below; scratch space comes from the
 *     caller's workspace, sized by moe_workspace_bytes().
 *   - Every pointer must be 16-byte aligned (MOE_ERR_ALIGNMENT otherwise).
 *   - All work is enqueued on `stream` (a cudaStream_t passed as void*, NULL = legacy default
 *     stream), and for the layer calls also on the caller's optional side stream
 *     (moe_side_stream), and is asynchronous with respect to the host.  The library owns no
 *     stream, event or global switch, and calls keep no state between them; two calls may run
 *     concurrently on different streams if their buffers, workspaces and side streams are
 *     distinct.  (moe_route_topk_noalloc is the one exception: its scratch is shared; see it.)
 *   - Row-major dense layouts; T tokens, d = d_model, E experts, k experts per token,
 *     f = expert ffn width, f_s = shared expert ffn width, N = T*k routed rows.
 *   - Activations and weights are in cfg->dtype (bf16 or fp32).  Router logits, gates and
 *     all weight gradients are fp32.  Weight gradients are overwritten, not accumulated.
 *   - Return value: MOE_OK (0) or a negative moe_status.  Argument errors are detected on the
 *     host before anything is enqueued.  MOE_ERR_CUDA means a launch failed; the message is
 *     in moe_last_error().  A kernel that detects an inconsistency at run time (a bounded wait
 *     that ran out, an index out of range) records it in a device error word that
 *     moe_check_device_error() reads.
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
  MOE_ERR_INVALID_ARG = -1,   /* null where a buffer is required, negative size, k > E ... */
  MOE_ERR_UNSUPPORTED = -2,   /* E > 256, k > 8, d or f not a multiple of 8, ...           */
  MOE_ERR_WORKSPACE = -3,     /* workspace null or smaller than moe_workspace_bytes()      */
  MOE_ERR_ALIGNMENT = -4,     /* a pointer is not 16-byte aligned                          */
  MOE_ERR_CUDA = -5,          /* a CUDA call or launch failed (see moe_last_error())       */
  MOE_ERR_DEVICE_CHECK = -6   /* a kernel reported a run-time inconsistency                */
} moe_status;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 };
/* What the router bias b_r [E] does (cfg->bias_mode). */
enum {
  MOE_BIAS_LOGIT = 0,   /* added to the logits: moves the selection and the gates alike       */
  MOE_BIAS_SELECT = 1   /* expert-bias correction: added to the scores (softmax over E, or
                           sigmoid) for the selection only; the gates never see it            */
};

/* Limits checked by every entry point. */
enum { MOE_MAX_EXPERTS = 256, MOE_MAX_TOPK = 8 };

/* Layer configuration, passed by pointer to every call.
 *   score_fn   MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID ("moe_router_score_function").
 *   renorm     1: the k selected gates are divided by their sum (softmax+renorm equals the
 *              softmax over the k selected logits); 0: raw softmax-over-E / sigmoid scores.
 *   f_shared   0: no shared expert.
 *   shared_gate 1: the shared expert's output is scaled by sigmoid(w_sg . x_t).
 *   dtype      MOE_DTYPE_BF16 (tensor-core path, fp32 accumulation) or MOE_DTYPE_F32
 *              (fp32 CUDA-core path, for exact-tolerance checks).
 *   bias_mode  MOE_BIAS_LOGIT or MOE_BIAS_SELECT (the expert-bias correction of sigmoid
 *              routing, "moe_router_enable_expert_bias"); see moe_route_topk.
 *   aux_coeff  coefficient of the load-balancing loss ("moe_aux_loss_coeff", 1e-4 on the
 *              pages); 0 disables it.  Must be finite and >= 0.  See moe_router_aux_loss. */
typedef struct moe_cfg {
  int32_t T, d, E, k, f, f_shared;
  int32_t score_fn;
  int32_t renorm;
  int32_t shared_gate;
  int32_t dtype;
  int32_t bias_mode;
  float aux_coeff;
} moe_cfg;

/* Which call a workspace is sized for. */
enum {
  MOE_WS_ROUTE = 0,       /* moe_route_topk                           */
  MOE_WS_FFN_FWD = 1,     /* moe_grouped_swiglu_fwd                   */
  MOE_WS_FFN_BWD = 2,     /* moe_grouped_swiglu_bwd                   */
  MOE_WS_LAYER_FWD = 3,   /* moe_layer_fwd                            */
  MOE_WS_LAYER_BWD = 4,   /* moe_layer_bwd                            */
  MOE_WS_FFN_BWD_FP8 = 5, /* moe_grouped_swiglu_bwd_fp8               */
  MOE_WS_LAYER_BWD_FP8 = 6, /* moe_layer_bwd_fp8                      */
  MOE_WS_WGRAD_MXFP8 = 7  /* moe_grouped_swiglu_wgrad_mxfp8; moe_mxfp8_dgrad.wgrad_ws */
};

/* Bytes of caller workspace the call `which` needs for cfg (0 if cfg is invalid). */
size_t moe_workspace_bytes(const moe_cfg* cfg, int which);

/* Router + top-k + routing maps (one GPU's stand-in for the expert-parallel dispatch plan).
 * "Megatron-Bridge 深度剖析", §Expert Parallel 基础 (Step 1, Router(x) -> TopK scores) and
 * §核心模块架构 (moe_router_topk, moe_router_score_function).
 *   x [T,d], W_r [E,d] (dtype); b_r [E] fp32 or NULL: with MOE_BIAS_LOGIT added to the
 *     logits; with MOE_BIAS_SELECT the expert bias of the selection (below).
 *   logits_in [T,E] fp32 or NULL: if set, the router GEMM is skipped and these logits are
 *     routed (a MOE_BIAS_LOGIT b_r is then ignored; a MOE_BIAS_SELECT b_r still applies).
 *   logits_out [T,E] fp32 or NULL: receives the router logits (x.W_r^T, + b_r with
 *     MOE_BIAS_LOGIT, fp32).
 *   Outputs: idx [T,k] int32 -- selected experts, by descending key, equal keys -> lower
 *     expert index first; the key is the fp32 logit, or with MOE_BIAS_SELECT the fp32 score
 *     plus b_r[e] (score = softmax over all E, or sigmoid, of the fp32 logits: "Megatron-
 *     Bridge 深度剖析", §Nemotron-3-Nano 配置, sigmoid routing with expert-bias correction as
 *     in DeepSeek V3); gate [T,k] fp32 -- combine weights (softmax / sigmoid, renorm per
 *     cfg); counts [E], offsets [E+1] int32 (offsets[0]=0, offsets[E]=N); slot_of_pair [T,k],
 *     token_of_slot [N] int32: pair (t,j) sits in row slot_of_pair[t,j] of the expert-sorted
 *     layout; inside one expert's rows the tokens ascend.
 *   Selection is made on fp32 keys and is bit-for-bit deterministic for given logits. */
int moe_route_topk(const moe_cfg* cfg, const void* x, const void* W_r, const float* b_r,
                   const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                   int32_t* counts, int32_t* offsets, int32_t* slot_of_pair,
                   int32_t* token_of_slot, void* ws, size_t ws_bytes, void* stream);

/* Routing without a workspace.  The pages have no counterpart: this entry point serves callers
 * that cannot allocate device memory and cannot lend the library a workspace (for example a
 * runtime that owns all device memory through its own arena, or a plugin interface that passes
 * only input and output tensors).  Arguments, outputs and errors are those of moe_route_topk,
 * without ws / ws_bytes, and with one more requirement: logits_in or logits_out must be set
 * (the router logits need a caller buffer; MOE_ERR_INVALID_ARG otherwise).
 *   Scratch: a fixed 128 KB array inside the library (the expert histogram: one row of E16 bytes
 *   per 128 tokens, E16 = E rounded up to a power of two of at least 16), held on every GPU that
 *   loads it until the process exits.  ceil(T/128) * E16 must not exceed 131072 (e.g. T = 65536
 *   tokens with E = 256, or T = 131072 with E = 128); larger calls return MOE_ERR_UNSUPPORTED.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress),
 *   and so does the first call after the device's context was replaced (cudaDeviceReset): make
 *   those calls before any stream capture.
 *   All calls share the one array and every call overwrites what it reads, so nothing needs
 *   clearing; but calls whose GPU work overlaps (different streams or host threads without
 *   ordering between them) race on it and give wrong results: order them.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
int moe_route_topk_noalloc(const moe_cfg* cfg, const void* x, const void* W_r, const float* b_r,
                           const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                           int32_t* counts, int32_t* offsets, int32_t* slot_of_pair,
                           int32_t* token_of_slot, void* stream);

/* Permute: x_perm[s] = x[token_of_slot[s]] for s < N.  "Megatron-Bridge 深度剖析",
 * §Permute Fusion (tokens regrouped by expert: one memory copy).
 *   x [T,d], x_perm [N,d] (dtype); slot_of_pair [T,k] from moe_route_topk. */
int moe_permute(const moe_cfg* cfg, const void* x, const int32_t* slot_of_pair, void* x_perm,
                void* stream);

/* Grouped SwiGLU experts, forward.  "Megatron-Bridge 深度剖析", §计算融合 / Grouped GEMM and
 * §权重映射策略 (GatedMLPMapping: fc1 = [gate; up]).  For every expert e and every row s in
 * [offsets[e], offsets[e+1]):
 *   [a | u] = x_perm[s] . W1[e]^T,  h[s] = SiLU(a) * u,  y_perm[s] = h[s] . W2[e]^T.
 *   x_perm [N,d]; W1 [E,2f,d] (rows 0..f-1 gate, f..2f-1 up); W2 [E,d,f]; offsets [E+1].
 *   Outputs (dtype): h [N,f]; act [N,2f] = [a | u] (pre-activations, kept for the backward;
 *   may be NULL if no backward follows); y_perm [N,d].
 *   The number of rows N is cfg->T*cfg->k (offsets[E] must equal it). */
int moe_grouped_swiglu_fwd(const moe_cfg* cfg, const void* x_perm, const int32_t* offsets,
                           const void* W1, const void* W2, void* h, void* act, void* y_perm,
                           void* ws, size_t ws_bytes, void* stream);

/* Grouped SwiGLU experts, backward (chain rule of moe_grouped_swiglu_fwd).
 *   Inputs: x_perm, offsets, W1, W2, act, h as in the forward; dy_perm [N,d] (dtype).
 *   Outputs: dx_perm [N,d] (dtype); dW1 [E,2f,d], dW2 [E,d,f] fp32 (experts with no rows
 *   get zeros).  The gradient of [a | u] is formed in the workspace. */
int moe_grouped_swiglu_bwd(const moe_cfg* cfg, const void* x_perm, const int32_t* offsets,
                           const void* W1, const void* W2, const void* act, const void* h,
                           const void* dy_perm, void* dx_perm, float* dW1, float* dW2,
                           void* ws, size_t ws_bytes, void* stream);

/* The same two calls with the permutation folded into the operand loads ("Megatron-Bridge
 * 深度剖析", §Permute Fusion): instead of x_perm they take x [T,d] and token_of_slot [N] (from
 * moe_route_topk) and gather row token_of_slot[s] of x wherever x_perm[s] would be read (fc1's
 * A operand and fc1's weight-gradient operand), with TMA tile::gather4 copies.  Results are
 * bit-identical to moe_permute followed by the x_perm calls.  bf16 only (MOE_ERR_UNSUPPORTED
 * for fp32); a token index outside [0, T) is recorded in the device error word and row 0 is
 * read instead.  Slower than the explicit permute on GB300 (the gathered copies move 512 bytes
 * each): kept for callers that cannot hold x_perm's N*d elements. */
int moe_grouped_swiglu_fwd_gathered(const moe_cfg* cfg, const void* x,
                                    const int32_t* token_of_slot, const int32_t* offsets,
                                    const void* W1, const void* W2, void* h, void* act,
                                    void* y_perm, void* ws, size_t ws_bytes, void* stream);
int moe_grouped_swiglu_bwd_gathered(const moe_cfg* cfg, const void* x,
                                    const int32_t* token_of_slot, const int32_t* offsets,
                                    const void* W1, const void* W2, const void* act,
                                    const void* h, const void* dy_perm, void* dx_perm,
                                    float* dW1, float* dW2, void* ws, size_t ws_bytes,
                                    void* stream);

/* E4M3 tensorwise quantisation ("Megatron-Bridge 深度剖析", §FP8 训练: FP8 E4M3 with the
 * "tensorwise" scaling recipe; the pages give no formula, this is the plain reading).  x holds
 * `groups` consecutive tensors of elems_per_group bf16 values each (an activation matrix is one
 * group; W1 [E,2f,d] is E groups of 2f*d).  Per group:
 *   amax[g] = max |x|;  q = E4M3(x * (448 / amax))  (fp32 quotient and product, round to nearest
 *   even, saturating to +-448; the sign of zero kept);  scale[g] = amax / 448 (dequantisation).
 * amax = 0 gives inv = scale = 1.  q: uint8 codes, same layout as x; scale, amax: fp32 [groups]
 * (amax is scratch that also returns the maxima).  elems_per_group must be a multiple of 16.
 * No moe_cfg: the call only needs the sizes. */
int moe_quantize_e4m3(const void* x, int64_t elems_per_group, int32_t groups, uint8_t* q,
                      float* scale, float* amax, void* stream);

/* Permute + E4M3 quantisation in one pass: amax over x [T,d] (every token is routed k >= 1
 * times, so it is the permuted matrix's amax too), then x_perm_q[slot_of_pair[t,j]] =
 * E4M3(x[t] * (448 / amax)) as moe_quantize_e4m3 would give for the permuted bf16 matrix;
 * x_scale[0] = amax / 448, x_amax[0] = amax.  bf16 x, d a multiple of 16. */
int moe_permute_quantize_e4m3(const moe_cfg* cfg, const void* x, const int32_t* slot_of_pair,
                              uint8_t* x_perm_q, float* x_scale, float* x_amax, void* stream);

/* Grouped SwiGLU forward on E4M3 operands ("Megatron-Bridge 深度剖析", §FP8 训练: FP8 doubles the
 * tensor-core rate and halves the bytes of the 128-expert grouped GEMM).  For rows s of expert e:
 *   [a | u] = x_scale * W1_scale[e] * (dec(x_perm_q[s]) . dec(W1_q[e])^T)   (fp32 accumulation)
 *   h = SiLU(a) * u  (bf16, and [a | u] in act unless NULL);  h is quantised as one tensor
 *   (as moe_quantize_e4m3 does, with its amax taken in fc1's epilogue) into h_q, h_scale[0]
 *   (h_amax[0]: its amax);
 *   y_perm[s] = h_scale * W2_scale[e] * (dec(h_q[s]) . dec(W2_q[e])^T)  (bf16).
 * x_perm_q [N,d], W1_q [E,2f,d], W2_q [E,d,f]: uint8 E4M3 codes from moe_quantize_e4m3 (W1_q and
 * W2_q with E groups, x_perm_q with one); scales fp32 device values.  d and f must be multiples
 * of 16; cfg->dtype must be MOE_DTYPE_BF16.  moe_grouped_swiglu_bwd_fp8 is its backward. */
int moe_grouped_swiglu_fwd_fp8(const moe_cfg* cfg, const uint8_t* x_perm_q, const float* x_scale,
                               const int32_t* offsets, const uint8_t* W1_q, const float* W1_scale,
                               const uint8_t* W2_q, const float* W2_scale, void* h, void* act,
                               uint8_t* h_q, float* h_scale, float* h_amax, void* y_perm,
                               void* stream);

/* Grouped SwiGLU backward on E4M3 operands ("Megatron-Bridge 深度剖析", §FP8 训练: E4M3 with
 * tensorwise scaling, weight gradients in FP8 as well).  Takes the forward's quantised tensors
 * (x_perm_q, h_q with their scales; W1_q, W2_q with one scale per expert) and its bf16 [a | u]
 * (act [N,2f]); for rows s of expert e:
 *   dy_perm [N,d] (bf16) is quantised as one tensor (moe_quantize_e4m3) into dy_q, dy_scale[0],
 *     dy_amax[0];
 *   dh[s] = dy_scale * W2_scale[e] * (dec(dy_q[s]) . dec(W2_q[e]))          (fp32 accumulation)
 *   dH1[s] = [da | du] = SwiGLU backward of dh[s] at act[s] (bf16 [N,2f], as moe_grouped_swiglu_bwd);
 *     dH1 is quantised as one tensor (its amax taken in the same epilogue, dH1_amax[0]) into
 *     dH1_q [N,2f], dH1_scale[0];
 *   dx_perm[s] = dH1_scale * W1_scale[e] * (dec(dH1_q[s]) . dec(W1_q[e]))   (bf16 [N,d])
 *   dW1[e] = dH1_scale * x_scale * dec(dH1_q[rows of e])^T . dec(x_perm_q[rows of e])  (fp32)
 *   dW2[e] = dy_scale * h_scale * dec(dy_q[rows of e])^T . dec(h_q[rows of e])         (fp32)
 * The weights' codes are read in their stored [E,2f,d] / [E,d,f] layouts (no transposed copies);
 * experts without rows get zero weight gradients.  dy_q [N,d] and dH1_q are caller buffers of
 * uint8; scales and amaxes one fp32 each.  Workspace MOE_WS_FFN_BWD_FP8.  d and f multiples of
 * 16; cfg->dtype MOE_DTYPE_BF16. */
int moe_grouped_swiglu_bwd_fp8(const moe_cfg* cfg, const uint8_t* x_perm_q, const float* x_scale,
                               const int32_t* offsets, const uint8_t* W1_q, const float* W1_scale,
                               const uint8_t* W2_q, const float* W2_scale, const void* act,
                               const uint8_t* h_q, const float* h_scale, const void* dy_perm,
                               uint8_t* dy_q, float* dy_scale, float* dy_amax, void* dH1,
                               uint8_t* dH1_q, float* dH1_scale, float* dH1_amax, void* dx_perm,
                               float* dW1, float* dW2, void* ws, size_t ws_bytes, void* stream);

/* MXFP8: microscaled FP8 ("Megatron-Bridge 深度剖析", §新硬件适配: Blackwell's microscaling FP8,
 * with scale factors finer grained than per tensor; element and scale formats are the OCP
 * Microscaling ones).  A block is 32 consecutive elements along a product's reduction dimension:
 *   e = floor(log2(max |x| over the block)) - 8, clamped to [-127, 127] (-127 for an all-zero
 *   block); code = E4M3(x * 2^-e) (round to nearest even, saturating at +-448); scale byte
 *   (E8M0) = e + 127, so x ~ E4M3value(code) * 2^(byte - 127).
 * The GEMMs read block scales in packed layouts sized by moe_mxfp8_scale_bytes:
 *   MOE_MX_SCALES_X / _H: the permuted activations x_perm [N,d] / h [N,f], in 512-byte chunks of
 *     128 rows x 128 elements.  Chunk (mt, kc) starts at (mt * ceil(K/128) + kc) * 512, where the
 *     row tile mt of slot s (expert e, rows [off_e, off_e+1)) is sum_{e'<e} ceil(n_e'/128) +
 *     (s - off_e) / 128, and the scale of the tile's row r, block j (of the chunk's four) is byte
 *     (r % 32) * 16 + (r / 32) * 4 + j.  Rows past an expert's end are left unwritten; blocks past K
 *     are 127.
 *   MOE_MX_SCALES_W1 / _W2: each expert's weights, per output tile of 192 B-rows (fc1 tile t: gate
 *     rows 96t..96t+95 then up rows f+96t..f+96t+95; fc2 tile t: rows 192t..192t+191) and per
 *     128-element K chunk kc, two such chunks (tile rows 0..127, 128..255) at
 *     ((e * tiles + t) * ceil(K/128) + kc) * 1024; rows and blocks past the weight are 127. */
enum { MOE_MX_SCALES_X = 0, MOE_MX_SCALES_H = 1, MOE_MX_SCALES_W1 = 2, MOE_MX_SCALES_W2 = 3,
       MOE_MX_SCALES_DH1 = 4, MOE_MX_SCALES_W1C = 5, MOE_MX_SCALES_W2C = 6,
       MOE_MX_SCALES_TOK_D = 7, MOE_MX_SCALES_TOK_F = 8, MOE_MX_SCALES_TOK_2F = 9 };
/* The data gradients' layouts: MOE_MX_SCALES_DH1 is [da | du] [N,2f] in the activation layout
 * (K = 2f).  MOE_MX_SCALES_W1C / _W2C are the weights blocked down their rows (W1 [2f,d] along 2f,
 * W2 [d,f] along d, as moe_mxfp8_prepare_dgrad_weights makes them): per expert, per tile of
 * columns (256 of d for W1, 128 of f for W2) and per 128-row K chunk, one 512-byte chunk per 128
 * columns of the tile, at ((e * tiles + t) * ceil(K/128) + kc) * (512 per 128 tile columns), byte
 * (c % 32) * 16 + (c % 128 / 32) * 4 + j for column c and block j of the K chunk; columns and
 * blocks past the weight are 127. */
/* The weight gradients' layouts (their reduction dimension is the tokens):
 * MOE_MX_SCALES_TOK_D / _F / _2F hold an [N, C] operand (C = d: x_perm or dy_perm; f: h; 2f:
 * [da | du]) blocked down its columns in 32-row blocks counted from each expert segment's first
 * row (a segment's last block may be short).  Per 128-column tile ct and 128-token chunk kc of
 * the expert segments -- chunk kc of rows s of expert e is cbase[e] + (s - off_e) / 128, cbase[e]
 * = sum_{e'<e} ceil(n_e' / 128) -- one 512-byte chunk at (ct * (N / 128 + E) + kc) * 512, byte
 * (c % 32) * 16 + (c % 128 / 32) * 4 + j for column c and block j of the chunk; the blocks of a
 * segment's last chunk past its rows are 127. */
/* Bytes of one packed scale buffer for cfg (0 for an invalid cfg or `which`). */
size_t moe_mxfp8_scale_bytes(const moe_cfg* cfg, int which);

/* MXFP8 quantisation of `rows` rows of `cols` bf16 values along each row (cols a multiple of
 * 32): q uint8 codes in x's layout, scales uint8 [rows, cols/32] row-major (plain layout, not
 * packed).  Quantise a weight along its reduction dimension: W1 [E,2f,d] as E*2f rows of d, W2
 * [E,d,f] as E*d rows of f.  All pointers device, 16-byte aligned. */
int moe_quantize_mxfp8(const void* x, int64_t rows, int32_t cols, uint8_t* q, uint8_t* scales,
                       void* stream);

/* Row-major expert weight scales (from moe_quantize_mxfp8: W1_s [E,2f,d/32], W2_s [E,d,f/32]) ->
 * the packed layouts MOE_MX_SCALES_W1 (W1_sp) and MOE_MX_SCALES_W2 (W2_sp).  Done once per
 * weight update; the codes keep their [E,2f,d] / [E,d,f] layouts. */
int moe_mxfp8_pack_expert_scales(const moe_cfg* cfg, const uint8_t* W1_s, const uint8_t* W2_s,
                                 uint8_t* W1_sp, uint8_t* W2_sp, void* stream);

/* Permute + MXFP8 quantisation in one pass: x_perm_q[slot_of_pair[t,j]] = the codes of x[t]
 * (moe_quantize_mxfp8 of row t), the scales into x_perm_s in the MOE_MX_SCALES_X layout (row tiles
 * from offsets [E+1], the routing's).  bf16 x [T,d]; d a multiple of 32. */
int moe_permute_quantize_mxfp8(const moe_cfg* cfg, const void* x, const int32_t* slot_of_pair,
                               const int32_t* offsets, uint8_t* x_perm_q, uint8_t* x_perm_s,
                               void* stream);

/* Grouped SwiGLU forward on MXFP8 operands, block-scaled tensor-core products (every K-block of
 * 32 carries its A-row and B-row scales).  For rows s of expert e:
 *   [a | u] = dec(x_perm_q[s], x_perm_s) . dec(W1_q[e], W1_sp)^T   (fp32 accumulation)
 *   h = SiLU(a) * u, rounded to bf16 (written to h [N,f] unless NULL; [a | u] to act [N,2f] unless
 *     NULL), then quantised to MXFP8 along f in the same epilogue: codes h_q [N,f], scales h_s in
 *     the MOE_MX_SCALES_H layout;
 *   y_perm[s] = dec(h_q[s], h_s) . dec(W2_q[e], W2_sp)^T                 (bf16 [N,d])
 * W1_q [E,2f,d] and W2_q [E,d,f] are codes from moe_quantize_mxfp8, W1_sp / W2_sp their packed
 * scales (moe_mxfp8_pack_expert_scales).  d and f multiples of 32; cfg->dtype MOE_DTYPE_BF16. */
int moe_grouped_swiglu_fwd_mxfp8(const moe_cfg* cfg, const uint8_t* x_perm_q,
                                 const uint8_t* x_perm_s, const int32_t* offsets,
                                 const uint8_t* W1_q, const uint8_t* W1_sp, const uint8_t* W2_q,
                                 const uint8_t* W2_sp, void* h, void* act, uint8_t* h_q,
                                 uint8_t* h_s, void* y_perm, void* stream);

/* MXFP8 state of the routed experts for moe_layer_fwd_mxfp8.  Caller-owned device buffers:
 *   W1_q [E,2f,d], W2_q [E,d,f]: codes from moe_quantize_mxfp8 (W1 blocked along d, W2 along f);
 *   W1_sp, W2_sp: their packed scales (moe_mxfp8_pack_expert_scales); read only;
 *   x_perm_q [N,d], x_perm_s (MOE_MX_SCALES_X bytes), h_q [N,f], h_s (MOE_MX_SCALES_H bytes): the
 *   layer forward's MXFP8 activations, written by the call. */
typedef struct moe_mxfp8_experts {
  const uint8_t* W1_q;
  const uint8_t* W1_sp;
  const uint8_t* W2_q;
  const uint8_t* W2_sp;
  uint8_t* x_perm_q;
  uint8_t* x_perm_s;
  uint8_t* h_q;
  uint8_t* h_s;
} moe_mxfp8_experts;

/* The data gradients' copies of the expert weights, blocked along the dimension the data
 * gradients reduce over: W1 [E,2f,d] in 32-row blocks along 2f, W2 [E,d,f] in 32-row blocks along d
 * (codes W1c_q / W2c_q in the weights' layouts; plain scales W1c_s [E,2f/32,d], W2c_s [E,d/32,f];
 * packed W1c_sp (MOE_MX_SCALES_W1C bytes), W2c_sp (MOE_MX_SCALES_W2C)).  Done once per weight
 * update, beside moe_quantize_mxfp8 / moe_mxfp8_pack_expert_scales for the forward's copies. */
int moe_mxfp8_prepare_dgrad_weights(const moe_cfg* cfg, const void* W1, const void* W2,
                                    uint8_t* W1c_q, uint8_t* W1c_s, uint8_t* W1c_sp,
                                    uint8_t* W2c_q, uint8_t* W2c_s, uint8_t* W2c_sp, void* stream);

/* The routed experts' data gradients on MXFP8 operands: dy_perm [N,d] (bf16, rows in expert order)
 * quantised along d into dy_q, dy_s (MOE_MX_SCALES_X layout); for rows s of expert e
 *   dh[s] = dec(dy_q[s], dy_s) . decc(W2c_q[e], W2c_sp)       (fp32 accumulation)
 *   [da | du] = SwiGLU backward of dh at act[s] ([a | u], bf16 [N,2f]), rounded to bf16: written to
 *     dH1 [N,2f] unless NULL, and quantised along 2f into dH1_q, dH1_s (MOE_MX_SCALES_DH1);
 *   dx_perm[s] = dec(dH1_q[s], dH1_s) . decc(W1c_q[e], W1c_sp)  (bf16 [N,d])
 * with the weights' column-blocked copies (moe_mxfp8_prepare_dgrad_weights).  d and f multiples of
 * 32; cfg->dtype MOE_DTYPE_BF16. */
int moe_grouped_swiglu_dgrad_mxfp8(const moe_cfg* cfg, const void* dy_perm, const int32_t* offsets,
                                   const void* act, const uint8_t* W1c_q, const uint8_t* W1c_sp,
                                   const uint8_t* W2c_q, const uint8_t* W2c_sp, uint8_t* dy_q,
                                   uint8_t* dy_s, void* dH1, uint8_t* dH1_q, uint8_t* dH1_s,
                                   void* dx_perm, void* stream);

/* MXFP8 data-gradient state for moe_layer_bwd_mxfp8: the weights' column-blocked copies (read
 * only) and the buffers the backward writes (dy_q [N,d], dy_s MOE_MX_SCALES_X bytes, dH1_q
 * [N,2f], dH1_s MOE_MX_SCALES_DH1 bytes). */
typedef struct moe_mxfp8_dgrad {
  const uint8_t* W1c_q;
  const uint8_t* W1c_sp;
  const uint8_t* W2c_q;
  const uint8_t* W2c_sp;
  uint8_t* dy_q;
  uint8_t* dy_s;
  uint8_t* dH1_q;
  uint8_t* dH1_s;
  /* Scratch for MXFP8 weight gradients (moe_workspace_bytes(cfg, MOE_WS_WGRAD_MXFP8) bytes):
   * when set, the routed experts' dW1 and dW2 run as moe_grouped_swiglu_wgrad_mxfp8 does; NULL:
   * they run on the bf16 operands. */
  void* wgrad_ws;
  size_t wgrad_ws_bytes;
} moe_mxfp8_dgrad;

/* MXFP8 weight gradients: "Megatron-Bridge 深度剖析", §FP8 训练 (the weight gradient in FP8,
 * fp8_wgrad) and §新硬件适配 (MXFP8).  Their reduction dimension is each expert's tokens, so the
 * operands are blocked along the tokens inside every expert segment.
 * moe_mxfp8_quantize_tokens: x [N, cols] bf16 (cols a multiple of 32) -> codes q [N, cols] and
 *   scales s in the token-chunk layout (MOE_MX_SCALES_TOK_*, for cols = d, f or 2f; in general
 *   ceil(cols/128) * (N/128 + E) * 512 bytes), cbase [E+1] int32 the segments' first chunks.
 *   offsets [E+1] as from routing (non-decreasing, from 0 to at most N; MOE_ERR_DEVICE_CHECK from
 *   moe_check_device_error otherwise, nothing written).
 * moe_grouped_swiglu_wgrad_mxfp8: for the rows s of expert e (offsets),
 *     dW1[e] = dec(dH1 blocks)^T . dec(x_perm blocks)   [2f, d]
 *     dW2[e] = dec(dy_perm blocks)^T . dec(h blocks)    [d, f]
 *   fp32 accumulation; every operand [N, .] bf16 is quantised by moe_mxfp8_quantize_tokens into
 *   the workspace (MOE_WS_WGRAD_MXFP8).  An expert without rows gets zero blocks.  cfg->dtype
 *   MOE_DTYPE_BF16, d and f multiples of 32. */
int moe_mxfp8_quantize_tokens(const moe_cfg* cfg, const void* x, int32_t cols,
                              const int32_t* offsets, uint8_t* q, uint8_t* s, int32_t* cbase,
                              void* stream);
int moe_grouped_swiglu_wgrad_mxfp8(const moe_cfg* cfg, const int32_t* offsets, const void* x_perm,
                                   const void* h, const void* dy_perm, const void* dH1,
                                   float* dW1, float* dW2, void* ws, size_t ws_bytes,
                                   void* stream);

/* Unpermute + weighted combine: "Megatron-Bridge 深度剖析", §Expert Parallel 基础 (Step 3,
 * results sent back to token order) and §Shared Expert Overlap (shared output added).
 *   y[t] = sum_{j<k} gate[t,j] * y_perm[slot_of_pair[t,j]]  (+ c_t * shared_out[t])
 *   accumulated in fp32 in ascending j, the shared term last, rounded once to dtype.
 *   shared_out [T,d] (dtype) or NULL; shared_coef [T] fp32 or NULL (c_t = 1). */
int moe_unpermute_combine(const moe_cfg* cfg, const void* y_perm, const float* gate,
                          const int32_t* slot_of_pair, const void* shared_out,
                          const float* shared_coef, void* y, void* stream);

/* Backward of moe_unpermute_combine.
 *   dy_perm[slot(t,j)] = gate[t,j] * dy[t];  dgate[t,j] = <dy[t], y_perm[slot(t,j)]> (fp32);
 *   with shared_out: dshared[t] = c_t * dy[t] (dtype) and, if shared_coef is set,
 *   dcoef[t] = <dy[t], shared_out[t]> (fp32).  dshared / dcoef may be NULL when unused. */
int moe_unpermute_combine_bwd(const moe_cfg* cfg, const void* dy, const void* y_perm,
                              const float* gate, const int32_t* slot_of_pair,
                              const void* shared_out, const float* shared_coef, void* dy_perm,
                              float* dgate, void* dshared, float* dcoef, void* stream);

/* Buffers a forward pass leaves for the backward.  All are caller-owned device buffers with
 * the shapes given; dtype means cfg->dtype.  The s_* members are used only with a shared
 * expert (f_s > 0) and s_coef only with the shared gate. */
typedef struct moe_saved {
  float* logits;          /* [T,E]  fp32                                       */
  int32_t* idx;           /* [T,k]                                             */
  float* gate;            /* [T,k]  fp32                                       */
  int32_t* counts;        /* [E]                                               */
  int32_t* offsets;       /* [E+1]                                             */
  int32_t* slot_of_pair;  /* [T,k]                                             */
  int32_t* token_of_slot; /* [N]                                               */
  void* x_perm;           /* [N,d]   dtype (unused, may be NULL, by a bf16 library built with
                             the permutation folded into its GEMMs: MOE_FUSE_PERMUTE=1) */
  void* act;              /* [N,2f]  dtype  ([a | u] pre-activations)          */
  void* h;                /* [N,f]   dtype                                     */
  void* y_perm;           /* [N,d]   dtype                                     */
  void* s_act;            /* [T,2f_s] dtype                                    */
  void* s_h;              /* [T,f_s]  dtype                                    */
  void* s_out;            /* [T,d]    dtype                                    */
  float* s_coef;          /* [T]  fp32, c_t = sigmoid(w_sg . x_t)              */
  float* aux_loss;        /* [1]  fp32 load-balancing loss (cfg->aux_coeff > 0) */
} moe_saved;

/* Load-balancing loss of one batch: "Megatron-Bridge 深度剖析", §Nemotron-3-Nano 配置
 * (moe_aux_loss_coeff: a loss that pushes tokens to spread evenly over the experts and keeps
 * them from collapsing onto a few).  The pages give no formula; this is the switch-style loss
 *   L = aux_coeff * E * sum_e f_e * P_e,  f_e = counts[e] / (T*k),  P_e = (1/T) sum_t p[t,e],
 * with p[t,:] the softmax of the logits (softmax routing) or s/sum(s), s = sigmoid(logits)
 * (sigmoid routing).  It equals aux_coeff when p is uniform.
 *   logits [T,E] fp32 (as routed: with a MOE_BIAS_LOGIT bias already in them); counts [E]
 *   from moe_route_topk; aux_loss [1] fp32 output.  Fixed-order sums: deterministic.
 *   Workspace: MOE_WS_ROUTE.  MOE_ERR_INVALID_ARG if cfg->aux_coeff is 0. */
int moe_router_aux_loss(const moe_cfg* cfg, const float* logits, const int32_t* counts,
                        float* aux_loss, void* ws, size_t ws_bytes, void* stream);

/* Expert-bias correction after a step (the auxiliary-loss-free balancing of DeepSeek V3 that
 * "Megatron-Bridge 深度剖析", §Nemotron-3-Nano 配置 turns on with moe_router_enable_expert_bias):
 *   e_bias[e] += rate * sign(T*k/E - counts[e])   (fp32; sign(0) = 0),
 * so an expert above the mean load loses selection priority and one below gains it.
 *   counts [E] int32 (one batch, from moe_route_topk or moe_layer_fwd's saved counts);
 *   e_bias [E] fp32, updated in place; the b_r of a MOE_BIAS_SELECT layer.  rate finite. */
int moe_expert_bias_update(const moe_cfg* cfg, const int32_t* counts, float* e_bias, float rate,
                           void* stream);

/* The layer calls' second stream, owned by the caller ("Megatron-Bridge 深度剖析", §Shared
 * Expert Overlap: the shared expert's work runs beside the routed experts' instead of after
 * them).  Given one, moe_layer_fwd* run the shared expert (and its gate) on `stream` while
 * routing, permute and the routed experts run on the call's stream, and moe_layer_bwd* run the
 * shared expert's backward and the router's backward on it while the routed experts' backward
 * runs; the call's stream then waits for it before the combine (forward) or the dx gather
 * (backward).
 *   stream: a cudaStream_t (as void*) other than the call's stream;
 *   fork, join: two distinct cudaEvent_t (as void*; cudaEventDisableTiming suffices), which the
 *     call records and waits on.
 * All three are created and destroyed by the caller; the library keeps no reference once the
 * call returns, and the side stream's work is ordered before the call's stream continues.  One
 * moe_side_stream must not serve two calls whose work can overlap (their event records would
 * interleave): give each concurrent caller its own.  NULL (the pointer): everything runs on the
 * call's stream in order.  Results are bit-identical either way.  MOE_ERR_INVALID_ARG if a
 * field is NULL, fork == join, or stream is the call's stream. */
typedef struct moe_side_stream {
  void* stream;
  void* fork;
  void* join;
} moe_side_stream;

/* Whole layer forward: route, permute, grouped SwiGLU, shared expert, combine.
 *   x [T,d]; W_r [E,d]; b_r [E] fp32 or NULL (cfg->bias_mode says how it acts);
 *   W1 [E,2f,d]; W2 [E,d,f];
 *   Ws1 [2f_s,d], Ws2 [d,f_s] (NULL without shared expert); w_sg [d] (NULL without gate).
 *   y [T,d].  `saved` receives everything the backward needs, and with cfg->aux_coeff > 0
 *   the load-balancing loss in saved->aux_loss (moe_router_aux_loss).  side: see
 *   moe_side_stream (NULL: one stream). */
int moe_layer_fwd(const moe_cfg* cfg, const void* x, const void* W_r, const float* b_r,
                  const void* W1, const void* W2, const void* Ws1, const void* Ws2,
                  const void* w_sg, void* y, const moe_saved* saved, void* ws, size_t ws_bytes,
                  void* stream, const moe_side_stream* side);

/* Whole layer backward, for the upstream gradient dy [T,d].  No gradient flows through the
 * expert selection (it is piecewise constant in the logits); b_r gets none (an input).
 * With cfg->aux_coeff > 0 the gradient of the load-balancing loss (weight 1, counts held
 * fixed) is added to the router's logit gradient:
 *   w_e = aux_coeff*E*counts[e]/(k*T^2),  G_t = sum_e p[t,e] w_e,
 *   softmax: dl[t,e] += p[t,e] (w_e - G_t);  sigmoid: dl[t,e] += s(1-s)(w_e - G_t)/sum_e s.
 *   Outputs: dx [T,d] (dtype); dW_r [E,d], dW1 [E,2f,d], dW2 [E,d,f], dWs1 [2f_s,d],
 *   dWs2 [d,f_s], dw_sg [d] -- all fp32 (the shared ones NULL when absent).
 *   side: see moe_side_stream (NULL: one stream). */
int moe_layer_bwd(const moe_cfg* cfg, const void* dy, const void* x, const void* W_r,
                  const void* W1, const void* W2, const void* Ws1, const void* Ws2,
                  const void* w_sg, const moe_saved* saved, void* dx, float* dW_r, float* dW1,
                  float* dW2, float* dWs1, float* dWs2, float* dw_sg, void* ws, size_t ws_bytes,
                  void* stream, const moe_side_stream* side);

/* The experts of a layer in FP8 ("Megatron-Bridge 深度剖析", §FP8 训练: E4M3, tensorwise
 * scaling, FP8 parameters, weight gradients in FP8).  Caller-owned device buffers:
 *   W1_q [E,2f,d], W2_q [E,d,f]: E4M3 codes of the routed experts' weights with one fp32 scale
 *     per expert (W1_scale [E], W2_scale [E]) -- moe_quantize_e4m3 with E groups; read only;
 *   x_perm_q [N,d], h_q [N,f]: the E4M3 activations moe_layer_fwd_fp8 leaves for the backward;
 *   scales [16] fp32, written by the calls, scale then amax of: [0] x, [2] h, [4] dy_perm,
 *     [6] [da | du] (routed), [8] the shared expert's h, [10] its upstream gradient, [12] its
 *     [da | du];
 *   Ws1_q [2f_s,d], Ws2_q [d,f_s] with Ws1_scale [1], Ws2_scale [1]: the shared expert's E4M3
 *     weights, or Ws1_q = NULL to keep the shared expert in bf16 (then the layer calls take Ws1,
 *     Ws2); with them, x_q [T,d] (x's codes in token order, same scale) and s_h_q [T,f_s] are
 *     written by the forward. */
typedef struct moe_fp8_experts {
  const uint8_t* W1_q;
  const float* W1_scale;
  const uint8_t* W2_q;
  const float* W2_scale;
  uint8_t* x_perm_q;
  uint8_t* h_q;
  float* scales;
  const uint8_t* Ws1_q;
  const float* Ws1_scale;
  const uint8_t* Ws2_q;
  const float* Ws2_scale;
  uint8_t* x_q;
  uint8_t* s_h_q;
} moe_fp8_experts;

/* The layer forward with its routed experts on MXFP8 operands: moe_layer_fwd, except that x is
 * permuted and block-quantised in one pass (moe_permute_quantize_mxfp8) and the routed experts run
 * as moe_grouped_swiglu_fwd_mxfp8 on mx's weights and buffers.  Router, shared expert (bf16 Ws1,
 * Ws2), shared gate and combine are those of moe_layer_fwd.  Routing, y_perm and the shared
 * expert's buffers are written as by moe_layer_fwd.  saved.x_perm, saved.act and saved.h may be
 * NULL (inference: not written); when given, the forward writes the permuted bf16 rows of x, the
 * bf16 [a | u] of the MXFP8 products and the bf16 h, and moe_layer_bwd (the bf16 backward, with
 * the bf16 weights) then runs on this forward's state: MXFP8 forward, bf16 data and weight
 * gradients.  Workspace MOE_WS_LAYER_FWD; d and f multiples of 32; cfg->dtype MOE_DTYPE_BF16. */
int moe_layer_fwd_mxfp8(const moe_cfg* cfg, const void* x, const void* W_r, const float* b_r,
                        const moe_mxfp8_experts* mx, const void* Ws1, const void* Ws2,
                        const void* w_sg, void* y, const moe_saved* saved, void* ws,
                        size_t ws_bytes, void* stream, const moe_side_stream* side);

/* The layer backward after moe_layer_fwd_mxfp8 (given saved.x_perm, act and h): moe_layer_bwd,
 * except that the routed experts' data gradients run on MXFP8 operands
 * (moe_grouped_swiglu_dgrad_mxfp8 on mxd's weights and buffers).  Their weight gradients run in
 * MXFP8 too when mxd->wgrad_ws is set (moe_grouped_swiglu_wgrad_mxfp8 on the saved bf16 x_perm and
 * h and the bf16 dy_perm and [da | du]); otherwise they are bf16 products of those operands (fp32
 * out).  The router's and the shared expert's backward stay bf16.  Workspace MOE_WS_LAYER_BWD. */
int moe_layer_bwd_mxfp8(const moe_cfg* cfg, const void* dy, const void* x, const void* W_r,
                        const moe_mxfp8_dgrad* mxd, const void* Ws1, const void* Ws2,
                        const void* w_sg, const moe_saved* saved, void* dx, float* dW_r,
                        float* dW1, float* dW2, float* dWs1, float* dWs2, float* dw_sg, void* ws,
                        size_t ws_bytes, void* stream, const moe_side_stream* side);

/* moe_layer_fwd with the routed experts on E4M3 operands: x is permuted and quantised in one
 * pass (moe_permute_quantize_e4m3) and the experts run as moe_grouped_swiglu_fwd_fp8 does, with
 * fp8's weights -- the shared expert too when fp8 holds its weights (an FP8 dense SwiGLU on
 * x_q); routing, the shared gate and the combine are those of moe_layer_fwd.  saved is filled
 * as by moe_layer_fwd except saved.x_perm (unused, may be NULL).  Workspace MOE_WS_LAYER_FWD.
 * cfg->dtype MOE_DTYPE_BF16; d, f (and f_s for an FP8 shared expert) multiples of 16. */
int moe_layer_fwd_fp8(const moe_cfg* cfg, const void* x, const void* W_r, const float* b_r,
                      const moe_fp8_experts* fp8, const void* Ws1, const void* Ws2,
                      const void* w_sg, void* y, const moe_saved* saved, void* ws, size_t ws_bytes,
                      void* stream, const moe_side_stream* side);

/* moe_layer_bwd after moe_layer_fwd_fp8: the routed experts' backward runs as
 * moe_grouped_swiglu_bwd_fp8 does (dy_perm and [da | du] quantised, both data gradients and
 * both weight gradients on E4M3 operands), the shared expert's likewise when it is in FP8;
 * the rest is that of moe_layer_bwd.  Outputs as moe_layer_bwd.  Workspace
 * MOE_WS_LAYER_BWD_FP8. */
int moe_layer_bwd_fp8(const moe_cfg* cfg, const void* dy, const void* x, const void* W_r,
                      const moe_fp8_experts* fp8, const void* Ws1, const void* Ws2,
                      const void* w_sg, const moe_saved* saved, void* dx, float* dW_r, float* dW1,
                      float* dW2, float* dWs1, float* dWs2, float* dw_sg, void* ws,
                      size_t ws_bytes, void* stream, const moe_side_stream* side);

/* Message of the last error on this host thread ("" if none). */
const char* moe_last_error(void);

/* Synchronises `stream`, reads and clears the device error word of the current device.
 * Returns MOE_OK, MOE_ERR_DEVICE_CHECK (with the kernel's code in *code if code != NULL),
 * or MOE_ERR_CUDA.  Codes (the first one recorded wins): 1 a bounded wait ran out, 2 an expert
 * index outside [0, E), 3 a slot outside [0, N), 4 offsets not monotone or not ending at N,
 * 5 dynamic shared memory not 1024-byte aligned, 6 a gathered token index outside [0, T). */
int moe_check_device_error(void* stream, int32_t* code);

/* Launch accounting and per-kernel timing (tracing).  moe_trace_enable(1) makes every
 * launch of this library record CUDA events around itself on its stream; moe_trace_read()
 * synchronises the device and returns, per kernel kind, launches and total milliseconds.
 * moe_launch_count() is the number of kernels this library launched in this process. */
uint64_t moe_launch_count(void);
int moe_trace_enable(int on);
/* Fills up to `cap` entries; returns the number of kernel kinds seen (or < 0 on error). */
int moe_trace_read(char* names, int name_stride, int* launches, double* total_ms, int cap);

/* GEMM pipeline wait statistics (tracing; a build option: the library built with
 * -DMOE_WAIT_STATS=1, e.g. MOE_NVCC_EXTRA=-DMOE_WAIT_STATS=1 for build.py; otherwise this
 * returns MOE_ERR_UNSUPPORTED and reads nothing).  Every tensor-core GEMM CTA adds, for its kernel
 * kind, SM clock cycles summed over CTAs: [0] its TMA producer waiting for a free ring stage, [1]
 * its MMA warp waiting for a loaded stage, [2] its MMA warp waiting for a free accumulator, [3]
 * its first epilogue warp waiting for a finished accumulator, [4] the CTA's own cycles; then [5]
 * the k-blocks its MMA warp consumed and [6] 1 (the CTA).  Kind k's seven values are
 * out[7k .. 7k+6].  One-CTA kernel: k = (A MN-major) + 2 (B MN-major) + 4 (reduction ragged per
 * group, the weight gradients) + 8 * epilogue (0 bf16 store, 1 fp32, 2 SwiGLU forward, 3 SwiGLU
 * backward) + 32 (8-bit operands); tall row tiles (fc2 and the data gradients in bf16): k = 48 +
 * (B MN-major).  The CTA-pair kernels are not counted.  Synchronises the device, copies the 64
 * kinds (448 values; cap >= 448), clears them and returns 64. */
int moe_gemm_wait_stats(uint64_t* out, int cap);

/* Self-test of the failure path of the pipelined kernels: launches one block that waits, through
 * the same bounded mbarrier wait as every GEMM pipeline (here with a 50 ms limit), on a barrier
 * that nothing arrives on.  The wait gives up, the kernel raises its abort flag, records
 * device error code 1 (a bounded wait ran out) in the device error word and returns.
 *   observed (device int32): bit 0 = the wait reported success (expected 0), bit 1 = the abort
 *   flag was raised (expected 1).
 * The caller then reads the code with moe_check_device_error (which clears it); the context stays
 * usable. */
int moe_selftest_wait_timeout(int32_t* observed, void* stream);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
