// Host-side interfaces between the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_gb300.h"

namespace moe {

// ------------------------------------------------------------------ launch bookkeeping
// Every kernel of the library is launched through launch(): it counts the launch and,
// when tracing is on, brackets it with CUDA events on its stream.
void trace_before(const char* name, cudaStream_t s);
void trace_after(const char* name, cudaStream_t s);
void count_launch();
void set_error(const char* fmt, ...);
int* device_error_word();   // per-device error word (nullptr if CUDA is unusable)
int num_sms();
// Device address of a __device__ variable of this library in the current context.  Addresses
// are cached per device together with the unique id of the context they were looked up in, and
// looked up again when the current context differs (after cudaDeviceReset the module is loaded
// into a new context and its variables may sit elsewhere).  The lookup initialises the device's
// primary context if needed, so make the first call on a device before any stream capture.
// MOE_OK or MOE_ERR_CUDA (message set).
struct SymbolCache {
  void* ptr[64];
  unsigned long long ctx[64];
};
int symbol_address(const void* symbol, SymbolCache* cache, void** out, const char* what);

template <typename... KArgs, typename... Args>
int launch(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
           cudaStream_t st, Args&&... args) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return MOE_OK;
  trace_before(name, st);
  kern<<<grid, block, smem, st>>>(std::forward<Args>(args)...);
  cudaError_t e = cudaGetLastError();
  trace_after(name, st);
  count_launch();
  if (e != cudaSuccess) {
    set_error("launch of %s failed: %s", name, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// The same, for a kernel launched in clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
int launch_clusters(const char* name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                    unsigned cluster_x, cudaStream_t st, Args&&... args) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return MOE_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before(name, st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e == cudaSuccess) e = cudaGetLastError();
  trace_after(name, st);
  count_launch();
  if (e != cudaSuccess) {
    set_error("launch of %s (clusters of %u) failed: %s", name, cluster_x, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

#define MOE_TRY(x)                 \
  do {                             \
    int _st = (x);                 \
    if (_st != MOE_OK) return _st; \
  } while (0)

// ------------------------------------------------------------------ routing (route.cu)
// Balancing-loss partial sums: one block per 256 tokens.
constexpr int ROUTE_TOK_PER_BLOCK = 256;
inline int route_blocks(int T) { return (T + ROUTE_TOK_PER_BLOCK - 1) / ROUTE_TOK_PER_BLOCK; }

// Expert histogram: one row per 128 tokens (a router GEMM row tile), one byte per expert (a row
// counts at most 128 tokens), rows of route_ldh(E) bytes (E rounded up to a power of two of at
// least 16, so that a row is whole 16-byte chunks and a warp covers whole rows).
constexpr int ROUTE_HIST_TOK = 128;
constexpr int ROUTE_SLOT_TOK = 256;          // tokens per block of the slots kernel
// Largest histogram every slots block reads whole; past it a scan kernel forms the per-row
// prefixes first (into rowpre: E * route_rows(T) int32).
constexpr int64_t ROUTE_DIRECT_BYTES = 131072;
inline int route_rows(int T) { return (T + ROUTE_HIST_TOK - 1) / ROUTE_HIST_TOK; }
inline int route_ldh(int E) {
  int l = 16;
  while (l < E) l <<= 1;
  return l;
}
inline int64_t route_hist_bytes(int T, int E) {
  return static_cast<int64_t>(route_rows(T)) * route_ldh(E);
}
inline bool route_hist_direct(int T, int E) { return route_hist_bytes(T, E) <= ROUTE_DIRECT_BYTES; }

// Per-token selection and gates (sel_bias: selection-only expert bias [E], keys = score + bias;
// null: keys = logits), and the histogram rows.
int launch_topk(const float* logits, int T, int E, int k, int score_fn, int renorm,
                const float* sel_bias, int32_t* idx, float* gate, uint8_t* hist, cudaStream_t st);
// Load-balancing loss; partial: route_blocks(T) * E floats of scratch.
int launch_aux_loss(const float* logits, const int32_t* counts, int T, int E, int k, int score_fn,
                    float coeff, float* partial, float* out, cudaStream_t st);
int launch_bias_update(const int32_t* counts, float* bias, int T, int k, int E, float rate,
                       cudaStream_t st);
// counts, offsets (the exclusive scan of counts, E+1 entries) and both slot maps from the
// histogram and idx.  rowpre (E * route_rows(T) int32) is used only when the histogram is larger
// than ROUTE_DIRECT_BYTES (may be null otherwise).
int launch_slots(const int32_t* idx, int T, int k, int E, const uint8_t* hist, int32_t* rowpre,
                 int32_t* counts, int32_t* offsets, int32_t* slot_of_pair, int32_t* token_of_slot,
                 cudaStream_t st);

// ------------------------------------------------------------------ row kernels (rowops.cu)
int launch_permute(int dtype, const void* x, const int32_t* slot_of_pair, void* x_perm, int T,
                   int d, int k, cudaStream_t st);
int launch_combine(int dtype, const void* y_perm, const float* gate, const int32_t* slot_of_pair,
                   const void* shared_out, const float* shared_coef, void* y, int T, int d, int k,
                   cudaStream_t st);
int launch_combine_bwd(int dtype, const void* dy, const void* y_perm, const float* gate,
                       const int32_t* slot_of_pair, const void* shared_out,
                       const float* shared_coef, void* dy_perm, float* dgate, void* dshared,
                       float* dcoef, int T, int d, int k, cudaStream_t st, float* amax_dy = nullptr,
                       float* amax_ds = nullptr);
// As launch_combine_bwd (bf16 only), and dy_perm's MXFP8 codes and packed scales as it stores it.
int launch_combine_bwd_mx(const void* dy, const void* y_perm, const float* gate,
                          const int32_t* sop, const void* shared_out, const float* shared_coef,
                          void* dy_perm, float* dgate, void* dshared, float* dcoef, int T, int d,
                          int k, const int32_t* offsets, int E, uint8_t* dy_q, uint8_t* dy_s,
                          cudaStream_t st);
int launch_gather_sum(int dtype, const void* dx_perm, const int32_t* slot_of_pair,
                      const void* dx_shared, const void* dx_router, const float* dz,
                      const void* w_sg, void* dx, int T, int d, int k, cudaStream_t st);
int launch_shared_gate(int dtype, const void* x, const void* w_sg, float* coef, int T, int d,
                       cudaStream_t st);
int launch_router_bwd(int dtype, const float* logits, const int32_t* idx, const float* gate,
                      const float* dgate, const float* dcoef, const float* coef, void* dl_ext,
                      float* dz, int T, int E, int k, int ld_ext, int score_fn, int renorm,
                      const int32_t* aux_counts, float aux_w, cudaStream_t st);
int launch_split_reduce(const float* part, int S, int rows, int cols, float* out_main,
                        int main_rows, float* out_extra, cudaStream_t st);

// ------------------------------------------------------------------ grouped GEMMs
// Scheduling of a grouped GEMM C_g = A_g . B_g^T over groups g < G.
//   RAGGED_M: rows of group g are [off[g], off[g+1]) of A and of C (offsets on the device; a
//             null offsets pointer means one group of rows [0, M)).  B_g is the g-th block of
//             b_group_rows rows of B.  K fixed.
//   RAGGED_K: C_g is a fixed M x N block (stored at out + g*out_group_stride); the reduction
//             runs over rows [off[g], off[g+1]) of A and B (null offsets: K split evenly
//             into G chunks).
enum Sched { RAGGED_M = 0, RAGGED_K = 1 };
// Epilogues.
enum Epi {
  EPI_STORE = 0,        // C in the activation dtype (bf16 / fp32)
  EPI_F32 = 1,          // C in fp32 (+ bias[n] if bias != null)
  EPI_SWIGLU_FWD = 2,   // acc = [gate | up] columns: h = SiLU(a)*u -> out, [a | u] -> out2
  EPI_SWIGLU_BWD = 3,   // acc = dh: reads [a | u] from aux, writes [da | du] -> out
};

// One operand: element (row, col) at base[row*ld + col]; `rows`/`cols` are the extents of
// the whole array as seen by this GEMM.  A K-major operand has the reduction index as col;
// an MN-major one has it as row.
struct Operand {
  const void* base;
  int64_t rows, cols, ld;
  bool mn_major;
};

// The router GEMM's epilogue routes its tokens: idx and gate [T, k] and the expert histogram
// rows of its row tiles (hist: [route_rows(T)][ldh] bytes), as launch_topk would from the logits.
struct RouterEpi {
  int32_t* idx;
  float* gate;
  uint8_t* hist;
  const float* sel_bias;   // selection-only expert bias [E] or null
  int k, score_fn, renorm, ldh;
};

struct GemmDesc {
  const char* name;        // trace name (kernel kind) of this product
  int sched;
  int epi;
  int G;
  const int32_t* offsets;
  int M, N, K;             // see Sched
  Operand A, B;
  int64_t b_group_rows;    // RAGGED_M: row offset of group g inside B
  int64_t b_up_rows;       // EPI_SWIGLU_FWD: row offset of the up half inside a group
  int f;                   // SwiGLU width (EPI_SWIGLU_*)
  void* out;
  int64_t ldo, out_group_stride;
  void* out2;
  int64_t ldo2;
  const void* aux;
  int64_t ld_aux;
  const float* bias;
  int* tile_ctr;           // RAGGED_K: two device counters (8 bytes, 8-byte aligned) for
                           // run-time tile scheduling
  // Gathered operand (bf16 only): row s of the operand is row gather[s] of the tensor the
  // Operand describes (A for RAGGED_M, with M rows; B for RAGGED_K, with K rows).  Null: plain.
  const int32_t* gather;
  // FP8 (E4M3) operands: A and B hold E4M3 codes; the product is scaled by a_scale[0] *
  // b_scale[g] (b_scale[0] with b_scale_scalar: both operands one tensor each, as in a weight
  // gradient) before the epilogue.
  bool fp8;
  const float* a_scale;
  const float* b_scale;
  bool b_scale_scalar;
  float* amax_out;         // FP8 SwiGLU forward / backward: receives max |h| or max |[da | du]|
                           // over the bf16 values written (zeroed by the caller)
  // MXFP8 operands (with fp8): E4M3 codes whose E8M0 block scales (one per 32 K-elements of each
  // row) sfa / sfb hold in the packed layouts below; the MMAs apply them, the epilogue none.
  bool mx;
  const uint8_t* sfa;
  const uint8_t* sfb;
  // MXFP8 weight gradients (RAGGED_K): the first 128-token chunk of each group's rows in the
  // token-chunk scale layouts of sfa / sfb; those layouts hold mx_tok_chunks(K, G) chunks per
  // 128-row tile.
  const int32_t* mx_cbase;
  // MXFP8 SwiGLU forward: h as MXFP8 codes [rows, f] and its packed block scales (the A-operand
  // layout, row tiles as this product's); `out` (bf16 h) and `out2` ([a | u]) may be null.
  uint8_t* q_out;
  uint8_t* q_sf;
  // Router top-k in the epilogue (RAGGED_M fp32 logits, bf16 operands, E <= the tile's width so
  // that one column tile holds a token's every logit): rt.idx null = off.
  RouterEpi rt;
};

// ------------------------------------------------------------------ MXFP8 packed scales
// Block scales of 128 operand rows x 128 K-elements (four 32-blocks per row) form one 512-byte
// chunk in the order the tensor cores read them from TMEM: the scale of row r, block j sits at
// byte (r % 32) * 16 + (r / 32) * 4 + j.
//   activation operand [N rows, K]: chunk (mt, kc) at (mt * kch + kc) * 512, where mt is the row
//     tile -- the tiles of earlier experts (sum of ceil(rows_e / 128)) plus the row's offset
//     inside its expert / 128 -- and kc = K-element / 128, kch = ceil(K / 128);
//   weight operand: per expert e and output tile nt, for every kc, MX_SFB_CHUNKS chunks (tile rows
//     0..127, 128..255) at ((e * NT + nt) * kch + kc) * MX_SFB_BYTES.  fc1 tile nt holds gate rows
//     nt*96 .. +95 then up rows f + nt*96 .. +95 (NT = ceil(f / 96)); fc2 tile nt holds rows
//     nt*192 .. +191 (NT = ceil(d / 192)).
// Scales of rows or blocks past the operand's end are 127 (2^0) in weight chunks; activation
// chunks leave rows past an expert's end unwritten (their products are never stored) and set
// blocks past K to 127.
constexpr int MX_BN = 192;                 // output columns of an MXFP8 forward tile
// MXFP8 data-gradient tiles (MN-major weights come in 128-column chunks): fc1's 256 columns wide
// with one accumulator (fewer operand bytes per FLOP); fc2's, whose SwiGLU-backward epilogue is
// long, 128 wide with two, so that the epilogue overlaps the next tile's MMAs.
constexpr int MX_BN_DGRAD1 = 256;
constexpr int MX_BN_DGRAD2 = 128;
constexpr int MX_CHUNK = 512;
constexpr int MX_SFB_CHUNKS = (MX_BN + 127) / 128;
constexpr int MX_SFB_BYTES = MX_SFB_CHUNKS * MX_CHUNK;
inline int64_t mx_kch(int64_t K) { return (K + 127) / 128; }
// Token-direction operands of the MXFP8 weight gradients: 128-token chunks of the expert segments
// (at most N / 128 + E of them), per 128-column tile one 512-byte chunk each.
inline int64_t mx_tok_chunks(int64_t N, int E) { return N / 128 + E; }
inline int64_t mx_tok_scale_bytes(int64_t N, int E, int64_t C) {
  return ((C + 127) / 128) * mx_tok_chunks(N, E) * MX_CHUNK;
}
// an upper bound of sum_e ceil(rows_e / 128) for N rows over E experts
inline int64_t mx_row_tiles(int64_t N, int E) { return (N + 127 * static_cast<int64_t>(E)) / 128 + 1; }
inline int64_t mx_act_scale_bytes(int64_t N, int E, int64_t K) {
  return mx_row_tiles(N, E) * mx_kch(K) * MX_CHUNK;
}
inline int64_t mx_fc1_tiles(int f) { return (f + MX_BN / 2 - 1) / (MX_BN / 2); }
inline int64_t mx_fc2_tiles(int d) { return (d + MX_BN - 1) / MX_BN; }

// Argument checks and the routing stages (capi.cu), for entry points defined elsewhere.
int validate_cfg(const moe_cfg* c);
int validate_ptr(const void* p, const char* name, bool required);
int route_stages(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                 const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                 int32_t* counts, int32_t* offsets, int32_t* slot_of_pair, int32_t* token_of_slot,
                 uint8_t* hist, int32_t* rowpre, cudaStream_t st);

// E4M3 tensorwise quantisation of `groups` blocks of per_group bf16 values (fp8.cu).
int launch_quantize_e4m3(const void* x, int64_t per_group, int groups, uint8_t* q, float* scale,
                         float* amax, cudaStream_t st);
// The cast alone, with amax already computed (e.g. by the producing GEMM's epilogue).
int launch_quant_e4m3_given_amax(const void* x, int64_t per_group, int groups, uint8_t* q,
                                 float* scale, const float* amax, cudaStream_t st);
// amax of x [T,d] and the permuted E4M3 rows x_perm_q[slot_of_pair[t,j]] = E4M3(x[t] * inv)
// (and x_q[t], the same codes in token order, if x_q is not NULL).
int launch_permute_quant_e4m3(const void* x, const int32_t* sop, uint8_t* xq, uint8_t* x_q,
                              float* scale, float* amax, int T, int d, int k, cudaStream_t st);

// MXFP8 quantisation (mxfp8.cu).  Rows of `cols` bf16 values (cols % 32 == 0) -> E4M3 codes and
// row-major E8M0 scales [rows, cols / 32].
int launch_mx_quantize(const void* x, int64_t rows, int cols, uint8_t* q, uint8_t* s,
                       cudaStream_t st);
// Weight scales -> the packed weight layout with tiles of tile_rows B-rows; swiglu_f > 0: fc1
// tiles over R = 2 * swiglu_f rows, 0: plain tiles over R B-rows.  Row-major scales [E, R, K/32]
// (blocks along each B-row's K), or with cols scales [E, K/32, R] of a weight whose columns are
// the B-rows (blocks along its rows, as the data gradients read W1 and W2).
int launch_mx_pack_weight_scales(const uint8_t* s, int E, int R, int K, int swiglu_f,
                                 uint8_t* packed, cudaStream_t st, int tile_rows = MX_BN,
                                 int cols = 0);
// G groups of R x C bf16 rows quantised in 32-row blocks down each column: codes in x's layout,
// scales [G, R/32, C].
// Token-direction blocks of x [N, C] bf16 inside the expert segments given by offsets [E+1]:
// codes q [N, C], scales in the packed token-chunk layout (mx_tok_scale_bytes), chunk bases
// cbase [E+1] (sum of ceil(n_e / 128) over the experts before e).
int launch_mx_quantize_tokens(const void* x, int64_t N, int C, const int32_t* offsets, int E,
                              uint8_t* q, uint8_t* s, int32_t* cbase, cudaStream_t st);
int launch_mx_quantize_cols(const void* x, int G, int R, int C, uint8_t* q, uint8_t* s,
                            cudaStream_t st);
// Permute + quantise: x_perm_q[slot(t, j)] = MXFP8 codes of x[t], scales in the packed
// activation layout (row tiles from the routing offsets); xp (optional): the bf16 rows too.
// sop = NULL (with k = 1): row t is slot t (quantising rows already in expert order).
int launch_permute_quant_mx(const void* x, const int32_t* sop, const int32_t* offsets,
                            uint8_t* xq, uint8_t* xs, int T, int d, int k, int E, cudaStream_t st,
                            void* xp = nullptr);

int gemm_tc(const GemmDesc& g, cudaStream_t st);     // bf16 tcgen05 path (gemm_tc.cu)
int gemm_simt(const GemmDesc& g, cudaStream_t st);   // fp32 CUDA-core path (gemm_simt.cu)

}  // namespace moe
