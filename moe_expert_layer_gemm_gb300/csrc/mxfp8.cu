// MXFP8 quantisation: E4M3 elements with one shared E8M0 (power-of-two) scale per 32 consecutive
// elements along a product's reduction dimension ("Megatron-Bridge 深度剖析", §新硬件适配:
// Blackwell's microscaling FP8, scale factors finer than per tensor; the element and scale
// formats are the OCP Microscaling ones).
//
// Per block of 32 values: e = floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for amax = 0),
// code = E4M3(x * 2^-e) (round to nearest even, saturating at +-448), scale byte = e + 127.
// The multiply is by an exact power of two, so the codes depend on the input alone.
//
// Kernels:
//   mx_quant_kernel        rows of a matrix, row-major scales [rows, cols / 32] (weights; any
//                          matrix)
//   mx_pack_wscales_kernel row-major weight scales -> the packed per-tile layout the GEMMs read
//   permute_quant_mx_kernel  x [T, d] -> the permuted codes x_perm_q[slot] and its scales in the
//                          packed activation layout (row tiles from the routing offsets), and
//                          optionally the permuted bf16 rows themselves (for a bf16 backward)
//   mx_quant_tokens_kernel the weight gradients' operands [N, C]: blocks of 32 rows down each
//                          column inside every expert segment (the tokens are their reduction
//                          dimension), codes in place, scales in the packed token-chunk layout
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// One 32-block: 32 bf16 values in, 32 codes and the exponent out.
__device__ __forceinline__ int quant_block32(const float (&v)[32], uint32_t (&w)[8]) {
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
  const int e = mx_exponent(am);
  const float inv = mx_inv_scale(e);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = cvt_e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv);
    const uint32_t hi = cvt_e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv);
    w[j] = lo | (hi << 16);
  }
  return e;
}

// One thread per 32-block of a row-major [rows, cols] bf16 matrix (cols % 32 == 0).
__global__ void __launch_bounds__(256) mx_quant_kernel(const bf16* __restrict__ x, int64_t nblk,
                                                       uint8_t* __restrict__ q,
                                                       uint8_t* __restrict__ s) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk;
       b += stride) {
    const bf16* src = x + b * 32;
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) unpack16(ld_nc16(src + 8 * j), v + 8 * j, static_cast<const bf16*>(nullptr));
    uint32_t w[8];
    const int e = quant_block32(v, w);
    uint4* dst = reinterpret_cast<uint4*>(q + b * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    s[b] = static_cast<uint8_t>(e + 127);
  }
}

// One thread per byte of a packed weight-scale layout (internal.h): E experts x NT tiles of TR
// B-rows x kch chunks x ceil(TR / 128) chunks of 512 bytes.  Byte pos of chunk ch holds tile row
// ch * 128 + (pos / 4) % 4 * 32 + pos / 16, block kc * 4 + pos % 4.  B-row r of expert e is
// weight row r (scales s[e][r][block], blocks along the weight's rows' K) or, with cols, weight
// column r (scales s[e][block][r], blocks along its columns).
__global__ void __launch_bounds__(256) mx_pack_wscales_kernel(const uint8_t* __restrict__ s, int E,
                                                              int R, int nb, int swiglu_f, int NT,
                                                              int kch, int TR, int cols,
                                                              uint8_t* __restrict__ out) {
  const int CH = (TR + 127) / 128;
  const int64_t total = static_cast<int64_t>(E) * NT * kch * CH * MX_CHUNK;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int pos = static_cast<int>(i % MX_CHUNK);
    int64_t rest = i / MX_CHUNK;
    const int ch = static_cast<int>(rest % CH);
    rest /= CH;
    const int kc = static_cast<int>(rest % kch);
    rest /= kch;
    const int nt = static_cast<int>(rest % NT);
    const int e = static_cast<int>(rest / NT);
    const int rt = ch * 128 + ((pos >> 2) & 3) * 32 + (pos >> 4);   // row inside the tile
    const int blk = kc * 4 + (pos & 3);
    int row = -1;
    if (rt < TR) {
      if (swiglu_f > 0) {
        const int half = TR / 2;
        const int hc = nt * half + (rt < half ? rt : rt - half);   // h column of this B row
        if (hc < swiglu_f) row = rt < half ? hc : swiglu_f + hc;
      } else {
        const int r = nt * TR + rt;
        if (r < R) row = r;
      }
    }
    const int64_t src = cols ? (static_cast<int64_t>(e) * nb + blk) * R + row
                             : (static_cast<int64_t>(e) * R + row) * nb + blk;
    out[i] = (row >= 0 && blk < nb) ? s[src] : static_cast<uint8_t>(127);
  }
}

// One thread per (group g, 32-row block b, column c) of G groups of R x C bf16 rows (R % 32 ==
// 0): the block's 32 values down column c, codes in x's layout, scales s[g][b][c].  Consecutive
// threads take consecutive columns, so every row access is coalesced.
__global__ void __launch_bounds__(256) mx_quant_cols_kernel(const bf16* __restrict__ x, int G, int R,
                                                            int C, uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ s) {
  const int64_t nbr = R / 32;
  const int64_t total = static_cast<int64_t>(G) * nbr * C;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int c = static_cast<int>(i % C);
    const int64_t gb = i / C;                      // g * nbr + b
    const int64_t r0 = gb * 32;                    // first row of the block in the G*R rows
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __bfloat162float(x[(r0 + j) * C + c]);
    uint32_t w[8];
    const int e = quant_block32(v, w);
#pragma unroll
    for (int j = 0; j < 32; ++j) q[(r0 + j) * C + c] = static_cast<uint8_t>(w[j >> 2] >> (8 * (j & 3)));
    s[gb * C + c] = static_cast<uint8_t>(e + 127);
  }
}

// Permute + quantise, one warp per token: lane L quantises columns 8L.. of each 256-column step,
// four lanes make one 32-block (amax over the four by shuffles).  Codes go to every slot of the
// token; the block's scale byte to each slot's place in the packed activation layout; with xp,
// the bf16 row to each slot too.
constexpr int MXP_THREADS = 256;
__global__ void __launch_bounds__(MXP_THREADS) permute_quant_mx_kernel(
    const bf16* __restrict__ x, const int32_t* __restrict__ sop, const int32_t* __restrict__ offsets,
    uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, bf16* __restrict__ xp, int Tn, int d, int k,
    int E, int* err) {
  __shared__ int s_off[MOE_MAX_EXPERTS + 1];
  __shared__ int s_pre[MOE_MAX_EXPERTS + 1];
  const int lane = threadIdx.x & 31;
  mx_tile_prefix(offsets, E, s_off, s_pre);
  const int64_t N = static_cast<int64_t>(Tn) * k;
  const int kch = (d + 127) / 128;
  const int nb = d / 32;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int t = gw; t < Tn; t += nw) {
    int my_slot = -1;
    int64_t my_sf = 0;
    if (lane < k) {
      my_slot = sop ? sop[static_cast<int64_t>(t) * k + lane] : t;   // no map: row t is slot t
      if (my_slot < 0 || my_slot >= N || my_slot >= s_off[E]) {
        record_error(err, DEVERR_BAD_SLOT);
        my_slot = -1;
      } else {
        my_sf = mx_row_scale_base(my_slot, s_off, s_pre, E, kch);
      }
    }
    int slot[MOE_MAX_TOPK];
    int64_t sfb[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
      sfb[j] = __shfl_sync(0xffffffffu, my_sf, j);
    }
    const bf16* src = x + static_cast<int64_t>(t) * d;
    for (int c0 = 0; c0 < d; c0 += 256) {
      const int c = c0 + lane * 8;
      const bool act = c < d;   // d % 32 == 0: a 4-lane group is all in or all out
      float f[8];
      const uint4 raw = act ? ld_nc16(src + c) : make_uint4(0, 0, 0, 0);
      unpack16(raw, f, static_cast<const bf16*>(nullptr));
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = act ? fmaxf(m, fabsf(f[i])) : m;
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (!act) continue;
      const int e = mx_exponent(m);
      const float inv = mx_inv_scale(e);
      uint32_t w[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = cvt_e4m3x2(f[4 * j] * inv, f[4 * j + 1] * inv);
        const uint32_t hi = cvt_e4m3x2(f[4 * j + 2] * inv, f[4 * j + 3] * inv);
        w[j] = lo | (hi << 16);
      }
      const int blk = c >> 5;
      const bool writes_scale = (lane & 3) == 0;
      const bool pads = writes_scale && blk == nb - 1 && (nb & 3) != 0;
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        if (j >= k) break;
        if (slot[j] < 0) continue;
        *reinterpret_cast<uint2*>(xq + static_cast<int64_t>(slot[j]) * d + c) = make_uint2(w[0], w[1]);
        if (xp) *reinterpret_cast<uint4*>(xp + static_cast<int64_t>(slot[j]) * d + c) = raw;
        if (writes_scale) {
          uint8_t* sf = xs + sfb[j] + (blk >> 2) * MX_CHUNK;
          sf[blk & 3] = static_cast<uint8_t>(e + 127);
          if (pads)
            for (int q = (blk & 3) + 1; q < 4; ++q) sf[q] = 127;   // blocks past d: 2^0
        }
      }
    }
  }
}

// Token-direction blocks of the weight gradients' operands: one thread per (32-row block of an
// expert segment, 2 adjacent columns) of x [N, C] bf16 (C % 32 == 0).  The blocks of expert e are
// counted from its first row; its last block may be short (the missing rows are zeros for the
// amax and store nothing).  Codes go to q in x's layout.  A block's scale byte goes to the packed
// layout: 128-token chunk kc = cbase[e] + b / 4 of the expert segments (cbase[e] = sum_{e'<e}
// ceil(n_e' / 128)), column tile c / 128, chunk at ((c / 128) * kct + kc) * 512, byte (c % 32) *
// 16 + (c % 128 / 32) * 4 + b % 4; the later blocks of a segment's last chunk (no rows) get 127.
// Block 0 writes cbase.  A warp covers 64 adjacent columns: 128-byte row reads, 64-byte code
// rows.  The block's 32 rows are held as packed bf16 pairs between the amax and the rounding.
constexpr int MXT_COLS = 2;   // columns per thread
__global__ void __launch_bounds__(256) mx_quant_tokens_kernel(const bf16* __restrict__ x,
                                                              const int32_t* __restrict__ offsets,
                                                              int E, int C, int64_t N, int64_t kct,
                                                              uint8_t* __restrict__ q,
                                                              uint8_t* __restrict__ s,
                                                              int32_t* __restrict__ cbase,
                                                              int* err) {
  __shared__ int s_off[MOE_MAX_EXPERTS + 1], s_bp[MOE_MAX_EXPERTS + 1], s_cp[MOE_MAX_EXPERTS + 1];
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    int bp = 0, cp = 0, bad = offsets[0] != 0;
    for (int e = 0; e <= E; ++e) {
      const int o = offsets[e];
      s_off[e] = o;
      s_bp[e] = bp;
      s_cp[e] = cp;
      if (e < E) {
        const int n = offsets[e + 1] - o;
        if (n < 0) bad = 1;
        bp += (n + 31) / 32;
        cp += (n + 127) / 128;
      }
    }
    if (s_off[E] > N || cp > kct) bad = 1;
    if (bad) record_error(err, DEVERR_BAD_OFFSETS);
    s_bad = bad;
  }
  __syncthreads();
  if (s_bad) return;
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) cbase[e] = s_cp[e];
  const int CG = C / MXT_COLS;   // column groups
  const int64_t total = static_cast<int64_t>(s_bp[E]) * CG;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int c0 = static_cast<int>(i % CG) * MXT_COLS;
    const int gb = static_cast<int>(i / CG);
    int lo = 0, hi = E;   // the expert of block gb: the largest e with s_bp[e] <= gb
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_bp[mid] <= gb) lo = mid;
      else hi = mid;
    }
    const int e = lo;
    const int b = gb - s_bp[e];
    const int n = s_off[e + 1] - s_off[e];
    const int64_t r0 = s_off[e] + 32 * static_cast<int64_t>(b);
    const int nr = min(32, n - 32 * b);
    uint32_t raw[32];   // row j: columns c0, c0+1 as a bf16 pair
#pragma unroll
    for (int j = 0; j < 32; ++j)
      raw[j] = j < nr ? __ldg(reinterpret_cast<const uint32_t*>(x + (r0 + j) * C + c0)) : 0u;
    float am[MXT_COLS] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      am[0] = fmaxf(am[0], fabsf(__uint_as_float(raw[j] << 16)));
      am[1] = fmaxf(am[1], fabsf(__uint_as_float(raw[j] & 0xffff0000u)));
    }
    int ex[MXT_COLS];
    float inv[MXT_COLS];
#pragma unroll
    for (int u = 0; u < MXT_COLS; ++u) {
      ex[u] = mx_exponent(am[u]);
      inv[u] = mx_inv_scale(ex[u]);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nr)
        *reinterpret_cast<uint16_t*>(q + (r0 + j) * C + c0) =
            cvt_e4m3x2(__uint_as_float(raw[j] << 16) * inv[0],
                       __uint_as_float(raw[j] & 0xffff0000u) * inv[1]);
    const int64_t kc = s_cp[e] + b / 4;
    const bool last = 32 * (b + 1) >= n;   // the segment's last block
#pragma unroll
    for (int u = 0; u < MXT_COLS; ++u) {
      const int c = c0 + u, rr = c & 127;
      uint8_t* row = s + ((c >> 7) * kct + kc) * MX_CHUNK + (rr & 31) * 16 + (rr >> 5) * 4;
      row[b & 3] = static_cast<uint8_t>(ex[u] + 127);
      if (last)   // the chunk's later blocks hold no rows
        for (int j4 = (b & 3) + 1; j4 < 4; ++j4) row[j4] = 127;
    }
  }
}

int grid_for(int64_t items, int per_block) {
  int64_t b = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (b > cap) b = cap;
  return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

int launch_mx_quantize(const void* x, int64_t rows, int cols, uint8_t* q, uint8_t* s,
                       cudaStream_t st) {
  const int64_t nblk = rows * (cols / 32);
  if (nblk == 0) return MOE_OK;
  return launch("mxfp8_quantize", mx_quant_kernel, dim3(grid_for(nblk, 256)), dim3(256), 0, st,
                static_cast<const bf16*>(x), nblk, q, s);
}

int launch_mx_pack_weight_scales(const uint8_t* s, int E, int R, int K, int swiglu_f,
                                 uint8_t* packed, cudaStream_t st, int tile_rows, int cols) {
  const int NT = static_cast<int>(swiglu_f > 0 ? (swiglu_f + tile_rows / 2 - 1) / (tile_rows / 2)
                                               : (R + tile_rows - 1) / tile_rows);
  const int kch = static_cast<int>(mx_kch(K));
  const int64_t total = static_cast<int64_t>(E) * NT * kch * ((tile_rows + 127) / 128) * MX_CHUNK;
  return launch("mxfp8_pack_scales", mx_pack_wscales_kernel, dim3(grid_for(total, 256)), dim3(256),
                0, st, s, E, R, K / 32, swiglu_f, NT, kch, tile_rows, cols, packed);
}

int launch_mx_quantize_cols(const void* x, int G, int R, int C, uint8_t* q, uint8_t* s,
                            cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(G) * (R / 32) * C;
  if (n == 0) return MOE_OK;
  return launch("mxfp8_quantize_cols", mx_quant_cols_kernel, dim3(grid_for(n, 256)), dim3(256), 0,
                st, static_cast<const bf16*>(x), G, R, C, q, s);
}

int launch_mx_quantize_tokens(const void* x, int64_t N, int C, const int32_t* offsets, int E,
                              uint8_t* q, uint8_t* s, int32_t* cbase, cudaStream_t st) {
  const int64_t items = (N / 32 + E) * static_cast<int64_t>(C / MXT_COLS);   // blocks <= N/32 + E
  return launch("mxfp8_quantize_tokens", mx_quant_tokens_kernel, dim3(grid_for(items, 256)),
                dim3(256), 0, st, static_cast<const bf16*>(x), offsets, E, C, N,
                mx_tok_chunks(N, E), q, s, cbase, device_error_word());
}

int launch_permute_quant_mx(const void* x, const int32_t* sop, const int32_t* offsets,
                            uint8_t* xq, uint8_t* xs, int T, int d, int k, int E, cudaStream_t st,
                            void* xp) {
  const int wpb = MXP_THREADS / 32;
  int rb = (T + wpb - 1) / wpb;
  if (rb > num_sms() * 8) rb = num_sms() * 8;
  return launch(sop ? "mxfp8_permute_quantize" : "mxfp8_quantize_rows", permute_quant_mx_kernel,
                dim3(rb), dim3(MXP_THREADS), 0,
                st, static_cast<const bf16*>(x), sop, offsets, xq, xs, static_cast<bf16*>(xp), T, d,
                k, E, device_error_word());
}

}  // namespace moe
