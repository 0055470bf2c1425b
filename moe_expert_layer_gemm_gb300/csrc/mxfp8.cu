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
