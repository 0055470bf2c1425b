// E4M3 tensorwise quantisation ("Megatron-Bridge 深度剖析", §FP8 训练: FP8 E4M3 with a
// "tensorwise" scaling recipe) and the FP8 grouped SwiGLU forward built on it.
//
// Per group of elements (one tensor: an activation matrix, or one expert's weight):
//   amax = max |x|;  inv = 448 / amax;  code = E4M3(x * inv)  (round to nearest even, saturating);
//   scale = amax / 448 (the dequantisation factor the GEMM epilogue applies).
// amax = 0 gives inv = scale = 1.  Both quotients are IEEE fp32 divisions and the product is one
// fp32 multiply, so the codes are a deterministic function of the input.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr float E4M3_MAX = 448.0f;

// amax of each group: grid (blocks, groups); 8 bf16 per 16-byte load.
__global__ void __launch_bounds__(256) amax_kernel(const bf16* __restrict__ x, int64_t per_group,
                                                   unsigned int* __restrict__ amax_bits) {
  __shared__ float wmax[8];
  const bf16* base = x + static_cast<int64_t>(blockIdx.y) * per_group;
  float m = 0.f;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < per_group;
       i += step) {
    float f[8];
    unpack16(ld_nc16(base + i), f, static_cast<const bf16*>(nullptr));
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = fmaxf(b, wmax[w]);
    // non-negative floats order like their bit patterns
    atomicMax(amax_bits + blockIdx.y, __float_as_uint(b));
  }
}

__global__ void __launch_bounds__(256) quant_kernel(const bf16* __restrict__ x, int64_t per_group,
                                                    const unsigned int* __restrict__ amax_bits,
                                                    uint8_t* __restrict__ q,
                                                    float* __restrict__ scale) {
  const int g = blockIdx.y;
  const float amax = __uint_as_float(amax_bits[g]);
  const float inv = amax > 0.f ? E4M3_MAX / amax : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) scale[g] = amax > 0.f ? amax / E4M3_MAX : 1.0f;
  const bf16* base = x + static_cast<int64_t>(g) * per_group;
  uint8_t* qb = q + static_cast<int64_t>(g) * per_group;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < per_group;
       i += step) {
    float f[8];
    unpack16(ld_nc16(base + i), f, static_cast<const bf16*>(nullptr));
    uint32_t w[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t lo = cvt_e4m3x2(__fmul_rn(f[4 * j], inv), __fmul_rn(f[4 * j + 1], inv));
      const uint32_t hi = cvt_e4m3x2(__fmul_rn(f[4 * j + 2], inv), __fmul_rn(f[4 * j + 3], inv));
      w[j] = lo | (hi << 16);
    }
    *reinterpret_cast<uint2*>(qb + i) = make_uint2(w[0], w[1]);
  }
}

// Permute + quantise: x_perm_q[slot(t, j)] = E4M3(x[t] * inv) for every pair (t, j), and
// x_q[t] the same codes in token order if x_q is given (the shared expert's input); x is read
// once per token (one warp per token).  Same codes as quantising the permuted matrix: the pairs'
// rows are exact copies of x's rows.
__global__ void __launch_bounds__(256) permute_quant_kernel(const bf16* __restrict__ x,
                                                            const int32_t* __restrict__ sop,
                                                            const unsigned int* __restrict__ amax_bits,
                                                            uint8_t* __restrict__ xq,
                                                            uint8_t* __restrict__ xq_tok,
                                                            float* __restrict__ scale, int Tn,
                                                            int d, int k, int* err) {
  const float amax = __uint_as_float(amax_bits[0]);
  const float inv = amax > 0.f ? E4M3_MAX / amax : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) scale[0] = amax > 0.f ? amax / E4M3_MAX : 1.0f;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int64_t N = static_cast<int64_t>(Tn) * k;
  for (int t = gw; t < Tn; t += nw) {
    int my_slot = -1;
    if (lane < k) {
      my_slot = sop[static_cast<int64_t>(t) * k + lane];
      if (my_slot < 0 || my_slot >= N) {
        record_error(err, DEVERR_BAD_SLOT);
        my_slot = -1;
      }
    }
    int slot[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
    const bf16* src = x + static_cast<int64_t>(t) * d;
    for (int c = lane * 8; c < d; c += 32 * 8) {
      float f[8];
      unpack16(ld_nc16(src + c), f, static_cast<const bf16*>(nullptr));
      uint32_t w[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(f[4 * j], inv), __fmul_rn(f[4 * j + 1], inv));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(f[4 * j + 2], inv), __fmul_rn(f[4 * j + 3], inv));
        w[j] = lo | (hi << 16);
      }
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        if (j >= k) break;
        if (slot[j] >= 0)
          *reinterpret_cast<uint2*>(xq + static_cast<int64_t>(slot[j]) * d + c) = make_uint2(w[0], w[1]);
      }
      if (xq_tok)
        *reinterpret_cast<uint2*>(xq_tok + static_cast<int64_t>(t) * d + c) = make_uint2(w[0], w[1]);
    }
  }
}

}  // namespace

int launch_quant_e4m3_given_amax(const void* x, int64_t per_group, int groups, uint8_t* q,
                                 float* scale, const float* amax, cudaStream_t st) {
  int64_t want = (per_group / 8 + 255) / 256;
  const int64_t cap = (static_cast<int64_t>(num_sms()) * 8 + groups - 1) / groups;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  const dim3 grid(static_cast<unsigned>(want), static_cast<unsigned>(groups));
  return launch("fp8_quantize", quant_kernel, grid, dim3(256), 0, st, static_cast<const bf16*>(x),
                per_group, reinterpret_cast<const unsigned int*>(amax), q, scale);
}

int launch_permute_quant_e4m3(const void* x, const int32_t* sop, uint8_t* xq, uint8_t* xq_tok,
                              float* scale, float* amax, int T, int d, int k, cudaStream_t st) {
  if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) {
    set_error("clearing the amax buffer failed");
    return MOE_ERR_CUDA;
  }
  const int64_t n = static_cast<int64_t>(T) * d;
  int64_t blocks = (n / 8 + 255) / 256;
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  if (blocks < 1) blocks = 1;
  MOE_TRY(launch("fp8_amax", amax_kernel, dim3(static_cast<unsigned>(blocks), 1), dim3(256), 0, st,
                 static_cast<const bf16*>(x), n, reinterpret_cast<unsigned int*>(amax)));
  int rb = (T + 7) / 8;
  if (rb > num_sms() * 8) rb = num_sms() * 8;
  return launch("fp8_permute_quantize", permute_quant_kernel, dim3(rb), dim3(256), 0, st,
                static_cast<const bf16*>(x), sop, reinterpret_cast<const unsigned int*>(amax), xq,
                xq_tok, scale, T, d, k, device_error_word());
}

int launch_quantize_e4m3(const void* x, int64_t per_group, int groups, uint8_t* q, float* scale,
                         float* amax, cudaStream_t st) {
  if (cudaMemsetAsync(amax, 0, sizeof(float) * groups, st) != cudaSuccess) {
    set_error("clearing the amax buffer failed");
    return MOE_ERR_CUDA;
  }
  int64_t want = (per_group / 8 + 255) / 256;
  const int64_t cap = (static_cast<int64_t>(num_sms()) * 8 + groups - 1) / groups;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  const dim3 grid(static_cast<unsigned>(want), static_cast<unsigned>(groups));
  MOE_TRY(launch("fp8_amax", amax_kernel, grid, dim3(256), 0, st, static_cast<const bf16*>(x),
                 per_group, reinterpret_cast<unsigned int*>(amax)));
  return launch("fp8_quantize", quant_kernel, grid, dim3(256), 0, st, static_cast<const bf16*>(x),
                per_group, reinterpret_cast<const unsigned int*>(amax), q, scale);
}

}  // namespace moe
