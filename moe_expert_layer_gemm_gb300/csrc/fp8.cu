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

// Two fp32 values -> two E4M3 codes (lo in the low byte).
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

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

}  // namespace

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
