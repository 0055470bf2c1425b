// Shared device/host helpers of the MoE layer library (no kernels here).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// Device error codes recorded in the error word (first error wins).
enum : int {
  DEVERR_NONE = 0,
  DEVERR_WAIT_TIMEOUT = 1,    // a bounded mbarrier wait ran out
  DEVERR_BAD_EXPERT = 2,      // an expert index outside [0, E)
  DEVERR_BAD_SLOT = 3,        // a slot outside [0, N)
  DEVERR_BAD_OFFSETS = 4,     // offsets not monotone or not ending at N
  DEVERR_SMEM_ALIGN = 5,      // dynamic shared memory not 1024-byte aligned
  DEVERR_BAD_TOKEN = 6,       // a gathered row (token index) outside [0, T)
};

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- element conversion
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<bf16> {
  static __device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ bf16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// A 16-byte vector of elements: 8 bf16 or 4 fp32.
template <typename T> struct Vec16 { static constexpr int n = 16 / sizeof(T); };

__device__ __forceinline__ void unpack16(const uint4& v, float* f, const bf16*) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack16(const uint4& v, float* f, const float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 pack16(const float* f, const bf16*) {
  uint4 v;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}
__device__ __forceinline__ uint4 pack16(const float* f, const float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

// A float as it reads back after being stored as T (round to nearest even for bf16).
__device__ __forceinline__ float as_stored(float v, const bf16*) {
  return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float as_stored(float v, const float*) { return v; }

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld16(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ void st16(void* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}
// Streaming store: written once, not re-read by this kernel.
__device__ __forceinline__ void st16_cs(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

// Two fp32 values -> two E4M3 codes (lo in the low byte): round to nearest even, saturating at
// +-448.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Shared exponent of an MXFP8 block with largest magnitude amax: floor(log2(amax)) - 8 (8: the
// exponent of E4M3's largest normal, 448 = 1.75 * 2^8), clamped to [-127, 127]; -127 for 0 (and
// for subnormal amax, whose floor(log2) is below -126).  Read off the fp32 exponent field.
__device__ __forceinline__ int mx_exponent(float amax) {
  const int fe = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  return fe == 0 ? -127 : max(fe - 135, -127);
}
// 2^-e for a shared exponent e from mx_exponent of a finite amax (e in [-127, 119]): an exact
// power of two and a normal fp32 value.
__device__ __forceinline__ float mx_inv_scale(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// MXFP8 activation scales are packed per 128-row tile of the expert-sorted rows (the GEMMs' row
// tiles).  s_off <- offsets[0..E]; s_pre[e] <- sum over e' < e of ceil(rows_e' / 128).  Called by
// every thread of the block (it synchronises); warp 0 scans.
__device__ __forceinline__ void mx_tile_prefix(const int32_t* offsets, int E, int* s_off,
                                               int* s_pre) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int local = 0;
    for (int e = lo; e < hi; ++e) local += (s_off[e + 1] - s_off[e] + 127) / 128;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = lo; e < hi; ++e) {
      s_pre[e] = run;
      run += (s_off[e + 1] - s_off[e] + 127) / 128;
    }
  }
  __syncthreads();
}
// Byte offset of row `slot`'s scales (its row of its tile's first 512-byte chunk) in the packed
// activation layout with kch 128-element chunks per row (slot < s_off[E]).
__device__ __forceinline__ int64_t mx_row_scale_base(int slot, const int* s_off, const int* s_pre,
                                                     int E, int kch) {
  int lo = 0, hi = E;   // the largest e with s_off[e] <= slot: the expert that holds it
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= slot) lo = mid; else hi = mid;
  }
  const int rr = slot - s_off[lo];
  return (static_cast<int64_t>(s_pre[lo]) + rr / 128) * kch * 512 + ((rr & 127) & 31) * 16 +
         ((rr & 127) >> 5) * 4;
}

}  // namespace moe
