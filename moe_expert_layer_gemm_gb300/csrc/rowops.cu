// Row kernels of the layer: permute, weighted combine and their backward, the shared-expert
// gate, the router's backward, and a fixed-order split reduction.  All are HBM-bound: one warp
// per token, 16-byte vector loads and stores along the row, fp32 arithmetic, fixed summation
// order (no float atomics, so results are bit-for-bit repeatable).
//
// "Megatron-Bridge 深度剖析", §Permute Fusion (tokens regrouped by expert: one memory copy),
// §Expert Parallel 基础 (Step 3: expert outputs sent back to token order and combined),
// §Shared Expert Overlap (shared expert output added to the routed output); the shared-expert
// gate: "Add Megatron-Core MTP training for Qwen3.5 MoE" (What's in it).
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int MAXK = MOE_MAX_TOPK;
constexpr int ROW_THREADS = 256;   // 8 warps per block, one token per warp at a time

// A slot read from memory, checked against [0, T*k): out-of-range values are reported and
// replaced by -1 (the row is then skipped), so a corrupt map cannot cause a wild access.
__device__ __forceinline__ int checked_slot(int s, int Tn, int k, int* err) {
  if (s < 0 || static_cast<int64_t>(s) >= static_cast<int64_t>(Tn) * k) {
    record_error(err, DEVERR_BAD_SLOT);
    return -1;
  }
  return s;
}

static inline dim3 row_grid(int T) {
  const int want = (T + 7) / 8;
  const int cap = num_sms() * 16;
  return dim3(want < cap ? want : cap);
}

// ----------------------------------------------------------------------------- permute
// Scatter by token: row x[t] is read once and written to its k slots (pair (t,j) -> row
// slot_of_pair[t,j] of x_perm).  Same result as gathering x_perm[s] = x[token_of_slot[s]],
// with x read from HBM once instead of k times.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) permute_kernel(const T* __restrict__ x,
                                                              const int32_t* __restrict__ sop,
                                                              T* __restrict__ x_perm, int Tn,
                                                              int d, int k, int* err) {
  constexpr int VE = Vec16<T>::n;
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vpr = d / VE;
  for (int t = gw; t < Tn; t += nw) {
    const int my_slot = lane < k ? checked_slot(sop[static_cast<int64_t>(t) * k + lane], Tn, k, err) : 0;
    int slot[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
    const char* src = reinterpret_cast<const char*>(x + static_cast<int64_t>(t) * d);
    for (int v0 = lane; v0 < vpr; v0 += 32 * U) {
      uint4 r[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * 32;
        if (v < vpr) r[u] = ld_nc16(src + static_cast<int64_t>(v) * 16);
      }
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j >= k) break;
        if (slot[j] < 0) continue;
        char* dst = reinterpret_cast<char*>(x_perm + static_cast<int64_t>(slot[j]) * d);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * 32;
          if (v < vpr) st16(dst + static_cast<int64_t>(v) * 16, r[u]);
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------- combine
// y[t] = sum_{j<k} gate[t,j] * y_perm[slot(t,j)]  (+ c_t * shared_out[t]); fp32, j ascending,
// the shared term last, one rounding.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS, 3) combine_kernel(
    const T* __restrict__ y_perm, const float* __restrict__ gate, const int32_t* __restrict__ sop,
    const T* __restrict__ shared_out, const float* __restrict__ shared_coef, T* __restrict__ y,
    int Tn, int d, int k, int* err) {
  constexpr int VE = Vec16<T>::n;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vpr = d / VE;
  for (int t = gw; t < Tn; t += nw) {
    const int64_t pk = static_cast<int64_t>(t) * k;
    const int my_slot = lane < k ? checked_slot(sop[pk + lane], Tn, k, err) : 0;
    const float my_g = lane < k ? gate[pk + lane] : 0.f;
    const float c = shared_coef ? shared_coef[t] : 1.0f;
    int slot[MAXK];
    float gj[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
      gj[j] = __shfl_sync(0xffffffffu, my_g, j);
    }
    for (int v = lane; v < vpr; v += 32) {
      uint4 raw[MAXK];
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k) {
          const int s = slot[j] < 0 ? 0 : slot[j];
          raw[j] = ld_nc16(reinterpret_cast<const char*>(y_perm + static_cast<int64_t>(s) * d) +
                           static_cast<int64_t>(v) * 16);
        }
      }
      uint4 raw_s = make_uint4(0, 0, 0, 0);   // requested with the routed rows, used last
      if (shared_out)
        raw_s = ld_nc16(reinterpret_cast<const char*>(shared_out + static_cast<int64_t>(t) * d) +
                        static_cast<int64_t>(v) * 16);
      float acc[VE];
#pragma unroll
      for (int i = 0; i < VE; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k) {
          const float g = gj[j];
          float val[VE];
          unpack16(raw[j], val, static_cast<const T*>(nullptr));
#pragma unroll
          for (int i = 0; i < VE; ++i) acc[i] = fmaf(g, val[i], acc[i]);
        }
      }
      if (shared_out) {
        float val[VE];
        unpack16(raw_s, val, static_cast<const T*>(nullptr));
#pragma unroll
        for (int i = 0; i < VE; ++i) acc[i] = fmaf(c, val[i], acc[i]);
      }
      st16(reinterpret_cast<char*>(y + static_cast<int64_t>(t) * d) + static_cast<int64_t>(v) * 16,
           pack16(acc, static_cast<const T*>(nullptr)));
    }
  }
}

// ----------------------------------------------------------------------------- combine bwd
// dy_perm[slot(t,j)] = gate[t,j] * dy[t];  dgate[t,j] = <dy[t], y_perm[slot(t,j)]>;
// dshared[t] = c_t * dy[t];  dcoef[t] = <dy[t], shared_out[t]>.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) combine_bwd_kernel(
    const T* __restrict__ dy, const T* __restrict__ y_perm, const float* __restrict__ gate,
    const int32_t* __restrict__ sop, const T* __restrict__ shared_out,
    const float* __restrict__ shared_coef, T* __restrict__ dy_perm, float* __restrict__ dgate,
    T* __restrict__ dshared, float* __restrict__ dcoef, int Tn, int d, int k, int* err,
    unsigned int* __restrict__ amax_dy, unsigned int* __restrict__ amax_ds) {
  constexpr int VE = Vec16<T>::n;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vpr = d / VE;
  // FP8 backward: max |value| of dy_perm and of dshared as stored (after rounding to T)
  float mdy = 0.f, mds = 0.f;
  auto stored = [](float v) { return fabsf(as_stored(v, static_cast<const T*>(nullptr))); };
  for (int t = gw; t < Tn; t += nw) {
    const int64_t pk = static_cast<int64_t>(t) * k;
    const int my_slot = lane < k ? checked_slot(sop[pk + lane], Tn, k, err) : 0;
    const float my_g = lane < k ? gate[pk + lane] : 0.f;
    const float c = shared_coef ? shared_coef[t] : 1.0f;
    int slot[MAXK];
    float gj[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
      gj[j] = __shfl_sync(0xffffffffu, my_g, j);
    }
    float dot[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) dot[j] = 0.f;
    float dotc = 0.f;
    const char* dyrow = reinterpret_cast<const char*>(dy + static_cast<int64_t>(t) * d);
    for (int v = lane; v < vpr; v += 32) {
      float g_in[VE];
      unpack16(ld_nc16(dyrow + static_cast<int64_t>(v) * 16), g_in, static_cast<const T*>(nullptr));
      uint4 raw[MAXK];
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k) {
          const int s = slot[j] < 0 ? 0 : slot[j];
          raw[j] = ld_nc16(reinterpret_cast<const char*>(y_perm + static_cast<int64_t>(s) * d) +
                           static_cast<int64_t>(v) * 16);
        }
      }
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k) {
          const int s = slot[j];
          const float g = gj[j];
          float yv[VE], o[VE];
          unpack16(raw[j], yv, static_cast<const T*>(nullptr));
#pragma unroll
          for (int i = 0; i < VE; ++i) {
            dot[j] = fmaf(g_in[i], yv[i], dot[j]);
            o[i] = g * g_in[i];
          }
          if (s >= 0) {
            st16(reinterpret_cast<char*>(dy_perm + static_cast<int64_t>(s) * d) +
                     static_cast<int64_t>(v) * 16,
                 pack16(o, static_cast<const T*>(nullptr)));
            if (amax_dy) {
#pragma unroll
              for (int i = 0; i < VE; ++i) mdy = fmaxf(mdy, stored(o[i]));
            }
          }
        }
      }
      if (shared_out) {
        if (dcoef) {
          float sv[VE];
          unpack16(ld_nc16(reinterpret_cast<const char*>(shared_out + static_cast<int64_t>(t) * d) +
                           static_cast<int64_t>(v) * 16),
                   sv, static_cast<const T*>(nullptr));
#pragma unroll
          for (int i = 0; i < VE; ++i) dotc = fmaf(g_in[i], sv[i], dotc);
        }
        if (dshared) {
          float o[VE];
#pragma unroll
          for (int i = 0; i < VE; ++i) o[i] = c * g_in[i];
          st16(reinterpret_cast<char*>(dshared + static_cast<int64_t>(t) * d) +
                   static_cast<int64_t>(v) * 16,
               pack16(o, static_cast<const T*>(nullptr)));
          if (amax_ds) {
#pragma unroll
            for (int i = 0; i < VE; ++i) mds = fmaxf(mds, stored(o[i]));
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (j < k) {
        const float s = warp_sum(dot[j]);
        if (lane == 0) dgate[pk + j] = s;
      }
    }
    if (shared_out && dcoef) {
      const float s = warp_sum(dotc);
      if (lane == 0) dcoef[t] = s;
    }
  }
  // non-negative floats order like their bit patterns
  if (amax_dy) {
    const float m = warp_max(mdy);
    if (lane == 0 && m > 0.f) atomicMax(amax_dy, __float_as_uint(m));
  }
  if (amax_ds) {
    const float m = warp_max(mds);
    if (lane == 0 && m > 0.f) atomicMax(amax_ds, __float_as_uint(m));
  }
}

// The combine backward of an MXFP8 data-gradient backward (bf16 only): as combine_bwd_kernel,
// and each dy_perm row it stores is also quantised to MXFP8 (blocks of 32 along d, from the bf16
// value stored) into dy_q [N, d], with its scales in dy_s in the packed activation layout of the
// routing's 128-row tiles: the fc2 data gradient's A operand, without a second pass over dy_perm.
// A 4-lane group holds one 32-block (8 values a lane), so a block's amax takes two shuffles.
__global__ void __launch_bounds__(ROW_THREADS, 2) combine_bwd_mx_kernel(
    const bf16* __restrict__ dy, const bf16* __restrict__ y_perm, const float* __restrict__ gate,
    const int32_t* __restrict__ sop, const bf16* __restrict__ shared_out,
    const float* __restrict__ shared_coef, bf16* __restrict__ dy_perm, float* __restrict__ dgate,
    bf16* __restrict__ dshared, float* __restrict__ dcoef, int Tn, int d, int k,
    const int32_t* __restrict__ offsets, int E, uint8_t* __restrict__ dy_q,
    uint8_t* __restrict__ dy_s, int* err) {
  __shared__ int s_off[MOE_MAX_EXPERTS + 1];
  __shared__ int s_pre[MOE_MAX_EXPERTS + 1];
  mx_tile_prefix(offsets, E, s_off, s_pre);
  constexpr int VE = 8;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vpr = d / VE;
  const int kch = (d + 127) / 128;
  const int nb = d / 32;
  const bf16* tag = nullptr;
  for (int t = gw; t < Tn; t += nw) {
    const int64_t pk = static_cast<int64_t>(t) * k;
    int my_slot = lane < k ? checked_slot(sop[pk + lane], Tn, k, err) : -1;
    int64_t my_sf = 0;
    if (my_slot >= s_off[E]) {   // beyond the routed rows: the map and the offsets disagree
      record_error(err, DEVERR_BAD_SLOT);
      my_slot = -1;
    }
    if (my_slot >= 0) my_sf = mx_row_scale_base(my_slot, s_off, s_pre, E, kch);
    const float my_g = lane < k ? gate[pk + lane] : 0.f;
    const float c = shared_coef ? shared_coef[t] : 1.0f;
    int slot[MAXK];
    float gj[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
      gj[j] = __shfl_sync(0xffffffffu, my_g, j);
    }
    float dot[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) dot[j] = 0.f;
    float dotc = 0.f;
    const char* dyrow = reinterpret_cast<const char*>(dy + static_cast<int64_t>(t) * d);
    for (int v0 = 0; v0 < vpr; v0 += 32) {   // every lane stays for the group shuffles
      const int v = v0 + lane;
      const bool act = v < vpr;   // d % 32 == 0: a 4-lane group is all in or all out
      float g_in[VE];
      unpack16(act ? ld_nc16(dyrow + static_cast<int64_t>(v) * 16) : make_uint4(0, 0, 0, 0), g_in,
               tag);
      uint4 raw[MAXK];
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k && act) {
          const int s = slot[j] < 0 ? 0 : slot[j];
          raw[j] = ld_nc16(reinterpret_cast<const char*>(y_perm + static_cast<int64_t>(s) * d) +
                           static_cast<int64_t>(v) * 16);
        }
      }
      const int blk = (v * VE) >> 5;
      const bool writes_scale = act && (lane & 3) == 0;
      const bool pads = writes_scale && blk == nb - 1 && (nb & 3) != 0;
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j >= k) break;
        const int s = slot[j];
        float o[VE];
        float m = 0.f;
        if (act) {
          float yv[VE];
          unpack16(raw[j], yv, tag);
#pragma unroll
          for (int i = 0; i < VE; ++i) {
            dot[j] = fmaf(g_in[i], yv[i], dot[j]);
            o[i] = as_stored(gj[j] * g_in[i], tag);   // the bf16 value dy_perm holds
            m = fmaxf(m, fabsf(o[i]));
          }
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int64_t sfb = __shfl_sync(0xffffffffu, my_sf, j);   // (re-read: fewer live registers)
        if (!act || s < 0) continue;
        const int64_t row = static_cast<int64_t>(s) * d;
        st16(reinterpret_cast<char*>(dy_perm + row) + static_cast<int64_t>(v) * 16, pack16(o, tag));
        const int e = mx_exponent(m);
        const float inv = mx_inv_scale(e);
        uint32_t w[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t lo = cvt_e4m3x2(o[4 * q] * inv, o[4 * q + 1] * inv);
          const uint32_t hi = cvt_e4m3x2(o[4 * q + 2] * inv, o[4 * q + 3] * inv);
          w[q] = lo | (hi << 16);
        }
        *reinterpret_cast<uint2*>(dy_q + row + static_cast<int64_t>(v) * VE) =
            make_uint2(w[0], w[1]);
        if (writes_scale) {
          uint8_t* sf = dy_s + sfb + (blk >> 2) * MX_CHUNK;
          sf[blk & 3] = static_cast<uint8_t>(e + 127);
          if (pads)
            for (int q = (blk & 3) + 1; q < 4; ++q) sf[q] = 127;   // blocks past d: 2^0
        }
      }
      if (shared_out && act) {
        if (dcoef) {
          float sv[VE];
          unpack16(ld_nc16(reinterpret_cast<const char*>(shared_out + static_cast<int64_t>(t) * d) +
                           static_cast<int64_t>(v) * 16),
                   sv, tag);
#pragma unroll
          for (int i = 0; i < VE; ++i) dotc = fmaf(g_in[i], sv[i], dotc);
        }
        if (dshared) {
          float o[VE];
#pragma unroll
          for (int i = 0; i < VE; ++i) o[i] = c * g_in[i];
          st16(reinterpret_cast<char*>(dshared + static_cast<int64_t>(t) * d) +
                   static_cast<int64_t>(v) * 16,
               pack16(o, tag));
        }
      }
    }
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (j < k) {
        const float s = warp_sum(dot[j]);
        if (lane == 0) dgate[pk + j] = s;
      }
    }
    if (shared_out && dcoef) {
      const float s = warp_sum(dotc);
      if (lane == 0) dcoef[t] = s;
    }
  }
}

// ----------------------------------------------------------------------------- permute bwd
// dx[t] = sum_j dx_perm[slot(t,j)] + dx_shared[t] + dx_router[t] + dz[t] * w_sg  (fp32, that
// order, one rounding).  Optional terms are skipped when their pointer is null.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS, 3) gather_sum_kernel(
    const T* __restrict__ dx_perm, const int32_t* __restrict__ sop, const T* __restrict__ dx_shared,
    const T* __restrict__ dx_router, const float* __restrict__ dz, const T* __restrict__ w_sg,
    T* __restrict__ dx, int Tn, int d, int k, int* err) {
  constexpr int VE = Vec16<T>::n;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vpr = d / VE;
  for (int t = gw; t < Tn; t += nw) {
    const int64_t pk = static_cast<int64_t>(t) * k;
    const int my_slot = lane < k ? checked_slot(sop[pk + lane], Tn, k, err) : 0;
    const float zt = dz ? dz[t] : 0.f;
    int slot[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) slot[j] = __shfl_sync(0xffffffffu, my_slot, j);
    for (int v = lane; v < vpr; v += 32) {
      uint4 raw[MAXK];
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k) {
          const int s = slot[j] < 0 ? 0 : slot[j];
          raw[j] = ld_nc16(reinterpret_cast<const char*>(dx_perm + static_cast<int64_t>(s) * d) +
                           static_cast<int64_t>(v) * 16);
        }
      }
      // the per-token terms are requested with the routed rows and added after them
      const int64_t ro = static_cast<int64_t>(t) * d * sizeof(T) + static_cast<int64_t>(v) * 16;
      uint4 raw_s = make_uint4(0, 0, 0, 0), raw_r = make_uint4(0, 0, 0, 0);
      if (dx_shared) raw_s = ld_nc16(reinterpret_cast<const char*>(dx_shared) + ro);
      if (dx_router) raw_r = ld_nc16(reinterpret_cast<const char*>(dx_router) + ro);
      float acc[VE];
#pragma unroll
      for (int i = 0; i < VE; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < k) {
          float val[VE];
          unpack16(raw[j], val, static_cast<const T*>(nullptr));
#pragma unroll
          for (int i = 0; i < VE; ++i) acc[i] += val[i];
        }
      }
      if (dx_shared) {
        float val[VE];
        unpack16(raw_s, val, static_cast<const T*>(nullptr));
#pragma unroll
        for (int i = 0; i < VE; ++i) acc[i] += val[i];
      }
      if (dx_router) {
        float val[VE];
        unpack16(raw_r, val, static_cast<const T*>(nullptr));
#pragma unroll
        for (int i = 0; i < VE; ++i) acc[i] += val[i];
      }
      if (dz) {
        float wv[VE];
        unpack16(ld_nc16(reinterpret_cast<const char*>(w_sg) + static_cast<int64_t>(v) * 16), wv,
                 static_cast<const T*>(nullptr));
#pragma unroll
        for (int i = 0; i < VE; ++i) acc[i] = fmaf(zt, wv[i], acc[i]);
      }
      st16(reinterpret_cast<char*>(dx) + ro, pack16(acc, static_cast<const T*>(nullptr)));
    }
  }
}

// ----------------------------------------------------------------------------- shared gate
// coef[t] = sigmoid(<x[t], w_sg>).
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) shared_gate_kernel(const T* __restrict__ x,
                                                                  const T* __restrict__ w_sg,
                                                                  float* __restrict__ coef, int Tn,
                                                                  int d) {
  constexpr int VE = Vec16<T>::n;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vpr = d / VE;
  for (int t = gw; t < Tn; t += nw) {
    float acc = 0.f;
    for (int v = lane; v < vpr; v += 32) {
      float xv[VE], wv[VE];
      unpack16(ld_nc16(reinterpret_cast<const char*>(x + static_cast<int64_t>(t) * d) +
                       static_cast<int64_t>(v) * 16),
               xv, static_cast<const T*>(nullptr));
      unpack16(ld_nc16(reinterpret_cast<const char*>(w_sg) + static_cast<int64_t>(v) * 16), wv,
               static_cast<const T*>(nullptr));
#pragma unroll
      for (int i = 0; i < VE; ++i) acc = fmaf(xv[i], wv[i], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) coef[t] = sigmoid_f(acc);
  }
}

// ----------------------------------------------------------------------------- router bwd
// dL/dlogits from dL/dgate through the gate function (selection carries no gradient):
//   softmax, renorm:    dl_j = g_j (dg_j - sum_i g_i dg_i)                    (selected j)
//   softmax, no renorm: dl_e = p_e (dG_e - sum_j g_j dg_j), dG_e = dg_j at e = idx_j, else 0
//   sigmoid, renorm:    dl_j = (dg_j - sum_i g_i dg_i) s_j (1 - s_j) / sum_i s_i
//   sigmoid, no renorm: dl_j = dg_j s_j (1 - s_j)
// Row t of dl_ext [T, ld_ext] holds dl[t, 0..E-1], then (shared gate) dz_t = dc_t c_t (1-c_t)
// in column E, then zeros.  dz is also written in fp32 to dz[t].
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS) router_bwd_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ gate, const float* __restrict__ dgate,
    const float* __restrict__ dcoef, const float* __restrict__ coef, T* __restrict__ dl_ext,
    float* __restrict__ dz, int Tn, int E, int k, int ld_ext, int score_fn, int renorm,
    const int32_t* __restrict__ aux_counts, float aux_w, int* err) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int t = gw; t < Tn; t += nw) {
    const int64_t pk = static_cast<int64_t>(t) * k;
    const float* lrow = logits + static_cast<int64_t>(t) * E;
    int my_e = -1;
    float my_g = 0.f, my_dg = 0.f;
    if (lane < k) {
      my_e = idx[pk + lane];
      if (my_e < 0 || my_e >= E) {
        record_error(err, DEVERR_BAD_EXPERT);
        my_e = 0;
      }
      my_g = gate[pk + lane];
      my_dg = dgate[pk + lane];
    }
    float my_s = 0.f;
    if (score_fn == MOE_SCORE_SIGMOID && lane < k) my_s = sigmoid_f(lrow[my_e]);
    // every lane gets the k selected (expert, gate, dgate, score); inner = sum_j g_j dg_j and
    // ssum = sum_j s_j in ascending j, identical on all lanes
    int sel_e[MAXK];
    float sel_g[MAXK], sel_dg[MAXK], sel_s[MAXK];
    float inner = 0.f, ssum = 0.f;
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      sel_e[j] = __shfl_sync(0xffffffffu, my_e, j);
      sel_g[j] = __shfl_sync(0xffffffffu, my_g, j);
      sel_dg[j] = __shfl_sync(0xffffffffu, my_dg, j);
      sel_s[j] = __shfl_sync(0xffffffffu, my_s, j);
      if (j < k) {
        inner = fmaf(sel_g[j], sel_dg[j], inner);
        ssum += sel_s[j];
      }
    }
    // softmax over all E (no renorm, or the balancing loss): row maximum and normaliser
    float m = 0.f, denom = 1.f;
    const bool full_softmax = score_fn == MOE_SCORE_SOFTMAX && (!renorm || aux_counts);
    if (full_softmax) {
      float mx = __int_as_float(0xff800000u);
      for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lrow[e]);
      m = warp_max(mx);
      float part = 0.f;
      for (int e = lane; e < E; e += 32) part += expf(lrow[e] - m);
      denom = warp_sum(part);
    }
    // Balancing loss (counts held fixed): w_e = aux_w * counts[e] = dL/dp[t,e],
    // G = sum_e p[t,e] w_e;  softmax: dl_e += p_e (w_e - G);
    // sigmoid (p = s / S): dl_e += s_e (1 - s_e) (w_e - G) / S.
    float aux_G = 0.f, aux_S = 1.f;
    if (aux_counts) {
      float pw = 0.f, ps = 0.f;
      for (int e = lane; e < E; e += 32) {
        const float w = aux_w * static_cast<float>(aux_counts[e]);
        const float v = score_fn == MOE_SCORE_SOFTMAX ? expf(lrow[e] - m) : sigmoid_f(lrow[e]);
        pw = fmaf(v, w, pw);
        ps += v;
      }
      pw = warp_sum(pw);
      if (score_fn == MOE_SCORE_SOFTMAX) {
        aux_G = pw / denom;
      } else {
        aux_S = warp_sum(ps);
        aux_G = pw / aux_S;
      }
    }
    float dzt = 0.f;
    if (dcoef) {
      const float c = coef[t];
      dzt = dcoef[t] * c * (1.0f - c);
      if (lane == 0) dz[t] = dzt;
    }
    T* orow = dl_ext + static_cast<int64_t>(t) * ld_ext;
    for (int c0 = 0; c0 < ld_ext; c0 += 32) {
      const int col = c0 + lane;
      float val = 0.f;
      if (col < E) {
        int jsel = -1;
        float dgj = 0.f, gj = 0.f, sj = 0.f;
#pragma unroll
        for (int j = 0; j < MAXK; ++j) {
          if (j < k && sel_e[j] == col) {
            jsel = j;
            dgj = sel_dg[j];
            gj = sel_g[j];
            sj = sel_s[j];
          }
        }
        if (score_fn == MOE_SCORE_SOFTMAX) {
          if (renorm) {
            if (jsel >= 0) val = gj * (dgj - inner);
          } else {
            const float p = expf(lrow[col] - m) / denom;
            val = p * ((jsel >= 0 ? dgj : 0.f) - inner);
          }
        } else if (jsel >= 0) {
          val = renorm ? (dgj - inner) * sj * (1.0f - sj) / ssum : dgj * sj * (1.0f - sj);
        }
        if (aux_counts) {
          const float w = aux_w * static_cast<float>(aux_counts[col]);
          if (score_fn == MOE_SCORE_SOFTMAX) {
            val += expf(lrow[col] - m) / denom * (w - aux_G);
          } else {
            const float sc = sigmoid_f(lrow[col]);
            val += sc * (1.0f - sc) * (w - aux_G) / aux_S;
          }
        }
      } else if (col == E && dcoef) {
        val = dzt;
      }
      if (col < ld_ext) orow[col] = Elem<T>::from_f(val);
    }
  }
}

// ----------------------------------------------------------------------------- split reduce
// out_main[r][c] = sum_{s<S} part[s][r][c] for r < main_rows; row main_rows -> out_extra[c].
__global__ void split_reduce_kernel(const float* __restrict__ part, int S, int rows, int cols,
                                    float* __restrict__ out_main, int main_rows,
                                    float* __restrict__ out_extra) {
  const int64_t n = static_cast<int64_t>(rows) * cols;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) acc += part[static_cast<int64_t>(s) * n + i];
    const int64_t r = i / cols, c = i % cols;
    if (r < main_rows)
      out_main[i] = acc;
    else if (r == main_rows && out_extra)
      out_extra[c] = acc;
  }
}

// ----------------------------------------------------------------------------- launchers
int launch_permute(int dtype, const void* x, const int32_t* sop, void* x_perm, int T, int d, int k,
                   cudaStream_t st) {
  if (dtype == MOE_DTYPE_BF16)
    return launch("permute", permute_kernel<bf16>, row_grid(T), dim3(ROW_THREADS), 0, st,
                  (const bf16*)x, sop, (bf16*)x_perm, T, d, k, device_error_word());
  return launch("permute", permute_kernel<float>, row_grid(T), dim3(ROW_THREADS), 0, st,
                (const float*)x, sop, (float*)x_perm, T, d, k, device_error_word());
}

int launch_combine(int dtype, const void* y_perm, const float* gate, const int32_t* sop,
                   const void* shared_out, const float* shared_coef, void* y, int T, int d, int k,
                   cudaStream_t st) {
  if (dtype == MOE_DTYPE_BF16)
    return launch("combine", combine_kernel<bf16>, row_grid(T), dim3(ROW_THREADS), 0, st,
                  (const bf16*)y_perm, gate, sop, (const bf16*)shared_out, shared_coef, (bf16*)y,
                  T, d, k, device_error_word());
  return launch("combine", combine_kernel<float>, row_grid(T), dim3(ROW_THREADS), 0, st,
                (const float*)y_perm, gate, sop, (const float*)shared_out, shared_coef, (float*)y,
                T, d, k, device_error_word());
}

int launch_combine_bwd(int dtype, const void* dy, const void* y_perm, const float* gate,
                       const int32_t* sop, const void* shared_out, const float* shared_coef,
                       void* dy_perm, float* dgate, void* dshared, float* dcoef, int T, int d, int k,
                       cudaStream_t st, float* amax_dy, float* amax_ds) {
  auto* ady = reinterpret_cast<unsigned int*>(amax_dy);
  auto* ads = reinterpret_cast<unsigned int*>(amax_ds);
  if (dtype == MOE_DTYPE_BF16)
    return launch("combine_bwd", combine_bwd_kernel<bf16>, row_grid(T), dim3(ROW_THREADS), 0, st,
                  (const bf16*)dy, (const bf16*)y_perm, gate, sop, (const bf16*)shared_out,
                  shared_coef, (bf16*)dy_perm, dgate, (bf16*)dshared, dcoef, T, d, k,
                  device_error_word(), ady, ads);
  return launch("combine_bwd", combine_bwd_kernel<float>, row_grid(T), dim3(ROW_THREADS), 0, st,
                (const float*)dy, (const float*)y_perm, gate, sop, (const float*)shared_out,
                shared_coef, (float*)dy_perm, dgate, (float*)dshared, dcoef, T, d, k,
                device_error_word(), ady, ads);
}

int launch_combine_bwd_mx(const void* dy, const void* y_perm, const float* gate,
                          const int32_t* sop, const void* shared_out, const float* shared_coef,
                          void* dy_perm, float* dgate, void* dshared, float* dcoef, int T, int d,
                          int k, const int32_t* offsets, int E, uint8_t* dy_q, uint8_t* dy_s,
                          cudaStream_t st) {
  return launch("combine_bwd_mxfp8", combine_bwd_mx_kernel, row_grid(T), dim3(ROW_THREADS), 0, st,
                (const bf16*)dy, (const bf16*)y_perm, gate, sop, (const bf16*)shared_out,
                shared_coef, (bf16*)dy_perm, dgate, (bf16*)dshared, dcoef, T, d, k, offsets, E,
                dy_q, dy_s, device_error_word());
}

int launch_gather_sum(int dtype, const void* dx_perm, const int32_t* sop, const void* dx_shared,
                      const void* dx_router, const float* dz, const void* w_sg, void* dx, int T,
                      int d, int k, cudaStream_t st) {
  if (dtype == MOE_DTYPE_BF16)
    return launch("permute_bwd", gather_sum_kernel<bf16>, row_grid(T), dim3(ROW_THREADS), 0, st,
                  (const bf16*)dx_perm, sop, (const bf16*)dx_shared, (const bf16*)dx_router, dz,
                  (const bf16*)w_sg, (bf16*)dx, T, d, k, device_error_word());
  return launch("permute_bwd", gather_sum_kernel<float>, row_grid(T), dim3(ROW_THREADS), 0, st,
                (const float*)dx_perm, sop, (const float*)dx_shared, (const float*)dx_router, dz,
                (const float*)w_sg, (float*)dx, T, d, k, device_error_word());
}

int launch_shared_gate(int dtype, const void* x, const void* w_sg, float* coef, int T, int d,
                       cudaStream_t st) {
  if (dtype == MOE_DTYPE_BF16)
    return launch("shared_gate", shared_gate_kernel<bf16>, row_grid(T), dim3(ROW_THREADS), 0, st,
                  (const bf16*)x, (const bf16*)w_sg, coef, T, d);
  return launch("shared_gate", shared_gate_kernel<float>, row_grid(T), dim3(ROW_THREADS), 0, st,
                (const float*)x, (const float*)w_sg, coef, T, d);
}

int launch_router_bwd(int dtype, const float* logits, const int32_t* idx, const float* gate,
                      const float* dgate, const float* dcoef, const float* coef, void* dl_ext,
                      float* dz, int T, int E, int k, int ld_ext, int score_fn, int renorm,
                      const int32_t* aux_counts, float aux_w, cudaStream_t st) {
  if (dtype == MOE_DTYPE_BF16)
    return launch("router_bwd", router_bwd_kernel<bf16>, row_grid(T), dim3(ROW_THREADS), 0, st,
                  logits, idx, gate, dgate, dcoef, coef, (bf16*)dl_ext, dz, T, E, k, ld_ext,
                  score_fn, renorm, aux_counts, aux_w, device_error_word());
  return launch("router_bwd", router_bwd_kernel<float>, row_grid(T), dim3(ROW_THREADS), 0, st,
                logits, idx, gate, dgate, dcoef, coef, (float*)dl_ext, dz, T, E, k, ld_ext,
                score_fn, renorm, aux_counts, aux_w, device_error_word());
}

int launch_split_reduce(const float* part, int S, int rows, int cols, float* out_main,
                        int main_rows, float* out_extra, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(rows) * cols;
  int64_t blocks = (n + 255) / 256;
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  return launch("split_reduce", split_reduce_kernel, dim3(static_cast<unsigned>(blocks)),
                dim3(256), 0, st, part, S, rows, cols, out_main, main_rows, out_extra);
}

}  // namespace moe
