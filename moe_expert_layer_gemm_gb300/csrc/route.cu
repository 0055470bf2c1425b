// Routing: top-k selection + gates, per-expert histogram, prefix sum, token<->slot maps.
//
// "Megatron-Bridge 深度剖析", §Expert Parallel 基础 (workflow figure, Step 1: the router
// picks the top-k experts of every token; Step 2: tokens are regrouped by expert).  On one GPU
// the dispatch plan of Step 2 is a stable counting sort of the (token, expert) pairs:
//   counts[e], offsets[e] = sum_{e'<e} counts[e'],
//   slot(t, j) = offsets[e] + #{t' < t : t' picked e},  e = idx[t, j].
//
// Four launches:
//   topk  -- one warp per token (grid-stride over all tokens): k rounds of a warp-wide argmax
//            over fp32 logits (ties -> lower expert index), gates in fp32.
//   hist  -- one block per 256 tokens: per-expert counts of the block, hist[e][block].
//   scan  -- one block: exclusive prefix over hist in expert-major order gives, for every
//            (expert, block), the first slot of that block's tokens of that expert.
//   slots -- per block: per-expert bitmasks of the block's tokens; the rank of token t among
//            the block's tokens of expert e is the popcount of the mask bits below t.
// All integer, so the result is exact and independent of scheduling.
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int TPB = ROUTE_TOK_PER_BLOCK;   // tokens per histogram / slot block
constexpr int MASK_WORDS = TPB / 32;        // 8 words of 32 token bits per expert
constexpr int MAXK = MOE_MAX_TOPK;
#define NEG_INF __int_as_float(0xff800000u)

template <int EPL>
__device__ __forceinline__ void load_logit_row(const float* __restrict__ logits, int t, int T,
                                               int E, int lane, float (&v)[EPL]) {
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = q * 32 + lane;
    v[q] = (t < T && e < E) ? __ldg(logits + static_cast<int64_t>(t) * E + e) : NEG_INF;
  }
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                   int k, int score_fn, int renorm,
                                                   int32_t* __restrict__ idx,
                                                   float* __restrict__ gate) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  float cur[EPL], nxt[EPL];
  load_logit_row<EPL>(logits, gw, T, E, lane, cur);

  for (int t = gw; t < T; t += nw) {
    load_logit_row<EPL>(logits, t + nw, T, E, lane, nxt);   // next token's row in flight

    // ---- selection: k rounds of warp argmax, key (logit desc, expert asc)
    uint32_t taken = 0u;
    float sel_v[MAXK];
    int sel_e[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      sel_v[j] = NEG_INF;
      sel_e[j] = 0;
      if (j < k) {
        float bv = NEG_INF;
        int be = INT_MAX;
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
          const int e = q * 32 + lane;
          if (!((taken >> q) & 1u) && e < E && (cur[q] > bv || (cur[q] == bv && e < be))) {
            bv = cur[q];
            be = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        sel_v[j] = bv;
        sel_e[j] = be;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
      }
    }

    // ---- gates (fp32)
    float g[MAXK];
    if (score_fn == MOE_SCORE_SOFTMAX) {
      const float m = sel_v[0];   // the top-1 logit is the row maximum
      float denom = 0.f;
      if (renorm) {
#pragma unroll
        for (int j = 0; j < MAXK; ++j)
          if (j < k) denom += expf(sel_v[j] - m);
      } else {
        float part = 0.f;
#pragma unroll
        for (int q = 0; q < EPL; ++q)
          if (q * 32 + lane < E) part += expf(cur[q] - m);
        denom = warp_sum(part);
      }
      const float inv = 1.0f / denom;
#pragma unroll
      for (int j = 0; j < MAXK; ++j) g[j] = expf(sel_v[j] - m) * inv;
    } else {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        g[j] = sigmoid_f(sel_v[j]);
        if (j < k) sum += g[j];
      }
      if (renorm) {
        const float inv = 1.0f / sum;
#pragma unroll
        for (int j = 0; j < MAXK; ++j) g[j] *= inv;
      }
    }

    // ---- outputs: lane j writes pair j
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (j < k && lane == j) {
        idx[static_cast<int64_t>(t) * k + j] = sel_e[j];
        gate[static_cast<int64_t>(t) * k + j] = g[j];
      }
    }
#pragma unroll
    for (int q = 0; q < EPL; ++q) cur[q] = nxt[q];
  }
}

// Per-block expert counts: hist[e][b] = number of tokens of block b (256 tokens) that picked e.
__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                   int E, int32_t* __restrict__ hist, int nblk,
                                                   int* err) {
  __shared__ int cnt[MOE_MAX_EXPERTS];
  const int tid = threadIdx.x;
  for (int i = tid; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * TPB + tid;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[static_cast<int64_t>(t) * k + j];
      if (e < 0 || e >= E) record_error(err, DEVERR_BAD_EXPERT);
      else atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) hist[static_cast<int64_t>(e) * nblk + blockIdx.x] = cnt[e];
}

// Exclusive prefix sum over hist[E][nblk] (expert-major) by one block of 1024 threads.
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ hist, int E,
                                                    int nblk, int32_t* __restrict__ base,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = E * nblk;
  const int chunk = (L + blockDim.x - 1) / blockDim.x;
  const int lo = min(L, tid * chunk), hi = min(L, lo + chunk);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += hist[i];
  // block-wide exclusive scan of `local`
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? warp_tot[lane] : 0;
    int s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    if (lane < nw) warp_tot[lane] = s - v;   // exclusive prefix of warp totals
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    base[i] = run;
    run += hist[i];
  }
  __syncthreads();
  int total = 0;
  if (L > 0) total = base[L - 1] + hist[L - 1];
  for (int e = tid; e < E; e += blockDim.x) {
    const int start = base[static_cast<int64_t>(e) * nblk];
    const int end = (e + 1 < E) ? base[static_cast<int64_t>(e + 1) * nblk] : total;
    counts[e] = end - start;
    offsets[e] = start;
  }
  if (tid == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(256) slots_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                    int E, const int32_t* __restrict__ base,
                                                    int nblk, int32_t* __restrict__ slot_of_pair,
                                                    int32_t* __restrict__ token_of_slot,
                                                    int* err) {
  __shared__ uint32_t mask[MOE_MAX_EXPERTS * MASK_WORDS];
  const int tid = threadIdx.x;
  for (int i = tid; i < E * MASK_WORDS; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  const int t = blockIdx.x * TPB + tid;
  const int w = tid >> 5, bit = tid & 31;
  int ev[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    ev[j] = -1;
    if (j < k && t < T) {
      int e = idx[static_cast<int64_t>(t) * k + j];
      if (e < 0 || e >= E) {
        record_error(err, DEVERR_BAD_EXPERT);
        e = -1;
      } else {
        atomicOr(&mask[e * MASK_WORDS + w], 1u << bit);
      }
      ev[j] = e;
    }
  }
  __syncthreads();
  const int64_t N = static_cast<int64_t>(T) * k;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    const int e = ev[j];
    if (e < 0) continue;
    int rank = __popc(mask[e * MASK_WORDS + w] & ((1u << bit) - 1u));
    for (int ww = 0; ww < w; ++ww) rank += __popc(mask[e * MASK_WORDS + ww]);
    const int s = base[static_cast<int64_t>(e) * nblk + blockIdx.x] + rank;
    if (s < 0 || s >= N) {
      record_error(err, DEVERR_BAD_SLOT);
      continue;
    }
    slot_of_pair[static_cast<int64_t>(t) * k + j] = s;
    token_of_slot[s] = t;
  }
}

int launch_topk(const float* logits, int T, int E, int k, int score_fn, int renorm, int32_t* idx,
                float* gate, int32_t* hist, cudaStream_t st) {
  const int nblk = route_blocks(T);
  int blocks = (T + 7) / 8;   // 8 warps per block, one token per warp at a time
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  const dim3 grid(blocks), block(256);
  int rc;
  if (E <= 32)
    rc = launch("route_topk", topk_kernel<1>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                idx, gate);
  else if (E <= 64)
    rc = launch("route_topk", topk_kernel<2>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                idx, gate);
  else if (E <= 128)
    rc = launch("route_topk", topk_kernel<4>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                idx, gate);
  else
    rc = launch("route_topk", topk_kernel<8>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                idx, gate);
  MOE_TRY(rc);
  return launch("route_hist", hist_kernel, dim3(nblk), dim3(TPB), 0, st, idx, T, k, E, hist, nblk,
                device_error_word());
}

int launch_scan(const int32_t* hist, int E, int nblk, int32_t* base, int32_t* counts,
                int32_t* offsets, cudaStream_t st) {
  return launch("route_scan", scan_kernel, dim3(1), dim3(1024), 0, st, hist, E, nblk, base,
                counts, offsets);
}

int launch_slots(const int32_t* idx, int T, int k, int E, const int32_t* base,
                 int32_t* slot_of_pair, int32_t* token_of_slot, cudaStream_t st) {
  const int nblk = route_blocks(T);
  return launch("route_slots", slots_kernel, dim3(nblk), dim3(256), 0, st, idx, T, k, E, base,
                nblk, slot_of_pair, token_of_slot, device_error_word());
}

}  // namespace moe
