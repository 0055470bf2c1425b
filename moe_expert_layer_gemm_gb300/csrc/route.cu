// Routing: top-k selection + gates, per-expert histogram, prefix sum, token<->slot maps.
//
// "Megatron-Bridge 深度剖析", §Expert Parallel 基础 (workflow figure, Step 1: the router
// picks the top-k experts of every token; Step 2: tokens are regrouped by expert).  On one GPU
// the dispatch plan of Step 2 is a stable counting sort of the (token, expert) pairs:
//   counts[e], offsets[e] = sum_{e'<e} counts[e'],
//   slot(t, j) = offsets[e] + #{t' < t : t' picked e},  e = idx[t, j].
//
// Four launches:
//   topk  -- one warp per token (grid-stride over all tokens): k rounds of a warp-wide max
//            (fp32 key, ties to the lower expert index), gates in fp32, lane j computing pair
//            j's.  The key is the logit,
//            or, with a selection-only expert bias ("Megatron-Bridge 深度剖析",
//            §Nemotron-3-Nano 配置: sigmoid routing with expert-bias correction as in DeepSeek
//            V3), the fp32 score (softmax over E, or sigmoid) plus the expert's bias.
//   hist  -- one block per 256 tokens: per-expert counts of the block, hist[e][block].
//   scan  -- one block per expert: the exclusive prefix of its row of hist (the first slot of
//            each block's tokens of that expert, counted from the expert's first slot) and
//            its count.
//   slots -- per block: offsets = the exclusive scan of counts (formed by every block, written
//            out by block 0); per-expert bitmasks of the block's tokens; the rank of token t
//            among the block's tokens of expert e is the popcount of the mask bits below t.
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

// A float as an unsigned integer with the same order (for single-instruction warp reductions);
// -0 becomes +0 first, so that the two zeros tie as they compare equal.
__device__ __forceinline__ unsigned ordered_key(float f) {
  unsigned b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Sum over lanes 0..7 (k <= 8 pairs live there, the other lanes hold zeros), result in lane 0
// and every lane of its group of eight.  The same value as a full-warp butterfly over those
// lanes: the skipped steps would only add zeros.
__device__ __forceinline__ float sum8(float v) {
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                   int k, int score_fn, int renorm,
                                                   const float* __restrict__ sel_bias,
                                                   int32_t* __restrict__ idx,
                                                   float* __restrict__ gate, int* err) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  float cur[EPL], nxt[EPL], bias[EPL];
  load_logit_row<EPL>(logits, gw, T, E, lane, cur);
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = q * 32 + lane;
    bias[q] = (sel_bias && e < E) ? __ldg(sel_bias + e) : 0.f;
  }

  for (int t = gw; t < T; t += nw) {
    load_logit_row<EPL>(logits, t + nw, T, E, lane, nxt);   // next token's row in flight

    // ---- selection keys: the logits, or score + expert bias (row max kept for the gates)
    float key[EPL];
    float rmax = NEG_INF;
    if (sel_bias) {
      if (score_fn == MOE_SCORE_SOFTMAX) {
#pragma unroll
        for (int q = 0; q < EPL; ++q) rmax = fmaxf(rmax, cur[q]);
        rmax = warp_max(rmax);
        float ex[EPL], part = 0.f;
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
          ex[q] = (q * 32 + lane < E) ? expf(cur[q] - rmax) : 0.f;
          part += ex[q];
        }
        const float z = warp_sum(part);
#pragma unroll
        for (int q = 0; q < EPL; ++q)
          key[q] = (q * 32 + lane < E) ? ex[q] / z + bias[q] : NEG_INF;
      } else {
#pragma unroll
        for (int q = 0; q < EPL; ++q)
          key[q] = (q * 32 + lane < E) ? sigmoid_f(cur[q]) + bias[q] : NEG_INF;
      }
    } else {
#pragma unroll
      for (int q = 0; q < EPL; ++q) key[q] = cur[q];
    }

    // ---- selection: k rounds of a warp-wide max, order (key desc, expert asc).  Each lane first
    // sorts its EPL (key, expert) pairs, so a round compares only the lanes' heads: the largest
    // key, then the lowest expert among the lanes holding it -- two single-instruction warp
    // reductions (redux.sync) on the keys as order-preserving integers.  The winning lane moves
    // on to its next pair.
    unsigned hk[EPL];
    int he[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = q * 32 + lane;
      // a NaN key (outside the inputs' contract) ranks as -inf, so every round still has a
      // maximum that some lane holds and the selection stays within [0, E)
      hk[q] = ordered_key((e < E && key[q] == key[q]) ? key[q] : NEG_INF);
      he[q] = e < E ? e : INT_MAX;
    }
#pragma unroll
    for (int i = 1; i < EPL; ++i)          // insertion sort, (key desc, expert asc)
#pragma unroll
      for (int q = i; q > 0; --q)
        if (hk[q] > hk[q - 1] || (hk[q] == hk[q - 1] && he[q] < he[q - 1])) {
          const unsigned tk = hk[q];
          hk[q] = hk[q - 1];
          hk[q - 1] = tk;
          const int te = he[q];
          he[q] = he[q - 1];
          he[q - 1] = te;
        }
    int my_e = 0;                          // lane j: the j-th selected expert
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (j < k) {
        const unsigned m = __reduce_max_sync(0xffffffffu, hk[0]);
        const int e = __reduce_min_sync(0xffffffffu, hk[0] == m ? he[0] : INT_MAX);
        if (lane == j) my_e = e;
        if ((e & 31) == lane) {            // the winner drops its head
#pragma unroll
          for (int q = 0; q + 1 < EPL; ++q) {
            hk[q] = hk[q + 1];
            he[q] = he[q + 1];
          }
          hk[EPL - 1] = 0u;   // below every key (-inf is 0x007FFFFF)
          he[EPL - 1] = INT_MAX;
        }
      }
    }

    // ---- gates (fp32), lane j for pair j: the selected expert's logit (in L1 from the row load)
    if (lane < k && (my_e < 0 || my_e >= E)) {   // cannot happen; never index with it
      record_error(err, DEVERR_BAD_EXPERT);
      my_e = 0;
    }
    const float lv = lane < k ? __ldg(logits + static_cast<int64_t>(t) * E + my_e) : NEG_INF;
    float g;
    if (score_fn == MOE_SCORE_SOFTMAX) {
      // shift: the row maximum (over all E without renorm, over the selected with it); without
      // a selection bias the top-1 logit is both
      float m;
      if (!sel_bias) m = __shfl_sync(0xffffffffu, lv, 0);
      else if (renorm) m = __shfl_sync(0xffffffffu, warp_max(lv), 0);
      else m = rmax;
      const float ex = lane < k ? expf(lv - m) : 0.f;
      float denom;
      if (renorm) {
        denom = sum8(ex);   // pairs live in lanes 0..k-1
      } else {
        float part = 0.f;
#pragma unroll
        for (int q = 0; q < EPL; ++q)
          if (q * 32 + lane < E) part += expf(cur[q] - m);
        denom = warp_sum(part);
      }
      denom = __shfl_sync(0xffffffffu, denom, 0);   // one value for every lane
      g = ex * (1.0f / denom);
    } else {
      g = lane < k ? sigmoid_f(lv) : 0.f;
      if (renorm) {
        const float sum = __shfl_sync(0xffffffffu, sum8(g), 0);
        g *= 1.0f / sum;
      }
    }

    // ---- outputs: lane j writes pair j
    if (lane < k) {
      idx[static_cast<int64_t>(t) * k + lane] = my_e;
      gate[static_cast<int64_t>(t) * k + lane] = g;
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

// Per expert e (one block each): the exclusive prefix of hist[e][0..nblk) -- the first slot of
// block b's tokens of expert e, counted from the expert's first slot -- and the row total
// counts[e].  Each thread takes 8 consecutive entries; a block-wide scan of the threads' sums
// gives their starts.  The experts' own offsets are the scan of counts, which every slots block
// forms itself (it needs all of them).
constexpr int RSCAN_THREADS = 256;
constexpr int RSCAN_PER = 8;

__global__ void __launch_bounds__(RSCAN_THREADS) row_scan_kernel(const int32_t* __restrict__ hist,
                                                                 int nblk,
                                                                 int32_t* __restrict__ rowpre,
                                                                 int32_t* __restrict__ counts) {
  __shared__ int warp_tot[RSCAN_THREADS / 32];
  __shared__ int chunk_tot;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* row = hist + static_cast<int64_t>(blockIdx.x) * nblk;
  int32_t* out = rowpre + static_cast<int64_t>(blockIdx.x) * nblk;
  int carry = 0;
  for (int c0 = 0; c0 < nblk; c0 += RSCAN_THREADS * RSCAN_PER) {
    const int i0 = c0 + tid * RSCAN_PER;
    int v[RSCAN_PER];
    int local = 0;
#pragma unroll
    for (int i = 0; i < RSCAN_PER; ++i) {
      v[i] = i0 + i < nblk ? row[i0 + i] : 0;
      local += v[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int w = 0; w < RSCAN_THREADS / 32; ++w) {
        const int t = warp_tot[w];
        warp_tot[w] = run;
        run += t;
      }
      chunk_tot = run;
    }
    __syncthreads();
    int run = carry + warp_tot[warp] + incl - local;
#pragma unroll
    for (int i = 0; i < RSCAN_PER; ++i) {
      if (i0 + i < nblk) out[i0 + i] = run;
      run += v[i];
    }
    carry += chunk_tot;
    __syncthreads();   // warp_tot and chunk_tot are rewritten by the next chunk
  }
  if (tid == 0) counts[blockIdx.x] = carry;
}

__global__ void __launch_bounds__(256) slots_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                    int E, const int32_t* __restrict__ rowpre,
                                                    const int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets, int nblk,
                                                    int32_t* __restrict__ slot_of_pair,
                                                    int32_t* __restrict__ token_of_slot,
                                                    int* err) {
  __shared__ uint32_t mask[MOE_MAX_EXPERTS * MASK_WORDS];
  __shared__ int s_off[MOE_MAX_EXPERTS + 1];
  const int tid = threadIdx.x;
  for (int i = tid; i < E * MASK_WORDS; i += blockDim.x) mask[i] = 0u;
  if (tid < 32) {
    // offsets = exclusive scan of counts (E <= 256: 8 experts per lane, in expert order)
    constexpr int PER = MOE_MAX_EXPERTS / 32;
    int v[PER];
    int local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid * PER + i;
      v[i] = e < E ? counts[e] : 0;
      local += v[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += u;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid * PER + i;
      if (e < E) s_off[e] = run;
      run += v[i];
    }
    if (tid == 31) s_off[E] = incl;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = tid; e <= E; e += blockDim.x) offsets[e] = s_off[e];
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
    const int s = s_off[e] + rowpre[static_cast<int64_t>(e) * nblk + blockIdx.x] + rank;
    if (s < 0 || s >= N) {
      record_error(err, DEVERR_BAD_SLOT);
      continue;
    }
    slot_of_pair[static_cast<int64_t>(t) * k + j] = s;
    token_of_slot[s] = t;
  }
}

// ----------------------------------------------------------------------------- balancing loss
// "Megatron-Bridge 深度剖析", §Nemotron-3-Nano 配置 (moe_aux_loss_coeff): the load-balancing loss
//   L = coeff * E / (k * T^2) * sum_e counts[e] * sum_t p[t, e],
// p[t,:] = softmax(l_t) (softmax routing) or s / sum(s), s = sigmoid(l_t) (sigmoid routing).
// Two launches: per-256-token-block column sums of p (each warp sums its tokens in order, the
// block adds its 8 warps in order), then one block adds the blocks in order and takes the dot
// with the counts in fp64.  Fixed order throughout: bit-identical reruns.
template <int EPL>
__global__ void __launch_bounds__(256) aux_partial_kernel(const float* __restrict__ logits, int T,
                                                          int E, int score_fn,
                                                          float* __restrict__ partial) {
  __shared__ float wsum[8][MOE_MAX_EXPERTS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[EPL];
#pragma unroll
  for (int q = 0; q < EPL; ++q) acc[q] = 0.f;
  const int t0 = blockIdx.x * TPB;
  for (int i = warp; i < TPB && t0 + i < T; i += 8) {
    float v[EPL];
    load_logit_row<EPL>(logits, t0 + i, T, E, lane, v);
    float p[EPL], part = 0.f;
    if (score_fn == MOE_SCORE_SOFTMAX) {
      float m = NEG_INF;
#pragma unroll
      for (int q = 0; q < EPL; ++q) m = fmaxf(m, v[q]);
      m = warp_max(m);
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        p[q] = (q * 32 + lane < E) ? expf(v[q] - m) : 0.f;
        part += p[q];
      }
    } else {
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        p[q] = (q * 32 + lane < E) ? sigmoid_f(v[q]) : 0.f;
        part += p[q];
      }
    }
    const float z = warp_sum(part);
#pragma unroll
    for (int q = 0; q < EPL; ++q) acc[q] += p[q] / z;
  }
#pragma unroll
  for (int q = 0; q < EPL; ++q)
    if (q * 32 + lane < E) wsum[warp][q * 32 + lane] = acc[q];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += wsum[w][e];
    partial[static_cast<int64_t>(blockIdx.x) * E + e] = sum;
  }
}

__global__ void __launch_bounds__(256) aux_finish_kernel(const float* __restrict__ partial, int nblk,
                                                         int E, const int32_t* __restrict__ counts,
                                                         double scale, float* __restrict__ out) {
  __shared__ double red[256];
  const int tid = threadIdx.x;
  double v = 0.0;
  for (int e = tid; e < E; e += blockDim.x) {
    double col = 0.0;
    for (int b = 0; b < nblk; ++b) col += partial[static_cast<int64_t>(b) * E + e];
    v += col * static_cast<double>(counts[e]);
  }
  red[tid] = v;
  __syncthreads();
  for (int h = blockDim.x / 2; h > 0; h >>= 1) {
    if (tid < h) red[tid] += red[tid + h];
    __syncthreads();
  }
  if (tid == 0) out[0] = static_cast<float>(scale * red[0]);
}

int launch_aux_loss(const float* logits, const int32_t* counts, int T, int E, int k, int score_fn,
                    float coeff, float* partial, float* out, cudaStream_t st) {
  const int nblk = route_blocks(T);
  const dim3 grid(nblk), block(256);
  int rc;
  if (E <= 32)
    rc = launch("aux_partial", aux_partial_kernel<1>, grid, block, 0, st, logits, T, E, score_fn, partial);
  else if (E <= 64)
    rc = launch("aux_partial", aux_partial_kernel<2>, grid, block, 0, st, logits, T, E, score_fn, partial);
  else if (E <= 128)
    rc = launch("aux_partial", aux_partial_kernel<4>, grid, block, 0, st, logits, T, E, score_fn, partial);
  else
    rc = launch("aux_partial", aux_partial_kernel<8>, grid, block, 0, st, logits, T, E, score_fn, partial);
  MOE_TRY(rc);
  const double scale = static_cast<double>(coeff) * E / (static_cast<double>(k) * T * T);
  return launch("aux_finish", aux_finish_kernel, dim3(1), dim3(256), 0, st, partial, nblk, E,
                counts, scale, out);
}

// ----------------------------------------------------------------------------- expert bias
// The expert-bias correction after a step (DeepSeek V3's auxiliary-loss-free balancing):
//   b[e] += rate * sign(mean - counts[e]),  mean = T*k / E (fp32).
__global__ void bias_update_kernel(const int32_t* __restrict__ counts, float* __restrict__ bias,
                                   int E, float mean, float rate) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const float dlt = mean - static_cast<float>(counts[e]);
  const float sg = dlt > 0.f ? 1.f : (dlt < 0.f ? -1.f : 0.f);
  bias[e] = bias[e] + rate * sg;
}

int launch_bias_update(const int32_t* counts, float* bias, int T, int k, int E, float rate,
                       cudaStream_t st) {
  const float mean = static_cast<float>(static_cast<int64_t>(T) * k) / static_cast<float>(E);
  return launch("expert_bias_update", bias_update_kernel, dim3((E + 255) / 256), dim3(256), 0, st,
                counts, bias, E, mean, rate);
}

int launch_topk(const float* logits, int T, int E, int k, int score_fn, int renorm,
                const float* sel_bias, int32_t* idx, float* gate, int32_t* hist, cudaStream_t st) {
  const int nblk = route_blocks(T);
  int blocks = (T + 7) / 8;   // 8 warps per block, one token per warp at a time
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  const dim3 grid(blocks), block(256);
  int rc;
  if (E <= 32)
    rc = launch("route_topk", topk_kernel<1>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                sel_bias, idx, gate, device_error_word());
  else if (E <= 64)
    rc = launch("route_topk", topk_kernel<2>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                sel_bias, idx, gate, device_error_word());
  else if (E <= 128)
    rc = launch("route_topk", topk_kernel<4>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                sel_bias, idx, gate, device_error_word());
  else
    rc = launch("route_topk", topk_kernel<8>, grid, block, 0, st, logits, T, E, k, score_fn, renorm,
                sel_bias, idx, gate, device_error_word());
  MOE_TRY(rc);
  return launch("route_hist", hist_kernel, dim3(nblk), dim3(TPB), 0, st, idx, T, k, E, hist, nblk,
                device_error_word());
}

int launch_scan(const int32_t* hist, int E, int nblk, int32_t* base, int32_t* counts,
                cudaStream_t st) {
  return launch("route_scan", row_scan_kernel, dim3(E), dim3(RSCAN_THREADS), 0, st, hist, nblk,
                base, counts);
}

int launch_slots(const int32_t* idx, int T, int k, int E, const int32_t* base,
                 const int32_t* counts, int32_t* offsets, int32_t* slot_of_pair,
                 int32_t* token_of_slot, cudaStream_t st) {
  const int nblk = route_blocks(T);
  return launch("route_slots", slots_kernel, dim3(nblk), dim3(256), 0, st, idx, T, k, E, base,
                counts, offsets, nblk, slot_of_pair, token_of_slot, device_error_word());
}

}  // namespace moe
