// Routing of one token by one thread: selection keys, the top-k in (key desc, expert asc) order,
// and the gates.  Shared by the standalone top-k kernel (logits read from global memory) and
// the router GEMM's epilogue (logits read from the tensor-memory accumulator), so both give
// bit-identical indices and gates from the same fp32 logits.
//
// "Megatron-Bridge 深度剖析", §Expert Parallel 基础 (workflow figure, Step 1: the router scores
// every token against the experts and keeps the top-k); §Nemotron-3-Nano 配置 (sigmoid routing
// with a selection-only expert bias, as in DeepSeek V3).
//   key[e] = l[e]                                   (no selection bias)
//          = softmax(l)[e] + b[e] | sigmoid(l[e]) + b[e]   (selection-only bias b)
//   gates:  softmax, renorm:    softmax over the k selected logits
//           softmax, no renorm: softmax over all E logits, at the selected experts
//           sigmoid, renorm:    sigmoid of the selected, divided by their sum
//           sigmoid, no renorm: sigmoid of the selected
// Row sums run over the experts in increasing order, in fp32.  A NaN key ranks as -inf (outside
// the inputs' contract; keeps the selection inside [0, E)).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {
namespace rrow {

#define RROW_NEG_INF __int_as_float(0xff800000u)

__device__ __forceinline__ float sigmoid(float z) { return 1.0f / (1.0f + expf(-z)); }

// A selection key as an unsigned integer with the same order.  NaN becomes -inf (max(NaN, -inf)
// is -inf) and -0 becomes +0 (-0 + 0 = +0), so the two zeros tie as they compare equal; then the
// sign bit is flipped for positive keys and every bit for negative ones.  -inf maps to
// 0x007FFFFF, so 0 lies below every key.
__device__ __forceinline__ unsigned ordered_key(float f) {
  const float g = fmaxf(f, RROW_NEG_INF) + 0.0f;
  const unsigned b = __float_as_uint(g);
  const unsigned m = static_cast<unsigned>(static_cast<int>(b) >> 31);
  return b ^ (m | 0x80000000u);
}

struct Rule {
  int E, k, score_fn, renorm;
  const float* sel_bias;   // selection-only expert bias [E] (global or shared), or null
};

// The KL best (key, expert) pairs seen so far, best first.  Experts arrive in increasing order,
// so a key equal to one already held goes behind it: ties keep the lower expert first.
template <int KL> struct TopList {
  unsigned key[KL];
  int ex[KL];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      key[j] = 0u;
      ex[j] = 0;
    }
  }
  // The new pair takes the first place whose key it beats; the places below it move down one.
  __device__ __forceinline__ void push(unsigned c, int e) {
    bool gt[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) gt[j] = c > key[j];
#pragma unroll
    for (int j = KL - 1; j > 0; --j) {
      key[j] = gt[j - 1] ? key[j - 1] : (gt[j] ? c : key[j]);
      ex[j] = gt[j - 1] ? ex[j - 1] : (gt[j] ? e : ex[j]);
    }
    key[0] = gt[0] ? c : key[0];
    ex[0] = gt[0] ? e : ex[0];
  }
};

// Src: chunk(q, v) fills v[0..31] with the logits of experts 32q .. 32q+31 (entries at or past E
// are never read); at(e) returns expert e's logit.  stg: 32 words of this thread's own scratch
// (shared memory, stride 1) for one chunk's keys.  Writes sel[j] (the j-th selected expert) and
// gate[j] for j < k.
//
// Two passes over the keys.  The first takes the largest key of each of 8 expert groups
// (e mod 8); the smallest of those 8 maxima, tau, is held by 8 distinct experts, so at least 8 >= k
// keys reach it and no key below it is among the k best.  The second inserts, in expert order,
// only the keys >= tau that also beat the list's current last key (typically a dozen or two of
// E): each chunk's keys are staged and the set bits of that mask walked.
template <int KL, class Src>
__device__ __forceinline__ void route_row(const Src& src, const Rule& r, unsigned* stg,
                                          int (&sel)[KL], float (&gate)[KL]) {
  const int nq = (r.E + 31) >> 5;
  const bool softmax = r.score_fn == MOE_SCORE_SOFTMAX;
  float v[32];
  // row maximum and the softmax denominator over all E (selection keys under a bias, or the
  // gates without renormalisation)
  float rmax = RROW_NEG_INF, z = 0.f;
  if (softmax && (r.sel_bias || !r.renorm)) {
    for (int q = 0; q < nq; ++q) {
      src.chunk(q, v);
      const int lim = r.E - q * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < lim) rmax = fmaxf(rmax, v[i]);
    }
    for (int q = 0; q < nq; ++q) {
      src.chunk(q, v);
      const int lim = r.E - q * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < lim) z += expf(v[i] - rmax);
    }
  }
  auto key_of = [&](float x, int e) -> unsigned {
    float key = x;
    if (r.sel_bias) key = (softmax ? expf(x - rmax) / z : sigmoid(x)) + r.sel_bias[e];
    return ordered_key(key);
  };
  unsigned gm[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) gm[g] = 0u;
  for (int q = 0; q < nq; ++q) {
    src.chunk(q, v);
    const int lim = r.E - q * 32;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < lim) gm[i & 7] = max(gm[i & 7], key_of(v[i], q * 32 + i));
  }
  unsigned tau = gm[0];   // (an empty group's 0 keeps every key: still exact)
#pragma unroll
  for (int g = 1; g < 8; ++g) tau = min(tau, gm[g]);
  TopList<KL> L;
  L.init();
  for (int q = 0; q < nq; ++q) {
    src.chunk(q, v);
    const int lim = r.E - q * 32;
    const unsigned thr = L.key[KL - 1];
    unsigned m = 0u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < lim) {
        const unsigned c = key_of(v[i], q * 32 + i);
        stg[i] = c;
        m |= (c >= tau && c > thr ? 1u : 0u) << i;
      }
    }
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1u;
      L.push(stg[i], q * 32 + i);
    }
  }
  float lv[KL];
#pragma unroll
  for (int j = 0; j < KL; ++j) {
    sel[j] = L.ex[j];
    lv[j] = j < r.k ? src.at(L.ex[j]) : 0.f;
  }
  if (softmax) {
    float m = rmax, den = z;
    if (r.renorm) {
      m = RROW_NEG_INF;
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < r.k) m = fmaxf(m, lv[j]);
      den = 0.f;
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < r.k) den += expf(lv[j] - m);
    }
#pragma unroll
    for (int j = 0; j < KL; ++j) gate[j] = j < r.k ? expf(lv[j] - m) / den : 0.f;
  } else {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      gate[j] = j < r.k ? sigmoid(lv[j]) : 0.f;
      s += gate[j];
    }
    if (r.renorm) {
#pragma unroll
      for (int j = 0; j < KL; ++j) gate[j] = gate[j] / s;
    }
  }
}

}  // namespace rrow
}  // namespace moe
