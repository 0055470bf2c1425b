// Routing: top-k selection + gates, per-expert histogram, prefix sums, token<->slot maps.
//
// "Megatron-Bridge 深度剖析", §Expert Parallel 基础 (workflow figure, Step 1: the router
// picks the top-k experts of every token; Step 2: tokens are regrouped by expert).  On one GPU
// the dispatch plan of Step 2 is a stable counting sort of the (token, expert) pairs:
//   counts[e], offsets[e] = sum_{e'<e} counts[e'],
//   slot(t, j) = offsets[e] + #{t' < t : t' picked e},  e = idx[t, j].
//
// Two launches (or, with bf16 operands, one plus the router GEMM, whose epilogue does the
// first one's work on the accumulator):
//   topk  -- one thread per token (route_row.cuh): selection keys, the k best in (key desc,
//            expert asc) order, gates in fp32; one block per 128 tokens also writes the block's
//            row of the expert histogram hist[row][e] (bytes: a row counts at most 128 tokens).
//   slots -- one block per 256 tokens, in clusters of 8.  A cluster reads the whole histogram
//            (it is small: T/128 rows of E bytes), each block an eighth, and shares the sums
//            through distributed shared memory: every block gets each expert's total and the
//            count of its tokens in earlier blocks; block 0 writes counts and offsets.  Per-expert
//            bitmasks of the block's tokens then give each token's rank among the block's tokens
//            of its expert, and the block writes its pairs' slots and its slots' tokens as
//            contiguous runs.
// Where the histogram is larger than ROUTE_DIRECT_BYTES, a scan kernel forms those per-block
// prefixes and the totals first (three launches).  All integer, so the result is exact and
// independent of scheduling.
#include <limits.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "route_row.cuh"

namespace moe {

constexpr int HT = ROUTE_HIST_TOK;            // tokens per histogram row (128)
constexpr int ST = ROUTE_SLOT_TOK;            // tokens per slots block (256)
constexpr int SWORDS = ST / 32;               // 32-token mask words per expert in a slots block
constexpr int SWARPS = ST / 32;               // warps of a slots block
static_assert(SWORDS <= 32 && (SWORDS & (SWORDS - 1)) == 0, "mask words per expert: a power of two");
constexpr int MAXK = MOE_MAX_TOPK;
constexpr int SCL = 8;                        // slots blocks per cluster
constexpr int SOWN = SCL * (ST / HT);         // histogram rows of a cluster's own tokens
constexpr int TPB = ROUTE_TOK_PER_BLOCK;   // tokens per block of the balancing-loss sums

// logits of one token from global memory (fp32 rows of E; 16-byte loads when rows are aligned)
struct GlobalRow {
  const float* row;
  int E;
  bool vec;
  __device__ __forceinline__ void chunk(int q, float (&v)[32]) const {
    const int e0 = q * 32;
    if (vec) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (e0 + 4 * i < E) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(row + e0) + i);
          v[4 * i] = f.x;
          v[4 * i + 1] = f.y;
          v[4 * i + 2] = f.z;
          v[4 * i + 3] = f.w;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (e0 + i < E) v[i] = __ldg(row + e0 + i);
    }
  }
  __device__ __forceinline__ float at(int e) const { return __ldg(row + e); }
};

// One thread per token, one block per histogram row.  KL: the selection list's length (>= k).
template <int KL>
__global__ void __launch_bounds__(HT) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                  int k, int score_fn, int renorm,
                                                  const float* __restrict__ sel_bias,
                                                  int32_t* __restrict__ idx,
                                                  float* __restrict__ gate,
                                                  uint8_t* __restrict__ hist, int ldh, int* err) {
  __shared__ int cnt[MOE_MAX_EXPERTS];
  __shared__ unsigned stg[HT * 33];   // each thread's staged keys (rows of 33: no bank conflicts)
  __shared__ float sbias[MOE_MAX_EXPERTS];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += HT) {
    cnt[e] = 0;
    sbias[e] = sel_bias ? sel_bias[e] : 0.f;
  }
  __syncthreads();
  const int t = blockIdx.x * HT + tid;
  if (t < T) {
    GlobalRow src;
    src.row = logits + static_cast<int64_t>(t) * E;
    src.E = E;
    src.vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
    rrow::Rule r;
    r.E = E;
    r.k = k;
    r.score_fn = score_fn;
    r.renorm = renorm;
    r.sel_bias = sel_bias ? sbias : nullptr;
    int sel[KL];
    float g[KL];
    rrow::route_row<KL>(src, r, stg + tid * 33, sel, g);
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      if (j < k) {
        int e = sel[j];
        if (e < 0 || e >= E) {   // cannot happen; never index with it
          record_error(err, DEVERR_BAD_EXPERT);
          e = 0;
        }
        idx[static_cast<int64_t>(t) * k + j] = e;
        gate[static_cast<int64_t>(t) * k + j] = g[j];
        atomicAdd(&cnt[e], 1);
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < ldh; e += HT)
    hist[static_cast<int64_t>(blockIdx.x) * ldh + e] = static_cast<uint8_t>(e < E ? cnt[e] : 0);
}

// Large histograms only: per expert e (one block each), rowpre[e][r] = the exclusive prefix of
// hist[.][e] over rows (the expert's tokens in rows before r) and counts[e] = the column total.
// Each thread takes 8 consecutive rows; a block-wide scan of the threads' sums gives their starts.
constexpr int RSCAN_THREADS = 256;
constexpr int RSCAN_PER = 8;

__global__ void __launch_bounds__(RSCAN_THREADS) col_scan_kernel(const uint8_t* __restrict__ hist,
                                                                 int ldh, int nrows,
                                                                 int32_t* __restrict__ rowpre,
                                                                 int32_t* __restrict__ counts) {
  __shared__ int warp_tot[RSCAN_THREADS / 32];
  __shared__ int chunk_tot;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x;
  int32_t* out = rowpre + static_cast<int64_t>(e) * nrows;
  int carry = 0;
  for (int c0 = 0; c0 < nrows; c0 += RSCAN_THREADS * RSCAN_PER) {
    const int i0 = c0 + tid * RSCAN_PER;
    int v[RSCAN_PER];
    int local = 0;
#pragma unroll
    for (int i = 0; i < RSCAN_PER; ++i) {
      v[i] = i0 + i < nrows ? hist[static_cast<int64_t>(i0 + i) * ldh + e] : 0;
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
      if (i0 + i < nrows) out[i0 + i] = run;
      run += v[i];
    }
    carry += chunk_tot;
    __syncthreads();   // warp_tot and chunk_tot are rewritten by the next chunk
  }
  if (tid == 0) counts[e] = carry;
}

// 32 x 32 bit matrix, row i in lane i (bit b = column b), transposed: lane i receives column i.
// Five rounds swap the off-diagonal blocks of size 16, 8, 4, 2, 1 between lane pairs.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
  const uint32_t lo_mask[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int j = 16 >> s;
    const uint32_t m = lo_mask[s];
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y & ~m) >> j)) : ((x & m) | ((y & m) << j));
  }
  return x;
}

// Shared memory of a slots block: phase 1 (the histogram's column sums) and phase 2 (the token
// bitmasks and their per-word prefix counts) use the same bytes.
struct SlotsSmem {
  int cpart[2][MOE_MAX_EXPERTS];   // this CTA's share of the sums before / after the cluster's rows
  int pre[MOE_MAX_EXPERTS];        // the expert's tokens in earlier blocks
  int off[MOE_MAX_EXPERTS + 1];    // offsets (exclusive scan of the totals)
  int boff[MOE_MAX_EXPERTS];       // the expert's first pair in the block's expert order
  int gbase[MOE_MAX_EXPERTS];      // global slot of block-order position p: gbase[e] + p
  union {
    int part[SWARPS][2][MOE_MAX_EXPERTS];   // per warp: sums over rows before / from the block's
    struct {
      // bit i of word w: token 32w + i picked e (rows padded by one word: a warp's stores of
      // 32 experts' words fall in distinct banks)
      uint32_t mask[MOE_MAX_EXPERTS][SWORDS + 1];
      int wpre[MOE_MAX_EXPERTS][SWORDS];        // tokens of e in words before w
    } m;
  } u;
  int sop[ST * MAXK];              // the block's slot_of_pair, as it lies in memory
  int tok[ST * MAXK];              // the block's pairs in expert order: token ...
  uint8_t ex[ST * MAXK];           // ... and expert
};

// rowpre/counts_in: null (the block sums the histogram itself) or the scan kernel's results.
__global__ void __launch_bounds__(ST) slots_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                   int E, const uint8_t* __restrict__ hist,
                                                   int ldh, int nrows,
                                                   const int32_t* __restrict__ rowpre,
                                                   const int32_t* __restrict__ counts_in,
                                                   int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ slot_of_pair,
                                                   int32_t* __restrict__ token_of_slot, int* err) {
  __shared__ SlotsSmem sm;
  __shared__ int wsum[SWARPS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r0 = blockIdx.x * (ST / HT);   // this block's first histogram row
  // this thread's token's experts, loaded first so that their latency overlaps the sums below
  const int t = blockIdx.x * ST + tid;
  int ev[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j)
    ev[j] = (j < k && t < T) ? __ldg(idx + static_cast<int64_t>(t) * k + j) : -1;
  if (!rowpre) {
    // ---- column sums of the histogram, split over the cluster: the rows before the cluster's
    // own (P) and after them (Q) are read by the cluster's SCL blocks in turn, each block sums its
    // rows, and every block then adds all SCL shares (distributed shared memory, fixed order);
    // the SOWN rows of the cluster's own tokens each block reads itself.
    // Lane -> 16-byte chunk c of a row (cpr chunks per row, a power of two) and one of the 32/cpr
    // rows a warp instruction covers.
    const int crank = static_cast<int>(ptx::cluster_ctarank());
    const int R0 = (blockIdx.x - crank) * (ST / HT);   // the cluster's first row
    const int cpr = ldh >> 4, rpi = 32 / cpr;
    const int c = lane & (cpr - 1), rsub = lane / cpr;
    // bytes summed in 16-bit lanes (a lane's rows count at most 32 x 128 tokens in a histogram
    // of ROUTE_DIRECT_BYTES): word x of a chunk holds experts 4x..4x+3; its even bytes go to
    // *_ev[x], its odd ones to *_od[x]
    uint32_t lo_ev[4], lo_od[4], hi_ev[4], hi_od[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) lo_ev[x] = lo_od[x] = hi_ev[x] = hi_od[x] = 0u;
    const int step = SCL * SWARPS * rpi;
    const uint4* h4 = reinterpret_cast<const uint4*>(hist) + c;
    const int ld4 = ldh >> 4;
    int r = (crank * SWARPS + warp) * rpi + rsub;
#pragma unroll 4
    for (; r < nrows && r < R0; r += step) {
      const uint4 w = __ldg(h4 + static_cast<int64_t>(r) * ld4);
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        lo_ev[x] += wv[x] & 0x00ff00ffu;
        lo_od[x] += (wv[x] >> 8) & 0x00ff00ffu;
      }
    }
    while (r < R0 + SOWN) r += step;   // (the cluster's own rows: below)
#pragma unroll 4
    for (; r < nrows; r += step) {
      const uint4 w = __ldg(h4 + static_cast<int64_t>(r) * ld4);
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        hi_ev[x] += wv[x] & 0x00ff00ffu;
        hi_od[x] += (wv[x] >> 8) & 0x00ff00ffu;
      }
    }
    // lanes sharing a chunk add their packed sums (a warp's rows count at most 128 x 128 tokens
    // per 16-bit lane in such a histogram), then unpack
    for (int o = cpr; o < 32; o <<= 1) {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        lo_ev[x] += __shfl_xor_sync(0xffffffffu, lo_ev[x], o);
        lo_od[x] += __shfl_xor_sync(0xffffffffu, lo_od[x], o);
        hi_ev[x] += __shfl_xor_sync(0xffffffffu, hi_ev[x], o);
        hi_od[x] += __shfl_xor_sync(0xffffffffu, hi_od[x], o);
      }
    }
    int lo[16], hi[16];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      lo[4 * x] = lo_ev[x] & 0xffffu;
      lo[4 * x + 1] = lo_od[x] & 0xffffu;
      lo[4 * x + 2] = lo_ev[x] >> 16;
      lo[4 * x + 3] = lo_od[x] >> 16;
      hi[4 * x] = hi_ev[x] & 0xffffu;
      hi[4 * x + 1] = hi_od[x] & 0xffffu;
      hi[4 * x + 2] = hi_ev[x] >> 16;
      hi[4 * x + 3] = hi_od[x] >> 16;
    }
    if (rsub == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        sm.u.part[warp][0][c * 16 + i] = lo[i];
        sm.u.part[warp][1][c * 16 + i] = hi[i];
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += ST) {
      int a = 0, b = 0;
#pragma unroll
      for (int w = 0; w < SWARPS; ++w) {
        a += sm.u.part[w][0][e];
        b += sm.u.part[w][1][e];
      }
      sm.cpart[0][e] = a;
      sm.cpart[1][e] = b;
    }
    ptx::cluster_sync();   // every block's share is in its shared memory
    for (int e = tid; e < E; e += ST) {
      int P = 0, Q = 0;
      const uint32_t a0 = ptx::smem_u32(&sm.cpart[0][e]), a1 = ptx::smem_u32(&sm.cpart[1][e]);
#pragma unroll
      for (int q = 0; q < SCL; ++q) {
        P += static_cast<int>(ptx::ld_cluster_u32(ptx::mapa(a0, q)));
        Q += static_cast<int>(ptx::ld_cluster_u32(ptx::mapa(a1, q)));
      }
      // the cluster's own rows: those before this block's, and all of them
      int own_before = 0, own_all = 0;
#pragma unroll 4
      for (int rr = R0; rr < R0 + SOWN && rr < nrows; ++rr) {
        const int v = hist[static_cast<int64_t>(rr) * ldh + e];
        own_all += v;
        if (rr < r0) own_before += v;
      }
      sm.pre[e] = P + own_before;
      sm.off[e] = P + own_all + Q;   // the total, until the scan below replaces it
    }
    ptx::cluster_sync();   // no block leaves or reuses its shares while another may read them
  } else {
    for (int e = tid; e < E; e += ST) {
      sm.pre[e] = r0 < nrows ? rowpre[static_cast<int64_t>(e) * nrows + r0] : 0;
      sm.off[e] = counts_in[e];
    }
  }
  __syncthreads();   // (phase 1's shared memory is reused below)
  // ---- offsets: the exclusive scan of the totals; each thread takes E/ST (at most one when
  // E <= ST, else a run of consecutive experts)
  {
    constexpr int PER = (MOE_MAX_EXPERTS + ST - 1) / ST;
    int v[PER], local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid * PER + i;
      v[i] = e < E ? sm.off[e] : 0;
      local += v[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    int run = before + incl - local;
    if (blockIdx.x == 0 && !rowpre) {
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (tid * PER + i < E) counts[tid * PER + i] = v[i];
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = tid * PER + i;
      if (e < E) sm.off[e] = run;
      run += v[i];
    }
    if (tid == ST - 1) sm.off[E] = run;   // the last thread's run ends at the grand total
    __syncthreads();
  }
  if (blockIdx.x == 0)
    for (int e = tid; e <= E; e += ST) offsets[e] = sm.off[e];
  // ---- this block's tokens: per expert, a bitmask of the warp's tokens that picked it.  Each
  // lane holds its token's experts as a bitset (word w: experts 32w .. 32w+31); transposing a
  // word across the warp gives lane i the mask of the tokens that picked expert 32w + i.
  uint32_t bs[MOE_MAX_EXPERTS / 32];
#pragma unroll
  for (int w = 0; w < MOE_MAX_EXPERTS / 32; ++w) bs[w] = 0u;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j < k) {
      int e = ev[j];
      if (e >= E || e < -1) {
        record_error(err, DEVERR_BAD_EXPERT);
        e = ev[j] = -1;
      }
#pragma unroll
      for (int w = 0; w < MOE_MAX_EXPERTS / 32; ++w)
        bs[w] |= (e >= 0 && (e >> 5) == w) ? 1u << (e & 31) : 0u;
      sm.sop[tid * k + j] = -1;   // (stays -1 only for a pair whose expert was out of range)
    }
  }
  const int nwords = (E + 31) >> 5;
#pragma unroll
  for (int w = 0; w < MOE_MAX_EXPERTS / 32; ++w) {
    if (w < nwords) {
      const uint32_t m = transpose32(bs[w], lane);
      if (w * 32 + lane < E) sm.u.m.mask[w * 32 + lane][warp] = m;
    }
  }
  __syncthreads();
  // per expert, the exclusive prefix of its words' popcounts (SWORDS lanes per expert; the loop
  // bound is the same for every thread, so each shuffle has the whole warp); the last word's
  // inclusive sum is the expert's pair count in this block
  for (int e0 = 0; e0 < E; e0 += ST / SWORDS) {
    const int e = e0 + tid / SWORDS, w = tid & (SWORDS - 1);
    const int c = e < E ? __popc(sm.u.m.mask[e][w]) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < SWORDS; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o, SWORDS);
      if (w >= o) incl += u;
    }
    if (e < E) {
      sm.u.m.wpre[e][w] = incl - c;
      if (w == SWORDS - 1) sm.boff[e] = incl;
    }
  }
  __syncthreads();
  // the block's expert order: boff = the exclusive scan of the experts' pair counts (one expert
  // per thread, E <= ST)
  int npairs;
  {
    const int ne = tid < E ? sm.boff[tid] : 0;
    int incl = ne;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < SWARPS; ++w) {
      if (w < warp) before += wsum[w];
      all += wsum[w];
    }
    npairs = all;
    if (tid < E) {
      const int bo = before + incl - ne;
      sm.boff[tid] = bo;
      sm.gbase[tid] = sm.off[tid] + sm.pre[tid] - bo;
    }
    __syncthreads();
  }
  const int64_t N = static_cast<int64_t>(T) * k;
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    const int e = ev[j];
    if (e < 0) continue;
    const int p = sm.boff[e] + sm.u.m.wpre[e][warp] + __popc(sm.u.m.mask[e][warp] & below);
    sm.sop[tid * k + j] = sm.gbase[e] + p;
    sm.tok[p] = t;
    sm.ex[p] = static_cast<uint8_t>(e);
  }
  __syncthreads();
  // ---- out: slot_of_pair of the block's tokens is one contiguous run; token_of_slot takes the
  // block's pairs in expert order, each expert's a contiguous run of slots
  const int t0 = blockIdx.x * ST;
  const int nt = min(ST, T - t0);
  int32_t* sop_out = slot_of_pair + static_cast<int64_t>(t0) * k;
  for (int i = tid; i < nt * k; i += ST) {
    const int sv = sm.sop[i];
    if (sv >= N) record_error(err, DEVERR_BAD_SLOT);
    sop_out[i] = sv < N ? sv : -1;
  }
  for (int i = tid; i < npairs; i += ST) {
    const int64_t sv = static_cast<int64_t>(sm.gbase[sm.ex[i]]) + i;
    if (sv < 0 || sv >= N) {
      record_error(err, DEVERR_BAD_SLOT);
      continue;
    }
    token_of_slot[sv] = sm.tok[i];
  }
}

// ----------------------------------------------------------------------------- balancing loss
#define NEG_INF __int_as_float(0xff800000u)

// Lane `lane` of a warp loads experts lane, lane + 32, ... of token t's logits (-inf past E or T).
template <int EPL>
__device__ __forceinline__ void load_logit_row(const float* __restrict__ logits, int t, int T,
                                               int E, int lane, float (&v)[EPL]) {
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = q * 32 + lane;
    v[q] = (t < T && e < E) ? __ldg(logits + static_cast<int64_t>(t) * E + e) : NEG_INF;
  }
}

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
                const float* sel_bias, int32_t* idx, float* gate, uint8_t* hist, cudaStream_t st) {
  const dim3 grid(route_rows(T)), block(HT);
  const int ldh = route_ldh(E);
  int* err = device_error_word();
  if (k <= 2)
    return launch("route_topk", topk_kernel<2>, grid, block, 0, st, logits, T, E, k, score_fn,
                  renorm, sel_bias, idx, gate, hist, ldh, err);
  if (k <= 4)
    return launch("route_topk", topk_kernel<4>, grid, block, 0, st, logits, T, E, k, score_fn,
                  renorm, sel_bias, idx, gate, hist, ldh, err);
  return launch("route_topk", topk_kernel<MAXK>, grid, block, 0, st, logits, T, E, k, score_fn,
                renorm, sel_bias, idx, gate, hist, ldh, err);
}

int launch_slots(const int32_t* idx, int T, int k, int E, const uint8_t* hist, int32_t* rowpre,
                 int32_t* counts, int32_t* offsets, int32_t* slot_of_pair, int32_t* token_of_slot,
                 cudaStream_t st) {
  const int nrows = route_rows(T), ldh = route_ldh(E);
  const bool direct = route_hist_direct(T, E);
  if (!direct) {
    if (!rowpre) {
      set_error("route_slots: a histogram of %lld bytes needs the row-prefix scratch",
                static_cast<long long>(nrows) * ldh);
      return MOE_ERR_INVALID_ARG;
    }
    MOE_TRY(launch("route_scan", col_scan_kernel, dim3(E), dim3(RSCAN_THREADS), 0, st, hist, ldh,
                   nrows, rowpre, counts));
  }
  // whole clusters: blocks past the tokens only take their share of the histogram sums
  const int nblk = (T + ST - 1) / ST;
  const int grid = (nblk + SCL - 1) / SCL * SCL;
  return launch_clusters("route_slots", slots_kernel, dim3(grid), dim3(ST), 0, SCL, st, idx, T, k,
                         E, hist, ldh, nrows, direct ? nullptr : rowpre,
                         direct ? nullptr : counts, counts, offsets, slot_of_pair, token_of_slot,
                         device_error_word());
}

}  // namespace moe
