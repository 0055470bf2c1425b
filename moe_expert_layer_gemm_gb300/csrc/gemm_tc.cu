// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 in (or E4M3 with
// a tensorwise scale, or MXFP8: E4M3 with an E8M0 scale per 32 K-elements), fp32 accumulate.
// One kernel template serves every matrix product of the layer:
//   fc1 + SwiGLU, fc2 (ragged rows per expert), their data gradients (ragged rows, weights read
//   MN-major), their weight gradients (ragged reduction per expert), the router and the
//   shared expert (one group).
// "Megatron-Bridge 深度剖析", §计算融合 / Grouped GEMM: every expert's GEMM in one launch over
// ragged per-expert token counts.  Here the ragged extents are read on the device from the
// routing offsets, so the host never synchronises on them.
//
// CTA organisation (persistent, one CTA per SM):
//   warp 0     TMA producer: loads A/B k-blocks into a STAGES-deep shared-memory ring
//   warp 1     MMA issuer: owns TMEM (2 accumulators of BN fp32 columns), issues
//              tcgen05.mma (M=128, N=BN, K=16 bf16 / 32 E4M3) per k-step, commits to the ring's
//              empty barriers; MXFP8: first copies the stage's block scales into a TMEM slot
//              (tcgen05.cp) for the block-scaled MMAs
//   warps 2..  epilogue (4 or 8 warps): TMEM -> registers (tcgen05.ld) -> fused epilogue ->
//              a swizzled shared-memory slab per warp (32 rows x 128 bytes) -> TMA bulk-tensor
//              store, overlapped with the next tile's MMAs through the second accumulator
// Tiles are BM=128 rows x BN columns x BK=64; a CTA walks tiles blockIdx.x, blockIdx.x +
// gridDim.x, ... or, for the weight gradients, claims them at run time.
// Beside it: tc_rows_tall_kernel (the bf16-store row-ragged products on 256 x 256 tiles, two
// MMAs per K step sharing each B stage), tc_wgrad_pair_kernel (one-group weight gradients on
// CTA pairs) and tc_rows_pair_kernel (a measured option, off).
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "route_row.cuh"

namespace moe {

// Pipeline wait statistics (build option MOE_WAIT_STATS=1, read by moe_gemm_wait_stats): per
// kernel kind, SM clock cycles summed over CTAs -- 0 producer waiting for a free ring stage,
// 1 MMA warp waiting for a loaded stage, 2 MMA warp waiting for a free accumulator, 3 the first
// epilogue warp waiting for a finished accumulator, 4 the CTAs' own cycles -- and 5 the k-blocks
// the MMA warps consumed, 6 the CTAs.
#ifndef MOE_WAIT_STATS
#define MOE_WAIT_STATS 0
#endif
constexpr int WAIT_KINDS = 64, WAIT_FIELDS = 7;
__device__ unsigned long long g_wait_stats[WAIT_KINDS * WAIT_FIELDS];

namespace {

struct WaitStats {
  unsigned long long t_start = 0, prod = 0, full = 0, acc = 0, epi = 0, kblocks = 0;
  __device__ __forceinline__ void start() {
    if (MOE_WAIT_STATS) t_start = clock64();
  }
  __device__ __forceinline__ unsigned long long now() const {
    return MOE_WAIT_STATS ? static_cast<unsigned long long>(clock64()) : 0ull;
  }
  __device__ __forceinline__ void since(unsigned long long& field, unsigned long long t0) const {
    if (MOE_WAIT_STATS) field += static_cast<unsigned long long>(clock64()) - t0;
  }
  // warp 0 lane 0 the producer, warp 1 lane 0 the MMA issuer, warp 2 lane 0 the first epilogue
  __device__ __forceinline__ void flush(int kind, int warp, int lane) const {
    if (!MOE_WAIT_STATS) return;
    unsigned long long* g = g_wait_stats + kind * WAIT_FIELDS;
    if (lane != 0) return;
    if (warp == 0) atomicAdd(g + 0, prod);
    if (warp == 1) {
      atomicAdd(g + 1, full);
      atomicAdd(g + 2, acc);
      atomicAdd(g + 5, kblocks);
    }
    if (warp == 2) atomicAdd(g + 3, epi);
  }
  // after the CTA's last barrier, by one thread: its cycles and the CTA count
  __device__ __forceinline__ void flush_cta(int kind) const {
    if (!MOE_WAIT_STATS) return;
    unsigned long long* g = g_wait_stats + kind * WAIT_FIELDS;
    atomicAdd(g + 4, static_cast<unsigned long long>(clock64()) - t_start);
    atomicAdd(g + 6, 1ull);
  }
};


constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MAXG = 256;             // groups per launch (experts, or K splits)
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int SLAB = 32 * 128;        // one warp's staging buffer: 32 rows x 128 bytes

// Router logits (fp32 rows of E columns, E not necessarily a multiple of 4) are written with
// direct stores; every other product goes out through the staged TMA path.
template <int SCHED, int EPI> struct OutPath {
  static constexpr bool tma = !(SCHED == RAGGED_M && EPI == EPI_F32);
};

#ifndef MOE_EPI8_SWIGLU_BWD
#define MOE_EPI8_SWIGLU_BWD 1
#endif
#ifndef MOE_EPI8_OTHER
#define MOE_EPI8_OTHER 0
#endif

#ifndef MOE_DYN_WGRAD
#define MOE_DYN_WGRAD 1
#endif

// Weight gradients with tiles handed out at run time.  Every tile writes a full fp32 block, but
// its reduction length is its expert's row count, and routing is skewed (a few experts hold most
// rows).  A static walk gives some CTAs far more reduction work than others and leaves the GPU
// draining a long tail.  Instead the experts are ordered by row count (most first) and each CTA
// claims the next tile of that list from a global counter when it is ready for one: the longest
// tiles start first and the short ones fill in behind them (longest-processing-time-first).
template <int SCHED, int EPI> struct DynMode {
  static constexpr bool on = SCHED == RAGGED_K && EPI == EPI_F32 && MOE_DYN_WGRAD != 0;
};

// MOE_WGRAD_ALTERNATE=1: each CTA alternates its claims between the heavy end and the light end
// of that list, so that a nearly empty expert's tile (a fp32 block to store, almost no MMAs)
// drains its stores while the next heavy tile's MMAs run on the other accumulator.  The two
// ends share one 64-bit counter (front count low, back count high); a claim is valid while
// front + back < tiles, so every tile is claimed exactly once.  Measured no faster than
// heaviest-first (fc1 weight gradient 1.92 ms either way on the 128-expert layer): an SM's
// operand loads and fp32 stores share its memory pipeline whatever the order, so it is off.
#ifndef MOE_WGRAD_ALTERNATE
#define MOE_WGRAD_ALTERNATE 0
#endif
__device__ __forceinline__ int claim_tile(int* ctr, int total, int& nclaims) {
  if (!MOE_WGRAD_ALTERNATE) {
    const int t = atomicAdd(ctr, 1);
    return t < total ? t : -1;
  }
  const bool back = (nclaims++ & 1) != 0;
  const unsigned long long old =
      atomicAdd(reinterpret_cast<unsigned long long*>(ctr), back ? (1ull << 32) : 1ull);
  const long long front_n = static_cast<long long>(old & 0xffffffffull);
  const long long back_n = static_cast<long long>(old >> 32);
  if (front_n + back_n >= total) return -1;   // the two ends have met: every tile is taken
  return back ? static_cast<int>(total - 1 - back_n) : static_cast<int>(front_n);
}

// L2 priorities of the weight gradients: their fp32 blocks are written once and never read
// back here, so they go out evict-first and do not push the operands (re-read by every tile of
// an expert) out of L2; the operands may be marked evict-last.
#ifndef MOE_WGRAD_STORE_HINT
#define MOE_WGRAD_STORE_HINT 1
#endif
#ifndef MOE_WGRAD_LOAD_HINT
#define MOE_WGRAD_LOAD_HINT 0
#endif

// 192-column output tiles where they pad the product's width less than 256 (build option:
// measured slower on GB300 -- fc1 dgrad 1.38 -> 1.55 ms, fc2 dgrad 0.97 -> 1.15 ms at d = 2688,
// f = 1856 -- the per-FLOP operand traffic and per-tile costs outweigh the saved padding).
// Weight-gradient fp32 blocks through the load/store units instead of TMA (the staged slab read
// back so that each warp store writes four whole 128-byte lines).  It tests whether the SM's TMA
// unit, which also brings in every operand k-block, is what the stores contend for.  Interleaved
// on GB300 it is no faster on uniform or 16-hot routing and 9% slower on the DeepSeek-style
// routing: the contention is further out (L2 / DRAM), so the stores stay on TMA.
#ifndef MOE_WGRAD_LSU_STORE
#define MOE_WGRAD_LSU_STORE 0
#endif

// Weight-gradient stores paced: for tiles whose reduction is 2..MOE_WGRAD_PACE_KB k-blocks, an
// epilogue warp issues its next fp32 slab only once its previous stores have landed in memory
// (one 4 KB store in flight per warp), rather than once the TMA engine has read them out of
// shared memory.  Such tiles' MMAs take about as long as their 128 KB of stores, and unpaced a
// burst of stores costs an SM about as long as its operand loads, with no overlap between the
// two.  Pacing every tile, on the 128-expert layer: uniform routing (768 rows per expert) fc1's
// weight gradient 1.74-1.75 -> 1.64 ms, fc2's 0.89 -> 0.85 ms; MTP-256e (about 1024 rows per
// expert) 0.95 -> 0.90 and 0.51 -> 0.49 ms; 64 rows per expert, 8 experts of 12288 rows and the
// DeepSeek-style routing unchanged or up to 2% slower -- hence the window (0: never paced).
#ifndef MOE_WGRAD_PACE_KB
#define MOE_WGRAD_PACE_KB 32
#endif

#ifndef MOE_TILE192
#define MOE_TILE192 0
#endif

constexpr int FEED = 8;   // depth of the ring that passes run-time tile indices to the consumers

// Staging slabs per epilogue warp: the SwiGLU backward takes one (32 columns of the saved a and
// of u side by side, 64-byte swizzle), which leaves room for a fourth ring stage -- with two
// slabs of 64 columns each the ring had three stages and fc2's data gradient on the 128-expert
// layer took 0.98 ms instead of 0.87 (MOE_SWIGLU_BWD_ONESLAB=0 keeps that form; the MXFP8
// backward keeps it too); weight gradients take MOE_WGRAD_SLABS (stores in flight per warp);
// with 8 epilogue warps the others make do with one so that the ring keeps four stages.
#ifndef MOE_WGRAD_SLABS
#define MOE_WGRAD_SLABS 2
#endif
#ifndef MOE_SWIGLU_BWD_ONESLAB
#define MOE_SWIGLU_BWD_ONESLAB 1
#endif
template <int SCHED, int EPI, int EPI_WARPS> struct SlabsPerWarp {
  static constexpr int n = EPI == EPI_SWIGLU_BWD ? (MOE_SWIGLU_BWD_ONESLAB ? 1 : 2)
                         : SCHED == RAGGED_K ? MOE_WGRAD_SLABS
                         : EPI_WARPS == 4 ? 2 : 1;
};

// Epilogue width: 4 warps (one per TMEM lane quadrant) or 8 (two per quadrant, each on half
// of the tile's columns) for products whose epilogue is long relative to their MMAs (the
// SwiGLU backward; the E4M3 SwiGLU forward, whose MMAs take half the bf16 time: 0.97 -> 0.82 ms
// on the 128-expert layer); 8 epilogue warps trade one pipeline stage for staging slabs.
// (8 warps split a tile's columns in two halves of 64-column steps: BN a multiple of 128.)
// Weight gradients keep 4: with 8 they were slower (fc1 1.86 -> 2.04 ms) and their fp32
// blocks differed between runs on the 128-expert routing, so that form was removed.
#ifndef MOE_EPI8_F8_FWD
#define MOE_EPI8_F8_FWD 1
#endif
template <int BN, int SCHED, int EPI, bool F8 = false> struct EpiWidth {
  static constexpr int warps =
      (!OutPath<SCHED, EPI>::tma || BN % 128 != 0) ? 4
      : (SCHED == RAGGED_K ? 4
                           : (EPI == EPI_SWIGLU_BWD ? (MOE_EPI8_SWIGLU_BWD ? 8 : 4)
                                                    : ((F8 && EPI == EPI_SWIGLU_FWD ? MOE_EPI8_F8_FWD
                                                                                    : MOE_EPI8_OTHER)
                                                           ? 8 : 4)));
  static constexpr int slabs = SlabsPerWarp<SCHED, EPI, warps>::n;
};

// SFS: bytes of MXFP8 block scales per stage (0 without); MAXST: most stages the ring may have;
// TCOLS: TMEM columns to allocate (0: the two accumulators' power of two).
// XTRA: bytes after the AUX block (the router epilogue's histogram buffers).
template <int BN, bool TMA_OUT, int EPI_WARPS, int SLABS, int SFS = 0, int MAXST = 6, int TCOLS = 0,
          int XTRA = 0>
struct TileCfg {
  static constexpr int B_STAGE = BN * BK * 2;
  static constexpr int STAGING = TMA_OUT ? EPI_WARPS * SLABS * SLAB : 0;
  static constexpr int AUX = 3072;   // barriers, TMEM address, flags, group tables
  static constexpr int MAX_SMEM = 232448;   // opt-in dynamic shared memory per block
  static constexpr int FIT = (MAX_SMEM - STAGING - AUX - XTRA) / (A_STAGE + B_STAGE + SFS);
  static constexpr int STAGES = FIT < MAXST ? FIT : MAXST;
  static constexpr int RING = STAGES * (A_STAGE + B_STAGE);
  static constexpr int SF_RING = STAGES * SFS;   // after the staging slabs
  static constexpr int SMEM = RING + STAGING + SF_RING + AUX + XTRA;
  // two accumulators of BN columns; allocations are powers of two of at least 32 columns
  static constexpr int ACC_COLS = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128
                                : 2 * BN <= 256 ? 256 : 512;
  static constexpr int TMEM_COLS = TCOLS ? TCOLS : ACC_COLS;
  static constexpr int ACC_STRIDE = ACC_COLS / 2;   // column of accumulator 1 (aligned)
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
};

// MXFP8 tiles: the accumulators, then a 16-column TMEM slot per ring stage for the stage's block
// scales (A: 4 columns, B: 4 per 128 rows of the tile, at +8), in a 512-column allocation.
// BN = 192: two accumulators 0..191 and 256..447, four stages' scales in 448..511.  BN = 256: one
// accumulator 0..255 (two would fill the 512 columns), scale slots from 256; the next tile's MMAs
// then wait for the epilogue to drain it.
constexpr int MX_SF_COLS = 16;
template <int BN> struct MxCfg {
  static constexpr int NACC = BN > 192 ? 1 : 2;               // accumulators
  static constexpr int SFB_CH = (BN + 127) / 128;             // 512-byte B chunks per stage
  static constexpr int SF_STAGE = MX_CHUNK * (1 + SFB_CH);    // A chunk, then B chunks
  static constexpr int ACC_STRIDE = 2 * BN <= 256 ? 128 : 256;
  static constexpr int SF_COL0 = NACC == 1 ? BN : ACC_STRIDE + BN;
  static constexpr int MAX_STAGES = (512 - SF_COL0) / MX_SF_COLS;
};
// Epilogue staging: the 256-column MXFP8 products keep one slab per warp, which leaves room for a
// fourth ring stage beside their block scales.
template <int BN, int SCHED, int EPI, bool F8, bool MX> struct EpiOf {
  static constexpr bool staged = OutPath<SCHED, EPI>::tma;
  static constexpr int slabs = (MX && BN == 256) ? 1
                              : (MX && EPI == EPI_SWIGLU_BWD) ? 2   // (the two-slab loop)
                                                              : EpiWidth<BN, SCHED, EPI, F8>::slabs;
  // the SwiGLU backward's one-slab loop (bf16 and tensorwise E4M3)
  static constexpr bool half_slabs = EPI == EPI_SWIGLU_BWD && !MX && MOE_SWIGLU_BWD_ONESLAB;
};
// The router product (fp32 logits, bf16 operands) routes its tokens in the epilogue.
template <int SCHED, int EPI, bool F8> struct RouterOf {
  static constexpr bool on = SCHED == RAGGED_M && EPI == EPI_F32 && !F8;
  // an mbarrier (64 bytes reserved), two tile histograms of MOE_MAX_EXPERTS ints, the logit bias
  // and the selection bias (MOE_MAX_EXPERTS floats each), and every epilogue thread's 32 staged
  // keys (rows of 33 words: a warp's stores of one key index fall in 32 distinct banks)
  static constexpr int HIST_OFF = 64;
  static constexpr int LBIAS_OFF = HIST_OFF + 2 * MOE_MAX_EXPERTS * 4;
  static constexpr int SBIAS_OFF = LBIAS_OFF + MOE_MAX_EXPERTS * 4;
  static constexpr int STG_OFF = SBIAS_OFF + MOE_MAX_EXPERTS * 4;
  static constexpr int STG_LD = 33;
  static constexpr int XTRA = on ? STG_OFF + BM * STG_LD * 4 : 0;
};
template <int BN, int SCHED, int EPI, bool F8, bool MX> struct CfgOf {
  using type = TileCfg<BN, EpiOf<BN, SCHED, EPI, F8, MX>::staged, EpiWidth<BN, SCHED, EPI, F8>::warps,
                       EpiOf<BN, SCHED, EPI, F8, MX>::slabs, MX ? MxCfg<BN>::SF_STAGE : 0,
                       MX ? (MxCfg<BN>::MAX_STAGES < 6 ? MxCfg<BN>::MAX_STAGES : 6) : 6,
                       MX ? 512 : 0, RouterOf<SCHED, EPI, F8>::XTRA>;
};

// The router epilogue's logits of one token (this thread's TMEM lane), 32 experts at a time, as
// the epilogue stores them (accumulator + logit bias); at(e) re-reads the stored value.
struct TmemLogits {
  uint32_t t_row;
  const float* bias;   // the logit bias in shared memory (zero past E), or null
  const float* row;    // this token's stored logits (null for a row past the tensor's end)
  __device__ __forceinline__ void chunk(int q, float (&v)[32]) const {
    uint32_t u[32];
    ptx::tmem_ld32(t_row + static_cast<uint32_t>(q * 32), u);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
    if (bias) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += bias[q * 32 + i];
    }
  }
  __device__ __forceinline__ float at(int e) const { return row ? row[e] : 0.f; }
};

struct KArgs {
  int G;
  const int32_t* offsets;
  int M, N, K;
  int64_t b_group_rows, b_up_rows;
  int f;
  void* out;
  int64_t ldo, out_group_stride;
  void* out2;
  int64_t ldo2;
  const void* aux;
  int64_t ld_aux;
  const float* bias;
  int* tile_ctr;    // run-time scheduling: the next unclaimed tile (zeroed before the launch)
  const int32_t* gather;   // gathered operand: source row of each operand row
  int gather_rows;         // rows of the gathered source tensor
  const float* a_scale;    // FP8: dequantisation scale of A (one value)
  const float* b_scale;    // FP8: dequantisation scale of B, one per group
  int b_scale_per_group;   // FP8: 0 -> b_scale[0] for every group
  float* amax_out;         // FP8 SwiGLU epilogues: max |h| or |[da | du]| (fp32 bits, raised)
  const uint8_t* sfa;      // MXFP8: packed block scales of A (activation layout)
  const uint8_t* sfb;      // MXFP8: packed block scales of B (weight layout)
  uint8_t* q_out;          // MXFP8 SwiGLU forward: h codes [rows, f]
  uint8_t* q_sf;           // MXFP8 SwiGLU forward: h block scales (activation layout)
  int kch;                 // MXFP8: 128-element K chunks of the operands (weight gradients:
                           // the token-chunk capacity of the scale layouts)
  const int32_t* cbase;    // MXFP8 weight gradients: each group's first token chunk
  int kch_out;             // MXFP8 SwiGLU forward: 128-element chunks of h's rows
  RouterEpi rt;            // router top-k in the epilogue (rt.idx null: off)
  int* err;
};

struct TileInfo {
  int g, m0, m_end, n0, k0, k_end, kblocks;
  int mt, nt;   // RAGGED_M: row tile (over all groups) and column tile
};

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + __expf(-a)); }
// Sigmoid of the SwiGLU backward.  With E4M3 operands its MMAs take half the bf16 time and the
// epilogue bounds the product; its results are rounded to bf16, so there the quotient is the
// approximate one (about 2 ulp of fp32) instead of the IEEE division's multi-instruction
// sequence: fc2 dgrad 0.78 -> 0.56 ms on the 128-expert layer (bf16: no change either way, so
// bf16 keeps the IEEE quotient).  A huge denominator (a below about -87) gives 0 either way.
#ifndef MOE_FAST_SIGMOID_F8
#define MOE_FAST_SIGMOID_F8 1
#endif
template <bool FAST>
__device__ __forceinline__ float sigmoid_f(float a) {
  return FAST ? __fdividef(1.0f, 1.0f + __expf(-a)) : 1.0f / (1.0f + __expf(-a));
}

template <int BN, int SCHED, int EPI, int TBM = BM, int BKE = BK>
struct Sched {
  // Number of output column tiles.
  __device__ static int n_tiles(const KArgs& p) {
    if (EPI == EPI_SWIGLU_FWD) return (p.f + BN / 2 - 1) / (BN / 2);
    return (p.N + BN - 1) / BN;
  }
  __device__ static int total(const KArgs& p, const int* s_pre) {
    if (SCHED == RAGGED_M) return s_pre[p.G] * n_tiles(p);
    return p.G * ((p.M + TBM - 1) / TBM) * n_tiles(p);
  }
  // s_ord (RAGGED_K, run-time scheduling): the groups in tile-list order; null: g ascending.
  __device__ static TileInfo decode(const KArgs& p, const int* s_off, const int* s_pre,
                                    const int* s_ord, int tile) {
    TileInfo ti;
    const int nt_count = n_tiles(p);
    if (SCHED == RAGGED_M) {
      const int mt = tile / nt_count, nt = tile - mt * nt_count;
      int lo = 0, hi = p.G;   // largest g with s_pre[g] <= mt
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid] <= mt) lo = mid; else hi = mid;
      }
      ti.g = lo;
      ti.m0 = s_off[lo] + (mt - s_pre[lo]) * TBM;
      ti.m_end = s_off[lo + 1];
      ti.n0 = nt * (EPI == EPI_SWIGLU_FWD ? BN / 2 : BN);
      ti.k0 = 0;
      ti.k_end = p.K;
      ti.mt = mt;
      ti.nt = nt;
    } else {
      const int mtc = (p.M + TBM - 1) / TBM;
      const int per = mtc * nt_count;
      const int pos = tile / per;
      const int r = tile - pos * per;
      ti.g = s_ord ? s_ord[pos] : pos;
      const int mt = r / nt_count, nt = r - mt * nt_count;
      ti.m0 = mt * TBM;
      ti.m_end = p.M;
      ti.n0 = nt * BN;
      ti.k0 = s_off[ti.g];
      ti.k_end = s_off[ti.g + 1];
      ti.mt = mt;
      ti.nt = nt;
    }
    ti.kblocks = (ti.k_end - ti.k0 + BKE - 1) / BKE;
    return ti;
  }
};

// ---------------------------------------------------------------- staging slab helpers
// A slab is 32 rows x 128 bytes laid out as the 128-byte-swizzled box of a TMA map: the 16-byte
// chunk j of row r sits at r*128 + ((j ^ (r & 7)) * 16).  Lane r owns row r.
__device__ __forceinline__ void slab_put(uint8_t* slab, int lane, int j, const uint4& v) {
  *reinterpret_cast<uint4*>(slab + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
}
__device__ __forceinline__ uint4 slab_get(const uint8_t* slab, int lane, int j) {
  return *reinterpret_cast<const uint4*>(slab + lane * 128 + ((j ^ (lane & 7)) << 4));
}
// A half slab is 32 rows x 64 bytes laid out as the 64-byte-swizzled box of a TMA map: the
// 16-byte chunk j (0..3) of row r sits at r*64 + ((j ^ ((r >> 1) & 3)) * 16).
__device__ __forceinline__ void half_put(uint8_t* h, int lane, int j, const uint4& v) {
  *reinterpret_cast<uint4*>(h + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
}
__device__ __forceinline__ uint4 half_get(const uint8_t* h, int lane, int j) {
  return *reinterpret_cast<const uint4*>(h + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4));
}
// Make the warp's slab writes visible to the TMA engine, then store the slab (lane 0).
__device__ __forceinline__ void slab_store_2d(const CUtensorMap* m, const uint8_t* slab, int lane,
                                              int c0, int c1) {
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(m, slab, c0, c1);
    ptx::bulk_commit();
  }
}

template <int BN, bool A_MN, bool B_MN, int SCHED, int EPI, bool GATHER = false, bool F8 = false,
          bool MX = false>
__global__ void __launch_bounds__(64 + 32 * EpiWidth<BN, SCHED, EPI, F8>::warps, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                   const __grid_constant__ CUtensorMap tmO2, const KArgs p) {
  constexpr bool TMA_OUT = OutPath<SCHED, EPI>::tma;
  constexpr int EPI_WARPS = EpiWidth<BN, SCHED, EPI, F8>::warps;
  constexpr int SLABS = EpiOf<BN, SCHED, EPI, F8, MX>::slabs;
  constexpr bool HALF_SLABS = EpiOf<BN, SCHED, EPI, F8, MX>::half_slabs;
  using C = typename CfgOf<BN, SCHED, EPI, F8, MX>::type;
  constexpr bool DYN = DynMode<SCHED, EPI>::on;
  // gathered operands: A of a row-ragged product (K-major) or B of a weight gradient (MN-major)
  static_assert(!GATHER || (SCHED == RAGGED_M && !A_MN) || (SCHED == RAGGED_K && B_MN),
                "unsupported gathered operand");
  constexpr int TM = BM;   // rows of one walker tile
  // K elements per stage: 128-byte rows hold 64 bf16 or 128 E4M3 values
  constexpr int BKE = F8 ? 2 * BK : BK;
  using S = Sched<BN, SCHED, EPI, TM, BKE>;
  // MN-major operand tiles are chunks of 128-byte rows along K: 64 bf16 or 128 E4M3 of M/N each
  constexpr int MNW = F8 ? 128 : 64;
  constexpr int MN_CHUNK = BKE * 128;   // bytes of one such chunk in a stage
  static_assert(!F8 || !GATHER, "FP8 operands: no gathered loads");
  // MXFP8: K-major E4M3 operands of a row-ragged product, or the MN-major token-blocked operands
  // of a weight gradient (128-wide tiles); one stage is one 128-element K chunk
  static_assert(!MX || (F8 &&
                        ((SCHED == RAGGED_M && !A_MN && (!B_MN || BN % 128 == 0)) ||
                         (SCHED == RAGGED_K && A_MN && B_MN && EPI == EPI_F32 && BN == 128)) &&
                        BN <= 256 &&
                        C::ACC_STRIDE == MxCfg<BN>::ACC_STRIDE &&
                        MxCfg<BN>::SF_COL0 + C::STAGES * MX_SF_COLS <= C::TMEM_COLS),
                "MXFP8 tile configuration");
  constexpr int STAGES = C::STAGES;
  constexpr uint32_t STAGE_TX = A_STAGE + C::B_STAGE + (MX ? MxCfg<BN>::SF_STAGE : 0);
  constexpr int NACC = MX ? MxCfg<BN>::NACC : 2;   // TMEM accumulators (tile i uses i % NACC)

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint8_t* staging = smem + C::RING;
  uint8_t* sSF = smem + C::RING + C::STAGING;   // MXFP8 block scales, one slot per stage
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING + C::STAGING + C::SF_RING);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* epi_bar = tempty + 2;    // one per epilogue warp (TMA loads of saved activations)
  uint64_t* feed_full = epi_bar + EPI_WARPS;   // run-time tile ring (DYN)
  uint64_t* feed_empty = feed_full + FEED;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(feed_empty + FEED);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_bad = reinterpret_cast<int*>(tmem_holder + 2);
  int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
  int* s_pre = s_off + (MAXG + 1);   // RAGGED_M: tile prefix; DYN: groups by row count
  volatile int* s_feed = s_pre + (MAXG + 1);
  const int* s_ord = DYN ? s_pre : nullptr;
  // router epilogue: the histogram barrier (one arrival per epilogue warp) and two histograms
  // (tiles alternate between them)
  constexpr bool ROUTER = RouterOf<SCHED, EPI, F8>::on && !MX;
  uint8_t* xtra = smem + C::RING + C::STAGING + C::SF_RING + C::AUX;
  uint64_t* hbar = reinterpret_cast<uint64_t*>(xtra);
  int* s_rhist = reinterpret_cast<int*>(xtra + RouterOf<SCHED, EPI, F8>::HIST_OFF);
  float* s_lbias = reinterpret_cast<float*>(xtra + RouterOf<SCHED, EPI, F8>::LBIAS_OFF);
  float* s_sbias = reinterpret_cast<float*>(xtra + RouterOf<SCHED, EPI, F8>::SBIAS_OFF);
  unsigned* s_stg = reinterpret_cast<unsigned*>(xtra + RouterOf<SCHED, EPI, F8>::STG_OFF);

  WaitStats wst;
  wst.start();
  constexpr int WAIT_KIND = (A_MN ? 1 : 0) | (B_MN ? 2 : 0) | (SCHED << 2) | (EPI << 3) | ((F8 || MX) ? 32 : 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Tile walker: one per CTA (static walk), or tiles claimed at run time (DYN).
  const int unit = static_cast<int>(blockIdx.x);
  const int units = static_cast<int>(gridDim.x);

  // 128-byte swizzled tiles need 1024-byte aligned shared memory.
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      ptx::mbar_init(&tempty[i], EPI_WARPS);
    }
    for (int i = 0; i < EPI_WARPS; ++i) ptx::mbar_init(&epi_bar[i], 1);
    if (ROUTER) ptx::mbar_init(hbar, EPI_WARPS);
    if (DYN) {
      for (int i = 0; i < FEED; ++i) {
        ptx::mbar_init(&feed_full[i], 1);
        ptx::mbar_init(&feed_empty[i], 1 + EPI_WARPS);   // the MMA warp and every epilogue warp
      }
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (ROUTER && p.rt.idx) {
    for (int i = threadIdx.x; i < 2 * MOE_MAX_EXPERTS; i += blockDim.x) s_rhist[i] = 0;
    for (int i = threadIdx.x; i < MOE_MAX_EXPERTS; i += blockDim.x) {
      s_lbias[i] = (p.bias && i < p.N) ? p.bias[i] : 0.f;
      s_sbias[i] = (p.rt.sel_bias && i < p.N) ? p.rt.sel_bias[i] : 0.f;
    }
  }
  // Group table: row (RAGGED_M) or reduction (RAGGED_K) offsets, and for RAGGED_M the prefix
  // of per-group row-tile counts.
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
    int v;
    if (p.offsets) v = p.offsets[i];
    else v = static_cast<int>((static_cast<int64_t>(SCHED == RAGGED_M ? p.M : p.K) * i) / p.G);
    s_off[i] = v;
  }
  __syncthreads();
  // The offsets must be non-decreasing and stay inside the operands (rows of A for RAGGED_M,
  // the reduction length for RAGGED_K); otherwise nothing is computed and the error recorded.
  if (threadIdx.x == 0) {
    const int cap = SCHED == RAGGED_M ? p.M : p.K;
    int bad = (s_off[0] < 0 || s_off[p.G] > cap) ? 1 : 0;
    for (int i = 0; i < p.G && !bad; ++i) bad = s_off[i + 1] < s_off[i];
    *s_bad = bad;
    if (bad) record_error(p.err, DEVERR_BAD_OFFSETS);
  }
  __syncthreads();
  if (*s_bad) return;
  if (SCHED == RAGGED_M && warp == 0) {
    // s_pre[g] = sum_{g' < g} ceil(rows_g' / TM): lane L scans groups [L*per, (L+1)*per)
    const int per = (p.G + 31) / 32;
    const int lo = min(p.G, lane * per), hi = min(p.G, lo + per);
    int local = 0;
    for (int g = lo; g < hi; ++g) local += (s_off[g + 1] - s_off[g] + TM - 1) / TM;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int g = lo; g < hi; ++g) {
      s_pre[g] = run;
      run += (s_off[g + 1] - s_off[g] + TM - 1) / TM;
    }
    if (lane == 31) s_pre[p.G] = incl;
  }
  if (DYN) {
    // groups by row count, most first (ties: lower index first)
    for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
      const int n = s_off[g + 1] - s_off[g];
      int rank = 0;
      for (int h = 0; h < p.G; ++h) {
        const int m = s_off[h + 1] - s_off[h];
        rank += (m > n || (m == n && h < g)) ? 1 : 0;
      }
      s_pre[rank] = g;
    }
  }
  __syncthreads();

  const int total = S::total(p, s_pre);
  // nothing for this CTA
  if (DYN ? total == 0 : unit >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 && GATHER) {
    // ------------------------------------------------------------ TMA producer, gathered rows
    // "Megatron-Bridge 深度剖析", §Permute Fusion: the permutation is folded into the operand
    // load.  The whole warp issues: lane 0 waits on the ring, arms each stage and loads the
    // plain operand; every lane gathers four of the gathered operand's rows per copy
    // (tile::gather4).  Rows past the operand's end read row 0 (their products are masked or
    // multiplied by zeroed rows).
    int stage = 0;
    uint32_t phase = 0;
    int armed[STAGES];
    for (int i = 0; i < STAGES; ++i) armed[i] = -1;
    bool ok = true;
    const int lim = SCHED == RAGGED_M ? p.M : p.K;   // operand rows
    auto src_row = [&](int s) -> int {
      if (s < 0 || s >= lim) return 0;
      const int r = __ldg(p.gather + s);
      if (r < 0 || r >= p.gather_rows) {
        record_error(p.err, DEVERR_BAD_TOKEN);
        return 0;
      }
      return r;
    };
    int nclaims = 0;
    auto claim = [&]() -> int { return claim_tile(p.tile_ctr, total, nclaims); };
    int fslot = 0;
    uint32_t fphase = 0;
    int next = (DYN && lane == 0) ? claim() : unit;
    for (int it = 0; ok; ++it) {
      int tile;
      if (DYN) {
        bool w = true;
        if (lane == 0) {
          w = ptx::mbar_wait(&feed_empty[fslot], fphase ^ 1u, abort_flag, p.err);
          if (w) {
            s_feed[fslot] = next;
            ptx::mbar_arrive(&feed_full[fslot]);
          }
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        tile = __shfl_sync(0xffffffffu, next, 0);
        if (!w) { ok = false; break; }
        if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
        if (tile < 0) break;
        if (lane == 0) next = claim();
      } else {
        tile = unit + it * units;
        if (tile >= total) break;
      }
      const TileInfo ti = S::decode(p, s_off, s_pre, s_ord, tile);
      // row-ragged: lane j owns rows 4j..4j+3 of the 128-row A tile for the whole tile
      int ar[4] = {0, 0, 0, 0};
      if (SCHED == RAGGED_M) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ar[i] = src_row(ti.m0 + 4 * lane + i);
      }
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        const int kk = ti.k0 + kb * BK;
        // weight gradient: lane j owns k-rows 4q..4q+3 (q = j mod 16) of this k-block, in the
        // 64-column chunks j/16, j/16 + 2, ...
        int br[4] = {0, 0, 0, 0};
        if (SCHED == RAGGED_K) {
#pragma unroll
          for (int i = 0; i < 4; ++i) br[i] = src_row(kk + 4 * (lane & 15) + i);
        }
        bool w = true;
        if (lane == 0) {
          w = ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err);
          if (w) {
            ptx::mbar_arrive_expect_tx(&full[stage], STAGE_TX);
            armed[stage] = static_cast<int>(phase);
          }
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) { ok = false; break; }
        uint8_t* a_dst = sA + stage * A_STAGE;
        uint8_t* b_dst = sB + stage * C::B_STAGE;
        if (SCHED == RAGGED_M) {
          ptx::tma_gather4_2d(a_dst + lane * 512, &tmA, &full[stage], kk, ar[0], ar[1], ar[2], ar[3]);
          if (lane == 0) {
            const int brow = static_cast<int>(ti.g * p.b_group_rows) + ti.n0;
            if (EPI == EPI_SWIGLU_FWD) {
              ptx::tma_load_2d(b_dst, &tmB, &full[stage], kk, brow);
              ptx::tma_load_2d(b_dst + (BN / 2) * 128, &tmB, &full[stage], kk,
                               brow + static_cast<int>(p.b_up_rows));
            } else {
              ptx::tma_load_2d(b_dst, &tmB, &full[stage], kk, brow);
            }
          }
        } else {
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              ptx::tma_load_2d(a_dst + c * (BK * 128), &tmA, &full[stage], ti.m0 + 64 * c, kk);
          }
          const int q = lane & 15;
#pragma unroll
          for (int c = lane >> 4; c < BN / 64; c += 2)
            ptx::tma_gather4_2d(b_dst + c * (BK * 128) + q * 512, &tmB, &full[stage],
                                ti.n0 + 64 * c, br[0], br[1], br[2], br[3]);
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // Unwinding: let every copy of an armed stage land before the CTA exits.
      for (int i = 0; i < STAGES; ++i) {
        if (armed[i] < 0) continue;
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&full[i], static_cast<uint32_t>(armed[i])) &&
               ptx::globaltimer() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
      for (int i = 0; i < STAGES; ++i) armed[i] = -1;
      bool ok = true;
      // Loads of k-block kb of tile ti into `stage`.
      auto issue = [&](const TileInfo& ti, int kb, int stg) {
        uint8_t* a_dst = sA + stg * A_STAGE;
        uint8_t* b_dst = sB + stg * C::B_STAGE;
        const int kk = ti.k0 + kb * BKE;
        const int m_cta = ti.m0;
        auto box = [&](void* dst, const CUtensorMap* m, int c0, int c1) {
          if (SCHED == RAGGED_K && MOE_WGRAD_LOAD_HINT)
            ptx::tma_load_2d_hint(dst, m, &full[stg], c0, c1, ptx::policy_evict_last());
          else
            ptx::tma_load_2d(dst, m, &full[stg], c0, c1);
        };
        if (!A_MN) {
          box(a_dst, &tmA, kk, m_cta);
        } else {
#pragma unroll
          for (int c = 0; c < BM / MNW; ++c) box(a_dst + c * MN_CHUNK, &tmA, m_cta + MNW * c, kk);
        }
        if (!B_MN) {
          const int brow = static_cast<int>(ti.g * p.b_group_rows) + ti.n0;
          if (EPI == EPI_SWIGLU_FWD) {
            box(b_dst, &tmB, kk, brow);
            box(b_dst + (BN / 2) * 128, &tmB, kk, brow + static_cast<int>(p.b_up_rows));
          } else {
            box(b_dst, &tmB, kk, brow);
          }
        } else {
          const int krow = (SCHED == RAGGED_M) ? static_cast<int>(ti.g * p.b_group_rows) + kk : kk;
#pragma unroll
          for (int c = 0; c < BN / MNW; ++c) box(b_dst + c * MN_CHUNK, &tmB, ti.n0 + MNW * c, krow);
        }
        if (MX) {
          // this K chunk's block scales: the A row tile's chunk, then the B tile's chunks
          uint8_t* sf_dst = sSF + stg * MxCfg<BN>::SF_STAGE;
          constexpr int SFB = MX_CHUNK * MxCfg<BN>::SFB_CH;
          if (SCHED == RAGGED_K) {
            // token chunk kb of group g's rows; A's and B's 128-row tiles
            const int64_t kc = __ldg(p.cbase + ti.g) + kb;
            ptx::bulk_load(sf_dst, p.sfa + (static_cast<int64_t>(ti.mt) * p.kch + kc) * MX_CHUNK,
                           MX_CHUNK, &full[stg]);
            ptx::bulk_load(sf_dst + MX_CHUNK,
                           p.sfb + (static_cast<int64_t>(ti.nt) * p.kch + kc) * MX_CHUNK, SFB,
                           &full[stg]);
          } else {
            ptx::bulk_load(sf_dst, p.sfa + (static_cast<int64_t>(ti.mt) * p.kch + kb) * MX_CHUNK,
                           MX_CHUNK, &full[stg]);
            const int64_t wt = static_cast<int64_t>(ti.g) * S::n_tiles(p) + ti.nt;
            ptx::bulk_load(sf_dst + MX_CHUNK, p.sfb + (wt * p.kch + kb) * SFB, SFB, &full[stg]);
          }
        }
      };
      // Run-time tiles: the next tile is claimed before the current one's loads are issued,
      // hiding the atomic's latency; -1 once the list is exhausted.
      int nclaims = 0;
      auto claim = [&]() -> int { return claim_tile(p.tile_ctr, total, nclaims); };
      int fslot = 0;
      uint32_t fphase = 0;
      int next = DYN ? claim() : unit;
      for (int it = 0; ok; ++it) {
        int tile;
        if (DYN) {
          tile = next;
          if (!ptx::mbar_wait(&feed_empty[fslot], fphase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          s_feed[fslot] = tile;
          ptx::mbar_arrive(&feed_full[fslot]);
          if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
          if (tile < 0) break;
          next = claim();
        } else {
          tile = unit + it * units;
          if (tile >= total) break;
        }
        const TileInfo ti = S::decode(p, s_off, s_pre, s_ord, tile);
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const unsigned long long w0 = wst.now();
          const bool freed = ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err);
          wst.since(wst.prod, w0);
          if (!freed) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&full[stage], STAGE_TX);
          armed[stage] = static_cast<int>(phase);
          issue(ti, kb, stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // Unwinding: let every copy this thread issued land before the CTA exits.
        for (int i = 0; i < STAGES; ++i) {
          if (armed[i] < 0) continue;
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(&full[i], static_cast<uint32_t>(armed[i])) &&
                 ptx::globaltimer() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t IDESC =
        F8 ? ptx::idesc_e4m3_f32(BM, BN, A_MN, B_MN) : ptx::idesc_bf16_f32(BM, BN, A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int fslot = 0;
    uint32_t fphase = 0;
    for (int it = 0; ok; ++it) {
      int tile;
      if (DYN) {
        if (!ptx::mbar_wait(&feed_full[fslot], fphase, abort_flag, p.err)) { ok = false; break; }
        tile = s_feed[fslot];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&feed_empty[fslot]);
        if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
        if (tile < 0) break;
      } else {
        tile = unit + it * units;
        if (tile >= total) break;
      }
      const TileInfo ti = S::decode(p, s_off, s_pre, s_ord, tile);
      if (ti.kblocks == 0) continue;
      const unsigned long long wa = wst.now();
      const bool drained = ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err);
      wst.since(wst.acc, wa);
      if (!drained) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::ACC_STRIDE);
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        const unsigned long long wf = wst.now();
        const bool landed = ptx::mbar_wait(&full[stage], phase, abort_flag, p.err);
        wst.since(wst.full, wf);
        ++wst.kblocks;
        if (!landed) { ok = false; break; }
        uint8_t* a_src = sA + stage * A_STAGE;
        uint8_t* b_src = sB + stage * C::B_STAGE;
        if (SCHED == RAGGED_K && kb == ti.kblocks - 1) {
          // Rows of this k-block past the group's end belong to the next group: zero them in
          // the A tile (MN-major: row r of chunk c is 128 contiguous bytes).
          const int valid = ti.k_end - (ti.k0 + kb * BKE);
          if (valid < BKE) {
            const int nbytes = (BKE - valid) * 128;
            for (int c = 0; c < BM / MNW; ++c) {
              uint8_t* base = a_src + c * MN_CHUNK + valid * 128;
              for (int o = lane * 16; o < nbytes; o += 32 * 16)
                *reinterpret_cast<uint4*>(base + o) = make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_smem();
          }
          __syncwarp();
        }
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(a_src), b_addr = ptx::smem_u32(b_src);
          // MXFP8: the stage's block scales into its TMEM slot (the copies and the MMAs below
          // execute in issue order; the slot's previous MMAs finished before this stage was
          // refilled, as they released it)
          const uint32_t sf_t = tmem_base + static_cast<uint32_t>(MX ? MxCfg<BN>::SF_COL0 + stage * MX_SF_COLS : 0);
          if (MX) {
            const uint32_t sf_s = ptx::smem_u32(sSF + stage * MxCfg<BN>::SF_STAGE);
            ptx::tmem_cp_32x128_x4(sf_t, ptx::smem_desc_plain(sf_s, 128));
#pragma unroll
            for (int ch = 0; ch < MxCfg<BN>::SFB_CH; ++ch)
              ptx::tmem_cp_32x128_x4(sf_t + 8 + 4 * ch,
                                     ptx::smem_desc_plain(sf_s + MX_CHUNK * (1 + ch), 128));
          }
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16) {
            // one instruction takes 32 bytes of K: 16 bf16 or 32 E4M3 -- along a K-major row, or
            // that many 128-byte rows of an MN-major chunk
            constexpr uint32_t MN_KSTEP = (F8 ? 32 : 16) * 128;
            const uint64_t ad = A_MN ? ptx::smem_desc_sw128(a_addr + k16 * MN_KSTEP, MN_CHUNK, 1024)
                                     : ptx::smem_desc_sw128(a_addr + k16 * 32, 16, 1024);
            const uint64_t bd = B_MN ? ptx::smem_desc_sw128(b_addr + k16 * MN_KSTEP, MN_CHUNK, 1024)
                                     : ptx::smem_desc_sw128(b_addr + k16 * 32, 16, 1024);
            if (MX)   // K slice k16 of the chunk: byte k16 of each row's scale column
              ptx::umma_mx(d_tmem, ad, bd, ptx::idesc_mx_e4m3(BM, BN, A_MN, B_MN, k16, k16), sf_t,
                           sf_t + 8, (kb | k16) != 0 ? 1u : 0u);
            else if (F8) ptx::umma_f8(d_tmem, ad, bd, IDESC, (kb | k16) != 0 ? 1u : 0u);
            else ptx::umma_bf16(d_tmem, ad, bd, IDESC, (kb | k16) != 0 ? 1u : 0u);
          }
          // frees the smem stage when these MMAs finish
          ptx::umma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) ptx::umma_commit(&tfull[acc]);   // accumulator ready for the epilogue
      __syncwarp();
      if (NACC == 2) acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..)
    const int e = warp - 2;          // epilogue warp index
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;     // row inside the tile
    // Accumulator columns of this warp: all of them (4 epilogue warps) or one half (8 warps).
    // For the SwiGLU forward the half is taken in h columns (gate and up halves together).
    constexpr int NPART = EPI_WARPS / 4;
    const int part = e / 4;
    const int span = (EPI == EPI_SWIGLU_FWD ? BN / 2 : BN) / NPART;
    const int c_lo = part * span, c_hi = c_lo + span;
    uint8_t* slabs = staging + e * (SLABS * SLAB);
    uint64_t* my_bar = &epi_bar[e];
    int slab_sel = 0;
    uint32_t ld_phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    // fp32 slab -> [g][row][col] (weight gradients: evict-first in L2)
    auto store_f32 = [&](const uint8_t* src, int col, int row, int g) {
      if (SCHED == RAGGED_K && MOE_WGRAD_STORE_HINT)
        ptx::tma_store_3d_hint(&tmO0, src, col, row, g, ptx::policy_evict_first());
      else
        ptx::tma_store_3d(&tmO0, src, col, row, g);
    };
    // fp32 slab (32 rows x 32 columns, swizzled) -> [g][row0 + r][col ..] with warp-wide
    // coalesced stores: lanes 8i..8i+7 write one 128-byte row segment; rows past `rows`
    // (the output's end) are skipped.  v == nullptr stores zeros.
    auto lsu_store = [&](const uint8_t* slab, int col, int row, int g, int rows) {
      float* base = static_cast<float*>(p.out) + static_cast<int64_t>(g) * p.out_group_stride;
      const int ch = lane & 7;
      const int c4 = col + ch * 4;
      if (c4 >= p.N) return;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + (lane >> 3);
        if (r >= rows) break;
        const uint4 v = slab ? slab_get(slab, r, ch) : make_uint4(0, 0, 0, 0);
        st16_cs(base + static_cast<int64_t>(row + r) * p.ldo + c4, v);
      }
    };
    // Next free staging slab of this warp: at most SLABS-1 earlier stores may still read theirs
    // (a paced weight-gradient tile: every earlier store has landed).
    bool pace = false;
    auto next_slab = [&]() -> uint8_t* {
      if (lane == 0) {
        if (SCHED == RAGGED_K && pace) ptx::bulk_wait<0>();
        else ptx::bulk_wait_read<SLABS - 1>();
      }
      __syncwarp();
      uint8_t* s = slabs + slab_sel * SLAB;
      if (++slab_sel == SLABS) slab_sel = 0;
      return s;
    };
    int fslot = 0;
    uint32_t fphase = 0;
    uint32_t hphase = 0;   // router: phase of the histogram barrier (tiles alternate buffers)
    for (int it = 0;; ++it) {
      int tile;
      if (DYN) {
        if (!ptx::mbar_wait(&feed_full[fslot], fphase, abort_flag, p.err)) break;
        tile = s_feed[fslot];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&feed_empty[fslot]);
        if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
        if (tile < 0) break;
      } else {
        tile = unit + it * units;
        if (tile >= total) break;
      }
      const TileInfo ti = S::decode(p, s_off, s_pre, s_ord, tile);
      pace = SCHED == RAGGED_K && ti.kblocks >= 2 && ti.kblocks <= MOE_WGRAD_PACE_KB;
      const int m_cta = ti.m0;                      // this CTA's rows of the tile
      const int row0 = m_cta + q * 32;              // first row of this warp's slab
      const int rows_here = min(32, ti.m_end - row0);
      const int row = m_cta + r;
      const bool valid = row < ti.m_end;
      if (ti.kblocks == 0) {
        // Empty reduction (an expert with no rows): its weight-gradient block is zero.  One
        // zeroed slab is stored to every 32-column chunk of this warp's rows.
        if (EPI == EPI_F32 && SCHED == RAGGED_K && MOE_WGRAD_LSU_STORE && rows_here > 0) {
          for (int c = c_lo; c < c_hi; c += 32) {
            if (ti.n0 + c >= p.N) break;
            lsu_store(nullptr, ti.n0 + c, row0, ti.g, rows_here);
          }
        } else if (EPI == EPI_F32 && SCHED == RAGGED_K && TMA_OUT && rows_here > 0) {
          uint8_t* z = next_slab();
#pragma unroll
          for (int j = 0; j < 8; ++j) slab_put(z, lane, j, make_uint4(0, 0, 0, 0));
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int c = c_lo; c < c_hi; c += 32) {
              if (ti.n0 + c >= p.N) break;
              store_f32(z, ti.n0 + c, row0, ti.g);
              ptx::bulk_commit();
            }
          }
          __syncwarp();
        }
        continue;
      }
      const unsigned long long we = wst.now();
      const bool ready = ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err);
      wst.since(wst.epi, we);
      if (!ready) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * C::ACC_STRIDE);
      // Full slabs go out through TMA (the maps clip at the tensors' edges).  For ragged rows a
      // slab that crosses the end of its expert's rows would overwrite the next expert's: it is
      // written with masked stores instead.
      // (the MXFP8 SwiGLU backward stages through slabs only when [da | du] is also stored in bf16)
      const bool tma_slab = TMA_OUT && (SCHED == RAGGED_K ? rows_here > 0 : rows_here == 32) &&
                            (!(MX && EPI == EPI_SWIGLU_BWD) || p.out != nullptr);
      // FP8: the accumulator holds products of decoded E4M3 values; both scales apply here
      // (MXFP8: the block scales were applied by the MMAs)
      const float sc = F8 && !MX ? __ldg(p.a_scale) * __ldg(p.b_scale + (p.b_scale_per_group ? ti.g : 0)) : 1.0f;
      // FP8 SwiGLU epilogues: max |.| over this warp's stored (bf16) values of h (forward) or
      // [da | du] (backward), for that tensor's own quantisation
      constexpr bool AMAX = F8 && !MX && (EPI == EPI_SWIGLU_FWD || EPI == EPI_SWIGLU_BWD);
      float hmax = 0.f;
      auto track = [&](float v) {
        if (AMAX) hmax = fmaxf(hmax, fabsf(__bfloat162float(__float2bfloat16_rn(v))));
      };
      bool aborted = false;

      if (rows_here <= 0) {
        // no row of this slab exists
      } else if (MX && EPI == EPI_SWIGLU_FWD) {
        // h quantised to MXFP8 where it is made: a thread holds 32 consecutive h values of its
        // row (one block along f, fc2's reduction dimension), rounded to bf16 first.  Codes and
        // the block's scale byte go straight out (32 bytes and 1 byte per block); bf16 h and
        // [a | u] only if asked for.
        bf16* hrow = p.out ? static_cast<bf16*>(p.out) + row * p.ldo : nullptr;
        bf16* arow = p.out2 ? static_cast<bf16*>(p.out2) + row * p.ldo2 : nullptr;
        uint8_t* qrow = p.q_out + static_cast<int64_t>(row) * p.f;
        uint8_t* sfrow = p.q_sf + static_cast<int64_t>(ti.mt) * p.kch_out * MX_CHUNK + (r & 31) * 16 +
                         (r >> 5) * 4;
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          uint32_t ga[32], up[32];
          ptx::tmem_ld32(t_row + c, ga);
          ptx::tmem_ld32(t_row + BN / 2 + c, up);
          ptx::tmem_ld_wait();
          if (!valid) continue;
          float hv[32];
          float am = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            hv[i] = __bfloat162float(__float2bfloat16_rn(
                silu_f(__uint_as_float(ga[i])) * __uint_as_float(up[i])));
            am = fmaxf(am, fabsf(hv[i]));
          }
          const int ex = mx_exponent(am);
          const float inv = mx_inv_scale(ex);
          uint32_t w[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t lo = cvt_e4m3x2(hv[4 * j] * inv, hv[4 * j + 1] * inv);
            const uint32_t hi = cvt_e4m3x2(hv[4 * j + 2] * inv, hv[4 * j + 3] * inv);
            w[j] = lo | (hi << 16);
          }
          *reinterpret_cast<uint4*>(qrow + col) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(qrow + col + 16) = make_uint4(w[4], w[5], w[6], w[7]);
          const int blk = col >> 5;
          uint8_t* sf = sfrow + (blk >> 2) * MX_CHUNK;
          sf[blk & 3] = static_cast<uint8_t>(ex + 127);
          if (col + 32 >= p.f) {
            for (int j = (blk & 3) + 1; j < 4; ++j) sf[j] = 127;   // blocks past f: 2^0
          }
          if (hrow) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              st16(hrow + col + v * 8, pack16(hv + 8 * v, static_cast<const bf16*>(nullptr)));
          }
          if (arow) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float av[8], uv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                av[i] = __uint_as_float(ga[8 * v + i]);
                uv[i] = __uint_as_float(up[8 * v + i]);
              }
              st16(arow + col + v * 8, pack16(av, static_cast<const bf16*>(nullptr)));
              st16(arow + p.f + col + v * 8, pack16(uv, static_cast<const bf16*>(nullptr)));
            }
          }
        }
      } else if (tma_slab && EPI == EPI_STORE) {
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 64) {
          const int col = ti.n0 + c;
          if (col >= p.N) break;
          uint32_t v0[32], v1[32];
          ptx::tmem_ld32(t_row + c, v0);
          ptx::tmem_ld32(t_row + c + 32, v1);
          ptx::tmem_ld_wait();
          uint8_t* slab = next_slab();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              a[i] = __uint_as_float(v0[8 * j + i]) * sc;
              b[i] = __uint_as_float(v1[8 * j + i]) * sc;
            }
            slab_put(slab, lane, j, pack16(a, static_cast<const bf16*>(nullptr)));
            slab_put(slab, lane, 4 + j, pack16(b, static_cast<const bf16*>(nullptr)));
          }
          slab_store_2d(&tmO0, slab, lane, col, row0);
        }
      } else if (tma_slab && EPI == EPI_F32) {
        // 32-column chunks; the TMEM load of chunk i+1 is in flight while chunk i is staged
        // and stored (two register sets, alternating).
        auto put = [&](const uint32_t (&v)[32], int col) {
          // FP8: both dequantisation scales applied to the fp32 result
          auto w = [&](int i) { return F8 ? __float_as_uint(__uint_as_float(v[i]) * sc) : v[i]; };
          if (SCHED == RAGGED_K && MOE_WGRAD_LSU_STORE) {
            // one slab: written, read back by the whole warp, then free again
#pragma unroll
            for (int j = 0; j < 8; ++j)
              slab_put(slabs, lane, j, make_uint4(w(4 * j), w(4 * j + 1), w(4 * j + 2), w(4 * j + 3)));
            __syncwarp();
            lsu_store(slabs, col, row0, ti.g, rows_here);
            __syncwarp();
            return;
          }
          uint8_t* slab = next_slab();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            slab_put(slab, lane, j, make_uint4(w(4 * j), w(4 * j + 1), w(4 * j + 2), w(4 * j + 3)));
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store_f32(slab, col, row0, ti.g);
            ptx::bulk_commit();
          }
        };
        auto has = [&](int c) { return c < c_hi && ti.n0 + c < p.N; };
        uint32_t va[32], vb[32];
        int c = c_lo;
        if (has(c)) {
          ptx::tmem_ld32(t_row + c, va);
          ptx::tmem_ld_wait(va);
        }
#pragma unroll 1
        while (has(c)) {
          const bool nb = has(c + 32);
          if (nb) ptx::tmem_ld32(t_row + c + 32, vb);
          put(va, ti.n0 + c);
          if (!nb) break;
          ptx::tmem_ld_wait(vb);
          c += 32;
          const bool na = has(c + 32);
          if (na) ptx::tmem_ld32(t_row + c + 32, va);
          put(vb, ti.n0 + c);
          if (!na) break;
          ptx::tmem_ld_wait(va);
          c += 32;
        }
      } else if (tma_slab && EPI == EPI_SWIGLU_FWD) {
        // acc columns [0, BN/2) are gate, [BN/2, BN) up, for h columns n0 .. n0+BN/2
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 64) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          uint8_t* slab = next_slab();
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t ga[32], up[32];
            ptx::tmem_ld32(t_row + c + 32 * hf, ga);
            ptx::tmem_ld32(t_row + BN / 2 + c + 32 * hf, up);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float hv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                hv[i] = silu_f(__uint_as_float(ga[8 * j + i]) * sc) * (__uint_as_float(up[8 * j + i]) * sc);
                if (col + 32 * hf + 8 * j + i < p.f) track(hv[i]);
              }
              slab_put(slab, lane, 4 * hf + j, pack16(hv, static_cast<const bf16*>(nullptr)));
            }
          }
          slab_store_2d(&tmO0, slab, lane, col, row0);
          if (p.out2) {
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {   // 0: gate pre-activation a, 1: up u
              uint8_t* s2 = next_slab();
#pragma unroll 1
              for (int hf = 0; hf < 2; ++hf) {
                uint32_t v[32];
                ptx::tmem_ld32(t_row + part * (BN / 2) + c + 32 * hf, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  float fv[8];
#pragma unroll
                  for (int i = 0; i < 8; ++i) fv[i] = __uint_as_float(v[8 * j + i]) * sc;
                  slab_put(s2, lane, 4 * hf + j, pack16(fv, static_cast<const bf16*>(nullptr)));
                }
              }
              slab_store_2d(part == 0 ? &tmO1 : &tmO2, s2, lane, col, row0);
            }
          }
        }
      } else if (MX && EPI == EPI_SWIGLU_BWD && !tma_slab) {
        // [da | du] from dh and the saved [a | u] of the row, written in bf16 (the weight
        // gradients' operand) when out is given and as MXFP8 codes and block scales along 2f
        // (fc1's data-gradient operand): a thread's 32 columns are one block of da and one of du
        const bf16* arow = static_cast<const bf16*>(p.aux) + row * p.ld_aux;
        bf16* drow = p.out ? static_cast<bf16*>(p.out) + row * p.ldo : nullptr;
        uint8_t* qrow = p.q_out + static_cast<int64_t>(row) * 2 * p.f;
        uint8_t* sfrow = p.q_sf + static_cast<int64_t>(ti.mt) * p.kch_out * MX_CHUNK + (r & 31) * 16 +
                         (r >> 5) * 4;
        const int nb2 = 2 * p.f / 32;   // blocks of a [da | du] row
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          uint32_t dh[32];
          ptx::tmem_ld32(t_row + c, dh);
          ptx::tmem_ld_wait();
          if (!valid) continue;
          float da[32], du[32];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float av[8], uv[8];
            unpack16(ld16(arow + col + v * 8), av, static_cast<const bf16*>(nullptr));
            unpack16(ld16(arow + p.f + col + v * 8), uv, static_cast<const bf16*>(nullptr));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float g = __uint_as_float(dh[v * 8 + i]);
              const float s = sigmoid_f<MOE_FAST_SIGMOID_F8 != 0>(av[i]);
              da[v * 8 + i] = __bfloat162float(__float2bfloat16_rn(g * uv[i] * (s + av[i] * s * (1.0f - s))));
              du[v * 8 + i] = __bfloat162float(__float2bfloat16_rn(g * av[i] * s));
            }
            if (drow) {
              st16(drow + col + v * 8, pack16(da + 8 * v, static_cast<const bf16*>(nullptr)));
              st16(drow + p.f + col + v * 8, pack16(du + 8 * v, static_cast<const bf16*>(nullptr)));
            }
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const float* vals = half ? du : da;
            float am = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(vals[i]));
            const int ex = mx_exponent(am);
            const float inv = mx_inv_scale(ex);
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t lo = cvt_e4m3x2(vals[4 * j] * inv, vals[4 * j + 1] * inv);
              const uint32_t hi = cvt_e4m3x2(vals[4 * j + 2] * inv, vals[4 * j + 3] * inv);
              w[j] = lo | (hi << 16);
            }
            const int qc = half * p.f + col;   // column of this block in [da | du]
            *reinterpret_cast<uint4*>(qrow + qc) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(qrow + qc + 16) = make_uint4(w[4], w[5], w[6], w[7]);
            const int blk = qc >> 5;
            uint8_t* sf = sfrow + (blk >> 2) * MX_CHUNK;
            sf[blk & 3] = static_cast<uint8_t>(ex + 127);
            if (blk == nb2 - 1) {
              for (int j = (blk & 3) + 1; j < 4; ++j) sf[j] = 127;   // blocks past 2f: 2^0
            }
          }
        }
      } else if (tma_slab && HALF_SLABS) {
        // acc = dh for f columns n0 .. n0+BN, 32 at a time.  The slab's two halves take the
        // saved a and u of those columns (TMA, map tmO2 over act with 32 x 32 boxes), then the
        // results da and du in their place, stored by TMA (maps tmO0, tmO1).
        uint8_t* ha = slabs;
        uint8_t* hu = slabs + SLAB / 2;
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          if (lane == 0) {
            ptx::bulk_wait_read<0>();   // the slab's previous stores have read it
            ptx::mbar_arrive_expect_tx(my_bar, SLAB);
            ptx::tma_load_2d(ha, &tmO2, my_bar, col, row0);
            ptx::tma_load_2d(hu, &tmO2, my_bar, p.f + col, row0);
          }
          __syncwarp();
          uint32_t dh[32];
          ptx::tmem_ld32(t_row + c, dh);   // in flight while the loads land
          const bool landed = ptx::mbar_wait(my_bar, ld_phase, abort_flag, p.err);
          ptx::tmem_ld_wait(dh);
          if (!landed) { aborted = true; break; }
          ld_phase ^= 1u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float av[8], uv[8], da[8], du[8];
            unpack16(half_get(ha, lane, j), av, static_cast<const bf16*>(nullptr));
            unpack16(half_get(hu, lane, j), uv, static_cast<const bf16*>(nullptr));
            // columns past f (an edge tile) are never stored: keep them out of the amax
            const bool live = col + 8 * j < p.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float g = __uint_as_float(dh[8 * j + i]) * sc;
              const float s = sigmoid_f<F8 && MOE_FAST_SIGMOID_F8>(av[i]);
              da[i] = g * uv[i] * (s + av[i] * s * (1.0f - s));
              du[i] = g * av[i] * s;
              if (live) {
                track(da[i]);
                track(du[i]);
              }
            }
            half_put(ha, lane, j, pack16(da, static_cast<const bf16*>(nullptr)));
            half_put(hu, lane, j, pack16(du, static_cast<const bf16*>(nullptr)));
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmO0, ha, col, row0);
            ptx::tma_store_2d(&tmO1, hu, col, row0);
            ptx::bulk_commit();
          }
        }
      } else if (tma_slab && EPI == EPI_SWIGLU_BWD) {
        // acc = dh for f columns n0 .. n0+BN.  The saved [a | u] of the slab are brought in by
        // TMA (map tmO2 over act), combined with dh, and [da | du] written back by TMA.
        uint8_t* sa = slabs;
        uint8_t* su = slabs + SLAB;
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 64) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          if (lane == 0) {
            ptx::bulk_wait_read<0>();   // both slabs free
            ptx::mbar_arrive_expect_tx(my_bar, 2 * SLAB);
            ptx::tma_load_2d(sa, &tmO2, my_bar, col, row0);
            ptx::tma_load_2d(su, &tmO2, my_bar, p.f + col, row0);
          }
          __syncwarp();
          if (!ptx::mbar_wait(my_bar, ld_phase, abort_flag, p.err)) { aborted = true; break; }
          ld_phase ^= 1u;
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t dh[32];
            ptx::tmem_ld32(t_row + c + 32 * hf, dh);
            ptx::tmem_ld_wait();
            float dav[MX ? 32 : 1], duv[MX ? 32 : 1];   // MXFP8: the block's bf16 values
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float av[8], uv[8], da[8], du[8];
              unpack16(slab_get(sa, lane, 4 * hf + j), av, static_cast<const bf16*>(nullptr));
              unpack16(slab_get(su, lane, 4 * hf + j), uv, static_cast<const bf16*>(nullptr));
              // columns past f (an edge tile) are never stored: keep them out of the amax
              const bool live = col + 32 * hf + 8 * j < p.f;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float g = __uint_as_float(dh[8 * j + i]) * sc;
                const float s = sigmoid_f<F8 && MOE_FAST_SIGMOID_F8>(av[i]);
                da[i] = g * uv[i] * (s + av[i] * s * (1.0f - s));
                du[i] = g * av[i] * s;
                if (live) {
                  track(da[i]);
                  track(du[i]);
                }
                if (MX) {
                  da[i] = __bfloat162float(__float2bfloat16_rn(da[i]));
                  du[i] = __bfloat162float(__float2bfloat16_rn(du[i]));
                  dav[MX ? 8 * j + i : 0] = da[i];
                  duv[MX ? 8 * j + i : 0] = du[i];
                }
              }
              slab_put(sa, lane, 4 * hf + j, pack16(da, static_cast<const bf16*>(nullptr)));
              slab_put(su, lane, 4 * hf + j, pack16(du, static_cast<const bf16*>(nullptr)));
            }
            const int qc0 = col + 32 * hf;   // MXFP8: this block's column in the da half
            if (MX && qc0 < p.f) {
              // the 32 values are one block of da and one of du along [da | du]: codes and scale
              uint8_t* qrow = p.q_out + static_cast<int64_t>(row) * 2 * p.f;
              uint8_t* sfrow = p.q_sf + static_cast<int64_t>(ti.mt) * p.kch_out * MX_CHUNK +
                               (r & 31) * 16 + (r >> 5) * 4;
              const int nb2 = 2 * p.f / 32;
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const float* vals = half ? duv : dav;
                float am = 0.f;
#pragma unroll
                for (int i = 0; i < (MX ? 32 : 1); ++i) am = fmaxf(am, fabsf(vals[i]));
                const int ex = mx_exponent(am);
                const float inv = mx_inv_scale(ex);
                uint32_t w[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                  const int b0 = MX ? 4 * jj : 0;
                  const uint32_t lo = cvt_e4m3x2(vals[b0] * inv, vals[MX ? b0 + 1 : 0] * inv);
                  const uint32_t hi = cvt_e4m3x2(vals[MX ? b0 + 2 : 0] * inv, vals[MX ? b0 + 3 : 0] * inv);
                  w[jj] = lo | (hi << 16);
                }
                const int qc = half * p.f + qc0;
                *reinterpret_cast<uint4*>(qrow + qc) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(qrow + qc + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                const int blk = qc >> 5;
                uint8_t* sfp = sfrow + (blk >> 2) * MX_CHUNK;
                sfp[blk & 3] = static_cast<uint8_t>(ex + 127);
                if (blk == nb2 - 1) {
                  for (int jj = (blk & 3) + 1; jj < 4; ++jj) sfp[jj] = 127;   // blocks past 2f
                }
              }
            }
          }
          slab_store_2d(&tmO0, sa, lane, col, row0);
          slab_store_2d(&tmO1, su, lane, col, row0);
        }
      } else if (EPI == EPI_SWIGLU_FWD) {
        // masked stores (a slab at the end of an expert's rows)
        bf16* hrow = static_cast<bf16*>(p.out) + row * p.ldo;
        bf16* arow = static_cast<bf16*>(p.out2) + row * p.ldo2;
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          uint32_t ga[32], up[32];
          ptx::tmem_ld32(t_row + c, ga);
          ptx::tmem_ld32(t_row + BN / 2 + c, up);
          ptx::tmem_ld_wait();
          if (valid) {
            const int ncol = min(32, p.f - col);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (v * 8 >= ncol) break;
              float hv[8], av[8], uv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                av[i] = __uint_as_float(ga[v * 8 + i]) * sc;
                uv[i] = __uint_as_float(up[v * 8 + i]) * sc;
                hv[i] = silu_f(av[i]) * uv[i];
                track(hv[i]);
              }
              st16(hrow + col + v * 8, pack16(hv, static_cast<const bf16*>(nullptr)));
              if (p.out2) {
                st16(arow + col + v * 8, pack16(av, static_cast<const bf16*>(nullptr)));
                st16(arow + p.f + col + v * 8, pack16(uv, static_cast<const bf16*>(nullptr)));
              }
            }
          }
        }
      } else if (EPI == EPI_SWIGLU_BWD) {
        const bf16* act = static_cast<const bf16*>(p.aux) + row * p.ld_aux;
        bf16* drow = static_cast<bf16*>(p.out) + row * p.ldo;
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.f) break;
          uint32_t dh[32];
          ptx::tmem_ld32(t_row + c, dh);
          ptx::tmem_ld_wait();
          if (valid) {
            const int ncol = min(32, p.f - col);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (v * 8 >= ncol) break;
              float av[8], uv[8], da[8], du[8];
              unpack16(ld16(act + col + v * 8), av, static_cast<const bf16*>(nullptr));
              unpack16(ld16(act + p.f + col + v * 8), uv, static_cast<const bf16*>(nullptr));
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float g = __uint_as_float(dh[v * 8 + i]) * sc;
                const float s = sigmoid_f<F8 && MOE_FAST_SIGMOID_F8>(av[i]);
                da[i] = g * uv[i] * (s + av[i] * s * (1.0f - s));
                du[i] = g * av[i] * s;
                track(da[i]);
                track(du[i]);
              }
              st16(drow + col + v * 8, pack16(da, static_cast<const bf16*>(nullptr)));
              st16(drow + p.f + col + v * 8, pack16(du, static_cast<const bf16*>(nullptr)));
            }
          }
        }
      } else {
        // EPI_STORE (bf16) or EPI_F32 (+bias), masked direct stores
#pragma unroll 1
        for (int c = c_lo; c < c_hi; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.N) break;
          uint32_t v32[32];
          ptx::tmem_ld32(t_row + c, v32);
          ptx::tmem_ld_wait();
          if (valid) {
            const int ncol = min(32, p.N - col);
            if (EPI == EPI_STORE) {
              bf16* o = static_cast<bf16*>(p.out) + row * p.ldo + col;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                if (v * 8 >= ncol) break;
                float fv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) fv[i] = __uint_as_float(v32[v * 8 + i]) * sc;
                st16(o + v * 8, pack16(fv, static_cast<const bf16*>(nullptr)));
              }
            } else {
              float* o = static_cast<float*>(p.out) + ti.g * p.out_group_stride + row * p.ldo + col;
              if ((p.ldo & 3) != 0 || (ncol & 3) != 0) {
                // unaligned rows (e.g. router logits with E % 4 != 0): scalar stores (unrolled,
                // so that v32 stays in registers)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  if (i < ncol) {
                    float fv = __uint_as_float(v32[i]);
                    if (p.bias) fv += p.bias[col + i];
                    o[i] = fv;
                  }
                }
                continue;
              }
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                if (v * 4 >= ncol) break;
                float4 fv = make_float4(__uint_as_float(v32[v * 4]), __uint_as_float(v32[v * 4 + 1]),
                                        __uint_as_float(v32[v * 4 + 2]),
                                        __uint_as_float(v32[v * 4 + 3]));
                if (p.bias) {
                  fv.x += p.bias[col + v * 4];
                  fv.y += p.bias[col + v * 4 + 1];
                  fv.z += p.bias[col + v * 4 + 2];
                  fv.w += p.bias[col + v * 4 + 3];
                }
                *reinterpret_cast<float4*>(o + v * 4) = fv;
              }
            }
          }
        }
      }
      if (AMAX && p.amax_out) {
        const float m = warp_max(hmax);   // non-negative floats order like their bit patterns
        if (lane == 0 && m > 0.f) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(m));
      }
      // Router: this thread's token -- selection, gates and its experts' counts for the tile's
      // histogram row.  The whole warp reads tensor memory (tcgen05.ld is warp-collective); only
      // rows inside the tensor are written.
      int rsel[MOE_MAX_TOPK];
      if (ROUTER && p.rt.idx && rows_here > 0) {
        TmemLogits src;
        src.t_row = t_row;
        src.bias = p.bias ? s_lbias : nullptr;
        src.row = valid ? static_cast<const float*>(p.out) + row * p.ldo : nullptr;
        rrow::Rule rule;
        rule.E = p.N;
        rule.k = p.rt.k;
        rule.score_fn = p.rt.score_fn;
        rule.renorm = p.rt.renorm;
        rule.sel_bias = p.rt.sel_bias ? s_sbias : nullptr;
        float rg[MOE_MAX_TOPK];
        rrow::route_row<MOE_MAX_TOPK>(src, rule, s_stg + r * RouterOf<SCHED, EPI, F8>::STG_LD,
                                      rsel, rg);
        if (valid) {
#pragma unroll
          for (int j = 0; j < MOE_MAX_TOPK; ++j) {
            if (j < p.rt.k) {
              p.rt.idx[static_cast<int64_t>(row) * p.rt.k + j] = rsel[j];
              p.rt.gate[static_cast<int64_t>(row) * p.rt.k + j] = rg[j];
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      if (aborted) break;
      if (ROUTER && p.rt.idx) {
        // the tile's histogram row: every epilogue warp adds its tokens' experts, arrives, and
        // after all four have arrived writes a quarter of the row and clears it for the tile
        // after next (which uses this buffer again only after the next tile's arrivals)
        int* h = s_rhist + (it & 1) * MOE_MAX_EXPERTS;
        if (rows_here > 0 && valid) {
#pragma unroll
          for (int j = 0; j < MOE_MAX_TOPK; ++j)
            if (j < p.rt.k) atomicAdd(&h[rsel[j]], 1);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(hbar);
        if (!ptx::mbar_wait(hbar, hphase, abort_flag, p.err)) break;
        hphase ^= 1u;
        uint8_t* hrow = p.rt.hist + static_cast<int64_t>(ti.mt) * p.rt.ldh;
        for (int x = e * 32 + lane; x < p.rt.ldh; x += EPI_WARPS * 32) {
          hrow[x] = static_cast<uint8_t>(x < p.N ? h[x] : 0);
          if (x < MOE_MAX_EXPERTS) h[x] = 0;
        }
      }
      if (NACC == 2) acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait_all();   // every store of this warp has landed
    __syncwarp();
  }

  wst.flush(WAIT_KIND, warp, lane);
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) wst.flush_cta(WAIT_KIND);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- weight gradients on CTA pairs
// A weight gradient of ONE group (dW = A^T . B over all K rows, fp32 block; the shared expert's)
// on 2-SM tensor-core instructions (tcgen05 cta_group::2).  A cluster of two CTAs owns a
// 256 x 256 output tile: each CTA loads its 128 rows of A and its 128 columns of B per k-block
// (32 KB), and the even CTA issues M = 256, N = 256 MMAs that read both CTAs' shared memory and
// leave output rows 0..127 in its TMEM and rows 128..255 in the other CTA's.  Per FLOP each SM
// takes in a third fewer operand bytes than with one-CTA 128 x 256 tiles (48 KB per k-block).
// The group's rows are all of A's and B's rows, so the last k-block reads zeros past their end
// (TMA fills rows outside the tensor with zeros): nothing to mask.
//
// Protocol (stage s of the operand ring, tile t):
//   * the even CTA's producer claims tiles (heaviest groups first, as the one-CTA kernel) and
//     hands each to both CTAs' consumers through a feed ring written into both CTAs;
//   * both producers wait for their own empty[s] (the even CTA's MMA commit arrives on both),
//     then load; the even one arms full[s] with both CTAs' bytes, the odd one's copies count
//     their bytes on the even CTA's full[s] (cta_group::2 copies), and it does not arrive;
//   * the MMAs' commit arrives on tfull in both CTAs; each CTA's epilogue stores its own 128
//     rows and arrives on the even CTA's tempty, which the MMA warp waits on before reusing an
//     accumulator.
// Every wait is bounded (abort flag and error word as in the one-CTA kernel).
// Build option (on): 0 runs one-group weight gradients on the one-CTA kernel too.  Several
// groups always take the one-CTA kernel: with skewed routing most of their tiles only store,
// and its two accumulators overlap one tile's stores with the next tile's MMAs.
#ifndef MOE_PAIR_WGRAD
#define MOE_PAIR_WGRAD 1
#endif

namespace pairk {
constexpr int BN2 = 256;                       // output columns per pair tile
constexpr int HB = BN2 / 2;                    // B columns per CTA
constexpr int A_ST = BM * BK * 2;              // 16 KB
constexpr int B_ST = HB * BK * 2;              // 16 KB
constexpr int EW = 4;                          // epilogue warps
#ifndef MOE_PAIR_SLABS
#define MOE_PAIR_SLABS 2
#endif
constexpr int SLABS_P = MOE_PAIR_SLABS;        // fp32 stores in flight per epilogue warp
constexpr int STAGING = EW * SLABS_P * SLAB;
constexpr int AUX = 3072;
constexpr int MAX_SMEM = 232448;
constexpr int FIT = (MAX_SMEM - STAGING - AUX) / (A_ST + B_ST);
#ifndef MOE_PAIR_MAX_STAGES
#define MOE_PAIR_MAX_STAGES 8
#endif
constexpr int STAGES = FIT < MOE_PAIR_MAX_STAGES ? FIT : MOE_PAIR_MAX_STAGES;
constexpr int RING = STAGES * (A_ST + B_ST);
constexpr int SMEM = RING + STAGING + AUX;
constexpr int THREADS = 64 + 32 * EW;
constexpr int TMEM_COLS = 512;                 // two accumulators of 256 fp32 columns
}  // namespace pairk

__global__ void __launch_bounds__(pairk::THREADS, 1)
    tc_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmO0, const KArgs p) {
  using namespace pairk;
  using S = Sched<BN2, RAGGED_K, EPI_F32, 2 * BM>;
  constexpr uint32_t IDESC = ptx::idesc_bf16_f32(2 * BM, BN2, true, true);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_ST;
  uint8_t* staging = smem + RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING + STAGING);   // even CTA's are used
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;           // even CTA's are used
  uint64_t* feed_full = tempty + 2;
  uint64_t* feed_empty = feed_full + FEED;   // even CTA's are used
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(feed_empty + FEED);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_bad = reinterpret_cast<int*>(tmem_holder + 2);
  int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
  int* s_ord = s_off + (MAXG + 1);
  volatile int* s_feed = s_ord + (MAXG + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool even = rank == 0;

  if ((ptx::smem_u32(smem) & 1023u) != 0) {   // the same in both CTAs: both return
    if (threadIdx.x == 0) record_error(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);     // the even producer's arrival (with both CTAs' bytes)
      ptx::mbar_init(&empty[i], 1);    // the pair's MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      ptx::mbar_init(&tempty[i], 2 * EW);   // both CTAs' epilogue warps
    }
    for (int i = 0; i < FEED; ++i) {
      ptx::mbar_init(&feed_full[i], 1);
      ptx::mbar_init(&feed_empty[i], 2 + 2 * EW);   // even MMA + odd producer + all epilogues
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
    int v;
    if (p.offsets) v = p.offsets[i];
    else v = static_cast<int>((static_cast<int64_t>(p.K) * i) / p.G);
    s_off[i] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bad = (s_off[0] < 0 || s_off[p.G] > p.K) ? 1 : 0;
    for (int i = 0; i < p.G && !bad; ++i) bad = s_off[i + 1] < s_off[i];
    *s_bad = bad;
    if (bad && even) record_error(p.err, DEVERR_BAD_OFFSETS);
  }
  // groups by row count, most first (ties: lower index first), identical in both CTAs
  for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
    const int n = s_off[g + 1] - s_off[g];
    int r = 0;
    for (int h = 0; h < p.G; ++h) {
      const int m = s_off[h + 1] - s_off[h];
      r += (m > n || (m == n && h < g)) ? 1 : 0;
    }
    s_ord[r] = g;
  }
  __syncthreads();
  if (*s_bad) return;                    // the same decision in both CTAs
  const int total = S::total(p, nullptr);
  if (total == 0) return;
  ptx::cluster_sync();                   // both CTAs' barriers exist before either touches them

  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // the even CTA's barriers as seen from the odd CTA
  auto even_addr = [&](const void* local) { return ptx::mapa(ptx::smem_u32(local), 0); };

  if (warp == 0) {
    // ------------------------------------------------------------ producers (lane 0)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fslot = 0;
      uint32_t fphase = 0;
      bool ok = true;
      int armed[STAGES];
      for (int i = 0; i < STAGES; ++i) armed[i] = -1;
      const int m_off = static_cast<int>(rank) * BM;    // this CTA's rows of the pair tile
      const int n_off = static_cast<int>(rank) * HB;    // this CTA's columns of B
      int next = even ? atomicAdd(p.tile_ctr, 1) : 0;
      for (;;) {
        // -------- the tile: claimed and published by the even CTA, received by the odd one
        int tile;
        if (even) {
          tile = next < total ? next : -1;
          if (!ptx::mbar_wait_cluster(&feed_empty[fslot], fphase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          s_feed[fslot] = tile;
          ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(const_cast<int*>(&s_feed[fslot])), 1),
                              static_cast<uint32_t>(tile));
          ptx::mbar_arrive(&feed_full[fslot]);
          ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_u32(&feed_full[fslot]), 1));
          if (tile >= 0) next = atomicAdd(p.tile_ctr, 1);
        } else {
          if (!ptx::mbar_wait_cluster(&feed_full[fslot], fphase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tile = s_feed[fslot];
          ptx::mbar_arrive_remote(even_addr(&feed_empty[fslot]));
        }
        if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
        if (tile < 0) break;
        const TileInfo ti = S::decode(p, s_off, nullptr, s_ord, tile);
        const CUtensorMap* ma = &tmA;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const int kk = ti.k0 + kb * BK;
          uint8_t* a_dst = sA + stage * A_ST;
          uint8_t* b_dst = sB + stage * B_ST;
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          if (even) {
            ptx::mbar_arrive_expect_tx(&full[stage], 2 * (A_ST + B_ST));
            armed[stage] = static_cast<int>(phase);
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              ptx::tma_load_2d(a_dst + c * (BK * 128), ma, &full[stage], ti.m0 + m_off + 64 * c, kk);
#pragma unroll
            for (int c = 0; c < HB / 64; ++c)
              ptx::tma_load_2d(b_dst + c * (BK * 128), &tmB, &full[stage], ti.n0 + n_off + 64 * c, kk);
          } else {
            const uint32_t fb = even_addr(&full[stage]);
#pragma unroll
            for (int c = 0; c < BM / 64; ++c)
              ptx::tma_load_2d_pair(a_dst + c * (BK * 128), ma, fb, ti.m0 + m_off + 64 * c, kk);
#pragma unroll
            for (int c = 0; c < HB / 64; ++c)
              ptx::tma_load_2d_pair(b_dst + c * (BK * 128), &tmB, fb, ti.n0 + n_off + 64 * c, kk);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if (!ok && even) {
        // Unwinding: let every copy into an armed stage land before the CTA exits (bounded).
        const uint64_t t0 = ptx::globaltimer();
        for (int i = 0; i < STAGES; ++i) {
          if (armed[i] < 0) continue;
          while (!ptx::mbar_try_wait_acq_cluster(&full[i], static_cast<uint32_t>(armed[i])) &&
                 ptx::globaltimer() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (even) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int fslot = 0;
      uint32_t fphase = 0;
      bool ok = true;
      for (;;) {
        if (!ptx::mbar_wait(&feed_full[fslot], fphase, abort_flag, p.err)) break;
        const int tile = s_feed[fslot];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&feed_empty[fslot]);
        if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
        if (tile < 0) break;
        const TileInfo ti = S::decode(p, s_off, nullptr, s_ord, tile);
        if (ti.kblocks == 0) continue;
        if (!ptx::mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN2);
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, abort_flag, p.err)) { ok = false; break; }
          ptx::tc_fence_after();
          if (lane == 0) {
            const uint32_t a_addr = ptx::smem_u32(sA + stage * A_ST);
            const uint32_t b_addr = ptx::smem_u32(sB + stage * B_ST);
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t ad = ptx::smem_desc_sw128(a_addr + k16 * 2048, BK * 128, 1024);
              const uint64_t bd = ptx::smem_desc_sw128(b_addr + k16 * 2048, BK * 128, 1024);
              ptx::umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb | k16) != 0 ? 1u : 0u);
            }
            // frees the stage in both CTAs
            ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&empty[stage]), 0));
            ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&empty[stage]), 1));
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) {   // both CTAs' epilogues
          ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&tfull[acc]), 0));
          ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&tfull[acc]), 1));
        }
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int e = warp - 2;
    const int q = warp & 3;
    uint8_t* slabs = staging + e * (SLABS_P * SLAB);
    int slab_sel = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    int fslot = 0;
    uint32_t fphase = 0;
    auto next_slab = [&]() -> uint8_t* {
      if (lane == 0) ptx::bulk_wait_read<SLABS_P - 1>();
      __syncwarp();
      uint8_t* s = slabs + slab_sel * SLAB;
      if (++slab_sel == SLABS_P) slab_sel = 0;
      return s;
    };
    auto store = [&](const uint8_t* src, int col, int row, int g) {
      if (MOE_WGRAD_STORE_HINT)
        ptx::tma_store_3d_hint(&tmO0, src, col, row, g, ptx::policy_evict_first());
      else
        ptx::tma_store_3d(&tmO0, src, col, row, g);
    };
    for (;;) {
      const bool got = even ? ptx::mbar_wait(&feed_full[fslot], fphase, abort_flag, p.err)
                            : ptx::mbar_wait_cluster(&feed_full[fslot], fphase, abort_flag, p.err);
      if (!got) break;
      const int tile = s_feed[fslot];
      __syncwarp();
      if (lane == 0) {
        if (even) ptx::mbar_arrive(&feed_empty[fslot]);
        else ptx::mbar_arrive_remote(even_addr(&feed_empty[fslot]));
      }
      if (++fslot == FEED) { fslot = 0; fphase ^= 1u; }
      if (tile < 0) break;
      const TileInfo ti = S::decode(p, s_off, nullptr, s_ord, tile);
      const int row0 = ti.m0 + static_cast<int>(rank) * BM + q * 32;
      const int rows_here = min(32, ti.m_end - row0);
      if (ti.kblocks == 0) {
        // a group without rows: its block is zero (one zeroed slab stored everywhere)
        if (rows_here > 0) {
          uint8_t* z = next_slab();
#pragma unroll
          for (int j = 0; j < 8; ++j) slab_put(z, lane, j, make_uint4(0, 0, 0, 0));
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int c = 0; c < BN2; c += 32) {
              if (ti.n0 + c >= p.N) break;
              store(z, ti.n0 + c, row0, ti.g);
              ptx::bulk_commit();
            }
          }
          __syncwarp();
        }
        continue;
      }
      if (!ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err)) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN2);
      if (rows_here > 0) {
        auto put = [&](const uint32_t (&v)[32], int col) {
          uint8_t* slab = next_slab();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            slab_put(slab, lane, j, make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store(slab, col, row0, ti.g);
            ptx::bulk_commit();
          }
        };
        auto has = [&](int c) { return c < BN2 && ti.n0 + c < p.N; };
        uint32_t va[32], vb[32];
        int c = 0;
        if (has(c)) {
          ptx::tmem_ld32(t_row + c, va);
          ptx::tmem_ld_wait(va);
        }
#pragma unroll 1
        while (has(c)) {
          const bool nb = has(c + 32);
          if (nb) ptx::tmem_ld32(t_row + c + 32, vb);
          put(va, ti.n0 + c);
          if (!nb) break;
          ptx::tmem_ld_wait(vb);
          c += 32;
          const bool na = has(c + 32);
          if (na) ptx::tmem_ld32(t_row + c + 32, va);
          put(vb, ti.n0 + c);
          if (!na) break;
          ptx::tmem_ld_wait(va);
          c += 32;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (even) ptx::mbar_arrive(&tempty[acc]);
        else ptx::mbar_arrive_remote(even_addr(&tempty[acc]));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // neither CTA leaves while the other may still use its barriers or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- row-ragged products, tall tiles
// A row-ragged product with bf16 output (fc2; the data gradient with MN-major weights) on tiles
// of 256 rows x 256 columns per CTA: per k-block the CTA loads two 128-row A boxes and one
// 256-row B stage (64 KB) and issues two M = 128, N = 256 MMAs per K step that share the B stage,
// one into each half of TMEM (rows 0..127 in columns 0..255, rows 128..255 in 256..511).  A
// one-CTA 128 x 256 tile takes 48 KB per 128 x 256 x 64 k-block; this takes 32 KB for the same
// work.  A group's rows are cut into 256-row tiles, and a last tile of at most 128 rows issues
// only the first half's MMAs (and loads only that half of A), so groups are padded as with
// 128-row tiles.  One accumulator set fills TMEM: each epilogue warp copies its 32 rows x 256
// columns into registers (bf16) and releases the accumulator before it stores them, so the next
// tile's MMAs wait only for those copies.  Ring: 3 stages of 64 KB; 8 epilogue warps (a TMEM
// lane quadrant and a half each), one staging slab each.
namespace tallk {
constexpr int TM = 2 * BM;                // rows of a tile
constexpr int BN2 = 256;                  // columns of a tile
constexpr int A_ST = TM * BK * 2;         // 32 KB (two 128-row boxes)
constexpr int B_ST = BN2 * BK * 2;        // 32 KB
constexpr int EW = 8;                     // epilogue warps
constexpr int STAGING = EW * SLAB;
constexpr int AUX = 3072;
constexpr int MAX_SMEM = 232448;
constexpr int STAGES = (MAX_SMEM - STAGING - AUX) / (A_ST + B_ST);
constexpr int RING = STAGES * (A_ST + B_ST);
constexpr int SMEM = RING + STAGING + AUX;
constexpr int THREADS = 64 + 32 * EW;
constexpr int TMEM_COLS = 512;
static_assert(STAGES >= 3, "tall tiles need three ring stages");
}  // namespace tallk

template <bool B_MN>
__global__ void __launch_bounds__(tallk::THREADS, 1)
    tc_rows_tall_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO0, const KArgs p) {
  using namespace tallk;
  using S = Sched<BN2, RAGGED_M, EPI_STORE, TM>;
  constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN2, false, B_MN);
  constexpr int MN_CHUNK = BK * 128;      // one 64-column MN-major chunk of a stage

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_ST;
  uint8_t* staging = smem + RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING + STAGING);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_bad = reinterpret_cast<int*>(tmem_holder + 2);
  int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
  int* s_pre = s_off + (MAXG + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WaitStats wst;
  wst.start();
  constexpr int WAIT_KIND = 48 + (B_MN ? 1 : 0);
  const int unit = static_cast<int>(blockIdx.x), units = static_cast<int>(gridDim.x);

  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(tempty, EW);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x)
    s_off[i] = p.offsets ? p.offsets[i] : static_cast<int>((static_cast<int64_t>(p.M) * i) / p.G);
  __syncthreads();
  if (threadIdx.x == 0) {
    int bad = (s_off[0] < 0 || s_off[p.G] > p.M) ? 1 : 0;
    for (int i = 0; i < p.G && !bad; ++i) bad = s_off[i + 1] < s_off[i];
    *s_bad = bad;
    if (bad) record_error(p.err, DEVERR_BAD_OFFSETS);
  }
  __syncthreads();
  if (*s_bad) return;
  if (warp == 0) {
    // s_pre[g] = sum_{g' < g} ceil(rows_g' / 256): lane L scans groups [L*per, (L+1)*per)
    const int per = (p.G + 31) / 32;
    const int lo = min(p.G, lane * per), hi = min(p.G, lo + per);
    int local = 0;
    for (int g = lo; g < hi; ++g) local += (s_off[g + 1] - s_off[g] + TM - 1) / TM;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int g = lo; g < hi; ++g) {
      s_pre[g] = run;
      run += (s_off[g + 1] - s_off[g] + TM - 1) / TM;
    }
    if (lane == 31) s_pre[p.G] = incl;
  }
  __syncthreads();
  const int total = S::total(p, s_pre);
  if (unit >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (lane 0)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
      for (int i = 0; i < STAGES; ++i) armed[i] = -1;
      bool ok = true;
      for (int tile = unit; tile < total && ok; tile += units) {
        const TileInfo ti = S::decode(p, s_off, s_pre, nullptr, tile);
        const bool tall = ti.m_end - ti.m0 > BM;
        const uint32_t tx = static_cast<uint32_t>((tall ? 2 : 1) * BM * BK * 2 + B_ST);
        const int brow = static_cast<int>(ti.g * p.b_group_rows);
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const int kk = kb * BK;
          const unsigned long long w0 = wst.now();
          const bool freed = ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err);
          wst.since(wst.prod, w0);
          if (!freed) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&full[stage], tx);
          armed[stage] = static_cast<int>(phase);
          uint8_t* a_dst = sA + stage * A_ST;
          uint8_t* b_dst = sB + stage * B_ST;
          ptx::tma_load_2d(a_dst, &tmA, &full[stage], kk, ti.m0);
          if (tall) ptx::tma_load_2d(a_dst + BM * BK * 2, &tmA, &full[stage], kk, ti.m0 + BM);
          if (!B_MN) {
            ptx::tma_load_2d(b_dst, &tmB, &full[stage], kk, brow + ti.n0);
          } else {
#pragma unroll
            for (int c = 0; c < BN2 / 64; ++c)
              ptx::tma_load_2d(b_dst + c * MN_CHUNK, &tmB, &full[stage], ti.n0 + 64 * c, brow + kk);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // Unwinding: let every copy this thread issued land before the CTA exits (bounded).
        for (int i = 0; i < STAGES; ++i) {
          if (armed[i] < 0) continue;
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(&full[i], static_cast<uint32_t>(armed[i])) &&
                 ptx::globaltimer() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += units) {
      const TileInfo ti = S::decode(p, s_off, s_pre, nullptr, tile);
      const bool tall = ti.m_end - ti.m0 > BM;
      const unsigned long long wa = wst.now();
      const bool drained = ptx::mbar_wait(tempty, acc_phase ^ 1u, abort_flag, p.err);
      wst.since(wst.acc, wa);
      if (!drained) break;
      ptx::tc_fence_after();
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        const unsigned long long wf = wst.now();
        const bool landed = ptx::mbar_wait(&full[stage], phase, abort_flag, p.err);
        wst.since(wst.full, wf);
        ++wst.kblocks;
        if (!landed) { ok = false; break; }
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(sA + stage * A_ST);
          const uint32_t b_addr = ptx::smem_u32(sB + stage * B_ST);
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16) {
            const uint64_t bd = B_MN ? ptx::smem_desc_sw128(b_addr + k16 * 2048, MN_CHUNK, 1024)
                                     : ptx::smem_desc_sw128(b_addr + k16 * 32, 16, 1024);
            const uint32_t accumulate = (kb | k16) != 0 ? 1u : 0u;
            ptx::umma_bf16(tmem_base, ptx::smem_desc_sw128(a_addr + k16 * 32, 16, 1024), bd, IDESC,
                           accumulate);
            if (tall)
              ptx::umma_bf16(tmem_base + BN2,
                             ptx::smem_desc_sw128(a_addr + BM * BK * 2 + k16 * 32, 16, 1024), bd,
                             IDESC, accumulate);
          }
          ptx::umma_commit(&empty[stage]);   // frees the stage when these MMAs finish
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) ptx::umma_commit(tfull);   // accumulator ready for the epilogue
      __syncwarp();
      acc_phase ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    const int e = warp - 2;
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int h = e >> 2;                 // accumulator half: rows 128*h .. 128*h + 127
    uint8_t* slab = staging + e * SLAB;
    uint32_t acc_phase = 0;
    for (int tile = unit; tile < total; tile += units) {
      const TileInfo ti = S::decode(p, s_off, s_pre, nullptr, tile);
      const int row0 = ti.m0 + h * BM + q * 32;   // this warp's first row
      const int rows_here = min(32, ti.m_end - row0);
      const unsigned long long we = wst.now();
      const bool ready = ptx::mbar_wait(tfull, acc_phase, abort_flag, p.err);
      wst.since(wst.epi, we);
      if (!ready) break;
      acc_phase ^= 1u;
      ptx::tc_fence_after();
      // the warp's 32 rows x 256 columns as bf16 pairs: pk[16 c + i] holds columns 32 c + 2 i, +1
      uint32_t pk[BN2 / 2];
      if (rows_here > 0) {
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(h * BN2);
#pragma unroll
        for (int c = 0; c < BN2 / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld32(t_row + 32 * c, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v[8 * j + i]);
            const uint4 u = pack16(f, static_cast<const bf16*>(nullptr));
            pk[16 * c + 4 * j + 0] = u.x;
            pk[16 * c + 4 * j + 1] = u.y;
            pk[16 * c + 4 * j + 2] = u.z;
            pk[16 * c + 4 * j + 3] = u.w;
          }
        }
      }
      // the accumulator may be overwritten once every warp holds its rows
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty);
      if (rows_here == 32) {
        // 64 columns per slab, out through TMA (the map clips at the tensor's columns)
#pragma unroll
        for (int s = 0; s < BN2 / 64; ++s) {
          const int col = ti.n0 + 64 * s;
          if (col >= p.N) break;
          if (lane == 0) ptx::bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            slab_put(slab, lane, j,
                     make_uint4(pk[32 * s + 4 * j], pk[32 * s + 4 * j + 1], pk[32 * s + 4 * j + 2],
                                pk[32 * s + 4 * j + 3]));
          slab_store_2d(&tmO0, slab, lane, col, row0);
        }
      } else if (rows_here > 0 && lane < rows_here) {
        // the group's last rows: masked stores (a whole slab would overwrite the next group's)
        bf16* o = static_cast<bf16*>(p.out) + static_cast<int64_t>(row0 + lane) * p.ldo + ti.n0;
#pragma unroll
        for (int v = 0; v < BN2 / 8; ++v) {
          if (ti.n0 + 8 * v < p.N)
            st16(o + 8 * v, make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]));
        }
      }
    }
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }

  wst.flush(WAIT_KIND, warp, lane);
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) wst.flush_cta(WAIT_KIND);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- row-ragged products on CTA pairs
// A row-ragged product with bf16 output (fc2; the data gradient with MN-major weights) on CTA
// pairs (tcgen05 cta_group::2): tiles of 256 rows (each CTA's 128, counted per group as in the
// one-CTA kernel, so a group's last tile may run past its rows) by 256 columns.  Per k-block each
// CTA loads its 128 A rows and 128 of the 256 B rows (K-major) or columns (MN-major): 32 KB per
// SM instead of 48 for the same outputs, a third fewer operand bytes per FLOP.  Both CTAs walk
// the same static tile sequence; the odd CTA's copies complete on the even CTA's barrier, the
// even CTA's MMA warp issues the pair's MMAs and commits each stage and accumulator to both CTAs;
// each CTA's epilogue stores its own 128 rows and releases the accumulator on the even CTA.
namespace rpairk {
constexpr int BN2 = 256;                  // output columns per pair tile
constexpr int HB = BN2 / 2;               // B rows (K-major) or columns (MN-major) per CTA
constexpr int A_ST = BM * BK * 2;         // 16 KB
constexpr int B_ST = HB * BK * 2;         // 16 KB
constexpr int EW = 4;                     // epilogue warps
constexpr int SLABS_R = 2;
constexpr int STAGING = EW * SLABS_R * SLAB;
constexpr int AUX = 3072;
constexpr int MAX_SMEM = 232448;
constexpr int FIT = (MAX_SMEM - STAGING - AUX) / (A_ST + B_ST);
constexpr int STAGES = FIT < 8 ? FIT : 8;
constexpr int RING = STAGES * (A_ST + B_ST);
constexpr int SMEM = RING + STAGING + AUX;
constexpr int THREADS = 64 + 32 * EW;
constexpr int TMEM_COLS = 512;            // two accumulators of 256 fp32 columns
}  // namespace rpairk

template <bool B_MN>
__global__ void __launch_bounds__(rpairk::THREADS, 1)
    tc_rows_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO0, const KArgs p) {
  using namespace rpairk;
  using S = Sched<BN2, RAGGED_M, EPI_STORE, 2 * BM>;
  constexpr int TM = 2 * BM;   // rows of a pair tile
  constexpr uint32_t IDESC = ptx::idesc_bf16_f32(2 * BM, BN2, false, B_MN);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_ST;
  uint8_t* staging = smem + RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING + STAGING);   // even CTA's are used
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;           // even CTA's are used
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_bad = reinterpret_cast<int*>(tmem_holder + 2);
  int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
  int* s_pre = s_off + (MAXG + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool even = rank == 0;
  const int cid = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);

  if ((ptx::smem_u32(smem) & 1023u) != 0) {   // the same in both CTAs: both return
    if (threadIdx.x == 0) record_error(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);     // the even producer's arrival (with both CTAs' bytes)
      ptx::mbar_init(&empty[i], 1);    // the pair's MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      ptx::mbar_init(&tempty[i], 2 * EW);   // both CTAs' epilogue warps
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  for (int i = threadIdx.x; i <= p.G; i += blockDim.x)
    s_off[i] = p.offsets ? p.offsets[i] : static_cast<int>((static_cast<int64_t>(p.M) * i) / p.G);
  __syncthreads();
  if (threadIdx.x == 0) {
    int bad = (s_off[0] < 0 || s_off[p.G] > p.M) ? 1 : 0;
    for (int i = 0; i < p.G && !bad; ++i) bad = s_off[i + 1] < s_off[i];
    *s_bad = bad;
    if (bad && even) record_error(p.err, DEVERR_BAD_OFFSETS);
  }
  __syncthreads();
  if (*s_bad) return;                    // the same decision in both CTAs
  if (warp == 0) {
    // s_pre[g] = sum_{g' < g} ceil(rows_g' / 256): lane L scans groups [L*per, (L+1)*per)
    const int per = (p.G + 31) / 32;
    const int lo = min(p.G, lane * per), hi = min(p.G, lo + per);
    int local = 0;
    for (int g = lo; g < hi; ++g) local += (s_off[g + 1] - s_off[g] + TM - 1) / TM;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int g = lo; g < hi; ++g) {
      s_pre[g] = run;
      run += (s_off[g + 1] - s_off[g] + TM - 1) / TM;
    }
    if (lane == 31) s_pre[p.G] = incl;
  }
  __syncthreads();
  const int total = S::total(p, s_pre);
  if (cid >= total) return;              // the same decision in both CTAs of the cluster
  ptx::cluster_sync();                   // both CTAs' barriers exist before either touches them

  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  auto even_addr = [&](const void* local) { return ptx::mapa(ptx::smem_u32(local), 0); };

  if (warp == 0) {
    // ------------------------------------------------------------ producers (lane 0)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int armed[STAGES];
      for (int i = 0; i < STAGES; ++i) armed[i] = -1;
      const int m_off = static_cast<int>(rank) * BM;    // this CTA's rows of the pair tile
      const int n_off = static_cast<int>(rank) * HB;    // this CTA's half of B
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileInfo ti = S::decode(p, s_off, s_pre, nullptr, tile);
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const int kk = kb * BK;
          uint8_t* a_dst = sA + stage * A_ST;
          uint8_t* b_dst = sB + stage * B_ST;
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          const uint32_t fb = even_addr(&full[stage]);
          if (even) {
            ptx::mbar_arrive_expect_tx(&full[stage], 2 * (A_ST + B_ST));
            armed[stage] = static_cast<int>(phase);
          }
          auto load = [&](void* dst, const CUtensorMap* m, int c0, int c1) {
            if (even) ptx::tma_load_2d(dst, m, &full[stage], c0, c1);
            else ptx::tma_load_2d_pair(dst, m, fb, c0, c1);
          };
          load(a_dst, &tmA, kk, ti.m0 + m_off);
          if (!B_MN) {
            load(b_dst, &tmB, kk, static_cast<int>(ti.g * p.b_group_rows) + ti.n0 + n_off);
          } else {
            const int krow = static_cast<int>(ti.g * p.b_group_rows) + kk;
#pragma unroll
            for (int c = 0; c < HB / 64; ++c) load(b_dst + c * (BK * 128), &tmB, ti.n0 + n_off + 64 * c, krow);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && even) {
        // Unwinding: let every copy into an armed stage land before the CTA exits (bounded).
        const uint64_t t0 = ptx::globaltimer();
        for (int i = 0; i < STAGES; ++i) {
          if (armed[i] < 0) continue;
          while (!ptx::mbar_try_wait_acq_cluster(&full[i], static_cast<uint32_t>(armed[i])) &&
                 ptx::globaltimer() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (even) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cid; tile < total && ok; tile += ncl) {
        const TileInfo ti = S::decode(p, s_off, s_pre, nullptr, tile);
        if (!ptx::mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN2);
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, abort_flag, p.err)) { ok = false; break; }
          ptx::tc_fence_after();
          if (lane == 0) {
            const uint32_t a_addr = ptx::smem_u32(sA + stage * A_ST);
            const uint32_t b_addr = ptx::smem_u32(sB + stage * B_ST);
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t ad = ptx::smem_desc_sw128(a_addr + k16 * 32, 16, 1024);
              const uint64_t bd = B_MN ? ptx::smem_desc_sw128(b_addr + k16 * 2048, BK * 128, 1024)
                                       : ptx::smem_desc_sw128(b_addr + k16 * 32, 16, 1024);
              ptx::umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb | k16) != 0 ? 1u : 0u);
            }
            // frees the stage in both CTAs
            ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&empty[stage]), 0));
            ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&empty[stage]), 1));
          }
          __syncwarp();
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) {   // both CTAs' epilogues
          ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&tfull[acc]), 0));
          ptx::umma_commit_pair(ptx::mapa(ptx::smem_u32(&tfull[acc]), 1));
        }
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int e = warp - 2;
    const int q = warp & 3;
    uint8_t* slabs = staging + e * (SLABS_R * SLAB);
    int slab_sel = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    auto next_slab = [&]() -> uint8_t* {
      if (lane == 0) ptx::bulk_wait_read<SLABS_R - 1>();
      __syncwarp();
      uint8_t* sl = slabs + slab_sel * SLAB;
      if (++slab_sel == SLABS_R) slab_sel = 0;
      return sl;
    };
    for (int tile = cid; tile < total; tile += ncl) {
      const TileInfo ti = S::decode(p, s_off, s_pre, nullptr, tile);
      const int row0 = ti.m0 + static_cast<int>(rank) * BM + q * 32;   // this warp's first row
      const int rows_here = min(32, ti.m_end - row0);
      const int row = row0 + lane;
      if (!ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err)) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN2);
      if (rows_here == 32) {
        // whole slabs out through TMA (the map clips at the tensor's columns)
#pragma unroll 1
        for (int c = 0; c < BN2; c += 64) {
          const int col = ti.n0 + c;
          if (col >= p.N) break;
          uint32_t v0[32], v1[32];
          ptx::tmem_ld32(t_row + c, v0);
          ptx::tmem_ld32(t_row + c + 32, v1);
          ptx::tmem_ld_wait();
          uint8_t* slab = next_slab();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              a[i] = __uint_as_float(v0[8 * j + i]);
              b[i] = __uint_as_float(v1[8 * j + i]);
            }
            slab_put(slab, lane, j, pack16(a, static_cast<const bf16*>(nullptr)));
            slab_put(slab, lane, 4 + j, pack16(b, static_cast<const bf16*>(nullptr)));
          }
          slab_store_2d(&tmO0, slab, lane, col, row0);
        }
      } else if (rows_here > 0) {
        // the group's last rows: masked stores (a whole slab would overwrite the next group's)
#pragma unroll 1
        for (int c = 0; c < BN2; c += 32) {
          const int col = ti.n0 + c;
          if (col >= p.N) break;
          uint32_t v32[32];
          ptx::tmem_ld32(t_row + c, v32);
          ptx::tmem_ld_wait();
          if (lane < rows_here) {
            const int ncol = min(32, p.N - col);
            bf16* o = static_cast<bf16*>(p.out) + row * p.ldo + col;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (v * 8 >= ncol) break;
              float fv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) fv[i] = __uint_as_float(v32[v * 8 + i]);
              st16(o + v * 8, pack16(fv, static_cast<const bf16*>(nullptr)));
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (even) ptx::mbar_arrive(&tempty[acc]);
        else ptx::mbar_arrive_remote(even_addr(&tempty[acc]));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // neither CTA leaves while the other may still use its barriers or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A tensor map with 128-byte (or the given) swizzle; out-of-bounds elements read as zero and are
// not written.
int encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
           const cuuint64_t* strides_bytes, const cuuint32_t* box,
           CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return MOE_ERR_CUDA;
  }
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides_bytes,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d): rank=%d dims=%llu,%llu box=%u,%u", (int)r, rank,
              (unsigned long long)dims[0], (unsigned long long)dims[1], box[0], box[1]);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// bf16 rows x cols with row pitch ld (elements); box = 64 columns x box_rows.
int map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box);
}

// bf16 rows x cols with row pitch ld (elements); box = 32 columns x 32 rows, 64-byte swizzle (a
// half slab).
int map_bf16_half(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {32u, 32u};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_64B);
}

// fp32 [G][rows][cols] (group stride gs, row pitch ld, elements); box = 32 x 32 x 1.
int map_f32_3d(CUtensorMap* m, const void* base, int64_t G, int64_t rows, int64_t cols, int64_t ld,
               int64_t gs) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(G)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4, static_cast<cuuint64_t>(gs) * 4};
  cuuint32_t box[3] = {32u, 32u, 1u};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box);
}

// 8-bit (E4M3) rows x cols with row pitch ld (elements = bytes); box = 128 columns x box_rows.
int map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box);
}

int map_operand(CUtensorMap* m, const Operand& op, int box_rows, bool f8 = false) {
  return f8 ? map_u8(m, op.base, op.rows, op.cols, op.ld, box_rows)
            : map_bf16(m, op.base, op.rows, op.cols, op.ld, box_rows);
}

template <int BN, bool A_MN, bool B_MN, int SCHED, int EPI, bool GATHER = false, bool F8 = false,
          bool MX = false>
int run(const GemmDesc& g, const char* kind, cudaStream_t st) {
  const char* name = g.name ? g.name : kind;
  using C = typename CfgOf<BN, SCHED, EPI, F8, MX>::type;
  auto kern = tc_gemm_kernel<BN, A_MN, B_MN, SCHED, EPI, GATHER, F8, MX>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr_err != cudaSuccess) {
    set_error("cudaFuncSetAttribute(%s, %d bytes): %s", name, C::SMEM, cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  CUtensorMap ma, mb, mo[3];
  memset(mo, 0, sizeof(mo));
  // gathered operands are read one row per box (four rows per tile::gather4 copy)
  // an MN-major box is one stage's K rows: 64 (bf16) or 128 (E4M3) of them
  constexpr int KROWS = F8 ? 2 * BK : BK;
  MOE_TRY(map_operand(&ma, g.A, (GATHER && SCHED == RAGGED_M) ? 1 : (A_MN ? KROWS : BM), F8));
  MOE_TRY(map_operand(&mb, g.B,
                      (GATHER && SCHED == RAGGED_K) ? 1
                      : B_MN ? KROWS
                             : (EPI == EPI_SWIGLU_FWD ? BN / 2 : BN),
                      F8));
  const int64_t rows = g.M;   // RAGGED_M: rows of the output (capacity)
  if (EPI == EPI_STORE) {
    MOE_TRY(map_bf16(&mo[0], g.out, rows, g.N, g.ldo, 32));
  } else if (EPI == EPI_F32 && SCHED == RAGGED_K) {
    MOE_TRY(map_f32_3d(&mo[0], g.out, g.G, g.M, g.N, g.ldo, g.out_group_stride));
  } else if (EPI == EPI_SWIGLU_FWD && !MX) {   // (MXFP8: direct stores, no maps)
    MOE_TRY(map_bf16(&mo[0], g.out, rows, g.f, g.ldo, 32));
    if (g.out2) {
      MOE_TRY(map_bf16(&mo[1], g.out2, rows, g.f, g.ldo2, 32));
      MOE_TRY(map_bf16(&mo[2], static_cast<const bf16*>(g.out2) + g.f, rows, g.f, g.ldo2, 32));
    }
  } else if (EpiOf<BN, SCHED, EPI, F8, MX>::half_slabs) {   // the SwiGLU backward, one slab
    MOE_TRY(map_bf16_half(&mo[0], g.out, rows, g.f, g.ldo));
    MOE_TRY(map_bf16_half(&mo[1], static_cast<const bf16*>(g.out) + g.f, rows, g.f, g.ldo));
    MOE_TRY(map_bf16_half(&mo[2], g.aux, rows, 2 * static_cast<int64_t>(g.f), g.ld_aux));
  } else if (EPI == EPI_SWIGLU_BWD && (!MX || g.out)) {   // (MXFP8 without bf16 out: direct stores)
    MOE_TRY(map_bf16(&mo[0], g.out, rows, g.f, g.ldo, 32));
    MOE_TRY(map_bf16(&mo[1], static_cast<const bf16*>(g.out) + g.f, rows, g.f, g.ldo, 32));
    MOE_TRY(map_bf16(&mo[2], g.aux, rows, 2 * static_cast<int64_t>(g.f), g.ld_aux, 32));
  }
  KArgs a;
  a.G = g.G;
  a.offsets = g.offsets;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.b_group_rows = g.b_group_rows;
  a.b_up_rows = g.b_up_rows;
  a.f = g.f;
  a.out = g.out;
  a.ldo = g.ldo;
  a.out_group_stride = g.out_group_stride;
  a.out2 = g.out2;
  a.ldo2 = g.ldo2;
  a.aux = g.aux;
  a.ld_aux = g.ld_aux;
  a.bias = g.bias;
  a.tile_ctr = g.tile_ctr;
  a.gather = g.gather;
  a.gather_rows = static_cast<int>(SCHED == RAGGED_M ? g.A.rows : g.B.rows);
  a.a_scale = g.a_scale;
  a.b_scale = g.b_scale;
  a.b_scale_per_group = g.b_scale_scalar ? 0 : 1;
  a.amax_out = g.amax_out;
  a.sfa = g.sfa;
  a.sfb = g.sfb;
  a.q_out = g.q_out;
  a.q_sf = g.q_sf;
  a.kch = static_cast<int>(SCHED == RAGGED_K ? mx_tok_chunks(g.K, g.G) : mx_kch(g.K));
  a.cbase = g.mx_cbase;
  a.kch_out = static_cast<int>(mx_kch(EPI == EPI_SWIGLU_BWD ? 2 * static_cast<int64_t>(g.f) : g.f));
  a.rt = g.rt;
  if (g.rt.idx) {
    const bool ok = RouterOf<SCHED, EPI, F8>::on && !MX && g.G == 1 && !g.offsets && g.N <= BN &&
                    g.N <= MOE_MAX_EXPERTS && g.rt.gate && g.rt.hist && g.rt.k >= 1 &&
                    g.rt.k <= MOE_MAX_TOPK && g.rt.k <= g.N && g.rt.ldh >= g.N &&
                    g.ldo == g.N;
    if (!ok) {
      set_error("%s: the router epilogue needs one group of fp32 logits whose E columns fit one "
                "tile, k in [1, min(E, %d)] and its idx, gate and histogram buffers", name,
                MOE_MAX_TOPK);
      return MOE_ERR_INVALID_ARG;
    }
  }
  if (F8 && !MX && (!g.a_scale || !g.b_scale)) {
    set_error("%s: FP8 operands need their scales", name);
    return MOE_ERR_INVALID_ARG;
  }
  if (MX) {
    const bool aligned = (reinterpret_cast<uintptr_t>(g.sfa) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(g.sfb) & 15u) == 0;
    const bool swiglu = EPI == EPI_SWIGLU_FWD || EPI == EPI_SWIGLU_BWD;
    if (!g.sfa || !g.sfb || !aligned || (SCHED == RAGGED_M && g.K % 32 != 0) ||
        (SCHED == RAGGED_K && (!g.mx_cbase || !g.offsets)) ||
        (swiglu && (!g.q_out || !g.q_sf || g.f % 32 != 0 ||
                    (reinterpret_cast<uintptr_t>(g.q_out) & 15u) != 0)) ||
        (EPI == EPI_SWIGLU_BWD && !g.aux)) {
      set_error("%s: MXFP8 operands need 16-byte aligned block scales, K (and f) multiples of 32 "
                "(weight gradients: the groups' offsets and token-chunk bases) and, for SwiGLU, "
                "h's code and scale buffers", name);
      return MOE_ERR_INVALID_ARG;
    }
  }
  a.err = device_error_word();
  if (GATHER != (g.gather != nullptr)) {
    set_error("%s: gathered-operand instantiation does not match the descriptor", name);
    return MOE_ERR_INVALID_ARG;
  }
  if (DynMode<SCHED, EPI>::on) {
    if (!g.tile_ctr) {
      set_error("%s: run-time tile scheduling needs its counter (GemmDesc.tile_ctr)", name);
      return MOE_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(g.tile_ctr) & 7u) != 0) {
      set_error("%s: the tile counter must be 8-byte aligned", name);
      return MOE_ERR_ALIGNMENT;
    }
    if (cudaMemsetAsync(g.tile_ctr, 0, 2 * sizeof(int), st) != cudaSuccess) {   // both ends
      set_error("%s: clearing the tile counter failed", name);
      return MOE_ERR_CUDA;
    }
  }
  return launch(name, kern, dim3(num_sms()), dim3(C::THREADS), C::SMEM, st, ma, mb, mo[0], mo[1],
                mo[2], a);
}

// CTA pairs of tc_wgrad_pair_kernel that can be resident at once on the current device (one per
// two SMs at most: a pair must sit in one GPC), so that the persistent grid is a single wave.
int pair_clusters() {
  static int cached[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev]) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms() & ~1);
    cfg.blockDim = dim3(pairk::THREADS);
    cfg.dynamicSmemBytes = pairk::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, tc_wgrad_pair_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();   // clear it: the launch reports any real problem
      n = num_sms() / 2;
    }
    cached[dev] = n < num_sms() / 2 ? n : num_sms() / 2;
  }
  return cached[dev];
}

// A one-group weight gradient on CTA pairs (tc_wgrad_pair_kernel).
int run_wgrad_pair(const GemmDesc& g, cudaStream_t st) {
  using namespace pairk;
  const char* name = g.name ? g.name : "gemm_wgrad";
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(tc_wgrad_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM);
  });
  if (attr_err != cudaSuccess) {
    set_error("cudaFuncSetAttribute(%s, %d bytes): %s", name, SMEM, cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  if (!g.tile_ctr) {
    set_error("%s: run-time tile scheduling needs its counter (GemmDesc.tile_ctr)", name);
    return MOE_ERR_INVALID_ARG;
  }
  CUtensorMap ma, mb, mo;
  MOE_TRY(map_operand(&ma, g.A, BK));
  MOE_TRY(map_operand(&mb, g.B, BK));
  MOE_TRY(map_f32_3d(&mo, g.out, g.G, g.M, g.N, g.ldo, g.out_group_stride));
  KArgs a;
  memset(&a, 0, sizeof(a));
  a.G = g.G;
  a.offsets = g.offsets;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.out = g.out;
  a.ldo = g.ldo;
  a.out_group_stride = g.out_group_stride;
  a.tile_ctr = g.tile_ctr;
  a.err = device_error_word();
  if (cudaMemsetAsync(g.tile_ctr, 0, sizeof(int), st) != cudaSuccess) {
    set_error("%s: clearing the tile counter failed", name);
    return MOE_ERR_CUDA;
  }
  return launch_clusters(name, tc_wgrad_pair_kernel, dim3(2 * pair_clusters()), dim3(THREADS),
                         SMEM, 2, st, ma, mb, mo, a);
}

// Row-ragged bf16 products (fc2, the data gradients) on tall tiles (tc_rows_tall_kernel), on by
// default: interleaved on the 128-expert layer fc2 0.762-0.766 -> 0.735-0.740 ms, fc1 dgrad
// 1.432-1.446 -> 1.371-1.385 ms, shared fc1 dgrad 0.218-0.219 -> 0.205-0.208 ms.  0: the one-CTA
// 128 x 256 kernel.
#ifndef MOE_TALL_ROWS
#define MOE_TALL_ROWS 1
#endif
// Whole waves of tiles each form takes over the output's rows (the capacity, for grouped calls:
// their per-group tails add tiles to both forms), a tall tile costing 1.92 one-CTA tiles (the
// measured 4% gain per tile).  A one-group product of 4096 rows x 2688 columns is 176 tall tiles,
// two waves on 152 SMs, against three waves of 352 one-CTA tiles: the one-CTA form is faster there
// (shared fc2 on the 32-expert layer 35 us against 43 us tall).
bool tall_pays(const GemmDesc& g) {
  const int64_t sms = num_sms();
  const int64_t nt = (g.N + 255) / 256;
  const int64_t waves_tall = ((g.M + 255) / 256 * nt + sms - 1) / sms;
  const int64_t waves_one = ((g.M + 127) / 128 * nt + sms - 1) / sms;
  return waves_tall * 192 <= waves_one * 100;
}

template <bool B_MN>
int run_rows_tall(const GemmDesc& g, cudaStream_t st) {
  using namespace tallk;
  const char* name = g.name ? g.name : (B_MN ? "gemm_dgrad" : "gemm_fc2");
  auto kern = tc_rows_tall_kernel<B_MN>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (attr_err != cudaSuccess) {
    set_error("cudaFuncSetAttribute(%s, %d bytes): %s", name, SMEM, cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  CUtensorMap ma, mb, mo;
  MOE_TRY(map_operand(&ma, g.A, BM));
  MOE_TRY(map_operand(&mb, g.B, B_MN ? BK : BN2));
  MOE_TRY(map_bf16(&mo, g.out, g.M, g.N, g.ldo, 32));
  KArgs a;
  memset(&a, 0, sizeof(a));
  a.G = g.G;
  a.offsets = g.offsets;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.b_group_rows = g.b_group_rows;
  a.out = g.out;
  a.ldo = g.ldo;
  a.err = device_error_word();
  return launch(name, kern, dim3(num_sms()), dim3(THREADS), SMEM, st, ma, mb, mo, a);
}

// Row-ragged bf16 products (fc2, the data gradients) on CTA pairs (tc_rows_pair_kernel).
#ifndef MOE_PAIR_ROWS
#define MOE_PAIR_ROWS 0
#endif
template <bool B_MN>
int run_rows_pair(const GemmDesc& g, cudaStream_t st) {
  using namespace rpairk;
  const char* name = g.name ? g.name : (B_MN ? "gemm_dgrad" : "gemm_fc2");
  auto kern = tc_rows_pair_kernel<B_MN>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  static int clusters[64];
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (attr_err != cudaSuccess) {
    set_error("cudaFuncSetAttribute(%s, %d bytes): %s", name, SMEM, cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!clusters[dev]) {   // pairs resident at once: one persistent wave
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms() & ~1);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    clusters[dev] = n < num_sms() / 2 ? n : num_sms() / 2;
  }
  CUtensorMap ma, mb, mo;
  MOE_TRY(map_operand(&ma, g.A, BM));
  MOE_TRY(map_operand(&mb, g.B, B_MN ? BK : HB));
  MOE_TRY(map_bf16(&mo, g.out, g.M, g.N, g.ldo, 32));
  KArgs a;
  memset(&a, 0, sizeof(a));
  a.G = g.G;
  a.offsets = g.offsets;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.b_group_rows = g.b_group_rows;
  a.out = g.out;
  a.ldo = g.ldo;
  a.err = device_error_word();
  return launch_clusters(name, kern, dim3(2 * clusters[dev]), dim3(THREADS), SMEM, 2, st, ma, mb,
                         mo, a);
}

}  // namespace

int gemm_tc(const GemmDesc& g, cudaStream_t st) {
  if (g.G < 1 || g.G > MAXG) {
    set_error("gemm_tc: group count %d outside [1, %d]", g.G, MAXG);
    return MOE_ERR_UNSUPPORTED;
  }
  if (g.fp8 && g.mx) {
    // MXFP8 operands: the expert products of the forward
    if (!g.gather && g.sched == RAGGED_M && !g.A.mn_major && !g.B.mn_major) {
      if (g.epi == EPI_SWIGLU_FWD)
        return run<MX_BN, false, false, RAGGED_M, EPI_SWIGLU_FWD, false, true, true>(
            g, "gemm_fc1_swiglu_mxfp8", st);
      if (g.epi == EPI_STORE)
        return run<MX_BN, false, false, RAGGED_M, EPI_STORE, false, true, true>(g, "gemm_fc2_mxfp8",
                                                                               st);
    }
    // the data gradients: weights read MN-major (their stored layout), 128-column tiles
    if (!g.gather && g.sched == RAGGED_M && !g.A.mn_major && g.B.mn_major) {
      if (g.epi == EPI_SWIGLU_BWD)
        return run<MX_BN_DGRAD2, false, true, RAGGED_M, EPI_SWIGLU_BWD, false, true, true>(
            g, "gemm_fc2_dgrad_mxfp8", st);
      if (g.epi == EPI_STORE)
        return run<MX_BN_DGRAD1, false, true, RAGGED_M, EPI_STORE, false, true, true>(
            g, "gemm_fc1_dgrad_mxfp8", st);
    }
    // the weight gradients: token-blocked MN-major operands, 128 x 128 tiles (two accumulators)
    if (!g.gather && g.sched == RAGGED_K && g.A.mn_major && g.B.mn_major && g.epi == EPI_F32)
      return run<128, true, true, RAGGED_K, EPI_F32, false, true, true>(g, "gemm_wgrad_mxfp8", st);
    set_error("gemm_tc: unsupported MXFP8 combination sched=%d epi=%d a_mn=%d b_mn=%d", g.sched,
              g.epi, (int)g.A.mn_major, (int)g.B.mn_major);
    return MOE_ERR_UNSUPPORTED;
  }
  if (g.fp8) {
    // E4M3 operands: the expert products of the forward and the backward
    if (!g.gather && g.sched == RAGGED_M && !g.A.mn_major) {
      if (g.epi == EPI_SWIGLU_FWD && !g.B.mn_major)
        return run<256, false, false, RAGGED_M, EPI_SWIGLU_FWD, false, true>(g, "gemm_fc1_swiglu_fp8", st);
      if (g.epi == EPI_STORE && !g.B.mn_major)
        return run<256, false, false, RAGGED_M, EPI_STORE, false, true>(g, "gemm_fc2_fp8", st);
      if (g.epi == EPI_SWIGLU_BWD && g.B.mn_major)
        return run<256, false, true, RAGGED_M, EPI_SWIGLU_BWD, false, true>(g, "gemm_fc2_dgrad_fp8", st);
      if (g.epi == EPI_STORE && g.B.mn_major)
        return run<256, false, true, RAGGED_M, EPI_STORE, false, true>(g, "gemm_fc1_dgrad_fp8", st);
    }
    if (!g.gather && g.sched == RAGGED_K && g.A.mn_major && g.B.mn_major && g.epi == EPI_F32)
      return run<256, true, true, RAGGED_K, EPI_F32, false, true>(g, "gemm_wgrad_fp8", st);
    set_error("gemm_tc: unsupported FP8 combination sched=%d epi=%d a_mn=%d b_mn=%d", g.sched, g.epi,
              (int)g.A.mn_major, (int)g.B.mn_major);
    return MOE_ERR_UNSUPPORTED;
  }
  if (g.sched == RAGGED_M && !g.A.mn_major) {
    if (g.epi == EPI_SWIGLU_FWD && !g.B.mn_major)
      return g.gather ? run<256, false, false, RAGGED_M, EPI_SWIGLU_FWD, true>(g, "gemm_fc1_swiglu", st)
                      : run<256, false, false, RAGGED_M, EPI_SWIGLU_FWD>(g, "gemm_fc1_swiglu", st);
    if (g.gather) {
      set_error("gemm_tc: a gathered A operand is supported for fc1 + SwiGLU only");
      return MOE_ERR_UNSUPPORTED;
    }
    // Output tiles of 192 or 256 columns, whichever pads the product's width less (e.g.
    // d = 2688 is 14 x 192, f = 1856 is 10 x 192 - 64 but 8 x 256 - 192); ties take 256.
    const int ncols = g.epi == EPI_SWIGLU_BWD ? g.f : g.N;
    const bool n192 = MOE_TILE192 && (ncols + 191) / 192 * 192 < (ncols + 255) / 256 * 256;
    if (g.epi == EPI_SWIGLU_BWD && g.B.mn_major)
      return n192 ? run<192, false, true, RAGGED_M, EPI_SWIGLU_BWD>(g, "gemm_fc2_dgrad_swiglu_bwd", st)
                  : run<256, false, true, RAGGED_M, EPI_SWIGLU_BWD>(g, "gemm_fc2_dgrad_swiglu_bwd", st);
    if (MOE_TALL_ROWS && g.epi == EPI_STORE && !n192 && g.G <= MAXG && tall_pays(g))
      return g.B.mn_major ? run_rows_tall<true>(g, st) : run_rows_tall<false>(g, st);
    if (MOE_PAIR_ROWS && g.epi == EPI_STORE && !n192)
      return g.B.mn_major ? run_rows_pair<true>(g, st) : run_rows_pair<false>(g, st);
    if (g.epi == EPI_STORE && !g.B.mn_major)
      return n192 ? run<192, false, false, RAGGED_M, EPI_STORE>(g, "gemm_fc2", st)
                  : run<256, false, false, RAGGED_M, EPI_STORE>(g, "gemm_fc2", st);
    if (g.epi == EPI_STORE && g.B.mn_major)
      return n192 ? run<192, false, true, RAGGED_M, EPI_STORE>(g, "gemm_dgrad", st)
                  : run<256, false, true, RAGGED_M, EPI_STORE>(g, "gemm_dgrad", st);
    if (g.epi == EPI_F32 && !g.B.mn_major) {
      if (g.N <= 128) return run<128, false, false, RAGGED_M, EPI_F32>(g, "gemm_router", st);
      return run<256, false, false, RAGGED_M, EPI_F32>(g, "gemm_router", st);
    }
  }
  if (g.sched == RAGGED_K && g.A.mn_major && g.B.mn_major && g.epi == EPI_F32) {
    if (g.gather) return run<256, true, true, RAGGED_K, EPI_F32, true>(g, "gemm_wgrad", st);
    // one group whose rows are all of both operands' rows (the shared expert): CTA pairs
    if (MOE_PAIR_WGRAD && g.G == 1 && !g.offsets && g.M > 256 && g.A.rows == g.K && g.B.rows == g.K)
      return run_wgrad_pair(g, st);
    return run<256, true, true, RAGGED_K, EPI_F32>(g, "gemm_wgrad", st);
  }
  set_error("gemm_tc: unsupported combination sched=%d epi=%d a_mn=%d b_mn=%d", g.sched, g.epi,
            (int)g.A.mn_major, (int)g.B.mn_major);
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe

extern "C" int moe_gemm_wait_stats(uint64_t* out, int cap) {
  using namespace moe;
  if (!MOE_WAIT_STATS) {
    set_error("moe_gemm_wait_stats: the library was built without MOE_WAIT_STATS=1");
    return MOE_ERR_UNSUPPORTED;
  }
  if (!out || cap < WAIT_KINDS * WAIT_FIELDS) {
    set_error("moe_gemm_wait_stats: out must hold %d values", WAIT_KINDS * WAIT_FIELDS);
    return MOE_ERR_INVALID_ARG;
  }
  static unsigned long long zero[WAIT_KINDS * WAIT_FIELDS];
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(out, g_wait_stats, sizeof(zero)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_wait_stats, zero, sizeof(zero)) != cudaSuccess) {
    set_error("moe_gemm_wait_stats: %s", cudaGetErrorString(cudaGetLastError()));
    return MOE_ERR_CUDA;
  }
  return WAIT_KINDS;
}
