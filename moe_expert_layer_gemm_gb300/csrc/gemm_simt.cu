// Grouped GEMM on the CUDA cores in fp32, for layers whose dtype is fp32: the tensor cores'
// fp32-input mode (tf32) rounds operands to 10 mantissa bits, far outside an fp32 tolerance.
// Same scheduling and epilogues as the tensor-core path (gemm_tc.cu), 64x64 output tiles,
// 256 threads each computing 4x4 outputs, operands staged in shared memory.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int SBM = 64, SBN = 64, SBK = 16;
constexpr int SMAXG = 256;

struct SArgs {
  int sched, epi, G;
  const int32_t* offsets;
  int M, N, K;
  const float* A;
  int64_t lda;
  bool a_mn;
  const float* B;
  int64_t ldb;
  bool b_mn;
  int64_t b_rows;          // rows of the B array (bounds)
  int64_t b_group_rows, b_up_rows;
  int f;
  float* out;
  int64_t ldo, out_group_stride;
  float* out2;
  int64_t ldo2;
  const float* aux;
  int64_t ld_aux;
  const float* bias;
};

// A(m, k) for an operand stored K-major (m row, k col) or MN-major (k row, m col).
__device__ __forceinline__ float opnd(const float* base, int64_t ld, bool mn, int64_t m, int64_t k) {
  return mn ? base[k * ld + m] : base[m * ld + k];
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const SArgs p) {
  __shared__ int s_off[SMAXG + 1];
  __shared__ int s_pre[SMAXG + 1];
  __shared__ float sa[SBK][SBM + 1];
  __shared__ float sb[SBK][2 * SBN + 1];
  const int tid = threadIdx.x;
  for (int i = tid; i <= p.G; i += blockDim.x)
    s_off[i] = p.offsets ? p.offsets[i]
                         : static_cast<int>(static_cast<int64_t>(p.sched == RAGGED_M ? p.M : p.K) *
                                            i / p.G);
  __syncthreads();
  const bool swf = p.epi == EPI_SWIGLU_FWD;
  const int NT = swf ? (p.f + SBN - 1) / SBN : (p.N + SBN - 1) / SBN;
  if (tid == 0) {
    int run = 0;
    for (int g = 0; g < p.G; ++g) {
      s_pre[g] = run;
      run += p.sched == RAGGED_M ? (s_off[g + 1] - s_off[g] + SBM - 1) / SBM : 0;
    }
    s_pre[p.G] = run;
  }
  __syncthreads();
  int g, m0, m_end, n0, k0, k_end;
  if (p.sched == RAGGED_M) {
    const int total = s_pre[p.G] * NT;
    const int tile = blockIdx.x;
    if (tile >= total) return;
    const int mt = tile / NT, nt = tile % NT;
    g = 0;
    while (g + 1 < p.G && s_pre[g + 1] <= mt) ++g;
    m0 = s_off[g] + (mt - s_pre[g]) * SBM;
    m_end = s_off[g + 1];
    n0 = nt * SBN;
    k0 = 0;
    k_end = p.K;
  } else {
    const int MT = (p.M + SBM - 1) / SBM;
    const int tile = blockIdx.x;
    if (tile >= p.G * MT * NT) return;
    g = tile / (MT * NT);
    const int r = tile % (MT * NT);
    m0 = (r / NT) * SBM;
    m_end = p.M;
    n0 = (r % NT) * SBN;
    k0 = s_off[g];
    k_end = s_off[g + 1];
  }
  const int ty = tid / 16, tx = tid % 16;   // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4], acc2[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;
  const int nb_rows = swf ? 2 * SBN : SBN;
  for (int kk = k0; kk < k_end; kk += SBK) {
    for (int i = tid; i < SBK * SBM; i += blockDim.x) {
      const int kq = i / SBM, mq = i % SBM;
      const int64_t m = m0 + mq, k = kk + kq;
      float v = 0.f;
      if (m < m_end && k < k_end) v = opnd(p.A, p.lda, p.a_mn, m, k);
      sa[kq][mq] = v;
    }
    for (int i = tid; i < SBK * nb_rows; i += blockDim.x) {
      const int kq = i / nb_rows, nq = i % nb_rows;
      const int64_t k = kk + kq;
      float v = 0.f;
      int64_t brow;   // B row (n index inside the array)
      bool ok;
      if (swf) {
        const int h = nq < SBN ? n0 + nq : n0 + nq - SBN;
        ok = h < p.f;
        brow = g * p.b_group_rows + (nq < SBN ? 0 : p.b_up_rows) + h;
      } else {
        ok = n0 + nq < p.N;
        brow = (p.sched == RAGGED_M ? g * p.b_group_rows : 0) + n0 + nq;
      }
      if (p.sched == RAGGED_M && p.b_mn && g * p.b_group_rows + k >= p.b_rows) ok = false;
      if (ok && k < k_end) {
        // RAGGED_M: B_g(n, k) = B[g*b_group_rows + n][k] (K-major) or B[g*b_group_rows + k][n]
        // (MN-major); RAGGED_K: B(n, k) = B[k][n].
        if (p.sched == RAGGED_M) {
          v = p.b_mn ? p.B[(g * p.b_group_rows + k) * p.ldb + (n0 + nq)] : p.B[brow * p.ldb + k];
        } else {
          v = opnd(p.B, p.ldb, true, n0 + nq, k);
        }
      }
      sb[kq][nq] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kq = 0; kq < SBK; ++kq) {
      float a[4], b[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sa[kq][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b[j] = sb[kq][tx * 4 + j];
        b2[j] = swf ? sb[kq][SBN + tx * 4 + j] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (swf) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = m0 + ty * 4 + i;
    if (row >= m_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (swf) {
        if (col >= p.f) continue;
        const float a = acc[i][j], u = acc2[i][j];
        p.out[row * p.ldo + col] = a / (1.0f + expf(-a)) * u;
        if (p.out2) {
          p.out2[row * p.ldo2 + col] = a;
          p.out2[row * p.ldo2 + p.f + col] = u;
        }
      } else if (p.epi == EPI_SWIGLU_BWD) {
        if (col >= p.f) continue;
        const float dh = acc[i][j];
        const float a = p.aux[row * p.ld_aux + col], u = p.aux[row * p.ld_aux + p.f + col];
        const float s = 1.0f / (1.0f + expf(-a));
        p.out[row * p.ldo + col] = dh * u * (s + a * s * (1.0f - s));
        p.out[row * p.ldo + p.f + col] = dh * a * s;
      } else {
        if (col >= p.N) continue;
        float v = acc[i][j];
        if (p.bias) v += p.bias[col];
        p.out[g * p.out_group_stride + row * p.ldo + col] = v;
      }
    }
  }
}

}  // namespace

int gemm_simt(const GemmDesc& d, cudaStream_t st) {
  if (d.G < 1 || d.G > SMAXG) {
    set_error("gemm_simt: group count %d outside [1, %d]", d.G, SMAXG);
    return MOE_ERR_UNSUPPORTED;
  }
  SArgs a;
  a.sched = d.sched;
  a.epi = d.epi;
  a.G = d.G;
  a.offsets = d.offsets;
  a.M = d.M;
  a.N = d.N;
  a.K = d.K;
  a.A = static_cast<const float*>(d.A.base);
  a.lda = d.A.ld;
  a.a_mn = d.A.mn_major;
  a.B = static_cast<const float*>(d.B.base);
  a.ldb = d.B.ld;
  a.b_mn = d.B.mn_major;
  a.b_rows = d.B.rows;
  a.b_group_rows = d.b_group_rows;
  a.b_up_rows = d.b_up_rows;
  a.f = d.f;
  a.out = static_cast<float*>(d.out);
  a.ldo = d.ldo;
  a.out_group_stride = d.out_group_stride;
  a.out2 = static_cast<float*>(d.out2);
  a.ldo2 = d.ldo2;
  a.aux = static_cast<const float*>(d.aux);
  a.ld_aux = d.ld_aux;
  a.bias = d.bias;
  const int NT = d.epi == EPI_SWIGLU_FWD ? (d.f + SBN - 1) / SBN : (d.N + SBN - 1) / SBN;
  int64_t tiles;
  if (d.sched == RAGGED_M)
    tiles = (static_cast<int64_t>(d.M) + SBM - 1) / SBM * NT + static_cast<int64_t>(d.G) * NT;
  else
    tiles = static_cast<int64_t>(d.G) * ((d.M + SBM - 1) / SBM) * NT;
  if (tiles > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
  const char* name = d.name ? d.name : "simt_gemm";
  return launch(name, simt_gemm_kernel, dim3(static_cast<unsigned>(tiles)), dim3(256), 0, st, a);
}

}  // namespace moe
