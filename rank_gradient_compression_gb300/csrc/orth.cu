// Batched fp32 orthonormalisation of P (m x r, every matrix of the step at once):
// adaptive shifted CholeskyQR.
//
// The method is fixed as "Cholesky-QR or Gram-Schmidt in fp32". One pass forms the Gram
// matrix X^T X (row-chunk partial sums, then a fixed-order sum), factors it
// X^T X (+ s I) = R^T R on one CTA, and sets X <- X R^-1. A Cholesky that loses more
// than 16 bits on some pivot is redone with a shift s = 2^-20 sqrt(m) tr(X^T X).
// That is the shifted CholeskyQR of Fukaya et al. (2020), with the rounding-error term
// taken at its typical sqrt(m) growth, not the worst case. The factor-of-m worst case
// in fp32 would shift by more than the largest eigenvalue. A pass whose Cholesky is
// unshifted and shows a nearly orthonormal X (pivot ratios >= 1/2, diag(R) within a
// factor 2) is the last one. CholeskyQR2 (two passes) is the common case. Columns whose
// pivot vanishes are numerically dependent; their column of R^-1 is zeroed. That
// leaves a zero column in P^ and the projector P^ P^T onto span(P) unchanged.
//
// Device pass state: ostate[pass] = {final, dst buffer, shifted, dead columns}, written
// by the pass's Cholesky kernel. The next pass reads it after the launch boundary.
#include "handle.h"

namespace psgd {
namespace {

constexpr int kT = 256;

__device__ __forceinline__ float* buf_ptr(const MatMeta& mt, int idx) {
  return idx == 0 ? mt.P : idx == 1 ? mt.Xa : idx == 2 ? mt.Xb : mt.Phat;
}

// Power-of-two scale that brings max|P| into [1, 2): exact.
__device__ __forceinline__ float p_scale(const MatMeta& mt) {
  const unsigned bits = reinterpret_cast<const unsigned*>(mt.scal)[1];
  const int ex = (int)((bits >> 23) & 0xff);
  if (bits == 0u) return 1.0f;
  return exp2f((float)(127 - max(ex, 1)));
}

// A pass runs only when every earlier pass ran and was not final. The scan stops at the
// first final pass, so every entry it reads was written earlier in this same step; the
// entries of passes that did not run hold values from older steps and are never read.
__device__ __forceinline__ bool pass_skipped(const Plan& p, const MatMeta& mt, int pass) {
  if (p.skip[mt.b]) return true;
  for (int q = 0; q < pass; ++q)
    if (mt.ostate[q * 4 + 0] != 0) return true;
  return false;
}

// Gram partial sums over a row chunk: Gpart[c] = X_c^T X_c (rp x rp, r <= 128).
// grid = (max C, B*J).
__global__ void __launch_bounds__(kT) k_gram(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if ((int)blockIdx.x >= mt.C || pass_skipped(p, mt, pass)) return;
  const int64_t m = mt.m;
  const int r = p.r, rp = p.rp;
  const float* X = pass == 0 ? mt.P : buf_ptr(mt, mt.ostate[(pass - 1) * 4 + 1]);
  const float sc = pass == 0 ? p_scale(mt) : 1.0f;
  const int64_t rows_per = ((m + mt.C - 1) / mt.C + 31) / 32 * 32;
  const int64_t rbeg = (int64_t)blockIdx.x * rows_per, rend = min(m, rbeg + rows_per);
  __shared__ __align__(16) float Xs[32][128];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int64_t k0 = rbeg; k0 < rend; k0 += 32) {
    const int kk = tid >> 3, c = (tid & 7) * 16;
    const int64_t row = k0 + kk;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      Xs[kk][c + i] = (row < rend && c + i < r) ? X[row * rp + c + i] * sc : 0.f;
    __syncthreads();
#pragma unroll 4
    for (int q = 0; q < 32; ++q) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&Xs[q][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&Xs[q][ty * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Xs[q][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Xs[q][tx * 8 + 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = mt.Gpart + (size_t)blockIdx.x * rp * rp;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ii = ty * 8 + i;
    if (ii >= r) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int jj = tx * 8 + j;
      if (jj < r) out[ii * rp + jj] = acc[i][j];
    }
  }
}

// G = sum_c Gpart[c] into slot C of Gpart. Eight threads share an entry: thread k sums
// the partials c = k, k+8, ... in order, then the eight sums are added in a fixed tree
// order (deterministic). grid = (ceil(rp*rp/32), B*J).
__global__ void __launch_bounds__(kT) k_gsum(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (pass_skipped(p, mt, pass)) return;
  const int rp = p.rp;
  const int idx = blockIdx.x * (kT / 8) + (threadIdx.x >> 3);
  const int part = threadIdx.x & 7;
  const bool live = idx < rp * rp;
  const float* src = mt.Gpart + (live ? idx : 0);
  float s = 0.f;
  if (live)
    for (int c = part; c < mt.C; c += 8) s = __fadd_rn(s, __ldg(src + (size_t)c * rp * rp));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 4));
  if (live && part == 0) mt.Gpart[(size_t)mt.C * rp * rp + idx] = s;
}

// Load the summed Gram matrix (slot C of Gpart) into shared memory, plus its diagonal.
// Threads work on a 16 x 16 grid of (row, column) strides: no integer division.
__device__ void load_gram(const MatMeta& mt, int r, int rp, float* G, int ldg, float* diag0,
                          float shift) {
  const float* src = mt.Gpart + (size_t)mt.C * rp * rp;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  for (int i = ty; i < r; i += 16)
    for (int j = tx; j < r; j += 16) {
      float s = src[i * rp + j];
      if (i == j) { diag0[i] = s; s += shift; }
      G[i * ldg + j] = s;
    }
  __syncthreads();
}

constexpr int NB = 16;  // panel width of the blocked factorisations

// In-place blocked right-looking Cholesky of the upper triangle of G (r x r, shared
// memory): G = R^T R. Pivot k is dead when it is <= dead_tol * diag0[k] (or not finite):
// row k of R becomes e_k and column k takes no part in later updates. The pivot ratio
// pivot_k / diag0_k goes into ratio[k] (0 for dead columns). Per 16-wide panel: warp 0
// factors the diagonal block, the panel rows are solved column by column, then one
// rank-16 update of the trailing matrix: three barriers a panel.
__device__ void cholesky_smem(float* G, int ldg, int r, const float* diag0, float dead_tol,
                              float* ratio, int* dead) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  for (int kb = 0; kb < r; kb += NB) {
    const int nb = min(NB, r - kb);
    if (warp == 0) {
      for (int k = 0; k < nb; ++k) {
        const int kk = kb + k;
        float d = G[kk * ldg + kk];
        const bool bad = !(d > dead_tol * diag0[kk]) || !isfinite(d) || !(diag0[kk] > 0.f);
        const float rkk = bad ? 1.f : sqrtf(d);
        const float inv = 1.f / rkk;
        __syncwarp();
        if (lane == 0) {
          dead[kk] = bad;
          ratio[kk] = bad ? 0.f : d / diag0[kk];
          G[kk * ldg + kk] = rkk;
        }
        // row kk of the diagonal block
        if (lane > k && lane < nb) G[kk * ldg + kb + lane] = bad ? 0.f : G[kk * ldg + kb + lane] * inv;
        __syncwarp();
        if (!bad) {
          for (int q = lane; q < (nb - k - 1) * (nb - k - 1); q += 32) {
            const int i = kb + k + 1 + q / (nb - k - 1), j = kb + k + 1 + q % (nb - k - 1);
            if (j >= i) G[i * ldg + j] = fmaf(-G[kk * ldg + i], G[kk * ldg + j], G[i * ldg + j]);
          }
        }
        __syncwarp();
      }
    }
    __syncthreads();
    // panel rows kb..kb+nb-1, columns j >= kb+nb: solve D^T x = g column by column
    for (int j = kb + nb + threadIdx.x; j < r; j += blockDim.x) {
      float x[NB];
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        if (k >= nb) break;
        const int kk = kb + k;
        float v = G[kk * ldg + j];
        for (int q = 0; q < k; ++q) v = fmaf(-G[(kb + q) * ldg + kk], x[q], v);
        x[k] = dead[kk] ? 0.f : v / G[kk * ldg + kk];
        G[kk * ldg + j] = x[k];
      }
    }
    __syncthreads();
    // trailing update: G[i][j] -= sum_q R[kb+q][i] R[kb+q][j], kb+nb <= i <= j < r
    for (int i = kb + nb + ty; i < r; i += 16)
      for (int j = kb + nb + tx; j < r; j += 16) {
        if (j < i) continue;
        float v = G[i * ldg + j];
        for (int q = 0; q < nb; ++q) v = fmaf(-G[(kb + q) * ldg + i], G[(kb + q) * ldg + j], v);
        G[i * ldg + j] = v;
      }
    __syncthreads();
  }
}

// X = R^-1 (upper triangular, r x r, shared memory) by blocked back substitution: for the
// panels from the bottom, T = I - R[panel, below] X[below, :], then D X[panel, :] = T
// with the panel's diagonal block D. Two barriers a panel. X must start as zero.
__device__ void inverse_upper(const float* G, int ldg, int r, float* X) {
  const int last = ((r - 1) / NB) * NB;
  for (int kb = last; kb >= 0; kb -= NB) {
    const int nb = min(NB, r - kb);
    // T[i][j] for i in the panel, j >= kb (kept in X's panel rows)
    for (int q = threadIdx.x; q < nb * (r - kb); q += blockDim.x) {
      const int i = kb + q / (r - kb), j = kb + q % (r - kb);
      float v = (i == j) ? 1.f : 0.f;
      for (int l = kb + nb; l <= j; ++l) v = fmaf(-G[i * ldg + l], X[l * ldg + j], v);
      X[i * ldg + j] = v;
    }
    __syncthreads();
    // back substitution within the panel, one column per thread
    for (int j = kb + threadIdx.x; j < r; j += blockDim.x) {
      for (int k = nb - 1; k >= 0; --k) {
        const int i = kb + k;
        if (i > j) continue;
        float v = X[i * ldg + j];
        for (int q = k + 1; q < nb && kb + q <= j; ++q) v = fmaf(-G[i * ldg + kb + q], X[(kb + q) * ldg + j], v);
        X[i * ldg + j] = v / G[i * ldg + i];
      }
    }
    __syncthreads();
  }
}

// One CTA per matrix: factor the Gram matrix of this pass, decide shift/final, write R^-1.
__global__ void __launch_bounds__(kT) k_chol(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.x];
  if (pass_skipped(p, mt, pass)) return;
  const int r = p.r, rp = p.rp, ldg = kMaxRank + 1;
  extern __shared__ float sm[];
  float* G = sm;                          // [kMaxRank][kMaxRank + 1]
  float* diag0 = G + kMaxRank * ldg;      // [kMaxRank]
  float* ratio = diag0 + kMaxRank;        // [kMaxRank]
  int* dead = reinterpret_cast<int*>(ratio + kMaxRank);  // [kMaxRank]; R^-1 work after it
  __shared__ float s_trace, s_maxr, s_minr, s_minratio;
  __shared__ int s_ndead, s_retry;
  const bool last = pass == kMaxPasses - 1;
  int* st = mt.ostate + pass * 4;
  const int src = pass == 0 ? 0 : mt.ostate[(pass - 1) * 4 + 1];

  load_gram(mt, r, rp, G, ldg, diag0, 0.f);
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < r; ++k) t += diag0[k];
    s_trace = t;
  }
  __syncthreads();
  const float trace = s_trace;
  bool shifted = false;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  if (!(trace > 0.f) || !isfinite(trace)) {
    for (int k = threadIdx.x; k < r; k += blockDim.x) dead[k] = 1;
    for (int i = ty; i < r; i += 16)
      for (int j = tx; j < r; j += 16) G[i * ldg + j] = (i == j) ? 1.f : 0.f;
    __syncthreads();
  } else {
    cholesky_smem(G, ldg, r, diag0, last ? 0x1p-40f : 0x1p-16f, ratio, dead);
    if (threadIdx.x == 0) {
      int nd = 0;
      for (int k = 0; k < r; ++k) nd += dead[k];
      s_retry = (nd > 0 && !last) ? 1 : 0;
    }
    __syncthreads();
    if (s_retry) {
      shifted = true;
      const float shift = 0x1p-20f * sqrtf((float)mt.m) * trace;
      load_gram(mt, r, rp, G, ldg, diag0, shift);
      cholesky_smem(G, ldg, r, diag0, 0x1p-40f, ratio, dead);
    }
  }
  // statistics of the factor
  if (threadIdx.x == 0) {
    float mx = 0.f, mn = 3.4e38f, mr = 1.f;
    int nd = 0;
    for (int k = 0; k < r; ++k) {
      if (dead[k]) { ++nd; continue; }
      const float d = G[k * ldg + k];
      mx = fmaxf(mx, d); mn = fminf(mn, d); mr = fminf(mr, ratio[k]);
    }
    s_maxr = mx; s_minr = mn; s_minratio = mr; s_ndead = nd;
  }
  __syncthreads();
  // R^-1 (upper triangular), blocked, in shared memory
  float* X = ratio + kMaxRank + kMaxRank;  // [kMaxRank][ldg], after dead[]
  for (int i = ty; i < r; i += 16)
    for (int j = tx; j < r; j += 16) X[i * ldg + j] = 0.f;
  __syncthreads();
  inverse_upper(G, ldg, r, X);
  float* Ri = mt.Rinv;
  for (int i = ty; i < r; i += 16)
    for (int j = tx; j < r; j += 16) Ri[i * rp + j] = (j >= i && !dead[j]) ? X[i * ldg + j] : 0.f;
  if (threadIdx.x == 0) {
    const bool nearly_orth = !shifted && s_ndead == 0 && s_minratio >= 0.5f &&
                             s_maxr <= 2.f * s_minr;
    const bool all_dead = s_ndead == r;
    const int fin = (last || nearly_orth || all_dead) ? 1 : 0;
    st[0] = fin;
    st[1] = fin ? 3 : (src == 1 ? 2 : 1);
    st[2] = shifted ? 1 : 0;
    st[3] = s_ndead;
  }
}

// X <- X R^-1 on 64-row tiles (R^-1 upper triangular, r <= 128). grid = (ceil(m/64), B*J).
__global__ void __launch_bounds__(kT) k_apply(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (pass_skipped(p, mt, pass)) return;
  const int64_t m = mt.m;
  const int r = p.r, rp = p.rp;
  const int64_t row0 = (int64_t)blockIdx.x * 64;
  if (row0 >= m) return;
  const float* X = pass == 0 ? mt.P : buf_ptr(mt, mt.ostate[(pass - 1) * 4 + 1]);
  float* Y = buf_ptr(mt, mt.ostate[pass * 4 + 1]);
  const float sc = pass == 0 ? p_scale(mt) : 1.0f;
  __shared__ float As[32][64 + 4];
  __shared__ __align__(16) float Bs[32][128];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < r; k0 += 32) {
    {
      const int rr = tid >> 2, kk = (tid & 3) * 8;
      const int64_t row = row0 + rr;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + kk + i;
        As[kk + i][rr] = (row < m && k < r) ? X[row * rp + k] * sc : 0.f;
      }
    }
    {
      const int kk = tid >> 3, c = (tid & 7) * 16;
      const int k = k0 + kk;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        Bs[kk][c + i] = (k < r && c + i < r) ? mt.Rinv[k * rp + c + i] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 8 + 4]);
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = row0 + ty * 4 + i;
    if (row >= m) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = tx * 8 + j;
      if (c < rp) Y[row * rp + c] = c < r ? acc[i][j] : 0.f;
    }
  }
}

constexpr size_t kCholSmem = 2 * (size_t)kMaxRank * (kMaxRank + 1) * 4 + 3 * kMaxRank * 4;

}  // namespace

cudaError_t launch_orth(const Handle& h, const Plan& p, cudaStream_t s) {
  cudaFuncSetAttribute(k_chol, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCholSmem);
  const int BJ = p.B * p.J;
  for (int pass = 0; pass < kMaxPasses; ++pass) {
    k_gram<<<dim3(h.max_C, BJ), kT, 0, s>>>(p, pass);
    k_gsum<<<dim3((p.rp * p.rp + kT / 8 - 1) / (kT / 8), BJ), kT, 0, s>>>(p, pass);
    k_chol<<<BJ, kT, kCholSmem, s>>>(p, pass);
    k_apply<<<dim3(h.max_mtiles64, BJ), kT, 0, s>>>(p, pass);
    h.launches += 4;
  }
  return cudaGetLastError();
}

cudaError_t launch_orth_one(const Plan& p, int C, int mtiles64, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_chol, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kCholSmem);
  if (e != cudaSuccess) return e;
  for (int pass = 0; pass < kMaxPasses; ++pass) {
    k_gram<<<dim3(C, 1), kT, 0, s>>>(p, pass);
    k_gsum<<<dim3((p.rp * p.rp + kT / 8 - 1) / (kT / 8), 1), kT, 0, s>>>(p, pass);
    k_chol<<<1, kT, kCholSmem, s>>>(p, pass);
    k_apply<<<dim3(mtiles64, 1), kT, 0, s>>>(p, pass);
  }
  return cudaGetLastError();
}

}  // namespace psgd
