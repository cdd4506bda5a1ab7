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

__device__ __forceinline__ bool pass_skipped(const Plan& p, const MatMeta& mt, int pass) {
  if (p.skip[mt.b]) return true;
  return pass > 0 && mt.ostate[(pass - 1) * 4 + 0] != 0;
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

// G = sum_c Gpart[c] in chunk order, one element per thread, into slot C of Gpart.
// grid = (ceil(rp*rp/256), B*J).
__global__ void __launch_bounds__(kT) k_gsum(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (pass_skipped(p, mt, pass)) return;
  const int rp = p.rp;
  const int idx = blockIdx.x * kT + threadIdx.x;
  if (idx >= rp * rp) return;
  const float* src = mt.Gpart + idx;
  float s = 0.f;
#pragma unroll 8
  for (int c = 0; c < mt.C; ++c) s = __fadd_rn(s, __ldg(src + (size_t)c * rp * rp));
  mt.Gpart[(size_t)mt.C * rp * rp + idx] = s;
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

// In-place right-looking Cholesky of the upper triangle of G (r x r, shared memory).
// Pivot k is dead when it is <= dead_tol * diag0[k] (or not finite): row k of R
// becomes e_k and column k is left out of the trailing update. The pivot ratio
// pivot_k / diag0_k goes into ratio[k] (0 for dead columns).
__device__ void cholesky_smem(float* G, int ldg, int r, const float* diag0, float dead_tol,
                              float* ratio, int* dead) {
  __shared__ float s_inv;
  __shared__ int s_dead;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  for (int k = 0; k < r; ++k) {
    if (threadIdx.x == 0) {
      const float d = G[k * ldg + k];
      const bool bad = !(d > dead_tol * diag0[k]) || !isfinite(d) || !(diag0[k] > 0.f);
      s_dead = bad;
      dead[k] = bad;
      ratio[k] = bad ? 0.f : d / diag0[k];
      const float rkk = bad ? 1.f : sqrtf(d);
      G[k * ldg + k] = rkk;
      s_inv = 1.f / rkk;
    }
    __syncthreads();
    const bool isdead = s_dead != 0;
    const float inv = s_inv;
    for (int j = k + 1 + threadIdx.x; j < r; j += blockDim.x)
      G[k * ldg + j] = isdead ? 0.f : G[k * ldg + j] * inv;
    __syncthreads();
    if (!isdead) {
      for (int i = k + 1 + ty; i < r; i += 16) {
        const float gki = G[k * ldg + i];
        for (int j = k + 1 + tx; j < r; j += 16)
          if (j >= i) G[i * ldg + j] = fmaf(-gki, G[k * ldg + j], G[i * ldg + j]);
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
  // R^-1 (upper triangular) by right-looking elimination in shared memory: X = I, then
  // for l = r-1 .. 0: X[l,:] /= R[l,l]; X[k,:] -= R[k,l] X[l,:] for k < l. When row l is
  // finalised, every row below it has already contributed, so X[l,:] is row l of R^-1.
  float* X = ratio + kMaxRank + kMaxRank;  // [kMaxRank][ldg], after dead[]
  for (int i = ty; i < r; i += 16)
    for (int j = tx; j < r; j += 16) X[i * ldg + j] = (i == j) ? 1.f : 0.f;
  __syncthreads();
  for (int l = r - 1; l >= 0; --l) {
    const float inv = 1.f / G[l * ldg + l];
    for (int j = l + threadIdx.x; j < r; j += blockDim.x) X[l * ldg + j] *= inv;
    __syncthreads();
    for (int k = ty; k < l; k += 16) {
      const float gkl = G[k * ldg + l];
      for (int j = l + tx; j < r; j += 16) X[k * ldg + j] = fmaf(-gkl, X[l * ldg + j], X[k * ldg + j]);
    }
    __syncthreads();
  }
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
    k_gsum<<<dim3((p.rp * p.rp + kT - 1) / kT, BJ), kT, 0, s>>>(p, pass);
    k_chol<<<BJ, kT, kCholSmem, s>>>(p, pass);
    k_apply<<<dim3(h.max_mtiles64, BJ), kT, 0, s>>>(p, pass);
    h.launches += 4;
  }
  return cudaGetLastError();
}

}  // namespace psgd
