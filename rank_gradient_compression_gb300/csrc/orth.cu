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

// Gram partial sums over a row chunk: the upper triangle of Gpart[c] = X_c^T X_c
// (rp x rp, r <= 128) in 8 x 8 blocks, one block (bi <= bj) per thread; the lower
// triangle is neither written nor read. grid = (max C, B*J), block kGramThreads.
constexpr int kGramThreads = 160;  // >= 16 * 17 / 2 = 136 upper-triangle blocks
__global__ void __launch_bounds__(kGramThreads) k_gram(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if ((int)blockIdx.x >= mt.C || pass_skipped(p, mt, pass)) return;
  const int64_t m = mt.m;
  const int r = p.r, rp = p.rp;
  const float* X = pass == 0 ? mt.P : buf_ptr(mt, mt.ostate[(pass - 1) * 4 + 1]);
  const float sc = pass == 0 ? p_scale(mt) : 1.0f;
  const int64_t rows_per = ((m + mt.C - 1) / mt.C + 31) / 32 * 32;
  const int64_t rbeg = (int64_t)blockIdx.x * rows_per, rend = min(m, rbeg + rows_per);
  __shared__ __align__(16) float Xs[32][128];
  const int tid = threadIdx.x;
  // this thread's block (bi, bj), bi <= bj, of the nb x nb block grid
  const int nb = (r + 7) / 8;
  int bi = 0, rem = tid;
  while (bi < nb && rem >= nb - bi) { rem -= nb - bi; ++bi; }
  const bool live = bi < nb;
  const int bj = bi + rem;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int64_t k0 = rbeg; k0 < rend; k0 += 32) {
    for (int idx = tid; idx < 32 * 128; idx += kGramThreads) {
      const int kk = idx >> 7, c = idx & 127;
      const int64_t row = k0 + kk;
      Xs[kk][c] = (row < rend && c < r) ? X[row * rp + c] * sc : 0.f;
    }
    __syncthreads();
    if (live) {
#pragma unroll 4
      for (int q = 0; q < 32; ++q) {
        float a[8], b[8];
        const float4 a0 = *reinterpret_cast<const float4*>(&Xs[q][bi * 8]);
        const float4 a1 = *reinterpret_cast<const float4*>(&Xs[q][bi * 8 + 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Xs[q][bj * 8]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Xs[q][bj * 8 + 4]);
        a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
    }
    __syncthreads();
  }
  if (!live) return;
  float* out = mt.Gpart + (size_t)blockIdx.x * rp * rp;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ii = bi * 8 + i;
    if (ii >= r) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int jj = bj * 8 + j;
      if (jj < r && jj >= ii) out[ii * rp + jj] = acc[i][j];
    }
  }
}

// G = sum_c Gpart[c] into slot C of Gpart (upper triangle). Eight threads share an entry: thread k sums
// the partials c = k, k+8, ... in order, then the eight sums are added in a fixed tree
// order (deterministic). grid = (ceil(rp*rp/32), B*J).
__global__ void __launch_bounds__(kT) k_gsum(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (pass_skipped(p, mt, pass)) return;
  const int rp = p.rp;
  const int idx = blockIdx.x * (kT / 8) + (threadIdx.x >> 3);
  const int part = threadIdx.x & 7;
  const bool live = idx < rp * rp && idx % rp >= idx / rp;  // upper triangle only
  const float* src = mt.Gpart + (live ? idx : 0);
  float s = 0.f;
  if (live) {
#pragma unroll 8
    for (int c = part; c < mt.C; c += 8) s = __fadd_rn(s, __ldg(src + (size_t)c * rp * rp));
  }
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 4));
  if (live && part == 0) mt.Gpart[(size_t)mt.C * rp * rp + idx] = s;
}

// ---------------------------------------------------------------- Cholesky + R^-1
// One CTA of kCholWarps warps per matrix. The Gram matrix lives in registers: warp w owns
// the 8-row panel [8w, 8w + 8), and lane l holds columns l, l + 32, l + 64, l + 96 of
// those rows. r <= 128, so every row has an owner.
//
// Factorisation G = R^T R (right-looking, by panels): the owner warp factors its panel
// with shuffles only and writes the panel's 8 rows of R to shared memory; after one
// block barrier every later warp subtracts the rank-8 update from its rows. Pivot k is
// dead when it is <= dead_tol * diag0[k] (or not finite): row k of R becomes e_k and
// column k takes no part in later updates.
//
// R^-1 (upper triangular) by the same panels from the bottom: the owner warp finishes
// the rows of its panel, X_k = T_k / r_kk with T_k = e_k minus the contributions of the
// rows below, and publishes them; the warps above subtract R[i][panel] X[panel].
// Two block barriers per 8 rows in all, instead of one or two per row.
constexpr int kCholWarps = 16;
constexpr int kCholThreads = kCholWarps * 32;
constexpr int kPanel = 8;
static_assert(kCholWarps * kPanel >= kMaxRank, "every row needs an owner warp");
constexpr int kRsLd = kMaxRank + 1;  // row stride of R in shared memory

struct CholSmem {
  float R[kMaxRank * kRsLd];           // rows of R as they are finished
  float X[2][kPanel * kRsLd];          // published rows of R^-1 (ping-pong by panel)
  float diag0[kMaxRank];               // diagonal of the unshifted Gram matrix
  float ratio[kMaxRank];               // pivot / diag0 (0 for dead pivots)
  int dead[kMaxRank];
};

// Select a[q] for a warp-uniform q in 0..3 without dynamic register indexing.
__device__ __forceinline__ float pick4(const float a[4], int q) {
  return q == 0 ? a[0] : q == 1 ? a[1] : q == 2 ? a[2] : a[3];
}

// Load rows [8 warp, 8 warp + 8) of the summed Gram matrix (slot C of Gpart) into
// registers, zero outside r x r, and add `shift` to the diagonal. With record set, the
// unshifted diagonal goes to diag0.
__device__ __forceinline__ void load_gram_regs(const MatMeta& mt, int r, int rp, float a[kPanel][4],
                                               float shift, CholSmem& S, bool record) {
  const float* src = mt.Gpart + (size_t)mt.C * rp * rp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kPanel; ++t) {
    const int i = warp * kPanel + t;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      float v = (i < r && j < r && j >= i) ? src[(size_t)i * rp + j] : 0.f;  // upper triangle
      if (i == j && i < r) {
        if (record) S.diag0[i] = v;
        v += shift;
      }
      a[t][q] = v;
    }
  }
}

// Factor the registers' panels in place (rows of R) and fill S.R, S.dead, S.ratio.
__device__ void cholesky_panels(float a[kPanel][4], int r, float dead_tol, CholSmem& S) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npan = (r + kPanel - 1) / kPanel;
  for (int pn = 0; pn < npan; ++pn) {
    const int k0 = pn * kPanel;
    if (warp == pn) {
      const int qk = k0 >> 5;  // column group of this panel (panels never straddle 32)
#pragma unroll
      for (int t = 0; t < kPanel; ++t) {
        const int k = k0 + t;
        if (k < r) {
          const float d = __shfl_sync(0xffffffffu, pick4(a[t], qk), k & 31);
          const float d0 = S.diag0[k];
          const bool bad = !(d > dead_tol * d0) || !isfinite(d) || !(d0 > 0.f);
          const float rkk = bad ? 1.f : sqrtf(d);
          const float inv = __frcp_rn(rkk);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = lane + 32 * q;
            a[t][q] = j < k ? 0.f : (j == k ? rkk : (bad ? 0.f : a[t][q] * inv));
          }
          if (lane == 0) {
            S.dead[k] = bad;
            S.ratio[k] = bad ? 0.f : __fdividef(d, d0);  // statistics only
          }
          // the rows below k in this panel
#pragma unroll
          for (int t2 = t + 1; t2 < kPanel; ++t2) {
            const float c = __shfl_sync(0xffffffffu, pick4(a[t], qk), (k0 + t2) & 31);
#pragma unroll
            for (int q = 0; q < 4; ++q) a[t2][q] = fmaf(-c, a[t][q], a[t2][q]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kPanel; ++t)
        if (k0 + t < r) {
#pragma unroll
          for (int q = 0; q < 4; ++q) S.R[(k0 + t) * kRsLd + lane + 32 * q] = a[t][q];
        }
    }
    __syncthreads();
    if (warp > pn) {
      const int kend = min(kPanel, r - k0);
      const int i0 = warp * kPanel;
#pragma unroll
      for (int pp = 0; pp < kPanel; ++pp) {
        if (pp >= kend) break;
        const float* Rk = S.R + (k0 + pp) * kRsLd;
        float rj[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) rj[q] = Rk[lane + 32 * q];
#pragma unroll
        for (int t = 0; t < kPanel; ++t) {  // rows i >= r hold zeros and stay unused
          const float c = Rk[i0 + t];
#pragma unroll
          for (int q = 0; q < 4; ++q) a[t][q] = fmaf(-c, rj[q], a[t][q]);
        }
      }
    }
  }
}

// R^-1 into the registers (rows of this warp's panel), from S.R.
__device__ void inverse_panels(float a[kPanel][4], int r, CholSmem& S) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kPanel; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) a[t][q] = (warp * kPanel + t == lane + 32 * q) ? 1.f : 0.f;
  const int npan = (r + kPanel - 1) / kPanel;
  for (int pn = npan - 1; pn >= 0; --pn) {
    const int k0 = pn * kPanel;
    float* Xp = S.X[pn & 1];
    if (warp == pn) {
#pragma unroll
      for (int t = kPanel - 1; t >= 0; --t) {
        const int k = k0 + t;
        if (k < r) {
          const float inv = __frcp_rn(S.R[k * kRsLd + k]);
#pragma unroll
          for (int q = 0; q < 4; ++q) a[t][q] *= inv;
#pragma unroll
          for (int t2 = 0; t2 < t; ++t2) {
            const float c = S.R[(k0 + t2) * kRsLd + k];
#pragma unroll
            for (int q = 0; q < 4; ++q) a[t2][q] = fmaf(-c, a[t][q], a[t2][q]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kPanel; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q) Xp[t * kRsLd + lane + 32 * q] = a[t][q];
    }
    __syncthreads();
    if (warp < pn) {
      const int kend = min(kPanel, r - k0);
      const float* Ri = S.R + (warp * kPanel) * kRsLd + k0;
#pragma unroll
      for (int pp = 0; pp < kPanel; ++pp) {
        if (pp >= kend) break;
        float xj[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) xj[q] = Xp[pp * kRsLd + lane + 32 * q];
#pragma unroll
        for (int t = 0; t < kPanel; ++t) {
          const float c = Ri[t * kRsLd + pp];
#pragma unroll
          for (int q = 0; q < 4; ++q) a[t][q] = fmaf(-c, xj[q], a[t][q]);
        }
      }
    }
  }
}

// One CTA per matrix: factor the Gram matrix of this pass, decide shift/final, write R^-1.
__global__ void __launch_bounds__(kCholThreads) k_chol(Plan p, int pass) {
  const MatMeta& mt = p.meta[blockIdx.x];
  if (pass_skipped(p, mt, pass)) return;
  const int r = p.r, rp = p.rp;
  extern __shared__ __align__(16) unsigned char chol_smem[];
  CholSmem& S = *reinterpret_cast<CholSmem*>(chol_smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool last = pass == kMaxPasses - 1;
  int* st = mt.ostate + pass * 4;
  const int src = pass == 0 ? 0 : mt.ostate[(pass - 1) * 4 + 1];

  float a[kPanel][4];
  __shared__ float s_trace;
  load_gram_regs(mt, r, rp, a, 0.f, S, true);
  __syncthreads();
  if (warp == 0) {  // trace: fixed-order warp reduction
    float t = 0.f;
    for (int k = lane; k < r; k += 32) t += S.diag0[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) s_trace = t;
  }
  __syncthreads();
  const float trace = s_trace;
  bool shifted = false;
  if (!(trace > 0.f) || !isfinite(trace)) {
    for (int k = threadIdx.x; k < r; k += blockDim.x) { S.dead[k] = 1; S.ratio[k] = 0.f; }
    for (int idx = threadIdx.x; idx < r * kRsLd; idx += blockDim.x) {
      const int i = idx / kRsLd, j = idx - i * kRsLd;
      S.R[idx] = (i == j) ? 1.f : 0.f;
    }
    __syncthreads();
  } else {
    cholesky_panels(a, r, last ? 0x1p-40f : 0x1p-16f, S);
    __syncthreads();
    int nd = 0;
    for (int k = lane; k < r; k += 32) nd += S.dead[k];
    nd = __reduce_add_sync(0xffffffffu, nd);  // every warp computes the same count
    if (nd > 0 && !last) {
      shifted = true;
      const float shift = 0x1p-20f * sqrtf((float)mt.m) * trace;
      load_gram_regs(mt, r, rp, a, shift, S, false);
      __syncthreads();
      cholesky_panels(a, r, 0x1p-40f, S);
      __syncthreads();
    }
  }
  // statistics of the factor: warp 0 reduces over the pivots
  __shared__ float s_maxr, s_minr, s_minratio;
  __shared__ int s_ndead;
  if (warp == 0) {
    float mx = 0.f, mn = 3.4e38f, mr = 1.f;
    int nd = 0;
    for (int k = lane; k < r; k += 32) {
      if (S.dead[k]) { ++nd; continue; }
      const float d = S.R[k * kRsLd + k];
      mx = fmaxf(mx, d); mn = fminf(mn, d); mr = fminf(mr, S.ratio[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mr = fminf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
    }
    nd = __reduce_add_sync(0xffffffffu, nd);
    if (lane == 0) { s_maxr = mx; s_minr = mn; s_minratio = mr; s_ndead = nd; }
  }
  inverse_panels(a, r, S);
  // R^-1 to global, dead columns zeroed
  float* Ri = mt.Rinv;
#pragma unroll
  for (int t = 0; t < kPanel; ++t) {
    const int i = warp * kPanel + t;
    if (i < r) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = lane + 32 * q;
        if (j < r) Ri[i * rp + j] = (j >= i && !S.dead[j]) ? a[t][q] : 0.f;
      }
    }
  }
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
  __shared__ __align__(16) float As[32][64 + 4];
  __shared__ __align__(16) float Bs[32][128];
  // A warp owns a 16-column strip (tx = column block of 8, ty = group of 4 rows), so the
  // chunks of R^-1 below its strip (rows k > its last column: zero) are skipped whole.
  const int tid = threadIdx.x, tx = tid >> 4, ty = tid & 15;
  const int warp_last_col = (tid >> 5) * 16 + 15;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  // 16-byte loads and stores when the row pitch and the buffers allow them (always in
  // the step: pitch rp a multiple of 16, workspace buffers 256-byte aligned); scalar ones
  // otherwise (a caller's 4-byte-aligned matrix in the one-matrix entry point).
  const bool vec = (rp & 3) == 0 &&
                   ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y) |
                     reinterpret_cast<uintptr_t>(mt.Rinv)) & 15) == 0;
  for (int k0 = 0; k0 < r; k0 += 32) {
    {
      const int rr = tid >> 2, kk = (tid & 3) * 8;
      const int64_t row = row0 + rr;
      float x[8];
      if (vec) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int k = k0 + kk + 4 * h;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row < m && k < rp) v = *reinterpret_cast<const float4*>(X + row * rp + k);
          x[4 * h] = v.x; x[4 * h + 1] = v.y; x[4 * h + 2] = v.z; x[4 * h + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = (row < m && k0 + kk + i < r) ? X[row * rp + k0 + kk + i] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) As[kk + i][rr] = (k0 + kk + i < r) ? x[i] * sc : 0.f;
    }
    {
      const int kk = tid >> 3, c = (tid & 7) * 16;
      const int k = k0 + kk;
      const float* rrow = mt.Rinv + (size_t)k * rp;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int cc = c + 4 * h;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < r) {
          if (vec) {
            if (cc < rp) v = *reinterpret_cast<const float4*>(rrow + cc);
          } else {
            v.x = cc < r ? rrow[cc] : 0.f;
            v.y = cc + 1 < r ? rrow[cc + 1] : 0.f;
            v.z = cc + 2 < r ? rrow[cc + 2] : 0.f;
            v.w = cc + 3 < r ? rrow[cc + 3] : 0.f;
          }
        }
        Bs[kk][cc] = cc < r ? v.x : 0.f;
        Bs[kk][cc + 1] = cc + 1 < r ? v.y : 0.f;
        Bs[kk][cc + 2] = cc + 2 < r ? v.z : 0.f;
        Bs[kk][cc + 3] = cc + 3 < r ? v.w : 0.f;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      if (k0 > warp_last_col) break;  // warp-uniform: R^-1 rows k0.. are zero in this strip
      float a[4], b[8];
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      a[0] = av.x; a[1] = av.y; a[2] = av.z; a[3] = av.w;
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
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = tx * 8 + j < r ? acc[i][j] : 0.f;
    if (vec) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = tx * 8 + 4 * h;
        if (c < rp)
          *reinterpret_cast<float4*>(Y + row * rp + c) = make_float4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (tx * 8 + j < rp) Y[row * rp + tx * 8 + j] = y[j];
    }
  }
}

constexpr size_t kCholSmem = sizeof(CholSmem);

}  // namespace

cudaError_t launch_orth(const Handle& h, const Plan& p, cudaStream_t s) {
  cudaFuncSetAttribute(k_chol, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCholSmem);
  const int BJ = p.B * p.J;
  for (int pass = 0; pass < kMaxPasses; ++pass) {
    k_gram<<<dim3(h.max_C, BJ), kGramThreads, 0, s>>>(p, pass);
    k_gsum<<<dim3((p.rp * p.rp + kT / 8 - 1) / (kT / 8), BJ), kT, 0, s>>>(p, pass);
    k_chol<<<BJ, kCholThreads, kCholSmem, s>>>(p, pass);
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
    k_gram<<<dim3(C, 1), kGramThreads, 0, s>>>(p, pass);
    k_gsum<<<dim3((p.rp * p.rp + kT / 8 - 1) / (kT / 8), 1), kT, 0, s>>>(p, pass);
    k_chol<<<1, kCholThreads, kCholSmem, s>>>(p, pass);
    k_apply<<<dim3(mtiles64, 1), kT, 0, s>>>(p, pass);
  }
  return cudaGetLastError();
}

}  // namespace psgd
