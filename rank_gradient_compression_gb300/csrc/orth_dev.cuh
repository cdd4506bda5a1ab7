// Device code of the fp32 orthonormalisation passes (adaptive shifted CholeskyQR), shared by
// the separate pass kernels of orth.cu and the cooperative one-launch version of orth_coop.cu.
//
// Every function that a 256-thread group runs takes the group's thread index `tid`
// (0..255) and a barrier policy: CtaBar (__syncthreads, the whole CTA is the group) or
// HalfBar (a named barrier over one half of a 512-thread CTA). Data that another CTA may
// have written earlier in the same launch (the cooperative kernel's earlier phases) is
// read with ld.global.cg, at L2: the L1 caches of different SMs are not coherent.
#pragma once

#include "handle.h"

namespace psgd {
namespace orthdev {
namespace {  // internal linkage: each translation unit keeps its own copy

constexpr int kT = 256;  // threads of one work group

__device__ __forceinline__ int ld_int(const int* p) { return __ldcg(p); }

__device__ __forceinline__ float* buf_ptr(const MatMeta& mt, int idx) {
  return idx == 0 ? mt.P : idx == 1 ? mt.Xa : idx == 2 ? mt.Xb : mt.Phat;
}

// The block's columns in the buffer a pass reads: P (or, for a column block projected off
// the earlier blocks, Xa) in pass 0, else the previous pass's output.
__device__ __forceinline__ const float* pass_src(const Plan& p, const MatMeta& mt, int pass) {
  const float* base = pass == 0 ? (p.ob_src0 ? mt.Xa : mt.P) : buf_ptr(mt, ld_int(mt.ostate + (pass - 1) * 4 + 1));
  return base + p.ob_c0;
}

// Power-of-two scale that brings max|P| into [1, 2): exact.
__device__ __forceinline__ float p_scale(const MatMeta& mt) {
  const unsigned bits = __ldcg(reinterpret_cast<const unsigned*>(mt.scal) + 1);
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
    if (ld_int(mt.ostate + q * 4) != 0) return true;
  return false;
}

// Block b (0 <= b < nb (nb + 1) / 2) of the upper triangle of an nb x nb grid of 8 x 8
// blocks, numbered row by row: (bi, bj) with bi <= bj.
__device__ __forceinline__ void block_coords(int b, int nb, int& bi, int& bj) {
  int i = 0, rem = b;
  while (i < nb && rem >= nb - i) { rem -= nb - i; ++i; }
  bi = i;
  bj = i + rem;
}

// acc += rows [q0, q0 + 32) of Xs restricted to columns 8 bi.. x columns 8 bj.., row by
// row in order.
__device__ __forceinline__ void gram_block_rows(const float (*Xs)[128], int bi, int bj, int q0,
                                                float (&acc)[8][8]) {
#pragma unroll 4
  for (int q = q0; q < q0 + 32; ++q) {
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

__device__ __forceinline__ void gram_block_store(float* out, const float (&acc)[8][8], int bi,
                                                 int bj, int r, int rp) {
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

// Upper triangle of X^T X for one 64-row chunk held in shared memory (Xs: 64 x 128, zero
// past r and past the end of the matrix) into Gram partial `chunk`, in 8 x 8 blocks
// (nb = ceil(r / 8), nb (nb + 1) / 2 <= 136 blocks). All 256 threads of the group call it
// (it holds group barriers). Thread t takes block t mod 128 and sums rows
// [32 h, 32 h + 32) of the chunk in order, h = t / 128; the upper half's sums are added to
// the lower half's through `red` (32 x 128 floats), four rows of the block at a time.
// Blocks 128 and up (r > 120 only) are summed over all 64 rows by the upper half alone.
// The partial is a fixed function of the chunk, whichever kernel calls this.
template <class Bar>
__device__ void gram_tile(const MatMeta& mt, const float (*Xs)[128], float* red, int r, int rp,
                          int chunk, int tid, const Bar& bar) {
  const int nb = (r + 7) / 8, nblk = nb * (nb + 1) / 2;
  const int h = tid >> 7, b = tid & 127;
  float* out = mt.Gpart + (size_t)chunk * rp * rp;
  const bool live = b < nblk;
  int bi = 0, bj = 0;
  if (live) block_coords(b, nb, bi, bj);
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  if (live) gram_block_rows(Xs, bi, bj, 32 * h, acc);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (h == 1 && live) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) red[(i * 8 + j) * 128 + b] = acc[4 * half + i][j];
    }
    bar.sync();
    if (h == 0 && live) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          acc[4 * half + i][j] = __fadd_rn(acc[4 * half + i][j], red[(i * 8 + j) * 128 + b]);
    }
    bar.sync();
  }
  if (h == 0 && live) gram_block_store(out, acc, bi, bj, r, rp);
  if (h == 1 && 128 + b < nblk) {
    block_coords(128 + b, nb, bi, bj);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    gram_block_rows(Xs, bi, bj, 0, acc);
    gram_block_rows(Xs, bi, bj, 32, acc);
    gram_block_store(out, acc, bi, bj, r, rp);
  }
}

// Gram partial of 64-row chunk `chunk`: Gpart[chunk] = X_c^T X_c (upper triangle; the lower
// one is neither written nor read). The chunk is staged in shared memory (Xs: 64 x 128,
// red: 32 x 128 floats) with all of a thread's loads issued before its stores.
template <class Bar>
__device__ void gram_chunk(const Plan& p, const MatMeta& mt, int pass, int chunk, float (*Xs)[128],
                           float* red, int tid, const Bar& bar) {
  const int64_t m = mt.m;
  const int r = p.ob_r, rp = p.ob_rp, xl = p.rp;  // block width, Gram pitch, X row pitch
  const float* X = pass_src(p, mt, pass);
  const float sc = pass == 0 ? p_scale(mt) : 1.0f;
  const int64_t row0 = (int64_t)chunk * kGramRows;
  if ((xl & 3) == 0 && (reinterpret_cast<uintptr_t>(X) & 15) == 0) {
    float4 v[8];  // 64 rows x 32 float4
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int f = tid + kT * u, rr = f >> 5, c = (f & 31) * 4;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row0 + rr < m && c < r) v[u] = __ldcg(reinterpret_cast<const float4*>(X + (row0 + rr) * xl + c));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int f = tid + kT * u, rr = f >> 5, c = (f & 31) * 4;
      *reinterpret_cast<float4*>(&Xs[rr][c]) =
          make_float4(c < r ? v[u].x * sc : 0.f, c + 1 < r ? v[u].y * sc : 0.f,
                      c + 2 < r ? v[u].z * sc : 0.f, c + 3 < r ? v[u].w * sc : 0.f);
    }
  } else {
    float v[32];  // 64 rows x 128 floats
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int f = tid + kT * u, rr = f >> 7, c = f & 127;
      v[u] = (row0 + rr < m && c < r) ? __ldcg(X + (row0 + rr) * xl + c) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int f = tid + kT * u;
      Xs[f >> 7][f & 127] = v[u] * sc;
    }
  }
  bar.sync();
  gram_tile(mt, Xs, red, r, rp, chunk, tid, bar);
}

// Number of (row, 32-column segment) items of the Gram sum: rp * ceil(rp / 32).
__device__ __forceinline__ int gsum_items(int rp) { return rp * ((rp + 31) / 32); }

// G = sum_c Gpart[c] into slot C of Gpart (upper triangle), for item `blk`: 32 consecutive
// entries of one row of G. Warp w of the group sums the partials c = w, w + 8, ... in
// order (one 128-byte load per partial), and the eight warp sums are added in warp order
// through part (8 x 32 floats of shared memory).
template <class Bar>
__device__ void gsum_item(const Plan& p, const MatMeta& mt, int blk, float (*part)[32], int tid,
                          const Bar& bar) {
  const int rp = p.ob_rp;
  const int nseg = (rp + 31) / 32;
  const int i = blk / nseg, j0 = (blk - i * nseg) * 32;
  const bool any = i < rp && j0 + 31 >= i;  // not wholly below the diagonal (group-uniform)
  if (!any) return;
  const int warp = tid >> 5, lane = tid & 31;
  const int j = j0 + lane;
  const bool live = j < rp && j >= i;
  const size_t slot = (size_t)rp * rp;
  const float* src = mt.Gpart + (size_t)i * rp + j;
  float s = 0.f;
  if (live) {
    const int C = mt.C;
    for (int c0 = warp; c0 < C; c0 += 8 * 16) {  // 16 loads in flight, then 16 adds in order
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = c0 + 8 * u;
        v[u] = c < C ? __ldcg(src + (size_t)c * slot) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (c0 + 8 * u < C) s = __fadd_rn(s, v[u]);
    }
  }
  part[warp][lane] = s;
  bar.sync();
  if (warp == 0 && live) {
    float t = part[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) t = __fadd_rn(t, part[w][lane]);
    mt.Gpart[(size_t)mt.C * slot + (size_t)i * rp + j] = t;
  }
  bar.sync();  // part is reused by the group's next item
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
// R^-1 in the same sweep: elimination on [G | I] turns the identity into L^-1 = R^-T with
// L = R^T. Each warp also holds its rows of Z (initially I) in registers; the owner warp
// scales its Z rows by 1/r_kk and updates them with the same multipliers as its G rows,
// publishes them next to the R rows, and the later warps subtract the same multiples
// from their Z rows. R^-1 = Z^T. One block barrier per 8 rows in all.
constexpr int kCholWarps = 16;
constexpr int kCholThreads = kCholWarps * 32;
constexpr int kPanel = 8;
static_assert(kCholWarps * kPanel >= kRankBlock, "every row needs an owner warp");
constexpr int kRsLd = kRankBlock + 1;  // row stride of R in shared memory

struct CholSmem {
  float R[kRankBlock * kRsLd];           // rows of R as they are finished
  float X[2][kPanel * kRsLd];          // published rows of Z = R^-T (ping-pong by panel)
  float diag0[kRankBlock];               // diagonal of the unshifted Gram matrix
  float ratio[kRankBlock];               // pivot / diag0 (0 for dead pivots)
  int dead[kRankBlock];
  float trace, maxr, minr, minratio;    // block-wide scalars of one factorisation
  int ndead;
};

// Warp w holds rows i in [8w, 8w + 8) of G (becoming R) in a[t][q] and of Z = R^-T in
// z[t][q], column j = lane + 32 q. One code body for every warp, with the loops that
// only address shared memory kept rolled: a per-warp specialisation of the register
// arrays would be smaller in arithmetic but overflows the instruction cache.
__device__ __forceinline__ float sel4(const float (&v)[4], int q) {  // q warp-uniform
  return q == 0 ? v[0] : q == 1 ? v[1] : q == 2 ? v[2] : v[3];
}

__device__ __forceinline__ void load_gram_rows(const MatMeta& mt, int r, int rp,
                                               float (&a)[kPanel][4], float shift, CholSmem& S,
                                               bool record) {
  const float* src = mt.Gpart + (size_t)mt.C * rp * rp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kPanel; ++t) {  // all loads first (upper triangle)
    const int i = warp * kPanel + t;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      a[t][q] = (i < r && j < r && j >= i) ? __ldcg(src + (size_t)i * rp + j) : 0.f;
    }
  }
  const int qw = warp >> 2;  // the diagonal of row i sits in group i / 32 = warp / 4
#pragma unroll
  for (int t = 0; t < kPanel; ++t) {
    const int i = warp * kPanel + t;
    if (i < r && lane == (i & 31)) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q == qw) {
          if (record) S.diag0[i] = a[t][q];
          a[t][q] += shift;
        }
    }
  }
}

__device__ __forceinline__ void identity_rows(float (&z)[kPanel][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kPanel; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) z[t][q] = (warp * kPanel + t == lane + 32 * q) ? 1.f : 0.f;
}

// Factor the registers' panels in place (a: rows of G -> R; z: rows of I -> Z = R^-T) and
// fill S.R, S.dead, S.ratio.
__device__ void cholesky_panels(float (&a)[kPanel][4], float (&z)[kPanel][4], int r,
                                float dead_tol, CholSmem& S) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npan = (r + kPanel - 1) / kPanel;
  for (int pn = 0; pn < npan; ++pn) {
    const int k0 = pn * kPanel;
    const int qg = pn >> 2;  // column group of this panel's pivots
    float* Zp = S.X[pn & 1];
    if (warp == pn) {  // the owner
      // The panel's 8 x 8 diagonal block reaches every lane in one round of shuffles
      // (upper triangle; columns k0.. sit in group qg at lanes l0..l0+7), and every lane
      // factors it in registers: no shuffle lies on the chain of the 8 pivots.
      const int nk = min(kPanel, r - k0);
      const int l0 = k0 & 31;
      float D[kPanel][kPanel];
#pragma unroll
      for (int s = 0; s < kPanel; ++s) {
        const float v = sel4(a[s], qg);
#pragma unroll
        for (int t = s; t < kPanel; ++t) D[s][t] = __shfl_sync(0xffffffffu, v, l0 + t);
      }
      float inv[kPanel];
      bool dead[kPanel];
#pragma unroll
      for (int t = 0; t < kPanel; ++t) {
        inv[t] = 1.f;
        dead[t] = true;
        if (t < nk) {
          const float d = D[t][t];
          const float d0 = S.diag0[k0 + t];
          const bool bad = !(d > dead_tol * d0) || !isfinite(d) || !(d0 > 0.f);
          const float iv = bad ? 1.f : rsqrtf(d);
          inv[t] = iv;
          dead[t] = bad;
          D[t][t] = bad ? 1.f : d * iv;  // r_kk
#pragma unroll
          for (int u = t + 1; u < kPanel; ++u) D[t][u] = bad ? 0.f : D[t][u] * iv;  // R[t][u]
#pragma unroll
          for (int u = t + 1; u < kPanel; ++u)
#pragma unroll
            for (int v = u; v < kPanel; ++v) D[u][v] = fmaf(-D[t][u], D[t][v], D[u][v]);
          if (lane == 0) {
            S.dead[k0 + t] = bad;
            S.ratio[k0 + t] = bad ? 0.f : __fdividef(d, d0);  // statistics only
          }
        }
      }
      // The panel's rows of R and Z by forward substitution with the block's R: row t
      // loses R[s][t] times the finished row s (s < t), then is scaled by 1 / r_tt. These
      // are the right-looking panel updates, in the same order.
#pragma unroll
      for (int t = 0; t < kPanel; ++t) {
        if (t < nk) {
          const int k = k0 + t;
#pragma unroll
          for (int s2 = 0; s2 < t; ++s2) {
            const float c = D[s2][t];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              a[t][q] = fmaf(-c, a[s2][q], a[t][q]);
              z[t][q] = fmaf(-c, z[s2][q], z[t][q]);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = lane + 32 * q;
            a[t][q] = j < k ? 0.f : (j == k ? D[t][t] : (dead[t] ? 0.f : a[t][q] * inv[t]));
            z[t][q] *= inv[t];
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kPanel; ++t)
        if (k0 + t < r) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            S.R[(k0 + t) * kRsLd + lane + 32 * q] = a[t][q];
            Zp[t * kRsLd + lane + 32 * q] = z[t][q];
          }
        }
    }
    __syncthreads();
    if (warp > pn && warp * kPanel < r) {  // warps whose rows all lie past r have nothing to update
      const int kend = min(kPanel, r - k0);
      const int i0 = warp * kPanel;
      // Only columns j >= i0 of G's rows matter (upper triangle), and Z = R^-T's rows are 0
      // past column i0 + 7 (lower triangle, from identity rows). Both limits fall in column
      // group qa = i0 / 32, so G's groups below qa and Z's groups above it are left as
      // they are: 5 of the 8 groups are updated.
      const int qa = i0 >> 5;
#pragma unroll 1
      for (int pp = 0; pp < kend; ++pp) {
        const float* Rk = S.R + (k0 + pp) * kRsLd;
        const float* Zk = Zp + pp * kRsLd;
        float rj[4], zj[4], c[kPanel];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          rj[q] = q >= qa ? Rk[lane + 32 * q] : 0.f;
          zj[q] = q <= qa ? Zk[lane + 32 * q] : 0.f;
        }
#pragma unroll
        for (int t = 0; t < kPanel; ++t) c[t] = Rk[i0 + t];
#pragma unroll
        for (int t = 0; t < kPanel; ++t) {  // rows i >= r hold zeros and stay unused
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q >= qa) a[t][q] = fmaf(-c[t], rj[q], a[t][q]);
            if (q <= qa) z[t][q] = fmaf(-c[t], zj[q], z[t][q]);
          }
        }
      }
    }
  }
}

// One CTA (kCholThreads threads, the whole CTA) per matrix: factor the Gram matrix of this
// pass, decide shift/final, write R^-1 and the pass record. Every branch that holds a block
// barrier is uniform over the block. The caller has checked that the pass runs.
__device__ void chol_matrix(const Plan& p, const MatMeta& mt, int pass, CholSmem& S) {
  const int r = p.ob_r, rp = p.ob_rp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool last = pass == kMaxPasses - 1;
  int* st = mt.ostate + pass * 4;
  const int src = pass == 0 ? 0 : ld_int(mt.ostate + (pass - 1) * 4 + 1);

  float a[kPanel][4], z[kPanel][4];
  identity_rows(z);
  load_gram_rows(mt, r, rp, a, 0.f, S, true);
  __syncthreads();
  if (warp == 0) {  // trace: fixed-order warp reduction
    float t = 0.f;
    for (int k = lane; k < r; k += 32) t += S.diag0[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) S.trace = t;
  }
  __syncthreads();
  const float trace = S.trace;
  bool shifted = false;
  if (!(trace > 0.f) || !isfinite(trace)) {
    for (int k = threadIdx.x; k < r; k += blockDim.x) { S.dead[k] = 1; S.ratio[k] = 0.f; }
    for (int idx = threadIdx.x; idx < r * kRsLd; idx += blockDim.x) {
      const int i = idx / kRsLd, j = idx - i * kRsLd;
      S.R[idx] = (i == j) ? 1.f : 0.f;
    }
    __syncthreads();
  } else {
    cholesky_panels(a, z, r, last ? 0x1p-40f : 0x1p-16f, S);
    __syncthreads();
    int nd = 0;
    for (int k = lane; k < r; k += 32) nd += S.dead[k];
    nd = __reduce_add_sync(0xffffffffu, nd);  // every warp computes the same count
    if (nd > 0 && !last) {
      shifted = true;
      const float shift = 0x1p-20f * sqrtf((float)mt.m) * trace;
      load_gram_rows(mt, r, rp, a, shift, S, false);
      identity_rows(z);
      __syncthreads();
      cholesky_panels(a, z, r, 0x1p-40f, S);
      __syncthreads();
    }
  }
  // statistics of the factor: warp 0 reduces over the pivots
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
    if (lane == 0) { S.maxr = mx; S.minr = mn; S.minratio = mr; S.ndead = nd; }
  }
  // R^-1 = Z^T to global, dead columns zeroed: this warp's Z rows j = 8 warp + t are R^-1's
  // columns j, so each thread holds 8 consecutive entries of R^-1 rows i = lane + 32 q,
  // written as two 16-byte stores when the pitch and the base allow.
  float* Ri = mt.Rinv;
  const int j0 = warp * kPanel;
  if (j0 < r) {
    bool live[kPanel];
#pragma unroll
    for (int t = 0; t < kPanel; ++t) live[t] = j0 + t < r && S.dead[j0 + t] == 0;
    const bool vec = j0 + kPanel <= r && (rp & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(Ri) & 15) == 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = lane + 32 * q;
      if (i >= r) continue;
      float v[kPanel];
#pragma unroll
      for (int t = 0; t < kPanel; ++t) v[t] = (i <= j0 + t && live[t]) ? z[t][q] : 0.f;
      float* row = Ri + (size_t)i * rp + j0;
      if (vec) {
        *reinterpret_cast<float4*>(row) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(row + 4) = make_float4(v[4], v[5], v[6], v[7]);
      } else {
#pragma unroll
        for (int t = 0; t < kPanel; ++t)
          if (j0 + t < r) row[t] = v[t];
      }
    }
  }
  if (threadIdx.x == 0) {
    const bool nearly_orth = !shifted && S.ndead == 0 && S.minratio >= 0.5f &&
                             S.maxr <= 2.f * S.minr;
    const bool all_dead = S.ndead == r;
    const int fin = (last || nearly_orth || all_dead) ? 1 : 0;
    st[0] = fin;
    st[1] = fin ? 3 : (src == 1 ? 2 : 1);
    st[2] = shifted ? 1 : 0;
    st[3] = S.ndead;
  }
}


// X <- X R^-1 on the 64-row tile `tile` (R^-1 upper triangular, r <= 128), then, unless the
// pass is final, the next pass's Gram partial of the same rows. smem: 64 x 128 floats for
// the operand chunks (then the Y tile), red: gram_tile's 32 x 128 reduction buffer.
//
// kAcc: every entry of X R^-1 is accumulated as a compensated dot product (dot2_acc) and
// rounded once. The span of the result is what the step keeps: any invertible R leaves
// span(X R^-1) = span(X) in exact arithmetic, so only the rounding of this product can move
// the subspace. Plain fp32 sums lose up to u * |X| |R^-1| per entry, which is cond(X)
// times the entry itself when the columns of X are nearly dependent (a warm-started P at
// high rank, column-scaled condition number up to ~4e5 at r = 896 on a 1/k spectrum).
// Compensated, each output column is within about u of its exact value relative to its
// own size, the same as rounding P to fp32 once. The blocked orthonormalisation of ranks
// above 128 uses it; at r <= 128 (warm-started P nearly orthogonal, one pass) the plain sum
// is within the tolerance and half the instructions.
template <bool kAcc, class Bar>
__device__ void apply_tile(const Plan& p, const MatMeta& mt, int pass, int tile, float* smem_apply,
                           float* red_apply, int tid, const Bar& bar) {
  const int64_t m = mt.m;
  const int r = p.ob_r, rp = p.ob_rp, xl = p.rp;  // block width, R^-1 pitch, X/Y row pitch
  const int64_t row0 = (int64_t)tile * 64;
  if (row0 >= m) return;
  const float* X = pass_src(p, mt, pass);
  float* Y = buf_ptr(mt, ld_int(mt.ostate + pass * 4 + 1)) + p.ob_c0;
  const float sc = pass == 0 ? p_scale(mt) : 1.0f;
  // As and Bs hold the operand chunks of the product; afterwards the same shared memory
  // holds this tile of Y for the next pass's Gram partial.
  float (*As)[64 + 4] = reinterpret_cast<float (*)[64 + 4]>(smem_apply);
  float (*Bs)[128] = reinterpret_cast<float (*)[128]>(smem_apply + 32 * (64 + 4));
  float (*Ys)[128] = reinterpret_cast<float (*)[128]>(smem_apply);
  // A warp owns a 16-column strip (tx = column block of 8, ty = group of 4 rows), so the
  // chunks of R^-1 below its strip (rows k > its last column: zero) are skipped whole.
  const int tx = tid >> 4, ty = tid & 15;
  const int warp_last_col = (tid >> 5) * 16 + 15;
  float acc[4][8], lo[4][8];  // lo: compensation terms (kAcc only)
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = lo[i][j] = 0.f;
  // 16-byte loads and stores when the row pitch and the buffers allow them (always in
  // the step: pitch rp a multiple of 16, workspace buffers 256-byte aligned); scalar ones
  // otherwise (a caller's 4-byte-aligned matrix in the one-matrix entry point).
  const bool vec = (xl & 3) == 0 && (rp & 3) == 0 &&
                   ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y) |
                     reinterpret_cast<uintptr_t>(mt.Rinv)) & 15) == 0;
  // One 32-wide k chunk: this thread's 8 entries of X (row xr, columns k0 + xk ..) and 16
  // of R^-1 (row k0 + bk, columns bc ..). The next chunk's loads go out before the FMAs
  // of the current one, and every load of a chunk before its shared-memory stores.
  const int xr = tid >> 2, xk = (tid & 3) * 8, bk = tid >> 3, bc = (tid & 7) * 16;
  const int64_t xrow = row0 + xr;
  float xv[8], bv[16];
  auto load_chunk = [&](int k0) {
    const int k = k0 + bk;
    const float* rrow = mt.Rinv + (size_t)k * rp;
    if (vec) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kx = k0 + xk + 4 * h;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (xrow < m && kx < rp) v = __ldcg(reinterpret_cast<const float4*>(X + xrow * xl + kx));
        xv[4 * h] = v.x; xv[4 * h + 1] = v.y; xv[4 * h + 2] = v.z; xv[4 * h + 3] = v.w;
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int cc = bc + 4 * h;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < r && cc < rp) v = __ldcg(reinterpret_cast<const float4*>(rrow + cc));
        bv[4 * h] = v.x; bv[4 * h + 1] = v.y; bv[4 * h + 2] = v.z; bv[4 * h + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        xv[i] = (xrow < m && k0 + xk + i < r) ? __ldcg(X + xrow * xl + k0 + xk + i) : 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) bv[i] = (k < r && bc + i < r) ? __ldcg(rrow + bc + i) : 0.f;
    }
  };
  auto store_chunk = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) As[xk + i][xr] = (k0 + xk + i < r) ? xv[i] * sc : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) Bs[bk][bc + i] = bc + i < r ? bv[i] : 0.f;
  };
  load_chunk(0);
  for (int k0 = 0; k0 < r; k0 += 32) {
    store_chunk(k0);
    bar.sync();
    if (k0 + 32 < r) load_chunk(k0 + 32);
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
        for (int j = 0; j < 8; ++j) {
          if (kAcc) dot2_acc(acc[i][j], lo[i][j], a[i], b[j]);
          else acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    bar.sync();
  }
  if (kAcc) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = __fadd_rn(acc[i][j], lo[i][j]);
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
          *reinterpret_cast<float4*>(Y + row * xl + c) = make_float4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (tx * 8 + j < rp) Y[row * xl + tx * 8 + j] = y[j];
    }
  }
  // The next pass's Gram partial of this 64-row chunk (the Gram chunking is 64 rows, so
  // chunk = tile), unless this pass is the last one. Same rows, same order and same FMA
  // chains as k_gram would use on the stored Y: the partial is bit for bit the same.
  if (ld_int(mt.ostate + pass * 4) != 0 || pass + 1 >= kMaxPasses) return;
  bar.sync();  // As and Bs are dead; Ys overlays them
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = ty * 4 + i;
    const bool live_row = row0 + rr < m;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = tx * 8 + j;
      Ys[rr][c] = (live_row && c < r) ? acc[i][j] : 0.f;
    }
  }
  bar.sync();
  gram_tile(mt, Ys, red_apply, r, rp, tile, tid, bar);
}

}  // namespace
}  // namespace orthdev
}  // namespace psgd
