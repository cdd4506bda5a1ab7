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

// Column c of a row of the Gram staging tile sits at gram_slot(c): the first halves (4
// columns) of the 8-column blocks side by side, then the second halves. A warp's threads
// read the halves of up to 14 different blocks of one row, 16 bytes each, and in this
// order those are consecutive 16-byte words (no bank conflict); in plain column order
// every fourth block would share banks.
__device__ __forceinline__ int gram_slot(int c) { return ((c >> 2) & 1) * 64 + (c >> 3) * 4 + (c & 3); }

// acc += rows [q0, q0 + 32) of Xs restricted to columns 8 bi.. x columns 8 bj.., row by
// row in order.
__device__ __forceinline__ void gram_block_rows(const float (*Xs)[128], int bi, int bj, int q0,
                                                float (&acc)[8][8]) {
#pragma unroll 4
  for (int q = q0; q < q0 + 32; ++q) {
    float a[8], b[8];
    const float4 a0 = *reinterpret_cast<const float4*>(&Xs[q][bi * 4]);
    const float4 a1 = *reinterpret_cast<const float4*>(&Xs[q][64 + bi * 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&Xs[q][bj * 4]);
    const float4 b1 = *reinterpret_cast<const float4*>(&Xs[q][64 + bj * 4]);
    a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
    b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

// The whole 8 x 8 block, as two 16-byte stores per row when the pitch allows (rp is a
// multiple of 16 in the step). Entries past r or below the diagonal are sums like the
// others and are never read; rows and columns stay below rp (8 ceil(r / 8) <= rp).
__device__ __forceinline__ void gram_block_store(float* out, const float (&acc)[8][8], int bi,
                                                 int bj, int r, int rp) {
  if ((rp & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0 && bj * 8 + 8 <= rp && bi * 8 + 8 <= rp) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float* row = out + (size_t)(bi * 8 + i) * rp + bj * 8;
      *reinterpret_cast<float4*>(row) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(row + 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    return;
  }
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
      *reinterpret_cast<float4*>(&Xs[rr][gram_slot(c)]) =
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
      Xs[f >> 7][gram_slot(f & 127)] = v[u] * sc;
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
// One CTA of kCholWarps warps per matrix; r <= 128. The Gram matrix G sits in shared
// memory as A (both triangles), next to Z = I.
//
// Factorisation G = R^T R, right-looking by panels of 8 pivots:
//  1. Each of the 128 threads of warps 0..3 (the solver) factors the panel's 8 x 8 diagonal
//     block in its registers (all alike: no shuffle and no barrier on the chain of the 8
//     pivots). Pivot k is dead when it is <= dead_tol * diag0[k] (or not finite): row k of
//     R becomes e_k and column k takes no part in later updates.
//  2. The same threads solve for the panel's rows, one column each: R[k0+t][j] for j right
//     of the block (row t loses R[k0+s][k0+t] times the finished row s < t, then is
//     scaled by 1 / r_tt), and the panel's rows of Z with the same multipliers.
//     Elimination on [G | I] turns I into L^-1 = R^-T (L = R^T), so R^-1 = Z^T. Each
//     column's 8 entries of R also go to RT[j] (the panel rows, transposed), so that a
//     row's 8 multipliers below are two 16-byte loads.
//  3. Warps 4..15 subtract the rank-8 update from the rows below the panel, one row per
//     warp at a time: lane q owns the column quad [4q, 4q + 4) of [Z | A] (Z left of the
//     panel's end, A from there on, its upper triangle only) and keeps the panel's 8
//     entries of its quad in registers.
// One-panel lookahead: the update warps do the next panel's 8 rows first and signal the
// solver (named barrier 4: 384 arrivals, 128 waiting), which factors and solves the next
// panel while they update the remaining rows. One block barrier per panel.
constexpr int kCholWarps = 16;
constexpr int kCholThreads = kCholWarps * 32;
constexpr int kPanel = 8;
constexpr int kCLd = kRankBlock + 4;  // row pitch of A and Z in shared memory (16-byte rows)
static_assert(kRankBlock == 128 && kCholThreads >= kRankBlock, "one column per solver thread");

struct CholSmem {
  float A[kRankBlock * kCLd];  // G, rows turning into R
  float Z[kRankBlock * kCLd];  // I, rows turning into Z = R^-T
  float RT[2][kRankBlock][kPanel];  // panel p's rows of R, transposed, in RT[p % 2]: RT[.][j][t] = R[k0+t][j]
  float diag0[kRankBlock];     // diagonal of the unshifted Gram matrix
  float ratio[kRankBlock];     // pivot / diag0 (0 for dead pivots)
  int dead[kRankBlock];
  float trace, maxr, minr, minratio;  // block-wide scalars of one factorisation
  int ndead;
};

// A = G + shift I and Z = I on the leading r x r block, zeros elsewhere. The Gram sum holds
// the upper triangle; each thread mirrors the entries it loads. All of a thread's loads are
// issued before its first shared-memory store (a store between two loads through a plain
// pointer would make each load wait for the one before it).
__device__ __forceinline__ void chol_load(const MatMeta& mt, int r, int rp, float shift, CholSmem& S,
                                          bool record) {
  const float* src = mt.Gpart + (size_t)mt.C * rp * rp;
  constexpr int kPer = kRankBlock * kRankBlock / kCholThreads;  // 32 entries per thread
  float v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int idx = (int)threadIdx.x + kCholThreads * u, i = idx >> 7, j = idx & 127;
    v[u] = (j >= i && j < r) ? __ldcg(src + (size_t)i * rp + j) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int idx = (int)threadIdx.x + kCholThreads * u, i = idx >> 7, j = idx & 127;
    S.Z[i * kCLd + j] = (i == j && i < r) ? 1.f : 0.f;
    if (j >= i) {
      float g = v[u];
      if (i == j && i < r) {
        if (record) S.diag0[i] = g;
        g += shift;
      }
      S.A[i * kCLd + j] = g;
      S.A[j * kCLd + i] = g;
    }
  }
}

// Steps 1 and 2 for the panel at k0 (kb <= 8 pivots); threads 0..127, column c = thread.
__device__ __forceinline__ void chol_panel_solve(int k0, int kb, int r, float dead_tol, CholSmem& S) {
  float D[kPanel][kPanel], d0[kPanel];
  {  // the block's original diagonal, off the pivot chain
    const float4 lo = *reinterpret_cast<const float4*>(&S.diag0[k0]);
    const float4 hi = *reinterpret_cast<const float4*>(&S.diag0[k0 + 4]);
    d0[0] = lo.x; d0[1] = lo.y; d0[2] = lo.z; d0[3] = lo.w; d0[4] = hi.x; d0[5] = hi.y; d0[6] = hi.z; d0[7] = hi.w;
  }
#pragma unroll
  for (int s = 0; s < kPanel; ++s) {  // row s of the block: two 16-byte loads (k0 % 8 == 0)
    const float4 lo = *reinterpret_cast<const float4*>(&S.A[(k0 + s) * kCLd + k0]);
    const float4 hi = *reinterpret_cast<const float4*>(&S.A[(k0 + s) * kCLd + k0 + 4]);
    const float row[kPanel] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int t = 0; t < kPanel; ++t) D[s][t] = (t >= s && t < kb) ? row[t] : 0.f;
  }
  float inv[kPanel];
  bool dead[kPanel];
#pragma unroll
  for (int t = 0; t < kPanel; ++t) {
    inv[t] = 1.f;
    dead[t] = true;
    if (t < kb) {
      const float d = D[t][t];
      const bool bad = !(d > dead_tol * d0[t]) || !isfinite(d) || !(d0[t] > 0.f);
      const float iv = bad ? 1.f : rsqrtf(d);
      inv[t] = iv;
      dead[t] = bad;
      D[t][t] = bad ? 1.f : d * iv;  // r_kk
#pragma unroll
      for (int u = t + 1; u < kPanel; ++u) D[t][u] = bad ? 0.f : D[t][u] * iv;  // R[k0+t][k0+u]
#pragma unroll
      for (int u = t + 1; u < kPanel; ++u)
#pragma unroll
        for (int v = u; v < kPanel; ++v) D[u][v] = fmaf(-D[t][u], D[t][v], D[u][v]);
    }
  }
  const int c = threadIdx.x;
  if (c == 0) {  // the pivot records
#pragma unroll
    for (int t = 0; t < kPanel; ++t) {
      if (t < kb) {
        S.dead[k0 + t] = dead[t];
        S.ratio[k0 + t] = dead[t] ? 0.f : __fdividef(D[t][t] * D[t][t], d0[t]);  // statistics only
      }
    }
  }
  if (c < k0 + kPanel && c < r) {  // the panel's rows of Z (lower triangular: columns <= k0 + 7)
    float x[kPanel];
#pragma unroll
    for (int t = 0; t < kPanel; ++t) x[t] = t < kb ? S.Z[(k0 + t) * kCLd + c] : 0.f;
#pragma unroll
    for (int t = 0; t < kPanel; ++t) {
#pragma unroll
      for (int s2 = 0; s2 < t; ++s2) x[t] = fmaf(-D[s2][t], x[s2], x[t]);
      x[t] *= inv[t];
    }
#pragma unroll
    for (int t = 0; t < kPanel; ++t)
      if (t < kb) S.Z[(k0 + t) * kCLd + c] = x[t];
  }
  // The panel's rows of R from column k0 on, by forward substitution with the block's R.
  // Inside the block (c < k0 + 8) this repeats the factor's own FMAs in its order, so row
  // t <= c - k0 gets the block's value bit for bit (the diagonal: d / sqrt(d) as above);
  // rows below the block's diagonal get values that nothing reads.
  if (c >= k0 && c < r) {
    float x[kPanel];
#pragma unroll
    for (int t = 0; t < kPanel; ++t) x[t] = t < kb ? S.A[(k0 + t) * kCLd + c] : 0.f;
#pragma unroll
    for (int t = 0; t < kPanel; ++t) {
#pragma unroll
      for (int s2 = 0; s2 < t; ++s2) x[t] = fmaf(-D[s2][t], x[s2], x[t]);
      x[t] = (dead[t] && c != k0 + t) ? 0.f : (dead[t] ? 1.f : x[t] * inv[t]);
    }
#pragma unroll
    for (int t = 0; t < kPanel; ++t)
      if (t < kb) S.A[(k0 + t) * kCLd + c] = x[t];
    float* rt = S.RT[(k0 / kPanel) & 1][c];  // the update of this panel reads it while the next
    *reinterpret_cast<float4*>(rt) = make_float4(x[0], x[1], x[2], x[3]);  // panel's solve writes
    *reinterpret_cast<float4*>(rt + 4) = make_float4(x[4], x[5], x[6], x[7]);  // the other buffer
  }
}

// Step 3 for the full panel at k0 (8 pivots) on rows [i0, i1): A (upper triangle) and Z
// lose sum_t R[k0+t][i] times the panel's row t. The calling group of nw warps (w = this
// warp's index in it) takes rows i0 + w, i0 + w + nw, ... pv: the lane's quad of the
// panel's rows, loaded by chol_panel_quad.
__device__ __forceinline__ void chol_panel_quad(int k0, int r, CholSmem& S, float4 (&pv)[kPanel]) {
  const int c0 = 4 * (threadIdx.x & 31);
  const float* M = c0 < k0 + kPanel ? S.Z : S.A;
#pragma unroll
  for (int t = 0; t < kPanel; ++t)
    pv[t] = c0 < r ? *reinterpret_cast<const float4*>(&M[(k0 + t) * kCLd + c0]) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void chol_update_rows(int k0, int r, int i0, int i1, int w, int nw,
                                                 const float4 (&pv)[kPanel], CholSmem& S) {
  const int c0 = 4 * (threadIdx.x & 31);
  if (i0 >= i1 || c0 >= r) return;
  const bool zq = c0 < k0 + kPanel;
  float* M = zq ? S.Z : S.A;
  for (int i = i0 + w; i < i1; i += nw) {
    if (!zq && c0 + 3 < i) continue;  // wholly below the diagonal of A
    const float* rt = S.RT[(k0 / kPanel) & 1][i];
    const float4 cf0 = *reinterpret_cast<const float4*>(rt);  // R[k0 .. k0+3][i]
    const float4 cf1 = *reinterpret_cast<const float4*>(rt + 4);
    const float cf[kPanel] = {cf0.x, cf0.y, cf0.z, cf0.w, cf1.x, cf1.y, cf1.z, cf1.w};
    float4 v = *reinterpret_cast<const float4*>(&M[i * kCLd + c0]);
#pragma unroll
    for (int t = 0; t < kPanel; ++t) {
      v.x = fmaf(-cf[t], pv[t].x, v.x);
      v.y = fmaf(-cf[t], pv[t].y, v.y);
      v.z = fmaf(-cf[t], pv[t].z, v.z);
      v.w = fmaf(-cf[t], pv[t].w, v.w);
    }
    *reinterpret_cast<float4*>(&M[i * kCLd + c0]) = v;
  }
}

__device__ __forceinline__ void next_rows_ready_arrive() { asm volatile("bar.arrive 4, 512;" ::: "memory"); }
__device__ __forceinline__ void next_rows_ready_wait() { asm volatile("bar.sync 4, 512;" ::: "memory"); }

__device__ void chol_factor(int r, float dead_tol, CholSmem& S) {
  const int warp = threadIdx.x >> 5;
  const int npan = (r + kPanel - 1) / kPanel;
  if (threadIdx.x < kRankBlock) chol_panel_solve(0, min(kPanel, r), r, dead_tol, S);
  __syncthreads();
  for (int pn = 0; pn + 1 < npan; ++pn) {
    const int k0 = pn * kPanel, nxt = k0 + kPanel;
    const int nkb = min(kPanel, r - nxt);
    if (warp < 4) {
      next_rows_ready_wait();
      chol_panel_solve(nxt, nkb, r, dead_tol, S);
    } else {
      float4 pv[kPanel];
      chol_panel_quad(k0, r, S, pv);
      chol_update_rows(k0, r, nxt, nxt + nkb, warp - 4, kCholWarps - 4, pv, S);
      next_rows_ready_arrive();
      chol_update_rows(k0, r, nxt + kPanel, r, warp - 4, kCholWarps - 4, pv, S);
    }
    __syncthreads();
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

  chol_load(mt, r, rp, 0.f, S, true);
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
    __syncthreads();
  } else {
    chol_factor(r, last ? 0x1p-40f : 0x1p-16f, S);
    int nd = 0;
    for (int k = lane; k < r; k += 32) nd += S.dead[k];
    nd = __reduce_add_sync(0xffffffffu, nd);  // every warp computes the same count
    if (nd > 0 && !last) {
      shifted = true;
      const float shift = 0x1p-20f * sqrtf((float)mt.m) * trace;
      __syncthreads();  // every warp has read the dead flags
      chol_load(mt, r, rp, shift, S, false);
      __syncthreads();
      chol_factor(r, 0x1p-40f, S);
    }
  }
  // statistics of the factor: warp 0 reduces over the pivots
  if (warp == 0) {
    float mx = 0.f, mn = 3.4e38f, mr = 1.f;
    int nd = 0;
    for (int k = lane; k < r; k += 32) {
      if (S.dead[k]) { ++nd; continue; }
      const float d = S.A[k * kCLd + k];
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
  // R^-1 = Z^T to global, dead columns zeroed: R^-1[i][j] = Z[j][i] for j >= i, 0 below
  // the diagonal; r x r entries, four consecutive columns per thread.
  float* Ri = mt.Rinv;
  const bool vec = (rp & 3) == 0 && (reinterpret_cast<uintptr_t>(Ri) & 15) == 0;
  const int nq = (r + 3) / 4;
  for (int idx = threadIdx.x; idx < r * nq; idx += blockDim.x) {
    const int i = idx / nq, j0 = 4 * (idx - i * nq);
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      v[u] = (j < r && j >= i && S.dead[j] == 0) ? S.Z[j * kCLd + i] : 0.f;
    }
    float* row = Ri + (size_t)i * rp + j0;
    if (vec && j0 + 4 <= rp) {
      *reinterpret_cast<float4*>(row) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j0 + u < r) row[u] = v[u];
    }
  }
  __syncthreads();  // the statistics of warp 0
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
  // a strip wholly right of column r - 1 has no output: it skips every chunk
  const int warp_last_col = (tid >> 5) * 16 >= r ? -1 : (tid >> 5) * 16 + 15;
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
      Ys[rr][gram_slot(c)] = (live_row && c < r) ? acc[i][j] : 0.f;
    }
  }
  bar.sync();
  gram_tile(mt, Ys, red_apply, r, rp, tile, tid, bar);
}

}  // namespace
}  // namespace orthdev
}  // namespace psgd
