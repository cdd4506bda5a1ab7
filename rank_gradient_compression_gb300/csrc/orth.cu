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
// factor 2) is the last one. After a warm start P is usually close to orthogonal and one
// pass is final; otherwise CholeskyQR2 (two passes) is the common case. Columns whose
// pivot vanishes are numerically dependent; their column of R^-1 is zeroed. That
// leaves a zero column in P^ and the projector P^ P^T onto span(P) unchanged.
//
// Device pass state: ostate[pass] = {final, dst buffer, shifted, dead columns}, written
// by the pass's Cholesky kernel. The next pass reads it after the launch boundary.
#include <algorithm>

#include "orth_dev.cuh"

namespace psgd {
namespace {

using namespace orthdev;

// One kernel per phase of a pass (the step of ranks above 128, and the one-matrix entry
// point); the cooperative kernel of orth_coop.cu runs the same device code in one launch.

// Gram partial of one 64-row chunk. grid = (max C, B*J), block kT.
static_assert(kGramRows == 64, "gram_tile sums 64-row chunks");
__global__ void __launch_bounds__(kT) k_gram(Plan p, int pass) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  if ((int)blockIdx.x >= mt.C || pass_skipped(p, mt, pass)) return;
  __shared__ __align__(16) float Xs[kGramRows][128];
  __shared__ __align__(16) float red[32 * 128];
  gram_chunk(p, mt, pass, blockIdx.x, Xs, red, threadIdx.x, CtaBar{});
}

// G = sum of the Gram partials. grid = (gsum_items(rp), B*J).
__global__ void __launch_bounds__(kT) k_gsum(Plan p, int pass) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  if (pass_skipped(p, mt, pass)) return;
  __shared__ float part[8][32];
  gsum_item(p, mt, blockIdx.x, part, threadIdx.x, CtaBar{});
}

// Cholesky and R^-1, one CTA per matrix.
__global__ void __launch_bounds__(kCholThreads, 1) k_chol(Plan p, int pass) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.x];
  if (pass_skipped(p, mt, pass)) return;
  extern __shared__ __align__(16) unsigned char chol_smem[];
  chol_matrix(p, mt, pass, *reinterpret_cast<CholSmem*>(chol_smem));
}

// X <- X R^-1 on 64-row tiles (and the next pass's Gram partials). grid = (ceil(m/64), B*J).
template <bool kAcc>
__global__ void __launch_bounds__(kT) k_apply(Plan p, int pass) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  if (pass_skipped(p, mt, pass)) return;
  __shared__ __align__(16) float smem_apply[64 * 128];
  __shared__ __align__(16) float red_apply[32 * 128];
  apply_tile<kAcc>(p, mt, pass, blockIdx.x, smem_apply, red_apply, threadIdx.x, CtaBar{});
}

// ---------------------------------------------------------------- block Gram-Schmidt
// For r > kRankBlock the columns are orthonormalised in blocks of kRankBlock: block
// classical Gram-Schmidt with one re-orthogonalisation (the first projection is repeated
// on its own result), then the CholeskyQR passes above on the projected block. A
// projection of block [c0, c0 + rb) of a source S (P, or Xa) off the finished columns
// P^[:, 0 .. c0):
//   C = P^[:, <c0]^T S_blk (c0 x rb): row-chunk partials (the Gram chunking), summed in a
//       fixed order into the slot after the partials (Gpart holds them: c0 * 128 < rp^2);
//   Xa_blk = S_blk - P^[:, <c0] C.

// C partials of one row chunk, one 128 x 128 tile of C per CTA (16 x 16 threads, 8 x 8 each).
// grid = (max C, ceil(c0 / 128), B*J).
__global__ void __launch_bounds__(kT) k_proj_coef(Plan p, int c0, int rb, int src_xa) {
  const MatMeta& mt = p.meta[blockIdx.z];
  if ((int)blockIdx.x >= mt.C || p.skip[mt.b]) return;
  const int64_t m = mt.m;
  const int xl = p.rp;
  const int q0 = blockIdx.y * 128, qn = min(128, c0 - q0);
  const float* Qh = mt.Phat + q0;
  const float* S = (src_xa ? mt.Xa : mt.P) + c0;
  const int64_t rows_per = ((m + mt.C - 1) / mt.C + 31) / 32 * 32;
  const int64_t rbeg = (int64_t)blockIdx.x * rows_per, rend = min(m, rbeg + rows_per);
  __shared__ __align__(16) float As[32][128];
  __shared__ __align__(16) float Bs[32][128];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int64_t k0 = rbeg; k0 < rend; k0 += 32) {
    for (int idx = tid; idx < 32 * 128; idx += kT) {
      const int kk = idx >> 7, c = idx & 127;
      const int64_t row = k0 + kk;
      As[kk][c] = (row < rend && c < qn) ? Qh[row * xl + c] : 0.f;
      Bs[kk][c] = (row < rend && c < rb) ? S[row * xl + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int q = 0; q < 32; ++q) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&As[q][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[q][ty * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[q][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[q][tx * 8 + 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = mt.Gpart + (size_t)blockIdx.x * c0 * 128;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ii = ty * 8 + i;
    if (ii >= qn) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int jj = tx * 8 + j;
      if (jj < rb) out[(size_t)(q0 + ii) * 128 + jj] = acc[i][j];
    }
  }
}

// C = sum over the row chunks of the partials (fixed order) into the slot after them.
// grid = (ceil(c0 * 128 / 32), B*J); eight threads per entry as in k_gsum.
__global__ void __launch_bounds__(kT) k_proj_sum(Plan p, int c0, int rb) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const int idx = blockIdx.x * (kT / 8) + (threadIdx.x >> 3);
  const int part = threadIdx.x & 7;
  const bool live = idx < c0 * 128 && (idx & 127) < rb;
  const float* src = mt.Gpart + (live ? idx : 0);
  const size_t slot = (size_t)c0 * 128;
  float s = 0.f;
  if (live) {
#pragma unroll 8
    for (int c = part; c < mt.C; c += 8) s = __fadd_rn(s, __ldg(src + (size_t)c * slot));
  }
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2));
  s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 4));
  if (live && part == 0) mt.Gpart[(size_t)mt.C * slot + idx] = s;
}

// Xa_blk = S_blk - P^[:, <c0] C on 64-row tiles (16 x 16 threads: 4 rows x 8 columns
// each; K = c0 in chunks of 32). S may be Xa itself: a CTA reads the rows of S it writes
// only at its end, and no other CTA touches them. grid = (ceil(m / 64), B*J).
// Adding multiples of the finished columns to S_blk leaves span(P^[:, <c0], S_blk)
// unchanged whatever C is, so the subspace moves only by the rounding of this update. It
// is a compensated dot product (dot2_acc) and one exactly rounded subtraction (TwoSum),
// so each entry is within about u of S - P^ C relative to itself, also where the block
// is nearly inside the span of the finished columns and the subtraction cancels.
__global__ void __launch_bounds__(kT) k_proj_apply(Plan p, int c0, int rb, int src_xa) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const int64_t m = mt.m;
  const int xl = p.rp;
  const int64_t row0 = (int64_t)blockIdx.x * 64;
  if (row0 >= m) return;
  const float* S = (src_xa ? mt.Xa : mt.P) + c0;
  float* Y = mt.Xa + c0;
  const float* Cf = mt.Gpart + (size_t)mt.C * c0 * 128;  // c0 x 128, pitch 128
  __shared__ __align__(16) float As[32][64 + 4];
  __shared__ __align__(16) float Bs[32][128];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][8], lo[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = lo[i][j] = 0.f;
  for (int k0 = 0; k0 < c0; k0 += 32) {
    {
      const int rr = tid >> 2, kk = (tid & 3) * 8;
      const int64_t row = row0 + rr;
#pragma unroll
      for (int i = 0; i < 8; ++i) As[kk + i][rr] = row < m ? mt.Phat[row * xl + k0 + kk + i] : 0.f;
    }
    {
      const int kk = tid >> 3, c = (tid & 7) * 16;
#pragma unroll
      for (int i = 0; i < 16; ++i) Bs[kk][c + i] = c + i < rb ? Cf[(size_t)(k0 + kk) * 128 + c + i] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float a[4] = {av.x, av.y, av.z, av.w};
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 8 + 4]);
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) dot2_acc(acc[i][j], lo[i][j], a[i], b[j]);
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
      if (c < rb) {
        // (S - hi) exactly as a sum of two floats, then the small terms, one rounding each
        const float sv = S[row * xl + c], nh = -acc[i][j];
        const float d = __fadd_rn(sv, nh), z = __fsub_rn(d, sv);
        const float de = __fadd_rn(__fsub_rn(sv, __fsub_rn(d, z)), __fsub_rn(nh, z));
        Y[row * xl + c] = __fadd_rn(d, __fsub_rn(de, lo[i][j]));
      }
    }
  }
}

constexpr size_t kCholSmem = sizeof(CholSmem);
// k_gsum: one block per 32-entry segment of a row of G.
unsigned gsum_blocks(int rp) { return (unsigned)(rp * ((rp + 31) / 32)); }

}  // namespace

cudaError_t launch_orth(const Handle& h, const Plan& p, cudaStream_t s) {
  cudaFuncSetAttribute(k_chol, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCholSmem);
  const int BJ = p.B * p.J;
  const int nblk = (p.r + kRankBlock - 1) / kRankBlock;  // one block when r <= kRankBlock
  for (int k = 0; k < nblk; ++k) {
    Plan pb = p;
    pb.ob_c0 = k * kRankBlock;
    pb.ob_r = std::min(kRankBlock, p.r - pb.ob_c0);
    pb.ob_rp = std::min(kRankBlock, p.rp - pb.ob_c0);
    pb.ob_src0 = 0;
    if (k > 0) {  // project the block off the finished columns, twice
      const int c0 = pb.ob_c0, rb = pb.ob_r;
      for (int it = 0; it < 2; ++it) {
        k_proj_coef<<<dim3(h.max_C, (c0 + 127) / 128, BJ), kT, 0, s>>>(pb, c0, rb, it);
        k_proj_sum<<<dim3((c0 * 128 + kT / 8 - 1) / (kT / 8), BJ), kT, 0, s>>>(pb, c0, rb);
        k_proj_apply<<<dim3(h.max_mtiles64, BJ), kT, 0, s>>>(pb, c0, rb, it);
        h.launches += 3;
      }
      pb.ob_src0 = 1;
    }
    cudaError_t e = launch_orth_passes(h, pb, 0, kMaxPasses - 1, s);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// Passes first_pass..last_pass of the column block pb describes, as separate kernels.
cudaError_t launch_orth_passes(const Handle& h, const Plan& pb, int first_pass, int last_pass, cudaStream_t s) {
  cudaFuncSetAttribute(k_chol, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCholSmem);
  const int BJ = pb.B * pb.J;
  for (int pass = first_pass; pass <= last_pass; ++pass) {
    if (pass == 0) {  // later passes get their Gram partials from the previous k_apply
      launch_pdl(k_gram, dim3(h.max_C, BJ), dim3(kT), 0, s, pb, pass);
      h.launches += 1;
    }
    launch_pdl(k_gsum, dim3(gsum_blocks(pb.ob_rp), BJ), dim3(kT), 0, s, pb, pass);
    launch_pdl(k_chol, dim3(BJ), dim3(kCholThreads), kCholSmem, s, pb, pass);
    if (pb.r > kRankBlock) launch_pdl(k_apply<true>, dim3(h.max_mtiles64, BJ), dim3(kT), 0, s, pb, pass);
    else launch_pdl(k_apply<false>, dim3(h.max_mtiles64, BJ), dim3(kT), 0, s, pb, pass);
    h.launches += 3;
  }
  return cudaGetLastError();
}

cudaError_t launch_orth_one(const Plan& p, int C, int mtiles64, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_chol, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kCholSmem);
  if (e != cudaSuccess) return e;
  for (int pass = 0; pass < kMaxPasses; ++pass) {
    if (pass == 0) launch_pdl(k_gram, dim3(C, 1), dim3(kT), 0, s, p, pass);
    launch_pdl(k_gsum, dim3(gsum_blocks(p.ob_rp), 1), dim3(kT), 0, s, p, pass);
    launch_pdl(k_chol, dim3(1), dim3(kCholThreads), kCholSmem, s, p, pass);
    launch_pdl(k_apply<false>, dim3(mtiles64, 1), dim3(kT), 0, s, p, pass);
  }
  return cudaGetLastError();
}

}  // namespace psgd
