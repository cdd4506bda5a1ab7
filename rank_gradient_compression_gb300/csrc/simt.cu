// FFMA engine of the three matrix products of the step: P = (1/W) sum_w M_w Q,
// Q = (1/W) sum_w M_w^T P^ (split-K partials, then a fixed-order reduction), and
// G^ = P^ Q^T fused with the error update E_w = round_E(M_w - G^).
//
// This engine runs fp32 gradients and serves as the debug reference of the tensor
// engine (PSGD_FLAG_SIMT). All sums run in a fixed order, so results are
// deterministic.
#include "handle.h"

namespace psgd {
namespace {

constexpr int kT = 256;

template <typename T>
__device__ __forceinline__ float ldf(const T* p) { return to_f(*p); }

// P tile: 64 rows x 128 columns of r. grid = (ceil(m/64), ceil(r/128), B*J). Q is read
// scaled by the exact power of two 2^e that puts max|Q| in [2^14, 2^15) (from scal[2]),
// so P = (1/W) sum_w M_w Q 2^e. P^ does not depend on that scale, and M Q stays inside
// fp32's range when M and Q are both tiny.
// Two-level fp32 accumulation: FMAs go into `part` (a run of 32 terms), which is added
// into `acc` with a compensated (Kahan) sum, `cmp` holding the running compensation.
// A single chain over W * n (up to 1.3e5) terms would leave about sqrt of that times the
// unit roundoff; here it is about sqrt(16) for the runs plus O(1) for the total. At high
// rank the GEMM error is amplified by cond(P) (up to 2e6) in the span of P^.
__device__ __forceinline__ void flush_part(float acc[4][8], float cmp[4][8], float part[4][8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float y = __fsub_rn(part[i][j], cmp[i][j]);
      const float t = __fadd_rn(acc[i][j], y);
      cmp[i][j] = __fsub_rn(__fsub_rn(t, acc[i][j]), y);
      acc[i][j] = t;
      part[i][j] = 0.f;
    }
}

template <typename TE>
__global__ void __launch_bounds__(kT) k_pgemm(Plan p) {
  const MatMeta& mt = p.meta[blockIdx.z];
  if (p.skip[mt.b]) return;
  const int64_t m = mt.m, n = mt.n;
  const int r = p.r, rp = p.rp;
  const int row0 = blockIdx.x * 64;
  if (row0 >= m) return;
  const int col0 = blockIdx.y * 128;
  const float* Q = p.tab.q[blockIdx.z];
  const unsigned qbits = reinterpret_cast<const unsigned*>(mt.scal)[2];
  const int qex = qbits == 0u ? 0 : (int)((qbits >> 23) & 0xff) - 127;
  const int qsh = 14 - (qex < -126 ? -126 : qex);  // Q * 2^qsh: ldexpf keeps it exact
  __shared__ float As[32][64 + 4];
  __shared__ __align__(16) float Bs[32][128];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][8], cmp[4][8], part[4][8];  // total, its compensation, the current run
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = cmp[i][j] = part[i][j] = 0.f;
  for (int w = 0; w < p.W; ++w) {
    const TE* M = static_cast<const TE*>(mt.mscr) + (size_t)w * m * n;
    for (int64_t k0 = 0; k0 < n; k0 += 32) {
      {
        const int rr = tid >> 2, kk = (tid & 3) * 8;
        const int64_t row = row0 + rr;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t k = k0 + kk + i;
          As[kk + i][rr] = (row < m && k < n) ? ldf(M + row * n + k) : 0.f;
        }
      }
      {
        const int kk = tid >> 3, c = (tid & 7) * 16;
        const int64_t k = k0 + kk;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = col0 + c + i;
          Bs[kk][c + i] = (k < n && col < r) ? ldexpf(Q[k * r + col], qsh) : 0.f;
        }
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
          for (int j = 0; j < 8; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
      }
      __syncthreads();
      flush_part(acc, cmp, part);  // every 32 terms
    }
  }
  unsigned vmax = 0u;
  const float fw = p.mean_div;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = row0 + ty * 4 + i;
    if (row >= m) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = col0 + tx * 8 + j;
      if (col < r) {
        const float v = __fdiv_rn(acc[i][j], fw);
        mt.P[row * rp + col] = v;
        vmax = max(vmax, __float_as_uint(fabsf(v)));
      }
    }
  }
  vmax = __reduce_max_sync(0xffffffffu, vmax);
  if ((tid & 31) == 0 && vmax) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + 1, vmax);
}

// Q partials: Qpart[s][n-tile 64][r-tile 128] = sum_w sum_{rows of slice s} M_w^T P^.
// grid = (ceil(n/64), S * ceil(r/128), B*J).
template <typename TE>
__global__ void __launch_bounds__(kT) k_qgemm(Plan p) {
  const MatMeta& mt = p.meta[blockIdx.z];
  if (p.skip[mt.b]) return;
  const int64_t m = mt.m, n = mt.n;
  const int r = p.r, rp = p.rp;
  const int rtiles = (r + 127) / 128;
  const int s = blockIdx.y / rtiles, rt = blockIdx.y % rtiles;
  if (s >= mt.S) return;
  const int64_t n0 = (int64_t)blockIdx.x * 64;
  if (n0 >= n) return;
  const int col0 = rt * 128;
  const int64_t rows_per = ((m + mt.S - 1) / mt.S + 31) / 32 * 32;
  const int64_t rbeg = s * rows_per, rend = min(m, rbeg + rows_per);
  __shared__ float As[32][64 + 4];
  __shared__ __align__(16) float Bs[32][128];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][8], cmp[4][8], part[4][8];  // total, its compensation, the current run
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = cmp[i][j] = part[i][j] = 0.f;
  for (int w = 0; w < p.W; ++w) {
    const TE* M = static_cast<const TE*>(mt.mscr) + (size_t)w * m * n;
    for (int64_t k0 = rbeg; k0 < rend; k0 += 32) {
      {
        const int kk = tid >> 3, c = (tid & 7) * 8;
        const int64_t row = k0 + kk;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t col = n0 + c + i;
          As[kk][c + i] = (row < rend && col < n) ? ldf(M + row * n + col) : 0.f;
        }
      }
      {
        const int kk = tid >> 3, c = (tid & 7) * 16;
        const int64_t row = k0 + kk;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = col0 + c + i;
          Bs[kk][c + i] = (row < rend && col < r) ? mt.Phat[row * rp + col] : 0.f;
        }
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
          for (int j = 0; j < 8; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
      }
      __syncthreads();
      flush_part(acc, cmp, part);  // every 32 terms
    }
  }
  float* out = mt.Qpart + (size_t)s * n * rp;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t col = n0 + ty * 4 + i;
    if (col >= n) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = col0 + tx * 8 + j;
      if (c < r) out[col * rp + c] = acc[i][j];
    }
  }
}

// Q = (sum over slices of Qpart) * qscale / W -> the caller's fp32 Q state (n x r), and
// max|Q| -> scal[3]. qscale undoes the power-of-two scale of a split P^ (exact).
// Four warps share a row of Q: warp g sums the slices s = g, g + 4, ... in order (all of
// its loads in flight together), and the four sums are added in the order g = 0, 1, 2, 3,
// a fixed order whatever the run. Lane l takes 4 consecutive columns per 128-column
// chunk of the row (one 16-byte load per slice; rp is a multiple of 16).
// Flattened grid (flat_item): B * sum_j ceil(n_j / 2) blocks of 256 threads, two rows each.
constexpr int kQredSplit = 4;
__global__ void __launch_bounds__(256) k_qreduce(Plan p, float qscale) {
  pdl_wait();
  int t;
  int64_t item;
  flat_item(p, blockIdx.x, [](const MatMeta& m) { return (m.n + 1) / 2; }, t, item);
  const MatMeta& mt = p.meta[t];
  if (p.skip[mt.b]) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp & (kQredSplit - 1);
  const int64_t row = item * 2 + (warp >> 2);
  const float fw = p.mean_div;
  float* q = p.q_to_exchange ? mt.xq : p.tab.q[t];
  const int msh = reinterpret_cast<const int*>(mt.scal)[SC_MSHIFT];  // rescaled M: Q * 2^msh
  const size_t stride = (size_t)mt.n * p.rp;  // one slice of Qpart
  __shared__ float4 part[2][kQredSplit][32];
  unsigned vmax = 0u;
  for (int c0 = 0; c0 < p.r; c0 += 128) {
    const int c = c0 + lane * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < mt.n && c < p.r) {
      const float* src = mt.Qpart + (size_t)row * p.rp + c;
#pragma unroll 16
      for (int s = g; s < mt.S; s += kQredSplit) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(src + (size_t)s * stride));
        acc.x = __fadd_rn(acc.x, v.x); acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z); acc.w = __fadd_rn(acc.w, v.w);
      }
    }
    part[warp >> 2][g][lane] = acc;
    __syncthreads();
    if (g == 0 && row < mt.n && c < p.r) {
      float4 t = part[warp >> 2][0][lane];
#pragma unroll
      for (int k = 1; k < kQredSplit; ++k) {
        const float4 v = part[warp >> 2][k][lane];
        t.x = __fadd_rn(t.x, v.x); t.y = __fadd_rn(t.y, v.y);
        t.z = __fadd_rn(t.z, v.z); t.w = __fadd_rn(t.w, v.w);
      }
      const float a4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (c + i < p.r) {
          const float v = ldexpf(__fdiv_rn(a4[i] * qscale, fw), -msh);
          q[row * p.r + c + i] = v;
          vmax = max(vmax, __float_as_uint(fabsf(v)));
        }
      }
    }
    __syncthreads();
  }
  vmax = block_max_u32(vmax);
  if (threadIdx.x == 0 && vmax && !p.q_to_exchange) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + 3, vmax);
}

template <typename TE> struct V4;
template <> struct V4<float> { using T = float4; };
template <> struct V4<__half> { using T = uint2; };
template <> struct V4<__nv_bfloat16> { using T = uint2; };

// G^ tile 64 x 64 = P^ Q^T (K = r, fp32 FFMA), then for every worker
// E_w = round_E(M_w - G^) on the same tile. grid = (ceil(n/64), ceil(m/64), B*J).
template <typename TE>
__global__ void __launch_bounds__(kT) k_decomp(Plan p) {
  const MatMeta& mt = p.meta[blockIdx.z];
  const int64_t m = mt.m, n = mt.n;
  const int64_t row0 = (int64_t)blockIdx.y * 64, col0 = (int64_t)blockIdx.x * 64;
  if (row0 >= m || col0 >= n) return;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float* gh = p.tab.ghat[blockIdx.z];
  const bool skipped = p.skip[mt.b] != 0;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  if (!skipped) {
    const int r = p.r, rp = p.rp;
    const float* Q = p.tab.q[blockIdx.z];
    __shared__ float As[32][64 + 4];
    __shared__ float Bs[32][64 + 4];
    for (int k0 = 0; k0 < r; k0 += 32) {
      {
        const int rr = tid >> 2, kk = (tid & 3) * 8;
        const int64_t row = row0 + rr, col = col0 + rr;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int k = k0 + kk + i;
          As[kk + i][rr] = (row < m && k < r) ? mt.Phat[row * rp + k] : 0.f;
          Bs[kk + i][rr] = (col < n && k < r) ? Q[col * r + k] : 0.f;
        }
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }
  const int64_t c = col0 + tx * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = row0 + ty * 4 + i;
    if (row >= m) continue;
    if (c + 4 <= n) {
      *reinterpret_cast<float4*>(gh + row * n + c) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    } else {
      for (int j = 0; j < 4 && c + j < n; ++j) gh[row * n + c + j] = acc[i][j];
    }
  }
  if (skipped) return;
  for (int w = 0; w < p.W; ++w) {
    const TE* M = static_cast<const TE*>(mt.mscr) + (size_t)w * m * n;
    TE* E = static_cast<TE*>(p.tab.e[(size_t)blockIdx.z * p.W + w]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = row0 + ty * 4 + i;
      if (row >= m) continue;
      if (c + 4 <= n) {
        typename V4<TE>::T mv = *reinterpret_cast<const typename V4<TE>::T*>(M + row * n + c);
        const TE* mx = reinterpret_cast<const TE*>(&mv);
        TE ev[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) ev[j] = add_to<TE>(to_f(mx[j]), -acc[i][j]);
        *reinterpret_cast<typename V4<TE>::T*>(E + row * n + c) = *reinterpret_cast<const typename V4<TE>::T*>(ev);
      } else {
        for (int j = 0; j < 4 && c + j < n; ++j)
          E[row * n + c + j] = add_to<TE>(to_f(M[row * n + c + j]), -acc[i][j]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_pgemm_simt(const Handle& h, const Plan& p, cudaStream_t s) {
  dim3 grid(h.max_mtiles64, (p.r + 127) / 128, p.B * p.J);
  if (h.edt == DT_F16) k_pgemm<__half><<<grid, kT, 0, s>>>(p);
  else if (h.edt == DT_BF16) k_pgemm<__nv_bfloat16><<<grid, kT, 0, s>>>(p);
  else k_pgemm<float><<<grid, kT, 0, s>>>(p);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_qgemm_simt(const Handle& h, const Plan& p, cudaStream_t s) {
  dim3 grid(h.max_ntiles64, h.max_S * ((p.r + 127) / 128), p.B * p.J);
  if (h.edt == DT_F16) k_qgemm<__half><<<grid, kT, 0, s>>>(p);
  else if (h.edt == DT_BF16) k_qgemm<__nv_bfloat16><<<grid, kT, 0, s>>>(p);
  else k_qgemm<float><<<grid, kT, 0, s>>>(p);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_qreduce(const Handle& h, const Plan& p, cudaStream_t s) {
  int64_t per = 0;
  for (int j = 0; j < h.J; ++j) per += (h.meta[j].n + 1) / 2;
  launch_pdl(k_qreduce, dim3((unsigned)(per * p.B)), dim3(256), 0, s, p, h.tc ? 0x1p-14f : 1.0f);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_decomp_simt(const Handle& h, const Plan& p, cudaStream_t s) {
  dim3 grid(h.max_ntiles64, h.max_mtiles64, p.B * p.J);
  if (h.edt == DT_F16) k_decomp<__half><<<grid, kT, 0, s>>>(p);
  else if (h.edt == DT_BF16) k_decomp<__nv_bfloat16><<<grid, kT, 0, s>>>(p);
  else k_decomp<float><<<grid, kT, 0, s>>>(p);
  h.launches += 1;
  return cudaGetLastError();
}

}  // namespace psgd
