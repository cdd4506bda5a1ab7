// Kernels of the data-parallel exchange points (psgd_step_p / psgd_step_q / psgd_step_e).
//
// The method all-reduces the low-rank factors between machines instead of the gradient
// ("Zero-Shot Text-to-Image Generation - 中文验证版", §方法适配; the all-reduces are grouped,
// §证据). With several ranks, each holding some of the workers, the step stops at the two
// points where the worker means are taken: after P_r = sum over the rank's workers of
// M_w Q, and after Q_r = sum of M_w^T P^. The caller sums the exchange buffers over the
// ranks (NCCL, gloo, ...) and resumes; the library then divides by the total worker count.
// The skip decision waits for the counts summed over every rank, so every rank decides
// alike ("AIGC 基本功|混合精度与数值稳定性", §6.2).
#include <cmath>

#include "handle.h"

namespace psgd {
namespace {

// xp[t] (m x r, dense) = P[t] (m x rp): this rank's sum of M_w Q over its workers; and
// xcnt[b] = sum over this rank's workers of counts[b][w] (block (0, 0)).
__global__ void k_pack_p(Plan p, int64_t* xcnt) {
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      int64_t c = 0;
      for (int w = 0; w < p.W; ++w) c += p.counts[(int64_t)b * p.W + w];
      xcnt[b] = c;
    }
  const MatMeta& mt = p.meta[blockIdx.y];
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= mt.m * p.r) return;
  const int64_t row = i / p.r, c = i - row * p.r;
  mt.xp[i] = mt.P[row * p.rp + c];
}

// skip[b] from the nonfinite counts summed over every rank and worker (an integer
// comparison with ceil(T W_total numel_b), computed in IEEE double like the threshold of
// psgd_init), and the max|P| / max|Q| words cleared for the maxima of the summed factors.
__global__ void k_skip_global(Plan p, const int64_t* block_counts, double frac, int64_t numel_b, int w_total) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const int64_t thr = (int64_t)ceil(frac * (double)((int64_t)w_total * numel_b));
  p.skip[b] = (uint8_t)(block_counts[b] >= thr);
  for (int j = 0; j < p.J; ++j) {
    float* sc = p.meta[b * p.J + j].scal;
    sc[SC_MAXP] = 0.f;
    sc[SC_MAXQN] = 0.f;
  }
}

// P[t] (m x rp, columns r.. zero) = xp[t] / W_total, and max|P| -> scal[SC_MAXP].
__global__ void __launch_bounds__(256) k_unpack_p(Plan p, float div) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  if ((int64_t)blockIdx.x * blockDim.x >= mt.m * p.rp) return;  // whole block past the end
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  unsigned mx = 0u;
  if (i < mt.m * p.rp) {
    const int64_t row = i / p.rp, c = i - row * p.rp;
    const float v = c < p.r ? __fdiv_rn(mt.xp[row * p.r + c], div) : 0.f;
    mt.P[i] = v;
    mx = __float_as_uint(fabsf(v));
  }
  mx = block_max_u32(mx);
  if (threadIdx.x == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + SC_MAXP, mx);
}

// Q state[t] (n x r) = xq[t] / W_total, and max|Q| -> scal[SC_MAXQN].
__global__ void __launch_bounds__(256) k_unpack_q(Plan p, float div) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  if ((int64_t)blockIdx.x * blockDim.x >= mt.n * p.r) return;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  unsigned mx = 0u;
  if (i < mt.n * p.r) {
    const float v = __fdiv_rn(mt.xq[i], div);
    p.tab.q[blockIdx.y][i] = v;
    mx = __float_as_uint(fabsf(v));
  }
  mx = block_max_u32(mx);
  if (threadIdx.x == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + SC_MAXQN, mx);
}

}  // namespace

cudaError_t launch_pack_p(const Handle& h, const Plan& p, cudaStream_t s) {
  int64_t mx = 0;
  for (const MatMeta& mt : h.meta) mx = std::max<int64_t>(mx, mt.m * p.r);
  launch_pdl(k_pack_p, dim3((unsigned)((mx + 255) / 256), p.B * p.J), dim3(256), 0, s, p, h.d_xcnt);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_skip_global(const Handle& h, const Plan& p, const int64_t* block_counts, int w_total,
                               cudaStream_t s) {
  int64_t numel_b = h.cfg.unc_len;
  for (int j = 0; j < h.J; ++j) numel_b += h.shapes[j].m * h.shapes[j].n;
  k_skip_global<<<(p.B + 127) / 128, 128, 0, s>>>(p, block_counts, h.cfg.skip_fraction, numel_b, w_total);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_unpack_p(const Handle& h, const Plan& p, int w_total, cudaStream_t s) {
  int64_t mx = 0;
  for (const MatMeta& mt : h.meta) mx = std::max<int64_t>(mx, mt.m * p.rp);
  launch_pdl(k_unpack_p, dim3((unsigned)((mx + 255) / 256), p.B * p.J), dim3(256), 0, s, p, (float)w_total);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_unpack_q(const Handle& h, const Plan& p, int w_total, cudaStream_t s) {
  int64_t mx = 0;
  for (const MatMeta& mt : h.meta) mx = std::max<int64_t>(mx, mt.n * p.r);
  launch_pdl(k_unpack_q, dim3((unsigned)((mx + 255) / 256), p.B * p.J), dim3(256), 0, s, p, (float)w_total);
  h.launches += 1;
  return cudaGetLastError();
}

}  // namespace psgd
