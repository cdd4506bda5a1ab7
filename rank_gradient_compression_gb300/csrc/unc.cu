// Uncompressed fp32 reduction of the tensors the method leaves out of PowerSGD: the
// embedding and unembedding (vocabulary x d_model) and any other fp32 gradient outside a
// resblock's compressed matrices.
//
// "Zero-Shot Text-to-Image Generation - 中文验证版", §方法适配: embedding, unembedding,
// gains and biases are not compressed and are reduced in 32-bit precision. "[논문 정리]
// Zero-Shot Text-to-Image Generation", PowerSGD list: they are kept in 32-bit and not
// compressed; §Mixed-Precision Training: Inf/NaN entries become 0 when a gradient is
// unscaled. The arithmetic is that of the step's gains/biases:
//   out[i] = (sum_w zero_nonfinite(in_w[i] * (1/s))) / W,  fp32, workers in order w = 0..W-1
//   counts[w] = number of entries of in_w whose unscaled value is not finite.
//
// The pass is one HBM sweep: W reads of len floats and one write. A persistent grid of
// a few CTAs per SM walks 16-byte chunks of the output; each thread loads its chunk from
// every worker before it adds (W loads in flight), and keeps per-worker counts in
// registers until one atomic per (CTA, worker) at the end.
#include <algorithm>
#include <cmath>

#include "handle.h"

namespace psgd {
namespace {

constexpr int kUncThreads = 256;
constexpr int kUncMaxWorkers = PSGD_UNC_MAX_WORKERS;
static_assert(kUncMaxWorkers <= 16, "per-worker counters are held for at most 16 workers");

struct UncArgs {
  const float* in[kUncMaxWorkers];
  float* out;
  unsigned long long* counts;
  const uint8_t* skip;
  int64_t len;
  float inv_s;
  int32_t W;
};

template <int kW>
__device__ __forceinline__ void unc_body(const UncArgs& a) {
  const int W = kW > 0 ? kW : a.W;
  int cnt[16];
#pragma unroll
  for (int w = 0; w < 16; ++w) cnt[w] = 0;
  const bool skipped = a.skip != nullptr && *a.skip != 0;
  const int64_t nvec = a.len >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const float inv_s = a.inv_s;
  const float fw = (float)W;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    float4 x[kW > 0 ? kW : 16];
#pragma unroll
    for (int w = 0; w < (kW > 0 ? kW : 16); ++w)
      if (w < W) x[w] = __ldcs(reinterpret_cast<const float4*>(a.in[w]) + v);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < (kW > 0 ? kW : 16); ++w) {
      if (w >= W) break;
      const float e0 = x[w].x * inv_s, e1 = x[w].y * inv_s, e2 = x[w].z * inv_s, e3 = x[w].w * inv_s;
      const bool b0 = !isfinite(e0), b1 = !isfinite(e1), b2 = !isfinite(e2), b3 = !isfinite(e3);
      cnt[w] += (int)b0 + (int)b1 + (int)b2 + (int)b3;
      acc.x = __fadd_rn(acc.x, b0 ? 0.f : e0);
      acc.y = __fadd_rn(acc.y, b1 ? 0.f : e1);
      acc.z = __fadd_rn(acc.z, b2 ? 0.f : e2);
      acc.w = __fadd_rn(acc.w, b3 ? 0.f : e3);
    }
    float4 o;
    o.x = skipped ? 0.f : __fdiv_rn(acc.x, fw);
    o.y = skipped ? 0.f : __fdiv_rn(acc.y, fw);
    o.z = skipped ? 0.f : __fdiv_rn(acc.z, fw);
    o.w = skipped ? 0.f : __fdiv_rn(acc.w, fw);
    __stcs(reinterpret_cast<float4*>(a.out) + v, o);
  }
  // the last len % 4 entries: one thread
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int64_t i = nvec * 4; i < a.len; ++i) {
      float acc = 0.f;
      for (int w = 0; w < W; ++w) {
        const float e = a.in[w][i] * inv_s;
        const bool bad = !isfinite(e);
        cnt[w] += bad;
        acc = __fadd_rn(acc, bad ? 0.f : e);
      }
      a.out[i] = skipped ? 0.f : __fdiv_rn(acc, fw);
    }
  }
  __shared__ int s_cnt[kUncThreads / 32][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    if (w >= W) break;
    const int c = __reduce_add_sync(0xffffffffu, cnt[w]);
    if (lane == 0) s_cnt[warp][w] = c;
  }
  __syncthreads();
  if (threadIdx.x < W) {
    unsigned long long t = 0;
    for (int k = 0; k < kUncThreads / 32; ++k) t += (unsigned)s_cnt[k][threadIdx.x];
    if (t) atomicAdd(a.counts + threadIdx.x, t);
  }
}

template <int kW>
__global__ void __launch_bounds__(kUncThreads) k_unc_reduce(const __grid_constant__ UncArgs a) {
  unc_body<kW>(a);
}

}  // namespace
}  // namespace psgd

using namespace psgd;

extern "C" psgd_status psgd_reduce_uncompressed(int32_t num_workers, const float* const* in, int64_t len,
                                                float scale, float* out, int64_t* counts,
                                                const uint8_t* skip, void* stream) {
  if (num_workers < 1 || num_workers > kUncMaxWorkers)
    return report_error(PSGD_EINVAL, "num_workers must be in [1, PSGD_UNC_MAX_WORKERS]");
  if (!in || !out || !counts) return report_error(PSGD_EINVAL, "in, out and counts are required");
  if (len < 0) return report_error(PSGD_EINVAL, "len must be >= 0");
  if (!std::isfinite(scale) || !(scale > 0.0f)) return report_error(PSGD_EINVAL, "scale must be finite and > 0");
  if ((reinterpret_cast<uintptr_t>(out) & 15u) || (reinterpret_cast<uintptr_t>(counts) & 7u))
    return report_error(PSGD_EINVAL, "out must be 16-byte aligned and counts 8-byte aligned");
  UncArgs a{};
  for (int w = 0; w < num_workers; ++w) {
    if (!in[w]) return report_error(PSGD_EINVAL, "NULL input pointer");
    if (reinterpret_cast<uintptr_t>(in[w]) & 15u)
      return report_error(PSGD_EINVAL, "input pointers must be 16-byte aligned");
    a.in[w] = in[w];
  }
  a.out = out;
  a.counts = reinterpret_cast<unsigned long long*>(counts);
  a.skip = skip;
  a.len = len;
  a.inv_s = (float)(1.0 / (double)scale);
  a.W = num_workers;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int64_t) * (size_t)num_workers, s);
  if (e != cudaSuccess) return report_cuda_error(e, "psgd_reduce_uncompressed");
  if (len == 0) return PSGD_OK;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  const int64_t nvec = len >> 2;
  const int64_t want = (nvec + kUncThreads - 1) / kUncThreads;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 4));
  switch (num_workers) {
    case 8: k_unc_reduce<8><<<grid, kUncThreads, 0, s>>>(a); break;
    case 4: k_unc_reduce<4><<<grid, kUncThreads, 0, s>>>(a); break;
    case 2: k_unc_reduce<2><<<grid, kUncThreads, 0, s>>>(a); break;
    case 1: k_unc_reduce<1><<<grid, kUncThreads, 0, s>>>(a); break;
    default: k_unc_reduce<0><<<grid, kUncThreads, 0, s>>>(a); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return report_cuda_error(e, "psgd_reduce_uncompressed");
  return PSGD_OK;
}
