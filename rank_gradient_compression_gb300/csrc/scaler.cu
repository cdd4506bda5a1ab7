// Dynamic per-resblock gradient scale, kept on the device between steps.
//
// The rule ("AIGC 基本功|混合精度与数值稳定性", §3.2, the dynamic scaler): a scale S
// becomes beta S when the scaled gradient holds an Inf or NaN, gamma S after K
// consecutive finite steps, and otherwise stays. "Zero-Shot Text-to-Image Generation -
// 中文验证版" §方法适配 gives every resblock its own scale, so the rule runs per block,
// on the block's nonfinite count over all workers, the count psgd_step leaves in its
// counts output. That count is the same for every worker, which makes the decision the
// same everywhere ("AIGC 基本功|混合精度与数值稳定性", §6.2).
//
// psgd_scale_update applies the rule to S and the finite-step streak in place. The next
// psgd_step reads S through psgd_step_args.scales_device: k_inv_scale forms 1/S on the
// device, so the scale never goes through the host between steps.
#include <cmath>

#include "handle.h"

namespace psgd {
namespace {

// One thread per block b. The counts of a block are summed in worker order (int64, so
// the order does not matter); each product is one IEEE single multiply.
__global__ void k_scale_update(int B, int W, const int64_t* __restrict__ counts,
                               float* __restrict__ scale, int* __restrict__ streak,
                               float backoff, float growth, int interval) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int64_t c = 0;
  for (int w = 0; w < W; ++w) c += counts[(int64_t)b * W + w];
  float s = scale[b];
  int k = streak[b];
  // A product that is not a finite normal float (overflow, or below 2^-126) keeps S: a
  // scale of Inf or 0 would make 1/S zero or Inf in the next step.
  if (c > 0) {
    const float t = __fmul_rn(s, backoff);
    if (isfinite(t) && fabsf(t) >= 0x1p-126f) s = t;
    k = 0;
  } else if (++k >= interval) {
    const float t = __fmul_rn(s, growth);
    if (isfinite(t) && fabsf(t) >= 0x1p-126f) s = t;
    k = 0;
  }
  scale[b] = s;
  streak[b] = k;
}

// inv[b] = 1 / scale[b], rounded to nearest (exact for powers of two).
__global__ void k_inv_scale(int B, const float* __restrict__ scale, float* __restrict__ inv) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) inv[b] = __frcp_rn(scale[b]);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

cudaError_t launch_inv_scale(int B, const float* scale, float* inv, cudaStream_t s) {
  k_inv_scale<<<(B + 127) / 128, 128, 0, s>>>(B, scale, inv);
  return cudaGetLastError();
}

}  // namespace psgd

using namespace psgd;

extern "C" psgd_status psgd_scale_update(int32_t num_blocks, int32_t num_workers,
                                         const int64_t* counts, float* scale, int32_t* streak,
                                         double backoff, double growth, int32_t interval,
                                         void* stream) {
  if (num_blocks < 1 || num_workers < 1)
    return report_error(PSGD_EINVAL, "num_blocks and num_workers must be >= 1");
  if (!counts || !scale || !streak)
    return report_error(PSGD_EINVAL, "counts, scale and streak must be device pointers");
  if (!aligned(counts, 8) || !aligned(scale, 4) || !aligned(streak, 4))
    return report_error(PSGD_EINVAL, "counts, scale and streak must be aligned to their element size");
  // The checks apply to the factors as the kernel uses them, rounded to fp32.
  const float bf = (float)backoff, gf = (float)growth;
  if (!(backoff > 0.0 && backoff < 1.0) || !(bf > 0.0f && bf < 1.0f))
    return report_error(PSGD_EINVAL, "backoff must be in (0, 1) as an fp32 value");
  if (!(growth > 1.0) || !std::isfinite(growth) || !(gf > 1.0f) || !std::isfinite(gf))
    return report_error(PSGD_EINVAL, "growth must be finite and > 1 as an fp32 value");
  if (interval < 1) return report_error(PSGD_EINVAL, "interval must be >= 1");
  if ((int64_t)num_blocks * num_workers > ((int64_t)1 << 40))
    return report_error(PSGD_EINVAL, "num_blocks * num_workers is too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_scale_update<<<(num_blocks + 127) / 128, 128, 0, s>>>(
      num_blocks, num_workers, counts, scale, reinterpret_cast<int*>(streak), bf, gf, interval);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_cuda_error(e, "psgd_scale_update");
  return PSGD_OK;
}
