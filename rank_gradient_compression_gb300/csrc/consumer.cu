// Consumer of the decompressed gradient: global-norm clipping and one Adam step with
// fp32 moments, on the device.
//
// "Zero-Shot Text-to-Image Generation - 中文验证版", §方法适配: training used Adam with
// gradient clipping and a skip rule for nonfinite values (the moments' 16-bit format
// is not given, so the moments here are fp32). "AIGC 基本功|混合精度与数值稳定性", §6.2:
// the clipping norm is global, the root of the all-reduced local sums of squares, taken
// after unscaling; a skipped step updates nothing. The update is the published
// bias-corrected Adam rule (Kingma and Ba, 2015):
//   g' = c g with c = min(1, C / ||g||) (c = 1 when C <= 0 or ||g|| <= C)
//   m <- b1 m + (1 - b1) g';  v <- b2 v + (1 - b2) g'^2
//   theta <- theta - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
//
// Three kernels over chunks of kChunk elements (a chunk never spans two tensors):
//   k_sumsq   partial[c] = sum of squares of chunk c (fp32 per thread, fp64 across the
//             block, fixed order);
//   k_norm    one block: ||g|| = sqrt(sum_c partial[c]) in fp64, fixed order, and c;
//   k_adam    the element-wise update, skipped for tensors of skipped blocks.
// The tensor table travels as a kernel parameter (at most kMaxTensors entries).
#include <cmath>

#include "handle.h"

namespace psgd {
namespace {

constexpr int kChunk = 8192;       // elements per block of k_sumsq / k_adam
constexpr int kConsThreads = 256;  // kChunk / kConsThreads elements per thread
constexpr int kMaxTensors = PSGD_ADAM_MAX_TENSORS;

struct AdamEntry {
  const float* g;
  float* p;
  float* m;
  float* v;
  int64_t n;
  int32_t chunk0;  // first chunk of this tensor
  int32_t block;   // resblock index for the skip flags (-1: never skipped)
};
struct AdamTab {
  AdamEntry e[kMaxTensors];
  int32_t T, nchunks;
};

// The tensor that chunk c belongs to (chunk0 ascending): binary search.
__device__ __forceinline__ int tensor_of(const AdamTab& tab, int c) {
  int lo = 0, hi = tab.T - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab.e[mid].chunk0 <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ double block_sum_f64(double x) {
  __shared__ double s_part[kConsThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
  if (lane == 0) s_part[warp] = x;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kConsThreads / 32; ++w) t += s_part[w];
  return t;  // valid in thread 0
}

__global__ void __launch_bounds__(kConsThreads) k_sumsq(const __grid_constant__ AdamTab tab,
                                                         double* __restrict__ partial) {
  const int c = blockIdx.x;
  const AdamEntry& e = tab.e[tensor_of(tab, c)];
  const int64_t base = (int64_t)(c - e.chunk0) * kChunk;
  float s = 0.f;
#pragma unroll 8
  for (int k = threadIdx.x; k < kChunk; k += kConsThreads) {
    const int64_t i = base + k;
    if (i < e.n) {
      const float x = __ldg(e.g + i);
      s = fmaf(x, x, s);
    }
  }
  const double t = block_sum_f64((double)s);
  if (threadIdx.x == 0) partial[c] = t;
}

__global__ void __launch_bounds__(kConsThreads) k_norm(const double* __restrict__ partial,
                                                        int nchunks, double max_norm,
                                                        float* __restrict__ coef,
                                                        float* __restrict__ norm_out) {
  double s = 0.0;
  for (int c = threadIdx.x; c < nchunks; c += kConsThreads) s += partial[c];
  const double t = block_sum_f64(s);
  if (threadIdx.x == 0) {
    const double nrm = sqrt(t);
    coef[0] = (max_norm > 0.0 && nrm > max_norm) ? (float)(max_norm / nrm) : 1.0f;
    coef[1] = (float)nrm;
    if (norm_out) norm_out[0] = (float)nrm;
  }
}

__global__ void __launch_bounds__(kConsThreads) k_adam(const __grid_constant__ AdamTab tab,
                                                        const uint8_t* __restrict__ skip,
                                                        const float* __restrict__ coef,
                                                        float lr, float b1, float b2, float eps,
                                                        float bc1, float bc2) {
  const int c = blockIdx.x;
  const AdamEntry& e = tab.e[tensor_of(tab, c)];
  if (skip && e.block >= 0 && skip[e.block]) return;
  const float cf = coef[0];
  const int64_t base = (int64_t)(c - e.chunk0) * kChunk;
  for (int k = threadIdx.x; k < kChunk; k += kConsThreads) {
    const int64_t i = base + k;
    if (i >= e.n) break;
    const float g = __ldg(e.g + i) * cf;
    const float m = fmaf(b1, e.m[i], (1.f - b1) * g);
    const float v = fmaf(b2, e.v[i], (1.f - b2) * g * g);
    e.m[i] = m;
    e.v[i] = v;
    e.p[i] -= lr * (m / bc1) / (sqrtf(v / bc2) + eps);
  }
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int64_t chunks_of(int64_t n) { return (n + kChunk - 1) / kChunk; }

}  // namespace
}  // namespace psgd

using namespace psgd;

extern "C" size_t psgd_clip_adam_workspace_size(int32_t num_tensors, const int64_t* numel) {
  if (num_tensors < 1 || num_tensors > kMaxTensors || !numel) {
    report_error(PSGD_EINVAL, "num_tensors must be in [1, PSGD_ADAM_MAX_TENSORS] with numel given");
    return 0;
  }
  int64_t nch = 0;
  for (int t = 0; t < num_tensors; ++t) {
    if (numel[t] < 0) { report_error(PSGD_EINVAL, "numel must be >= 0"); return 0; }
    nch += chunks_of(numel[t]);
  }
  return (size_t)(256 + 8 * nch + 255) / 256 * 256;
}

extern "C" psgd_status psgd_clip_adam(const psgd_adam_args* a, void* workspace, size_t ws_bytes,
                                      void* stream) {
  if (!a || !workspace) return report_error(PSGD_EINVAL, "args and workspace are required");
  const int T = a->num_tensors;
  if (T < 1 || T > kMaxTensors) return report_error(PSGD_EINVAL, "num_tensors must be in [1, PSGD_ADAM_MAX_TENSORS]");
  if (!a->grads || !a->params || !a->exp_avg || !a->exp_avg_sq || !a->numel)
    return report_error(PSGD_EINVAL, "a tensor array is NULL");
  if (a->skip && (!a->block || a->num_blocks < 1))
    return report_error(PSGD_EINVAL, "skip needs block indices and num_blocks");
  if (!(a->lr >= 0.0) || !std::isfinite(a->lr) || !(a->beta1 >= 0.0 && a->beta1 < 1.0) ||
      !(a->beta2 >= 0.0 && a->beta2 < 1.0) || !(a->eps >= 0.0) || !std::isfinite(a->eps) ||
      !std::isfinite(a->max_norm) || a->step < 1)
    return report_error(PSGD_EINVAL, "lr, beta1, beta2, eps, max_norm or step out of range");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return report_error(PSGD_EINVAL, "workspace must be 256-byte aligned");
  if (a->norm_out && !aligned4(a->norm_out)) return report_error(PSGD_EINVAL, "norm_out must be 4-byte aligned");
  AdamTab tab;
  int64_t nch = 0;
  for (int t = 0; t < T; ++t) {
    AdamEntry& e = tab.e[t];
    e.g = a->grads[t]; e.p = a->params[t]; e.m = a->exp_avg[t]; e.v = a->exp_avg_sq[t];
    e.n = a->numel[t];
    if (e.n < 0) return report_error(PSGD_EINVAL, "numel must be >= 0");
    if (e.n > 0 && (!e.g || !e.p || !e.m || !e.v))
      return report_error(PSGD_EINVAL, "NULL tensor pointer");
    if (!aligned4(e.g) || !aligned4(e.p) || !aligned4(e.m) || !aligned4(e.v))
      return report_error(PSGD_EINVAL, "tensor pointers must be 4-byte aligned");
    e.block = a->block ? a->block[t] : -1;
    if (a->skip && (e.block < -1 || e.block >= a->num_blocks))
      return report_error(PSGD_EINVAL, "block index out of range");
    e.chunk0 = (int32_t)nch;
    nch += chunks_of(e.n);
    if (nch >= ((int64_t)1 << 31) - 1) return report_error(PSGD_EINVAL, "too many elements");
  }
  tab.T = T;
  tab.nchunks = (int32_t)nch;
  const size_t need = (size_t)(256 + 8 * nch + 255) / 256 * 256;
  if (ws_bytes < need) return report_error(PSGD_EINVAL, "workspace smaller than psgd_clip_adam_workspace_size");
  float* coef = static_cast<float*>(workspace);                       // [2]: c, ||g||
  double* partial = reinterpret_cast<double*>(static_cast<char*>(workspace) + 256);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nch > 0) k_sumsq<<<(unsigned)nch, kConsThreads, 0, s>>>(tab, partial);
  k_norm<<<1, kConsThreads, 0, s>>>(partial, (int)nch, a->max_norm, coef, a->norm_out);
  const double bc1 = 1.0 - std::pow(a->beta1, (double)a->step);
  const double bc2 = 1.0 - std::pow(a->beta2, (double)a->step);
  if (nch > 0)
    k_adam<<<(unsigned)nch, kConsThreads, 0, s>>>(tab, a->skip, coef, (float)a->lr, (float)a->beta1,
                                                  (float)a->beta2, (float)a->eps, (float)bc1, (float)bc2);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_cuda_error(e, "psgd_clip_adam");
  return PSGD_OK;
}
