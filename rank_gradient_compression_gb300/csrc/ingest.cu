// Ingest: unscale, nonfinite mask/count and error-buffer accumulation (one HBM sweep),
// then the per-block skip decision and the uncompressed gains/biases mean.
//
// "[논문 정리] Zero-Shot Text-to-Image Generation", §Mixed-Precision Training: a
// resblock's gradient is unscaled when backprop leaves the block, and Inf/NaN become 0.
// PowerSGD list: the gradient is accumulated into the error buffer. "Zero-Shot
// Text-to-Image Generation - 中文验证版", §方法适配: the skip-update rule for nonfinite
// values; gains/biases are reduced in 32-bit without compression.
//
// Memory-bound. Each thread moves 8 entries per iteration with 16-byte loads and
// stores; a CTA issues all of its loads before it computes.
#include "handle.h"

namespace psgd {
namespace {

struct Raw8 {
  uint4 v[2];  // 16 bytes for 16-bit types, 32 bytes for fp32
};

template <typename T>
__device__ __forceinline__ void load8(const T* p, Raw8& r) {
  r.v[0] = __ldcs(reinterpret_cast<const uint4*>(p));
  if (sizeof(T) == 4) r.v[1] = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
}

template <typename T>
__device__ __forceinline__ void unpack8(const Raw8& r, float f[8]) {
  if constexpr (sizeof(T) == 4) {
    const float* x = reinterpret_cast<const float*>(&r.v[0]);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = x[i];
  } else {
    const T* x = reinterpret_cast<const T*>(&r.v[0]);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = to_f(x[i]);
  }
}

template <typename T>
__device__ __forceinline__ void store8(T* p, const T v[8]) {
  if constexpr (sizeof(T) == 4) {
    reinterpret_cast<uint4*>(p)[0] = *reinterpret_cast<const uint4*>(&v[0]);
    reinterpret_cast<uint4*>(p)[1] = *reinterpret_cast<const uint4*>(&v[4]);
  } else {
    reinterpret_cast<uint4*>(p)[0] = *reinterpret_cast<const uint4*>(&v[0]);
  }
}

__device__ __forceinline__ int block_sum(int v, int* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  int t = 0;
  if (threadIdx.x < 32) {
    t = (threadIdx.x < (int)(blockDim.x >> 5)) ? sh[threadIdx.x] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  }
  return t;  // valid in thread 0
}

__device__ __forceinline__ unsigned block_max(unsigned v, unsigned* sh) {
  v = __reduce_max_sync(0xffffffffu, v);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  unsigned t = 0;
  if (threadIdx.x < 32) {
    t = (threadIdx.x < (int)(blockDim.x >> 5)) ? sh[threadIdx.x] : 0u;
    t = __reduce_max_sync(0xffffffffu, t);
  }
  return t;
}

__device__ __forceinline__ int find_seg(const IngestSeg* segs, int nseg, int64_t cta) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (segs[mid].cta_start <= cta) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One CTA = kIngestChunk consecutive entries of one (matrix, worker) or one gains/biases
// vector. Matrices: M = round_E(zero_nonfinite(G * (1/s_b)) + E), the nonfinite
// count of (b, w), optional mask bits, and max|M| of the matrix. Vectors: the count only.
template <typename TG, typename TE>
__global__ void __launch_bounds__(kIngestThreads)
k_ingest(Plan p, const IngestSeg* __restrict__ segs, int nseg, int64_t cta_offset) {
  __shared__ int sh_i[kIngestThreads / 32];
  __shared__ unsigned sh_u[kIngestThreads / 32];
  const int64_t cta = (int64_t)blockIdx.x + cta_offset;
  const IngestSeg sg = segs[find_seg(segs, nseg, cta)];
  const int64_t base = (cta - sg.cta_start) * kIngestChunk;
  const float inv_s = p.tab.inv_scale[sg.b];
  const int tid = threadIdx.x;
  int cnt = 0;
  unsigned mmax = 0u;

  if (sg.kind == 0) {
    const MatMeta& mt = p.meta[sg.t];
    const int64_t numel = sg.numel;
    const size_t slot = (size_t)sg.t * p.W + sg.w;
    const TG* g = static_cast<const TG*>(p.tab.g[slot]);
    TE* e = static_cast<TE*>(p.tab.e[slot]);
    TE* mo = static_cast<TE*>(mt.mscr) + (size_t)sg.w * (size_t)numel;
    uint32_t* mask = p.mask ? p.mask + p.mask_off[slot] : nullptr;

    Raw8 rg[kIngestIters], re[kIngestIters];
    bool full[kIngestIters];
#pragma unroll
    for (int it = 0; it < kIngestIters; ++it) {
      const int64_t idx = base + (int64_t)it * kIngestThreads * kIngestVec + tid * kIngestVec;
      full[it] = idx + kIngestVec <= numel;
      if (full[it]) {
        load8(g + idx, rg[it]);
        load8(e + idx, re[it]);
      }
    }
#pragma unroll
    for (int it = 0; it < kIngestIters; ++it) {
      const int64_t idx = base + (int64_t)it * kIngestThreads * kIngestVec + tid * kIngestVec;
      float gv[8], ev[8];
      unsigned bits = 0u;
      TE mv[8];
      if (full[it]) {
        unpack8<TG>(rg[it], gv);
        unpack8<TE>(re[it], ev);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float x = gv[i] * inv_s;
          const bool bad = !isfinite(x);
          bits |= (unsigned)bad << i;
          x = bad ? 0.0f : x;
          mv[i] = add_to<TE>(x, ev[i]);
          mmax = max(mmax, __float_as_uint(fabsf(to_f(mv[i]))));
        }
        store8(mo + idx, mv);
      } else if (idx < numel) {
        for (int i = 0; i < 8 && idx + i < numel; ++i) {
          float x = to_f(g[idx + i]) * inv_s;
          const bool bad = !isfinite(x);
          bits |= (unsigned)bad << i;
          x = bad ? 0.0f : x;
          TE m1 = add_to<TE>(x, to_f(e[idx + i]));
          mo[idx + i] = m1;
          mmax = max(mmax, __float_as_uint(fabsf(to_f(m1))));
        }
      }
      cnt += __popc(bits);
      if (mask) {
        unsigned wv = bits << ((tid & 3) * 8);
        wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
        wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
        if ((tid & 3) == 0 && idx < numel) mask[idx >> 5] = wv;
      }
    }
    const unsigned bm = block_max(mmax, sh_u);
    if (tid == 0 && bm) atomicMax(reinterpret_cast<unsigned*>(mt.scal), bm);
  } else {
    const float* u = p.tab.unc_in[(size_t)sg.b * p.W + sg.w];
    for (int it = 0; it < kIngestIters; ++it) {
      const int64_t idx = base + (int64_t)it * kIngestThreads * kIngestVec + tid * kIngestVec;
      for (int i = 0; i < 8 && idx + i < sg.numel; ++i)
        cnt += !isfinite(u[idx + i] * inv_s);
    }
  }
  const int tot = block_sum(cnt, sh_i);
  if (tid == 0 && tot)
    atomicAdd(reinterpret_cast<unsigned long long*>(p.counts + (size_t)sg.b * p.W + sg.w),
              (unsigned long long)tot);
}

// skip[b] = (sum_w counts[b][w] >= threshold[b]); an integer decision, the same for
// every worker ("AIGC 基本功|混合精度与数值稳定性", §6.2: all ranks decide alike).
__global__ void k_skip(Plan p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  long long s = 0;
  for (int w = 0; w < p.W; ++w) s += p.counts[(size_t)b * p.W + w];
  p.skip[b] = (uint8_t)(s >= p.threshold[b]);
}

// Gains/biases: u = (sum_w zero_nonfinite(U_w * (1/s_b))) / W in fp32, fixed worker
// order; 0 for a skipped block.
__global__ void k_unc_out(Plan p) {
  const int b = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.unc_len) return;
  float* out = p.tab.unc_out[b];
  if (p.skip[b]) { out[i] = 0.0f; return; }
  const float inv_s = p.tab.inv_scale[b];
  float acc = 0.0f;
  for (int w = 0; w < p.W; ++w) {
    float x = p.tab.unc_in[(size_t)b * p.W + w][i] * inv_s;
    acc = __fadd_rn(acc, isfinite(x) ? x : 0.0f);
  }
  out[i] = __fdiv_rn(acc, (float)p.W);
}

}  // namespace

cudaError_t launch_ingest_range(const Handle& h, const Plan& p, cudaStream_t s, int64_t first, int64_t count) {
  if (count <= 0) return cudaSuccess;
  const int nseg = (int)h.segs.size();
  dim3 grid((unsigned)count);
  if (h.gdt == DT_F16) k_ingest<__half, __half><<<grid, kIngestThreads, 0, s>>>(p, h.d_segs, nseg, first);
  else if (h.gdt == DT_BF16) k_ingest<__nv_bfloat16, __nv_bfloat16><<<grid, kIngestThreads, 0, s>>>(p, h.d_segs, nseg, first);
  else k_ingest<float, float><<<grid, kIngestThreads, 0, s>>>(p, h.d_segs, nseg, first);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_ingest(const Handle& h, const Plan& p, cudaStream_t s) {
  return launch_ingest_range(h, p, s, 0, h.ingest_ctas);
}

// Gains/biases only: their nonfinite counts, for the skip decision (matrices are
// ingested by the fused tensor-core kernel).
cudaError_t launch_unc_count(const Handle& h, const Plan& p, cudaStream_t s) {
  return launch_ingest_range(h, p, s, h.unc_cta_start, h.ingest_ctas - h.unc_cta_start);
}

cudaError_t launch_skip_and_unc(const Handle& h, const Plan& p, cudaStream_t s) {
  k_skip<<<(p.B + 127) / 128, 128, 0, s>>>(p);
  if (p.unc_len > 0) {
    dim3 grid((unsigned)((p.unc_len + 255) / 256), (unsigned)p.B);
    k_unc_out<<<grid, 256, 0, s>>>(p);
    h.launches += 1;
  }
  h.launches += 1;
  return cudaGetLastError();
}

}  // namespace psgd
