// The orthonormalisation passes of every P of a step (r <= 128) in one cooperative launch.
//
// The separate-kernel version (orth.cu) enqueues, per CholeskyQR pass, a Gram sum, a
// Cholesky and an X R^-1 kernel, and four passes always, since whether a pass runs is
// decided on the device. After a warm start one pass is final, so most of those launches
// return at once, and each costs a few microseconds of launch, drain and ramp. Here one
// kernel runs the phases back to back with grid-wide barriers between them. The step
// runs pass 0 as separate kernels (their several CTAs per SM hide latency better than
// this kernel's one 512-thread CTA per SM) and then this kernel from pass 1, which leaves
// at once when no matrix needs another pass. The kernel can also run everything:
//
//   [P = (sum of the P GEMM's partial sums) / W, max|P|]     (tensor engine)
//   Gram partials of pass 0
//   per pass: Gram sum | Cholesky + R^-1 (one CTA per matrix) | X R^-1 and the next
//             pass's Gram partials; stop when every matrix's last pass was final
//   [the Q GEMM's split P^ operand and the decompression's P^ operand]  (tensor engine)
//
// The phases run the device code of orth_dev.cuh and split_dev.cuh, so the arithmetic,
// its order and the results are those of the separate kernels, bit for bit. A CTA has 512
// threads: the Cholesky uses all of them, the other phases run two 256-thread groups per
// CTA, each with its own named barrier and shared memory. The launch is cooperative, so
// every CTA is resident at once and a grid barrier cannot wait on a CTA that never
// starts. Barrier waits are bounded: on expiry the kernel records DEVERR_TIMEOUT and every
// CTA leaves (psgd_check reports it).
#include <algorithm>

#include "orth_dev.cuh"
#include "split_dev.cuh"

namespace psgd {
namespace {

using namespace orthdev;
using namespace splitdev;

constexpr int kCoopThreads = kCholThreads;  // 512: the Cholesky's 16 warps, or 2 groups
static_assert(kCoopThreads == 2 * kT, "two 256-thread groups per CTA");
constexpr int kGroupSmem = (kGramRows * 128 + 32 * 128) * 4;  // gram / apply: 48 KB per group
constexpr int kPreduceVec = kCoopThreads * 4;                 // floats per P-reduce item
constexpr uint32_t kGridSpinLimit = 1u << 22;                 // polls of a barrier wait

struct CoopArgs {
  GridBarrier* gbar;  // zeroed before every launch
  int fused_preduce;  // tensor engine: form P from the P GEMM's partial sums first
  int do_psplit;      // tensor engine: write psplit / pdec at the end
  int kp;             // K pad of the decompression terms
  int pchunk_kb;      // P GEMM k-blocks per partial sum
  int start_pass;     // first pass to run; > 0: the earlier passes ran as separate kernels
};

// Grid-wide barrier. Thread 0 of every CTA arrives; the last arrival resets the count and
// advances the generation that the others poll. Memory written before the barrier by any
// CTA is visible after it (fences on both sides; the phases read it at L2).
__device__ bool grid_barrier(GridBarrier* gb, int* err) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile unsigned* vgen = &gb->gen;
    const unsigned g = *vgen;
    __threadfence();
    volatile unsigned* vabort = &gb->abort;
    if (atomicAdd(&gb->count, 1u) == gridDim.x - 1) {
      atomicExch(&gb->count, 0u);
      __threadfence();
      atomicAdd(&gb->gen, 1u);
    } else {
      for (uint32_t i = 0; *vgen == g; ++i) {
        if (*vabort) { ok = 0; break; }  // another CTA's wait expired: leave at once
        if (i >= kGridSpinLimit) {
          ok = 0;
          *vabort = 1u;
          atomicCAS(err, DEVERR_NONE, DEVERR_TIMEOUT);
          break;
        }
        if (i > 16) __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Item i of a phase whose matrix j (of every block) has count(j) items, blocks in order:
// returns the matrix t = b*J + j and the item's index k within that matrix.
template <typename F>
__device__ __forceinline__ void decode(const Plan& p, int64_t i, int per_block, F count, int& t, int& k) {
  const int b = (int)(i / per_block);
  int rem = (int)(i - (int64_t)b * per_block), j = 0;
  for (; j < p.J - 1; ++j) {
    const int c = count(j);
    if (rem < c) break;
    rem -= c;
  }
  t = b * p.J + j;
  k = rem;
}

template <typename F>
__device__ __forceinline__ int per_block_items(const Plan& p, F count) {
  int n = 0;
  for (int j = 0; j < p.J; ++j) n += count(j);
  return n;
}

template <typename TE>
__global__ void __launch_bounds__(kCoopThreads, 1) k_orth_coop(Plan p, CoopArgs ca) {
  extern __shared__ __align__(16) unsigned char coop_smem[];
  __shared__ int s_more;
  const int half = threadIdx.x >> 8, tid = threadIdx.x & (kT - 1);
  const HalfBar hb{1u + (unsigned)half};
  const int64_t grp = (int64_t)blockIdx.x * 2 + half, ngrp = (int64_t)gridDim.x * 2;
  unsigned char* gsm = coop_smem + (size_t)half * kGroupSmem;  // this group's shared memory
  int* err = p.err_word;
  const int T = p.B * p.J;
  auto chunks = [&](int j) { return p.meta[j].C; };
  auto mpad32 = [&](int j) { return (int)((p.meta[j].m + 127) / 128 * 4); };

  // Resumed after separate-kernel passes: leave at once (every CTA alike) when no matrix
  // needs the next pass, which after a warm start is the common case.
  if (ca.start_pass > 0) {
    if (threadIdx.x == 0) {
      int more = 0;
      for (int t = 0; t < T && !more; ++t) more = !pass_skipped(p, p.meta[t], ca.start_pass);
      s_more = more;
    }
    __syncthreads();
    if (!s_more && !ca.do_psplit) return;
  }

  // ---- P = (sum of the partial sums in chunk order) / W, and max|P| per matrix
  if (ca.fused_preduce) {
    auto pitems = [&](int j) { return (int)((p.meta[j].m * p.rp + kPreduceVec - 1) / kPreduceVec); };
    const int per = per_block_items(p, pitems);
    for (int64_t it = blockIdx.x; it < (int64_t)per * p.B; it += gridDim.x) {
      int t, k;
      decode(p, it, per, pitems, t, k);
      const MatMeta& mt = p.meta[t];
      unsigned mx = 0u;
      if (!p.skip[mt.b]) {
        const int64_t i = (int64_t)k * kPreduceVec + threadIdx.x * 4;
        if (i < mt.m * p.rp) {
          const int64_t mpad = (mt.m + 127) / 128 * 128;
          const int kch = (int)(((mt.n + 63) / 64 + ca.pchunk_kb - 1) / ca.pchunk_kb);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
          for (int c = 0; c < kch; ++c) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(mt.Ppart + (size_t)c * mpad * p.rp + i));
            acc.x = __fadd_rn(acc.x, v.x); acc.y = __fadd_rn(acc.y, v.y);
            acc.z = __fadd_rn(acc.z, v.z); acc.w = __fadd_rn(acc.w, v.w);
          }
          const float fw = p.mean_div;
          float4 o;
          o.x = __fdiv_rn(acc.x, fw); o.y = __fdiv_rn(acc.y, fw);
          o.z = __fdiv_rn(acc.z, fw); o.w = __fdiv_rn(acc.w, fw);
          *reinterpret_cast<float4*>(mt.P + i) = o;
          mx = max(max(__float_as_uint(fabsf(o.x)), __float_as_uint(fabsf(o.y))),
                   max(__float_as_uint(fabsf(o.z)), __float_as_uint(fabsf(o.w))));
        }
      }
      mx = block_max_u32(mx);
      if (threadIdx.x == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + SC_MAXP, mx);
      __syncthreads();  // block_max_u32's buffer is reused by the next item
    }
    if (!grid_barrier(ca.gbar, err)) return;
  }

  // ---- Gram partials of pass 0 (later passes get theirs from the X R^-1 phase)
  if (ca.start_pass == 0) {
    const int per = per_block_items(p, chunks);
    for (int64_t it = grp; it < (int64_t)per * p.B; it += ngrp) {
      int t, c;
      decode(p, it, per, chunks, t, c);
      const MatMeta& mt = p.meta[t];
      if (pass_skipped(p, mt, 0)) continue;
      float* f = reinterpret_cast<float*>(gsm);
      gram_chunk(p, mt, 0, c, reinterpret_cast<float (*)[128]>(f), f + kGramRows * 128, tid, hb);
      hb.sync();  // the group's shared memory is reused by its next item
    }
    if (!grid_barrier(ca.gbar, err)) return;
  }

  for (int pass = ca.start_pass; pass < kMaxPasses; ++pass) {
    if (pass == ca.start_pass && pass > 0 && !s_more) break;
    // ---- Gram sum
    {
      const int per_mat = gsum_items(p.ob_rp);
      for (int64_t it = grp; it < (int64_t)per_mat * T; it += ngrp) {
        const int t = (int)(it / per_mat), k = (int)(it - (int64_t)t * per_mat);
        const MatMeta& mt = p.meta[t];
        if (pass_skipped(p, mt, pass)) continue;
        gsum_item(p, mt, k, reinterpret_cast<float (*)[32]>(gsm), tid, hb);
      }
      if (!grid_barrier(ca.gbar, err)) return;
    }
    // ---- Cholesky and R^-1: one CTA per matrix
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      const MatMeta& mt = p.meta[t];
      if (pass_skipped(p, mt, pass)) continue;
      chol_matrix(p, mt, pass, *reinterpret_cast<CholSmem*>(coop_smem));
      __syncthreads();  // the Cholesky's shared memory is reused by the next matrix
    }
    if (!grid_barrier(ca.gbar, err)) return;
    // ---- X <- X R^-1, and the next pass's Gram partials where this pass is not final
    {
      const int per = per_block_items(p, chunks);
      for (int64_t it = grp; it < (int64_t)per * p.B; it += ngrp) {
        int t, tile;
        decode(p, it, per, chunks, t, tile);
        const MatMeta& mt = p.meta[t];
        if (pass_skipped(p, mt, pass)) continue;
        float* f = reinterpret_cast<float*>(gsm);
        apply_tile<false>(p, mt, pass, tile, f, f + kGramRows * 128, tid, hb);
        hb.sync();
      }
      if (!grid_barrier(ca.gbar, err)) return;
    }
    // ---- another pass? (the same answer in every CTA: it reads what the barrier published)
    if (threadIdx.x == 0) {
      int more = 0;
      if (pass + 1 < kMaxPasses)
        for (int t = 0; t < T && !more; ++t) more = !pass_skipped(p, p.meta[t], pass + 1);
      s_more = more;
    }
    __syncthreads();
    if (!s_more) break;
  }

  // ---- split P^ for the Q GEMM (psplit) and the decompression (pdec)
  if (ca.do_psplit) {
    const int per = per_block_items(p, mpad32);
    for (int64_t it = grp; it < (int64_t)per * p.B; it += ngrp) {
      int t, blk;
      decode(p, it, per, mpad32, t, blk);
      const MatMeta& mt = p.meta[t];
      if (p.skip[mt.b]) continue;
      psplit_rows<TE>(p, mt, ca.kp, blk, reinterpret_cast<float (*)[kRankBlock + 1]>(gsm), tid, hb);
    }
  }
}

constexpr size_t kCoopSmem = std::max<size_t>(sizeof(CholSmem), 2 * (size_t)kGroupSmem);

}  // namespace

// The kernel's grid: one CTA per SM, fewer if the device cannot hold one per SM (0 on error).
int orth_coop_grid() {
  static int grid = -1;
  if (grid >= 0) return grid;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaFuncSetAttribute(k_orth_coop<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCoopSmem) != cudaSuccess ||
      cudaFuncSetAttribute(k_orth_coop<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCoopSmem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_orth_coop<__half>, kCoopThreads, kCoopSmem) != cudaSuccess) {
    cudaGetLastError();
    return grid = 0;
  }
  return grid = (per_sm >= 1 && sms > 0) ? sms : 0;
}

cudaError_t launch_orth_coop(const Handle& h, const Plan& p, bool fused_preduce, bool do_psplit, int kp,
                             int pchunk_kb, int start_pass, cudaStream_t s) {
  const int grid = orth_coop_grid();
  if (grid <= 0) return cudaErrorCooperativeLaunchTooLarge;
  CoopArgs ca{h.d_gbar, fused_preduce ? 1 : 0, do_psplit ? 1 : 0, kp, pchunk_kb, start_pass};
  cudaError_t e = cudaMemsetAsync(h.d_gbar, 0, sizeof(GridBarrier), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCoopThreads);
  cfg.dynamicSmemBytes = kCoopSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (h.edt == DT_BF16) e = cudaLaunchKernelEx(&cfg, k_orth_coop<__nv_bfloat16>, p, ca);
  else e = cudaLaunchKernelEx(&cfg, k_orth_coop<__half>, p, ca);
  h.launches += 1;
  return e;
}

}  // namespace psgd
