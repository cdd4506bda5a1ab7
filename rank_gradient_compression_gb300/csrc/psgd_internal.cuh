// Internal declarations shared by the CUDA translation units of libpsgd.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "psgd.h"

namespace psgd {

enum : int { DT_F32 = PSGD_F32, DT_F16 = PSGD_F16, DT_BF16 = PSGD_BF16 };

// Device error word values (psgd_check maps them to psgd_status).
enum : int { DEVERR_NONE = 0, DEVERR_TIMEOUT = 1, DEVERR_BOUNDS = 2 };

// Per-matrix metadata, built once by psgd_init (t = b*J + j).
struct MatMeta {
  int64_t m, n;
  int32_t b, j;
  int32_t S;          // row slices of the Q GEMM (split-K over m)
  int32_t C;          // row chunks of the Gram matrix
  int32_t mtiles;     // 128-row tiles
  int32_t kchunks;    // column chunks of the P GEMM (tensor path)
  void* mscr;         // W consecutive m x n matrices, error dtype (M_w)
  float* P;           // m x rp fp32: P (mean over workers)
  float* Xa;          // m x rp fp32: orthonormalisation work buffers
  float* Xb;
  float* Phat;        // m x rp fp32: orthonormal basis
  int* ostate;        // [kMaxPasses][4]: final, dst buffer, shifted, dead columns
  float* Ppart;       // kchunks x mpad x rp fp32: P GEMM partial sums (tensor path)
  float* Qpart;       // S x n x rp fp32: Q GEMM partial sums
  float* Gpart;       // (C + 1) x rp x rp fp32: Gram partial sums, then their sum
  float* Rinv;        // rp x rp fp32: inverse Cholesky factor of the current pass
  uint16_t* qsplit;   // [2*rp][n] 16-bit: Q (scaled) hi rows then lo rows, K-major B
  uint16_t* psplit;   // [2*rp][mpad] 16-bit: P^ (scaled) hi rows then lo rows
  uint16_t* pdec;     // [mpad][3*rp] 16-bit: [P^hi | P^lo | P^hi] rows (decompress A)
  uint16_t* qdec;     // [npad][3*rp] 16-bit: [Q hi | Q hi | Q lo] rows (decompress B)
  float* xp;          // m x r fp32: exchange buffer of this rank's P sum (or NULL)
  float* xq;          // n x r fp32: exchange buffer of this rank's Q sum (or NULL)
  float* scal;        // [8] words, zeroed every step: max|M|, max|P|, max|Q| (state),
                      // max|Q| (new), the exponent shift of a rescaled M scratch (int)
};

constexpr int kMaxPasses = 4;  // CholeskyQR passes at most (shifted ones included)
constexpr int kRankBlock = 128;  // widest column block the orthonormalisation factors at once,
                                 // and the largest r of the tensor-core engine
constexpr int kMaxRank = 1024;   // largest r supported (the FFMA engine above kRankBlock)
constexpr int64_t kGramRows = 64;  // rows per partial sum of the Gram matrix X^T X

// Per-step device pointer tables (uploaded when they change).
struct StepTable {
  const void* const* g;          // [B*J*W]
  void* const* e;                // [B*J*W]
  float* const* q;               // [B*J]
  float* const* ghat;            // [B*J]
  const float* const* unc_in;    // [B*W] or null
  float* const* unc_out;         // [B] or null
  const float* inv_scale;        // [B]
  const void* ge_maps;           // [B*J*W][2] TMA maps of G and E (tensor engine) or null
};

// State of the cooperative orthonormalisation kernel's grid barrier (workspace; zeroed
// before every launch): arrivals, generation, and a flag that an expired wait raises.
struct GridBarrier {
  unsigned count, gen, abort, pad;
};

constexpr int kScalWords = 8;
enum { SC_MAXM = 0, SC_MAXP = 1, SC_MAXQ = 2, SC_MAXQN = 3, SC_MSHIFT = 4 };

struct Plan {
  int32_t B, J, W, r, rp;        // rp: r rounded up to a multiple of 16 (tensor path)
  int32_t gdt, edt;
  int64_t unc_len;
  const MatMeta* meta;           // [B*J]
  const int64_t* threshold;      // [B]
  StepTable tab;
  int64_t* counts;               // [B*W]
  uint8_t* skip;                 // [B]
  uint32_t* mask;                // bitmap or null
  const int64_t* mask_off;       // [B*J*W]
  int* err_word;
  // The column block the orthonormalisation kernels work on: width ob_r <= kRankBlock,
  // Gram / R^-1 pitch ob_rp, first column ob_c0 in the P / X buffers (pitch rp), and the
  // buffer pass 0 reads (0 = P, 1 = Xa, the block projected off the earlier blocks).
  // One block (ob_r = r, ob_rp = rp, ob_c0 = 0, ob_src0 = 0) when r <= kRankBlock.
  int32_t ob_r, ob_rp, ob_c0, ob_src0;
  int32_t debug_expire;          // PSGD_FLAG_DEBUG_EXPIRE_WAIT: the decompression kernel's
                                 // MMA thread waits on a barrier nothing completes
  float mean_div;                // divisor of the worker sums of P and Q: W, or 1 when the
                                 // sums go to the exchange buffers (psgd_step_p / _q)
  int32_t q_to_exchange;         // the Q reduction writes this rank's sum to MatMeta::xq
};

// Programmatic dependent launch. A kernel launched by launch_pdl may be scheduled while
// the kernel before it in the stream is still finishing; it calls pdl_wait() first, which
// returns once that kernel has completed and its memory operations are visible, so none
// of its reads or writes can overlap its predecessor's. Launched without the attribute,
// pdl_wait() returns at once. What the overlap saves is the launch latency between the
// short kernels of the step.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Flattened grids over the B*J matrices. Every block has the same J shapes, so matrix j of
// block 0 gives the item count of matrix j of every block: item i of the launch is item k
// of matrix t = b*J + j. A grid of B * sum_j count(j) blocks has no idle blocks, where a
// (max count, B*J) grid would launch, for every smaller matrix, blocks that leave at once.
template <typename F>
__device__ __forceinline__ void flat_item(const Plan& p, int64_t i, F count, int& t, int64_t& k) {
  int64_t per = 0;
  for (int j = 0; j < p.J; ++j) per += count(p.meta[j]);
  const int64_t b = i / per;
  int64_t rem = i - b * per;
  int j = 0;
  for (; j < p.J - 1; ++j) {
    const int64_t c = count(p.meta[j]);
    if (rem < c) break;
    rem -= c;
  }
  t = (int)b * p.J + j;
  k = rem;
}

// Barrier policies of device code that a group of threads runs: the whole CTA
// (__syncthreads), or one 256-thread half of a 512-thread CTA (named barrier 1 or 2).
struct CtaBar {
  __device__ __forceinline__ void sync() const { __syncthreads(); }
};
struct HalfBar {
  uint32_t id;
  __device__ __forceinline__ void sync() const { asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory"); }
};

// Max of v over the block, returned in thread 0 (every thread of the block must call it;
// blockDim.x a multiple of 32). One atomic per block instead of one per warp: atomics on
// one address serialise at its L2 slice.
__device__ __forceinline__ unsigned block_max_u32(unsigned v) {
  __shared__ unsigned s_wmax[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = __reduce_max_sync(0xffffffffu, v);
  if (lane == 0) s_wmax[warp] = v;
  __syncthreads();
  unsigned r = 0u;
  if (warp == 0) {
    r = lane < (int)(blockDim.x >> 5) ? s_wmax[lane] : 0u;
    r = __reduce_max_sync(0xffffffffu, r);
  }
  return r;
}

// Stages the first `count` floats of a contiguous run src[0 .. count) into a 32-row
// shared-memory tile xs (`len` entries per row, row stride kRankBlock + 1, count <= 32 *
// len, len <= kRankBlock) as xs[i / len][i % len] = f(src[i], i % len); every other entry
// of rows 0..31, columns 0..len-1 gets 0. Each thread issues all of its loads before its
// first store: interleaved, every load would wait for the shared-memory store before it,
// since the compiler cannot rule out that src points into shared memory. src is read
// through the read-only path (it is not written during the kernel).
template <int kThreads, typename F>
__device__ __forceinline__ void stage_rows(float (*xs)[kRankBlock + 1], const float* src,
                                           int count, int len, F f) {
  constexpr int kPer = (32 * kRankBlock + kThreads - 1) / kThreads;
  float v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = (int)threadIdx.x + u * kThreads;
    v[u] = i < count ? __ldg(src + i) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = (int)threadIdx.x + u * kThreads;
    if (i < 32 * len) {
      const int rr = i / len, c = i - rr * len;
      xs[rr][c] = i < count ? f(v[u], c) : 0.f;
    }
  }
}

// ---------------------------------------------------------------- numerics helpers
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// a + b rounded to odd in fp32. The two directed roundings bracket the exact sum: equal
// when it is exact, else adjacent floats, and exactly one of those has an odd
// significand. A second rounding of a round-to-odd result to a format with at most 22
// significant bits is the correctly rounded (RNE) sum in that format (Boldo &
// Melquiond, "When double rounding is odd"). This lets M = round_E(g + E) and
// E = round_E(M - G^) equal a single rounding of the exact fp32-operand sum.
__device__ __forceinline__ float add_round_odd(float a, float b) {
  const float up = __fadd_ru(a, b), dn = __fadd_rd(a, b);
  return (up == dn || (__float_as_uint(up) & 1u)) ? up : dn;
}

// hi + lo += a * b, with hi + lo an unevaluated sum of two floats. The product's rounding
// error comes out of one FMA (exact), the sum's from Knuth's branch-free TwoSum (exact), and
// both go into lo. A dot product accumulated this way is as accurate as one carried in
// twice the working precision and rounded once at the end (Ogita, Rump and Oishi,
// "Accurate sum and dot product", 2005, Dot2). The _rn intrinsics keep the compiler from
// contracting the error terms into FMAs.
__device__ __forceinline__ void dot2_acc(float& hi, float& lo, float a, float b) {
  const float p = __fmul_rn(a, b);
  const float pe = fmaf(a, b, -p);
  const float s = __fadd_rn(hi, p);
  const float z = __fsub_rn(s, hi);
  const float se = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, z)), __fsub_rn(p, z));
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(pe, se));
}

// round_E(a + b) with E = T; exact single rounding for 16-bit T, plain RN for fp32.
template <typename T> __device__ __forceinline__ T add_to(float a, float b) {
  return from_f<T>(add_round_odd(a, b));
}
template <> __device__ __forceinline__ float add_to<float>(float a, float b) {
  return __fadd_rn(a, b);
}

// Bounded spin: returns false after `limit` polls.
#define PSGD_SPIN_LIMIT (1u << 26)

}  // namespace psgd

// Launchers implemented in the .cu files (host side). Each returns cudaGetLastError().
namespace psgd {
struct Handle;
cudaError_t launch_ingest(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_unc_count(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_skip_and_unc(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_pgemm_simt(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_orth(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_qgemm_simt(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_qreduce(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_decomp_simt(const Handle& h, const Plan& p, cudaStream_t s);
}  // namespace psgd
