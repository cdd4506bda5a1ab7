// Tensor-core engine (tcgen05 + TMA, sm_103a) of the step's three matrix products.
//
//   P GEMM   P_part = sum_w M_w[rows, k-chunk] (Q_hi | Q_lo)[k-chunk]     A K-major
//   Q GEMM   Q_part = sum_w M_w[k-slice, cols]^T (P^_hi | P^_lo)[k-slice] A MN-major
//   G^       G^ = (P^_hi | P^_lo | P^_hi) (Q_hi | Q_hi | Q_lo)^T, then E_w = round_E(M_w - G^)
//
// M is exact in its 16-bit type. The fp32 operand (Q or P^) is scaled by a power of two
// and split into 16-bit terms: x*2^e = hi + lo for fp16 (~22 significant bits), and
// hi + mid + lo for bf16 (~24). One pass over M multiplies it by every term: the fused P
// GEMM issues one MMA per term into the same accumulator columns, and the Q GEMM one MMA
// of width 2 rp for the first two terms side by side (the epilogue adds the two column
// ranges). A plain 16-bit product would keep 11 (fp16) or 8 (bf16) bits. The decompression
// ("32-bit products for the decompressed gradient", "Zero-Shot Text-to-Image Generation -
// 中文验证版", §证据) uses three products of fp16 splits, so a dropped lo*lo term costs
// ~2^-22.
//
// Persistent kernels, one CTA per SM. Warp 0 issues TMA loads into a ring of
// shared-memory stages. Warp 1 owns TMEM and issues tcgen05.mma from one thread. Four
// (fused P GEMM) or eight (Q GEMM, G^) epilogue warps drain the accumulators, which are
// double buffered in TMEM so the next segment's MMAs overlap the epilogue. Every mbarrier wait is
// bounded. On expiry the kernel records DEVERR_TIMEOUT, waits (bounded) for its own
// TMA loads, releases TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <type_traits>
#include <vector>

#include "handle.h"
#include "split_dev.cuh"
#include "tc_ptx.cuh"

namespace psgd {
namespace {

using namespace tc;
using namespace splitdev;

constexpr int kDynSmemCap = 227 * 1024 - 256;  // dynamic shared memory of the persistent kernels
constexpr int BM = 128;                // MMA M and A-tile rows (MN extent)
constexpr int BK = 64;                 // K per stage (one 128-byte swizzle span)
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_STAGES = 2;
constexpr int PCHUNK_KB = 4;           // P GEMM: k-blocks of 64 columns per unit
// Accumulator segments. The tensor cores' fp32 accumulation loses about 2^-24 of the
// accumulator per chained MMA, and those losses add up (they do not cancel like
// round-to-nearest errors). So an accumulator chains a bounded number of MMAs: after each
// segment of (k-block, worker) steps the epilogue adds the accumulator into a running sum
// with round-to-nearest fp32 adds. The fused ingest kernel issues one MMA per split term of
// Q into the same accumulator of rp columns, so a (k-block, worker) step chains 8 (fp16)
// or 12 (bf16) MMAs and a segment of 4 steps 32; it keeps the running sum in TMEM next to
// two accumulators. The separate GEMM kernel multiplies the first two split terms in one
// MMA of width 2 rp (term 0's products in columns [0, rp), term 1's in [rp, 2 rp); bf16's
// third term goes onto term 0's columns), so a step chains 4 (fp16) or 8 (bf16) MMAs per
// column and a segment of 16 steps 64 (fp16); the epilogue adds the two column ranges and
// keeps the running sum in registers, with two accumulators in TMEM. P's segments are
// shorter than Q's: errors in P are amplified by
// cond(P) in the span of P^ (up to ~2e4 for a decaying spectrum at r = 112), errors in
// Q reach G^ and E directly.
constexpr int kGemmSegSteps = 16;
constexpr int kIngSegSteps = 4;
constexpr int QSLICE_ROWS = 256;       // Q GEMM: rows of m per unit (matches Qpart slices)
constexpr int DEC_NT = 128;            // G^ tile columns
constexpr int NMAPS = 6;               // tensor maps per matrix
enum { MAP_MP = 0, MAP_MQ = 1, MAP_QS = 2, MAP_PS = 3, MAP_PD = 4, MAP_QD = 5 };

struct Unit {
  int32_t t, tile, kb0, kb1, slot, pad;
};

struct TcPlan {
  CUtensorMap* d_maps = nullptr;   // [B*J*NMAPS]
  Unit* d_punits = nullptr;
  Unit* d_qunits = nullptr;
  Unit* d_dunits = nullptr;
  int np = 0, nq = 0, nd = 0;
  int kp = 0;                      // K pad of each decompression term (multiple of 64)
  int qkps = 1;                    // Q GEMM k-blocks per stage
  int grid = 0;
};

__host__ __device__ inline int kpad_of(int rp) { return (rp + 63) / 64 * 64; }

// ---------------------------------------------------------------- small kernels
// max|Q| of the caller's Q state -> scal[2] (bits). grid = (qmax_blocks, B*J). This and k_qsplit
// run for every matrix: they can precede the skip decision of the step.
__global__ void k_qmax(Plan p) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  const float* q = p.tab.q[blockIdx.y];
  const int64_t total = mt.n * p.r;
  unsigned mx = 0u;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
    mx = max(mx, __float_as_uint(fabsf(q[i])));
  mx = block_max_u32(mx);
  if (threadIdx.x == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + 2, mx);
}

// qsplit[terms*rp][n]: rows k*rp + c hold term k of Q[:, c] * 2^e (k = 0 hi, then mid
// for bf16, then lo); e puts max|Q| * 2^e in [2^14, 2^15). Padding rows are 0.
// A block stages 32 rows of Q (n x r row-major: one contiguous run) in shared memory,
// then writes 8 consecutive entries of one qsplit row per 16-byte store (n is a multiple
// of 8, so a group of 8 is wholly inside or outside the matrix). grid = (ceil(n/32), B*J).
template <typename T>
__global__ void __launch_bounds__(256) k_qsplit(Plan p) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  const int64_t j0 = (int64_t)blockIdx.x * 32;
  if (j0 >= mt.n) return;
  const int r = p.r, rp = p.rp;
  __shared__ float xs[32][kRankBlock + 1];
  const float* q = p.tab.q[blockIdx.y] + j0 * r;
  const int64_t left = mt.n - j0;
  const int nrows = left < 32 ? (int)left : 32;
  const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[2]);
  stage_rows<256>(xs, q, nrows * r, r, [e](float v, int) { return ldexpf(v, e); });
  __syncthreads();
  for (int it = threadIdx.x; it < rp * 4; it += blockDim.x) {
    const int c = it >> 2, g = it & 3;
    if (8 * g >= nrows) continue;
    __align__(16) uint16_t t0[8], t1[8], t2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      t0[i] = t1[i] = t2[i] = 0;
      if (c < r) {
        if (nterms<T>() == 3) split3<T>(xs[8 * g + i][c], t0[i], t1[i], t2[i]);
        else split2<T>(xs[8 * g + i][c], t0[i], t1[i]);
      }
    }
    const size_t col = (size_t)j0 + 8 * g;
    *reinterpret_cast<uint4*>(mt.qsplit + (size_t)c * mt.n + col) = *reinterpret_cast<const uint4*>(t0);
    *reinterpret_cast<uint4*>(mt.qsplit + (size_t)(rp + c) * mt.n + col) = *reinterpret_cast<const uint4*>(t1);
    if (nterms<T>() == 3)
      *reinterpret_cast<uint4*>(mt.qsplit + (size_t)(2 * rp + c) * mt.n + col) = *reinterpret_cast<const uint4*>(t2);
  }
}

// P = (sum_c Ppart[c]) / W in chunk order, plus max|P| -> scal[1]. P keeps the power-of-
// two scale 2^e of the split Q: P^ does not depend on it, and removing it would push P
// below fp32's range when both M and Q are tiny (deep blocks of the stack, M ~ Q ~ 2^-80).
// Flattened grid (flat_item): B * sum_j ceil(m_j rp / 1024) blocks of 256 threads.
__global__ void k_preduce(Plan p, int pchunk_kb) {
  pdl_wait();
  int t;
  int64_t item;
  flat_item(p, blockIdx.x, [&](const MatMeta& m) { return (m.m * p.rp + 1023) / 1024; }, t, item);
  const MatMeta& mt = p.meta[t];
  if (p.skip[mt.b]) return;
  const int rp = p.rp;
  const int64_t i = (item * blockDim.x + threadIdx.x) * 4;
  const int64_t mpad = (mt.m + 127) / 128 * 128;
  unsigned mx = 0u;
  if (i < mt.m * rp) {
    const int kch = (int)(((mt.n + 63) / 64 + pchunk_kb - 1) / pchunk_kb);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int c = 0; c < kch; ++c) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(mt.Ppart + (size_t)c * mpad * rp + i));
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
  mx = block_max_u32(mx);
  if (threadIdx.x == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + 1, mx);
}

// From P^ (m x rp fp32): the Q GEMM's split operand and the decompression's A operand,
// 32 rows of P^ per CTA (psplit_rows). Flattened grid: B * sum_j mpad_j / 32 blocks.
template <typename T>
__global__ void __launch_bounds__(256) k_psplit(Plan p, int kp) {
  pdl_wait();
  int t;
  int64_t item;
  flat_item(p, blockIdx.x, [](const MatMeta& m) { return (m.m + 127) / 128 * 4; }, t, item);
  const MatMeta& mt = p.meta[t];
  if (p.skip[mt.b]) return;
  __shared__ float xs[32][kRankBlock + 1];
  psplit_rows<T>(p, mt, kp, (int)item, xs, threadIdx.x, CtaBar{});
}

// qdec[npad][3 kp] = [hi | hi | lo] of the new Q * 2^e in fp16 (e from max|Q|, scal[3]).
// A block stages 32 rows of Q (n x r row-major) in shared memory and writes 8 columns
// per 16-byte store. grid = (npad / 32, B*J).
__global__ void __launch_bounds__(256) k_qdec(Plan p, int kp) {
  pdl_wait();
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const int64_t npad = (mt.n + DEC_NT - 1) / DEC_NT * DEC_NT;
  const int64_t row0 = (int64_t)blockIdx.x * 32;
  if (row0 >= npad) return;
  const int r = p.r;
  __shared__ float xs[32][kRankBlock + 1];
  const int64_t left = mt.n - row0;
  const int nrows = left <= 0 ? 0 : (left < 32 ? (int)left : 32);
  const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[3]);
  const float* q = p.tab.q[blockIdx.y] + row0 * r;
  stage_rows<256>(xs, q, nrows * r, r, [e](float v, int) { return ldexpf(v, e); });
  __syncthreads();
  const int gpr = kp / 8;
  for (int it = threadIdx.x; it < 32 * gpr; it += blockDim.x) {
    const int rr = it / gpr, c0 = (it - rr * gpr) * 8;
    __align__(16) uint16_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      split2<__half>((rr < nrows && c0 + i < r) ? xs[rr][c0 + i] : 0.f, hi[i], lo[i]);
    uint16_t* qd = mt.qdec + (size_t)(row0 + rr) * 3 * kp;
    *reinterpret_cast<uint4*>(qd + c0) = *reinterpret_cast<const uint4*>(hi);
    *reinterpret_cast<uint4*>(qd + kp + c0) = *reinterpret_cast<const uint4*>(hi);
    *reinterpret_cast<uint4*>(qd + 2 * kp + c0) = *reinterpret_cast<const uint4*>(lo);
  }
}

// ---------------------------------------------------------------- GEMM kernel
// Shared memory, carved at run time: a_stages A tiles (16 KB each), B_STAGES B tiles of
// b_stage bytes (1 KB multiples), then the barriers and the TMEM address slot.
constexpr int kMaxAStages = 12;
constexpr int kGemmAccs = 2;  // TMEM accumulators of the separate GEMMs (256 columns each)
struct GemmBars {
  uint64_t full_a[kMaxAStages], empty_a[kMaxAStages];
  uint64_t full_b[B_STAGES], empty_b[B_STAGES];
  uint64_t acc_full[kGemmAccs], acc_empty[kGemmAccs], done;
  uint32_t tmem;
};
struct GemmSmem {
  uint8_t* a0;
  uint8_t* b0;
  GemmBars* bar;
  uint32_t a_bytes;
  __device__ uint8_t* a(int s) const { return a0 + (size_t)s * a_bytes; }
  __device__ uint8_t* b(int s, uint32_t b_stage) const { return b0 + (size_t)s * b_stage; }
};

// A unit is left out for a skipped block, and, in the rerun over rescaled bf16
// matrices (only_shifted), for every matrix whose M scratch was not rescaled.
__device__ __forceinline__ bool unit_off(const Plan& p, const MatMeta& mt, int only_shifted) {
  if (p.skip[mt.b]) return true;
  return only_shifted && reinterpret_cast<const int*>(mt.scal)[SC_MSHIFT] == 0;
}

// The sequence of (unit, k-block, worker) A stages of a CTA's units, skipping units that are
// off; the Q GEMM's producer walks a copy of it kPrefetchStages ahead of its loads and
// prefetches those boxes into L2.
constexpr int kPrefetchStages = 3;
struct AStageIter {
  int u, u_end, u_step, kb, w;
  bool valid;
  __device__ void seek(const Plan& p, const Unit* units, int only_shifted);
  __device__ void next(const Plan& p, const Unit* units, int only_shifted, int kps) {
    if (++w < p.W) return;
    w = 0;
    kb += kps;
    if (kb < units[u].kb1) return;
    u += u_step;
    seek(p, units, only_shifted);
  }
};

__device__ void AStageIter::seek(const Plan& p, const Unit* units, int only_shifted) {
  for (; u < u_end; u += u_step)
    if (!unit_off(p, p.meta[units[u].t], only_shifted)) {
      kb = units[u].kb0;
      w = 0;
      valid = true;
      return;
    }
  valid = false;
}

// MN_A = false: P GEMM (A = M tile K-major, unit = row tile x k-chunk).
// MN_A = true:  Q GEMM (A = M^T tile MN-major, unit = column tile x m-slice).
// kps (Q GEMM): k-blocks per stage. With 2, an A stage is 128 rows of M (two 64 x 128-row
// boxes, 32 KB) and a B stage holds the two k-blocks' split P^ tiles. 128-row boxes read
// HBM at 5.7 TB/s where 64-row boxes of the same columns reach 3.6 (a pure TMA read of
// the M scratch on GB300). The MMA steps through the stage's k-blocks in order.
constexpr int kGemmThreads = 320;  // warps: 0 TMA, 1 MMA, 2..9 epilogue
constexpr int kGemmEpiWarps = 8;   // two per TMEM lane quarter, each with half the columns
template <bool MN_A, bool BF16>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_gemm(Plan p, const CUtensorMap* __restrict__ maps, const Unit* __restrict__ units, int nunits,
       int a_stages, uint32_t b_stage, int only_shifted, int seg, int kps, int contig) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t a_bytes = (uint32_t)kps * A_BYTES;  // one A stage
  GemmSmem S{base, base + (size_t)a_stages * a_bytes,
             reinterpret_cast<GemmBars*>(base + (size_t)a_stages * a_bytes + (size_t)B_STAGES * b_stage), a_bytes};
  GemmBars& sm = *S.bar;
  const int A_STAGES = a_stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int TERMS = BF16 ? 3 : 2;
  const int rp = p.rp, N = TERMS * rp;          // B rows: the split terms, rp rows each
  // One MMA of N = 2 rp multiplies the A tile by the first two split terms side by side
  // (B rows [0, 2 rp)), so the tensor core reads each A tile once per K step instead of
  // once per term: below N = 256 an MMA's time is set by the shared-memory bytes it reads.
  // Accumulator columns [0, rp) hold term 0's products, [rp, 2 rp) term 1's; the third
  // term of bf16 goes onto term 0's columns. The epilogue adds the two halves. Two
  // accumulators of 256 columns fit in TMEM: the MMA can run a segment ahead of the drain.
  constexpr int NACC = kGemmAccs;
  constexpr uint32_t kAccCols = 256;
  static_assert(NACC * kAccCols <= 512 && kAccCols >= 2 * kRankBlock, "accumulators fit in TMEM");
  const int NBOX = N <= 256 ? 1 : 2;            // TMA boxes per B tile (<= 256 rows each)
  const uint32_t b_bytes = (uint32_t)N * BK * 2;  // one k-block's B tile
  const uint32_t b_tile = b_stage / (uint32_t)kps;  // its slot in a B stage (1 KB multiple)
  int* err = p.err_word;
  // Units of this CTA: every gridDim.x-th one, or (contig) one contiguous range, so that
  // consecutive units can share the rows of M and with them the B operand.
  const int u_first = contig ? (int)((int64_t)blockIdx.x * nunits / gridDim.x) : (int)blockIdx.x;
  const int u_end = contig ? (int)((int64_t)(blockIdx.x + 1) * nunits / gridDim.x) : nunits;
  const int u_step = contig ? 1 : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < A_STAGES; ++i) { mbar_init(&sm.full_a[i], 1); mbar_init(&sm.empty_a[i], 1); }
    for (int i = 0; i < B_STAGES; ++i) { mbar_init(&sm.full_b[i], 1); mbar_init(&sm.empty_b[i], 1); }
    for (int i = 0; i < kGemmAccs; ++i) { mbar_init(&sm.acc_full[i], 1); mbar_init(&sm.acc_empty[i], kGemmEpiWarps); }
    mbar_init(&sm.done, 1);
    abort_reset();
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // M (A) is streamed once; the split B tiles are re-read by every column tile of a slice
      const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
      uint32_t ia = 0, ib = 0;
      static_assert(B_STAGES == 2, "two B tags");
      int64_t b_tag0 = -1, b_tag1 = -1;  // (matrix, first k-block) each B stage holds, -1: none
      bool ok = true;
      // L2 prefetch of the A boxes kPrefetchStages stages ahead (Q GEMM)
      AStageIter pf{u_first, u_end, u_step, 0, 0, false};
      auto prefetch_next = [&]() {
        if (!pf.valid) return;
        const Unit un = units[pf.u];
        const CUtensorMap* mm = maps + (size_t)un.t * NMAPS + MAP_MQ;
        tma_prefetch_3d(mm, un.tile * BM, pf.kb * BK, pf.w);
        tma_prefetch_3d(mm, un.tile * BM + 64, pf.kb * BK, pf.w);
        pf.next(p, units, only_shifted, kps);
      };
      if (MN_A) {
        pf.seek(p, units, only_shifted);
        for (int i = 0; i < kPrefetchStages; ++i) prefetch_next();
      }
      for (int u = u_first; u < u_end && ok; u += u_step) {
        const Unit un = units[u];
        const MatMeta& mt = p.meta[un.t];
        if (unit_off(p, mt, only_shifted)) continue;
        const CUtensorMap* mm = maps + (size_t)un.t * NMAPS + (MN_A ? MAP_MQ : MAP_MP);
        const CUtensorMap* mb = maps + (size_t)un.t * NMAPS + (MN_A ? MAP_PS : MAP_QS);
        for (int kb = un.kb0; kb < un.kb1 && ok; kb += kps) {
          const int nk = min(kps, un.kb1 - kb);  // k-blocks of this stage
          const int sb = ib % B_STAGES;
          ok = mbar_wait(&sm.empty_b[sb], ((ib / B_STAGES) & 1) ^ 1, err);
          if (!ok) break;
          const int64_t tag = ((int64_t)un.t << 32) | ((int64_t)kb << 8) | nk;
          if ((sb ? b_tag1 : b_tag0) == tag) {
            mbar_arrive(&sm.full_b[sb]);  // the stage still holds these k-blocks' B tiles
          } else {
            if (sb) b_tag1 = tag; else b_tag0 = tag;
            mbar_arrive_expect_tx(&sm.full_b[sb], (uint32_t)nk * b_bytes);
            for (int h = 0; h < nk; ++h)
              for (int x = 0; x < NBOX; ++x)
                tma_load_2d_hint(S.b(sb, b_stage) + h * b_tile + x * (N / NBOX) * BK * 2, mb, (kb + h) * BK,
                                 x * (N / NBOX), &sm.full_b[sb], pol_keep);
          }
          ++ib;
          for (int w = 0; w < p.W; ++w) {
            const int sa = ia % A_STAGES;
            ok = mbar_wait(&sm.empty_a[sa], ((ia / A_STAGES) & 1) ^ 1, err);
            if (!ok) break;
            // the boxes span kps k-blocks whatever nk is (rows past the matrix read as 0),
            // so the stage always receives a_bytes
            mbar_arrive_expect_tx(&sm.full_a[sa], a_bytes);
            if (!MN_A) {
              tma_load_3d(S.a(sa), mm, kb * BK, un.tile * BM, w, &sm.full_a[sa]);
            } else {
              tma_load_3d_hint(S.a(sa), mm, un.tile * BM, kb * BK, w, &sm.full_a[sa], pol_stream);
              tma_load_3d_hint(S.a(sa) + a_bytes / 2, mm, un.tile * BM + 64, kb * BK, w, &sm.full_a[sa], pol_stream);
              prefetch_next();
            }
            ++ia;
          }
        }
      }
      // wait (bounded) for every load this thread issued before the CTA may exit
      for (uint32_t k = (ia > A_STAGES ? ia - A_STAGES : 0); k < ia; ++k)
        mbar_drain(&sm.full_a[k % A_STAGES], (k / A_STAGES) & 1, err, 1u << 20);
      for (uint32_t k = (ib > B_STAGES ? ib - B_STAGES : 0); k < ib; ++k)
        mbar_drain(&sm.full_b[k % B_STAGES], (k / B_STAGES) & 1, err, 1u << 20);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The issue loop between two MMAs is kept to a few integer adds: the descriptors of a
    // stage are its base descriptor plus constant offsets (in 16-byte units), ring slots and
    // segment ends are counters. Each tcgen05.mma waits until the tensor pipe takes it, so
    // the work between two of them adds to every MMA's time.
    if (lane == 0) {
      const uint32_t idesc2 = idesc_f16(BM, 2 * rp, BF16, MN_A, false), idesc1 = idesc_f16(BM, rp, BF16, MN_A, false);
      const uint64_t a_base = MN_A ? smem_desc(smem_u32(S.a(0)), a_bytes / 2, 1024) : smem_desc(smem_u32(S.a(0)), 16, 1024);
      const uint64_t b_base = smem_desc(smem_u32(S.b(0, b_stage)), 16, 1024);
      const uint32_t a_stage16 = a_bytes >> 4, b_stage16 = b_stage >> 4, b_tile16 = b_tile >> 4;
      const uint32_t term16 = (uint32_t)rp * 8;  // rp rows of 128 bytes
      uint32_t sa = 0, pa = 0, sb = 0, pb = 0, ju = 0;
      bool ok = true;
      for (int u = u_first; u < u_end && ok; u += u_step) {
        const Unit un = units[u];
        if (unit_off(p, p.meta[un.t], only_shifted)) continue;
        int steps_left = (un.kb1 - un.kb0) * p.W, seg_left = 0, acc = 0;
        uint32_t d_tmem = tmem_base, accum = 0;
        for (int kb = un.kb0; kb < un.kb1 && ok; kb += kps) {
          const int nk = min(kps, un.kb1 - kb);
          ok = mbar_wait(&sm.full_b[sb], pb, err);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bd = b_base + (uint64_t)(sb * b_stage16);
          for (int w = 0; w < p.W && ok; ++w) {
            ok = mbar_wait(&sm.full_a[sa], pa, err);
            if (!ok) break;
            tc_fence_after();
            const uint64_t ad = a_base + (uint64_t)(sa * a_stage16);
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // one step per k-block of the stage
              if (h < nk && ok) {
                if (seg_left == 0) {  // open an accumulator segment
                  acc = (int)(ju % NACC);
                  ok = mbar_wait(&sm.acc_empty[acc], ((ju / NACC) & 1) ^ 1, err);
                  if (!ok) break;
                  tc_fence_after();
                  d_tmem = tmem_base + (uint32_t)acc * kAccCols;
                  accum = 0;
                  seg_left = seg;
                }
                const uint64_t bdh = bd + (uint64_t)(h * b_tile16);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                  // MN-major A: 64 x (64 kps)-row boxes, k-block h at h * 64 rows of 128 bytes
                  const uint64_t adk = ad + (uint64_t)(MN_A ? (h * 8192 + k * 2048) >> 4 : (k * 32) >> 4);
                  // B rows [0, 2 rp): terms 0 and 1; rows [2 rp, 3 rp): term 2 (bf16)
                  umma_f16(d_tmem, adk, bdh + (uint64_t)(k * 2), idesc2, accum);
                  if (TERMS == 3) umma_f16(d_tmem, adk, bdh + (uint64_t)(2 * term16 + k * 2), idesc1, 1u);
                  accum = 1;
                }
                --steps_left;
                if (--seg_left == 0 || steps_left == 0) {  // close the segment
                  umma_commit(&sm.acc_full[acc]);
                  ++ju;
                  seg_left = 0;
                }
              }
            }
            umma_commit(&sm.empty_a[sa]);
            if (++sa == (uint32_t)A_STAGES) { sa = 0; pa ^= 1; }
          }
          umma_commit(&sm.empty_b[sb]);
          if (++sb == (uint32_t)B_STAGES) { sb = 0; pb ^= 1; }
        }
      }
      umma_commit(&sm.done);
      mbar_drain(&sm.done, 0, err, 1u << 22);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    // A warp may read only its own TMEM lane quarter (warp index mod 4). Two warps share
    // a quarter: half 0 takes the first ceil(rp/32) 16-column chunks, half 1 the rest.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quarter * 32 + lane;
    const int nch = rp / 16, ch0 = half ? (nch + 1) / 2 : 0, ch1 = half ? nch : (nch + 1) / 2;
    uint32_t ju = 0;
    bool ok = true;
    for (int u = u_first; u < u_end && ok; u += u_step) {
      const Unit un = units[u];
      const MatMeta& mt = p.meta[un.t];
      if (unit_off(p, mt, only_shifted)) continue;
      // Running sum of this row's chunks over the unit's accumulator segments, added in
      // segment order with round-to-nearest fp32 adds.
      float run[kRankBlock / 2];
      const int nseg = ((un.kb1 - un.kb0) * p.W + seg - 1) / seg;
      for (int sg = 0; sg < nseg && ok; ++sg) {
        const int acc = (int)(ju % NACC);
        ok = mbar_wait(&sm.acc_full[acc], (ju / NACC) & 1, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t t_row = tmem_base + (uint32_t)acc * kAccCols + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
        for (int cc = 0; cc < kRankBlock / 32; ++cc) {  // a chunk's two term columns, one wait
          if (ch0 + cc < ch1) {
            const int c = (ch0 + cc) * 16;
            float t0[16], t1[16];
            tmem_ld16x2(t_row + c, t_row + rp + c, t0, t1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float v = __fadd_rn(t0[i], t1[i]);
              run[cc * 16 + i] = sg == 0 ? v : __fadd_rn(run[cc * 16 + i], v);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
        ++ju;
      }
      if (!ok) break;
      float* out;
      int64_t grow, limit;
      if (!MN_A) {
        const int64_t mpad = (mt.m + 127) / 128 * 128;
        grow = (int64_t)un.tile * BM + row_in_tile;
        limit = mpad;
        out = mt.Ppart + ((size_t)un.slot * mpad + grow) * rp;
      } else {
        grow = (int64_t)un.tile * BM + row_in_tile;
        limit = mt.n;
        out = mt.Qpart + ((size_t)un.slot * mt.n + grow) * rp;
      }
      if (grow < limit) {
#pragma unroll
        for (int cc = 0; cc < kRankBlock / 32; ++cc) {
          if (ch0 + cc < ch1) {
            const int c = (ch0 + cc) * 16;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(out + c + i) = make_float4(
                  run[cc * 16 + i], run[cc * 16 + i + 1], run[cc * 16 + i + 2], run[cc * 16 + i + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------- fused ingest + P GEMM
// One HBM sweep of the gradients. A TMA warp stages G_w and E_w tiles (128 rows x 64
// columns, 128-byte rows in the 128-byte swizzle, zero-filled past the matrix edge) into a
// shared-memory ring. Ingest warps form M_w = round_E(zero_nonfinite(G_w / s_b) + E_w)
// from the staged tiles, count nonfinite entries per (block, worker), store M_w to its
// scratch, and write the same tile into shared memory in the UMMA 128-byte-swizzle
// K-major layout. The MMA thread multiplies M_w by each split term of Q (Q_hi, Q_lo
// [, Q_lo2]) into one accumulator, over every worker and k-block of the unit, in
// segments; the epilogue sums the segments and writes the unit's P partial sums.
// Warps: 0 TMA (Q split tiles), 1 MMA, 2..5 epilogue, then kIngWarps ingest warps, then
// the TMA warp of the G/E tiles (kIngGeWarp).
// The ingest warps also record max|M| per matrix (for the bf16 subnormal rescale).
constexpr int kIngWarps = 16;                       // ingest warps: 8 or 16 (a divisor of 32)
constexpr int kIngGeWarp = 6 + kIngWarps;           // the G/E TMA warp, after the ingest warps
constexpr int kIngThreads = 32 * (kIngGeWarp + 1);
constexpr int kIngRowsPerPass = 4 * kIngWarps;      // tile rows the ingest warps cover at once
static_assert(128 % kIngRowsPerPass == 0, "ingest rows");
// A G/E stage holds `kps` (1 or 2) consecutive k-blocks of one worker's G and E: G boxes
// first, then E boxes, each a 128 x 64 tile in the 128-byte swizzle. Two k-blocks put 256
// contiguous bytes of every row in flight at once; a stream of 128-byte row pieces reads
// HBM markedly slower (measured on GB300: 4.4 against 6.1 TB/s for a pure TMA read of the
// same bytes).
constexpr int kMaxKps = 2;
constexpr int kIngPrefetch = 1;  // G/E stages prefetched into L2 ahead of their loads
__host__ __device__ constexpr int ge_bytes(int kps) { return 2 * kps * A_BYTES; }
constexpr int kMaxGeStages = 4;
struct IngBars {
  uint64_t full_a[kMaxAStages], empty_a[kMaxAStages];
  uint64_t full_b[B_STAGES], empty_b[B_STAGES];
  uint64_t full_ge[kMaxGeStages], empty_ge[kMaxGeStages];
  uint64_t acc_full[2], acc_empty[2], done;
  uint32_t tmem;
};

// Walk the (unit, worker, stage) sequence of this CTA, a stage being kps consecutive
// k-blocks of the unit (fewer at the unit's end). The stages of one worker come back to
// back: a row piece that starts off a 128-byte line (any n * 2 not a multiple of 128)
// shares its last line with the next stage's piece, which then still finds it in L2.
struct StageIter {
  int u, kb, nk, w;
  bool valid;
  Unit un;
  __device__ void set_nk(int kps) { nk = min(kps, un.kb1 - kb); }
  __device__ void start(const Unit* units, int nunits, int kps) {
    u = blockIdx.x; w = 0;
    valid = u < nunits;
    if (valid) { un = units[u]; kb = un.kb0; set_nk(kps); }
  }
  __device__ void next(const Unit* units, int nunits, int W, int kps) {
    kb += nk;
    if (kb < un.kb1) { set_nk(kps); return; }
    kb = un.kb0;
    if (++w < W) { set_nk(kps); return; }
    w = 0;
    u += gridDim.x;
    valid = u < nunits;
    if (valid) { un = units[u]; kb = un.kb0; set_nk(kps); }
  }
};

template <typename TE, bool kMask>
__global__ void __launch_bounds__(kIngThreads, 1)
k_ingest_p(Plan p, const CUtensorMap* __restrict__ maps, const Unit* __restrict__ units, int nunits,
           int a_stages, int ge_stages, int kps, uint32_t b_stage, int seg) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* a0 = base;
  uint8_t* b0 = a0 + (size_t)a_stages * A_BYTES;
  uint8_t* ge0 = b0 + (size_t)B_STAGES * b_stage;
  const int GE_BYTES = ge_bytes(kps);
  IngBars& sm = *reinterpret_cast<IngBars*>(ge0 + (size_t)ge_stages * GE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool BF16 = std::is_same<TE, __nv_bfloat16>::value;
  constexpr int TERMS = BF16 ? 3 : 2;
  const int rp = p.rp, N = TERMS * rp;
  const int NBOX = N <= 256 ? 1 : 2;
  // TMEM: accumulators at columns 0 and 128 (rp <= 128 each: the split terms of Q go
  // along K into the same accumulator), the running sum of the unit at column 256.
  constexpr int NACC = 2;
  constexpr uint32_t kAccCols = 128, kRunCol = 256;
  const uint32_t b_bytes = (uint32_t)N * BK * 2;
  int* err = p.err_word;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a_stages; ++i) { mbar_init(&sm.full_a[i], kIngWarps); mbar_init(&sm.empty_a[i], 1); }
    for (int i = 0; i < B_STAGES; ++i) { mbar_init(&sm.full_b[i], 1); mbar_init(&sm.empty_b[i], 1); }
    for (int i = 0; i < ge_stages; ++i) { mbar_init(&sm.full_ge[i], 1); mbar_init(&sm.empty_ge[i], kIngWarps); }
    for (int i = 0; i < 2; ++i) { mbar_init(&sm.acc_full[i], 1); mbar_init(&sm.acc_empty[i], 4); }
    mbar_init(&sm.done, 1);
    abort_reset();
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA: Q split tiles
    if (lane == 0) {
      uint32_t ib = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        const CUtensorMap* mb = maps + (size_t)un.t * NMAPS + MAP_QS;
        for (int w = 0; w < p.W && ok; ++w)  // one Q tile per (worker, k-block) step
          for (int kb = un.kb0; kb < un.kb1 && ok; ++kb) {
            const int sb = ib % B_STAGES;
            ok = mbar_wait(&sm.empty_b[sb], ((ib / B_STAGES) & 1) ^ 1, err);
            if (!ok) break;
            mbar_arrive_expect_tx(&sm.full_b[sb], b_bytes);
            for (int x = 0; x < NBOX; ++x)
              tma_load_2d(b0 + (size_t)sb * b_stage + x * (N / NBOX) * BK * 2, mb, kb * BK, x * (N / NBOX), &sm.full_b[sb]);
            ++ib;
          }
      }
      for (uint32_t k = (ib > B_STAGES ? ib - B_STAGES : 0); k < ib; ++k)
        mbar_drain(&sm.full_b[k % B_STAGES], (k / B_STAGES) & 1, err, 1u << 20);
    }
  } else if (warp == kIngGeWarp) {
    // ------------------------------------------------------------ TMA: G/E tiles
    if (lane == 0) {
      const CUtensorMap* gem = static_cast<const CUtensorMap*>(p.tab.ge_maps);
      StageIter ti;
      ti.start(units, nunits, kps);
      // L2 prefetch of the G/E boxes kIngPrefetch stages ahead of the loads
      StageIter pf;
      pf.start(units, nunits, kps);
      auto prefetch_next = [&]() {
        if (!pf.valid) return;
        const size_t slot = (size_t)pf.un.t * p.W + pf.w;
        for (int h = 0; h < pf.nk; ++h) {
          tma_prefetch_2d(gem + 2 * slot, (pf.kb + h) * BK, pf.un.tile * BM);
          tma_prefetch_2d(gem + 2 * slot + 1, (pf.kb + h) * BK, pf.un.tile * BM);
        }
        pf.next(units, nunits, p.W, kps);
      };
      for (int i = 0; i < kIngPrefetch; ++i) prefetch_next();
      uint32_t ig = 0;
      bool ok = true;
      while (ti.valid && ok) {
        const size_t slot = (size_t)ti.un.t * p.W + ti.w;
        const int s = ig % ge_stages;
        ok = mbar_wait(&sm.empty_ge[s], ((ig / ge_stages) & 1) ^ 1, err);
        if (!ok) break;
        mbar_arrive_expect_tx(&sm.full_ge[s], (uint32_t)(2 * ti.nk * A_BYTES));
        uint8_t* st = ge0 + (size_t)s * GE_BYTES;
        for (int h = 0; h < ti.nk; ++h)  // the G boxes of the stage's k-blocks, side by side
          tma_load_2d(st + h * A_BYTES, gem + 2 * slot, (ti.kb + h) * BK, ti.un.tile * BM, &sm.full_ge[s]);
        for (int h = 0; h < ti.nk; ++h)  // then the E boxes
          tma_load_2d(st + (kps + h) * A_BYTES, gem + 2 * slot + 1, (ti.kb + h) * BK, ti.un.tile * BM, &sm.full_ge[s]);
        prefetch_next();
        ++ig;
        ti.next(units, nunits, p.W, kps);
      }
      for (uint32_t k = (ig > (uint32_t)ge_stages ? ig - ge_stages : 0); k < ig; ++k)
        mbar_drain(&sm.full_ge[k % ge_stages], (k / ge_stages) & 1, err, 1u << 20);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Between two MMAs only integer adds (descriptor = stage base + constant offset), as in
    // the separate GEMM kernel.
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(BM, rp, BF16, false, false);
      const uint64_t a_base = smem_desc(smem_u32(a0), 16, 1024), b_base = smem_desc(smem_u32(b0), 16, 1024);
      const uint32_t b_stage16 = b_stage >> 4, term16 = (uint32_t)rp * 8;
      uint32_t sa = 0, pa = 0, sb = 0, pb = 0, ju = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        int steps_left = (un.kb1 - un.kb0) * p.W, seg_left = 0, acc = 0;
        uint32_t d_tmem = tmem_base, accum = 0;
        for (int w = 0; w < p.W && ok; ++w) {
          for (int kb = un.kb0; kb < un.kb1 && ok; ++kb) {
            ok = mbar_wait(&sm.full_b[sb], pb, err);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bd = b_base + (uint64_t)(sb * b_stage16);
            if (seg_left == 0) {  // open an accumulator segment
              acc = (int)(ju % NACC);
              ok = mbar_wait(&sm.acc_empty[acc], ((ju / NACC) & 1) ^ 1, err);
              if (!ok) break;
              tc_fence_after();
              d_tmem = tmem_base + (uint32_t)acc * kAccCols;
              accum = 0;
              seg_left = seg;
            }
            ok = mbar_wait(&sm.full_a[sa], pa, err);
            if (!ok) break;
            tc_fence_after();
            const uint64_t ad = a_base + (uint64_t)(sa * (A_BYTES >> 4));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
#pragma unroll
              for (int tm = 0; tm < TERMS; ++tm) {  // B rows [tm rp, (tm + 1) rp): term tm of Q
                umma_f16(d_tmem, ad + (uint64_t)(k * 2), bd + (uint64_t)(tm * term16 + k * 2), idesc, accum);
                accum = 1;
              }
            }
            umma_commit(&sm.empty_a[sa]);
            umma_commit(&sm.empty_b[sb]);
            if (++sa == (uint32_t)a_stages) { sa = 0; pa ^= 1; }
            if (++sb == (uint32_t)B_STAGES) { sb = 0; pb ^= 1; }
            --steps_left;
            if (--seg_left == 0 || steps_left == 0) {  // close the segment
              umma_commit(&sm.acc_full[acc]);
              ++ju;
              seg_left = 0;
            }
          }
        }
      }
      umma_commit(&sm.done);
      mbar_drain(&sm.done, 0, err, 1u << 22);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint32_t ju = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const Unit un = units[u];
      const MatMeta& mt = p.meta[un.t];
      const int64_t mpad = (mt.m + 127) / 128 * 128;
      const int64_t grow = (int64_t)un.tile * BM + row_in_tile;
      float* out = mt.Ppart + ((size_t)un.slot * mpad + grow) * rp;
      // Running sum of the unit's accumulator segments in TMEM (this thread's lane only),
      // added in segment order with round-to-nearest fp32 adds; the last segment writes
      // the unit's P partial row.
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const uint32_t t_run = tmem_base + kRunCol + lane_off;
      const int nseg = ((un.kb1 - un.kb0) * p.W + seg - 1) / seg;
      for (int sg = 0; sg < nseg && ok; ++sg) {
        const int acc = (int)(ju % NACC);
        ok = mbar_wait(&sm.acc_full[acc], (ju / NACC) & 1, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t t_acc = tmem_base + (uint32_t)acc * kAccCols + lane_off;
        const bool last_seg = sg == nseg - 1;
        for (int c = 0; c < rp; c += 16) {
          float v[16], o[16];
          if (sg == 0) {
            tmem_ld16(t_acc + c, v);
          } else {
            tmem_ld16x2(t_acc + c, t_run + c, v, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fadd_rn(o[i], v[i]);
          }
          if (last_seg) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(out + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          } else {
            tmem_st16(t_run + c, v);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
        ++ju;
      }
    }
  } else {
    // ------------------------------------------------------------ ingest (warps 6 ..)
    const int it = threadIdx.x - 6 * 32;          // 0 .. 32 kIngWarps - 1
    const int cq = it & 7;                        // 16-byte chunk within the 128-byte row
    const int rq = it >> 3;                       // first row; rows rq + kIngRowsPerPass k
    StageIter ti;
    ti.start(units, nunits, kps);
    uint32_t ia = 0, ig = 0;
    bool ok = true;
    while (ti.valid && ok) {
      const MatMeta& mt = p.meta[ti.un.t];
      const int sg = ig % ge_stages;
      ok = mbar_wait(&sm.full_ge[sg], (ig / ge_stages) & 1, err);
      if (!ok) break;
      const uint8_t* gstage = ge0 + (size_t)sg * GE_BYTES;
      const float inv_s = p.tab.inv_scale[mt.b];
      // fp16 with a power-of-two 1/s in [2^-24, 1]: 1/s is exact in fp16 (a subnormal at
      // the low end) and g / s cannot overflow. One fp16 FMA then gives M = round_E(g / s + E)
      // with a single rounding of the exact value (IEEE fused multiply-add, subnormals
      // kept), two entries per instruction. An entry is nonfinite exactly when g's
      // exponent bits are all ones, and a zeroed entry gives M = E. Other scales and bf16
      // take the fp32 path with the round-to-odd sum.
      const bool h2_path = !BF16 && (__float_as_uint(inv_s) & 0x7fffffu) == 0u && inv_s <= 1.0f &&
                           inv_s >= 0x1p-24f;
      const __half2 inv2 = __float2half2_rn(inv_s);
      TE* mo = static_cast<TE*>(mt.mscr) + (size_t)ti.w * mt.m * mt.n;
      // nonfinite mask (PSGD_FLAG_MASK): n is a multiple of 8, so a thread's 8 entries are
      // one byte of the row-major, LSB-first bitmap
      uint8_t* mbits = kMask ? reinterpret_cast<uint8_t*>(p.mask + p.mask_off[(size_t)ti.un.t * p.W + ti.w]) : nullptr;
      int cnt = 0;
      unsigned mmax = 0u;
      for (int h = 0; h < ti.nk && ok; ++h) {  // the stage's k-blocks, one A tile each
        const int sa = ia % a_stages;
        ok = mbar_wait(&sm.empty_a[sa], ((ia / a_stages) & 1) ^ 1, err);
        if (!ok) break;
        uint8_t* tile = a0 + (size_t)sa * A_BYTES;
        const uint8_t* gs = gstage + h * A_BYTES;           // G box of k-block kb + h
        const uint8_t* es = gstage + (kps + h) * A_BYTES;   // E box of k-block kb + h
        const int64_t col = (int64_t)(ti.kb + h) * BK + cq * 8;
#pragma unroll
        for (int k = 0; k < 128 / kIngRowsPerPass; ++k) {
          const int rl = rq + kIngRowsPerPass * k;
          const int64_t row = (int64_t)ti.un.tile * BM + rl;
          uint4 mv = make_uint4(0u, 0u, 0u, 0u);
          if (row < mt.m && col < mt.n) {
            const int so = rl * 128 + ((cq ^ (rl & 7)) << 4);  // 128-byte swizzle of the staged tiles
            const uint4 gv = *reinterpret_cast<const uint4*>(gs + so);
            const uint4 ev = *reinterpret_cast<const uint4*>(es + so);
            const TE* gx = reinterpret_cast<const TE*>(&gv);
            const TE* ex = reinterpret_cast<const TE*>(&ev);
            TE* mx = reinterpret_cast<TE*>(&mv);
            uint32_t mbyte = 0u;
            if (h2_path) {
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, ew[4] = {ev.x, ev.y, ev.z, ev.w};
              uint32_t mw[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t xe = gw[i] & 0x7C007C00u;  // exponent fields of the two entries
                const uint32_t bad = ((xe & 0xFFFFu) == 0x7C00u ? 0x0000FFFFu : 0u) |
                                     ((xe >> 16) == 0x7C00u ? 0xFFFF0000u : 0u);
                cnt += __popc(bad) >> 4;
                if (kMask) mbyte |= ((bad & 1u) | ((bad >> 15) & 2u)) << (2 * i);
                __half2 gh, eh;
                memcpy(&gh, &gw[i], 4);
                memcpy(&eh, &ew[i], 4);
                const __half2 r = __hfma2(gh, inv2, eh);
                uint32_t rw;
                memcpy(&rw, &r, 4);
                mw[i] = (rw & ~bad) | (ew[i] & bad);
              }
              mv = make_uint4(mw[0], mw[1], mw[2], mw[3]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float x = to_f(gx[i]) * inv_s;
                const bool bad = !isfinite(x);
                cnt += bad;
                if (kMask) mbyte |= (uint32_t)bad << i;
                mx[i] = add_to<TE>(bad ? 0.0f : x, to_f(ex[i]));
                if (BF16) mmax = max(mmax, __float_as_uint(fabsf(to_f(mx[i]))));
              }
            }
            __stcg(reinterpret_cast<uint4*>(mo + row * mt.n + col), mv);
            if (kMask) mbits[(row * mt.n + col) >> 3] = (uint8_t)mbyte;
          }
          *reinterpret_cast<uint4*>(tile + rl * 128 + ((cq ^ (rl & 7)) << 4)) = mv;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.full_a[sa]);
        ++ia;
      }
      if (!ok) break;
      cnt = __reduce_add_sync(0xffffffffu, cnt);
      if (BF16) mmax = __reduce_max_sync(0xffffffffu, mmax);
      if (lane == 0 && cnt)
        atomicAdd(reinterpret_cast<unsigned long long*>(p.counts + (size_t)mt.b * p.W + ti.w),
                  (unsigned long long)cnt);
      if (BF16 && lane == 0 && mmax)  // only the bf16 subnormal rescale reads max|M|
        atomicMax(reinterpret_cast<unsigned*>(mt.scal) + SC_MAXM, mmax);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty_ge[sg]);
      ++ig;
      ti.next(units, nunits, p.W, kps);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// Stage counts of the fused kernel: A stages for the MMA, G/E staging stages.
// Two k-blocks per G/E stage when two such stages fit next to two A stages; otherwise
// (the bf16 case, whose three split terms make the B stages larger) one k-block per stage.
void ingest_stages(int edt, uint32_t b_stage, int* a_st, int* ge_st, int* kps, size_t* smem) {
  const size_t budget = kDynSmemCap - 1024 - sizeof(IngBars) - (size_t)B_STAGES * b_stage;
  int a = 2, k = kMaxKps;
  int ge = (int)std::min<size_t>(kMaxGeStages, (budget - (size_t)a * A_BYTES) / ge_bytes(k));
  if (ge < 2) {
    k = 1;
    a = edt == DT_BF16 ? 2 : 3;
    ge = (int)std::min<size_t>(kMaxGeStages, (budget - (size_t)a * A_BYTES) / ge_bytes(k));
  }
  *a_st = a;
  *ge_st = ge;
  *kps = k;
  *smem = 1024 + (size_t)a * A_BYTES + (size_t)B_STAGES * b_stage + (size_t)ge * ge_bytes(k) + sizeof(IngBars);
}

// ---------------------------------------------------------------- decompression kernel
constexpr int DEC_STAGES = 2;   // P^ / Q operand stages of the G^ MMA
constexpr int DEC_MSTAGES = 4;  // M_w tile ring (E is formed in place and stored from it;
                                // G^ goes out through the same ring, 64 fp32 columns a stage)
constexpr int DEC_MSTAGE_BYTES = 2 * A_BYTES;
constexpr int kDecPrefetch = 2;  // M tiles prefetched into L2 ahead of their loads
constexpr int DEC_THREADS = 352;
struct DecSmem {
  alignas(1024) uint8_t a[DEC_STAGES][A_BYTES];          // P^ split tiles, 128 x 64
  alignas(1024) uint8_t b[DEC_STAGES][DEC_NT * BK * 2];  // Q split tiles, 128 x 64
  alignas(1024) uint8_t mt[DEC_MSTAGES][2 * A_BYTES];    // M_w tile 128 x 128: two swizzled boxes
  uint64_t full[DEC_STAGES], empty[DEC_STAGES];
  uint64_t acc_full[2], acc_empty[2], done;
  uint64_t mfull[DEC_MSTAGES], mdone[DEC_MSTAGES];
  uint64_t never;  // no thread arrives on it (the PSGD_FLAG_DEBUG_EXPIRE_WAIT test wait)
  uint32_t tmem;
};

// G^ tile 128 x 128 = A B^T over K = 3 kp (tensor cores, accumulated in TMEM). The
// epilogue warps read it once from TMEM into registers (two warps per TMEM lane
// quarter, 64 columns each), write G^, and then, for every worker, form
// E_w = round_E(M_w - G^) in place in the staged M_w tile. A TMA warp streams the M_w
// tiles through a ring of shared-memory stages and stores the E_w tiles from them.
// Warps: 0 TMA (operands), 1 MMA, 2..9 epilogue, 10 TMA (M_w in, E_w out).
template <typename TE>
__global__ void __launch_bounds__(DEC_THREADS, 1)
k_decomp_tc(Plan p, const CUtensorMap* __restrict__ maps, const Unit* __restrict__ units, int nunits, int kp) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  DecSmem& sm = *reinterpret_cast<DecSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = 3 * kp / BK;
  int* err = p.err_word;
  constexpr uint32_t STAGE_TX = A_BYTES + DEC_NT * BK * 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < DEC_STAGES; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&sm.acc_full[i], 1); mbar_init(&sm.acc_empty[i], 8); }
    for (int i = 0; i < DEC_MSTAGES; ++i) { mbar_init(&sm.mfull[i], 1); mbar_init(&sm.mdone[i], 8); }
    mbar_init(&sm.never, 1);
    mbar_init(&sm.done, 1);
    abort_reset();
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA: G^ operands
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        if (p.skip[p.meta[un.t].b]) continue;
        const CUtensorMap* ma = maps + (size_t)un.t * NMAPS + MAP_PD;
        const CUtensorMap* mb = maps + (size_t)un.t * NMAPS + MAP_QD;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          const int s = it % DEC_STAGES;
          ok = mbar_wait(&sm.empty[s], ((it / DEC_STAGES) & 1) ^ 1, err);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.full[s], STAGE_TX);
          tma_load_2d(sm.a[s], ma, kb * BK, un.tile * BM, &sm.full[s]);
          tma_load_2d(sm.b[s], mb, kb * BK, un.kb0 * DEC_NT, &sm.full[s]);
          ++it;
        }
      }
      for (uint32_t k = (it > DEC_STAGES ? it - DEC_STAGES : 0); k < it; ++k)
        mbar_drain(&sm.full[k % DEC_STAGES], (k / DEC_STAGES) & 1, err, 1u << 20);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(BM, DEC_NT, false, false, false);
      uint32_t it = 0, ju = 0;
      bool ok = true;
      // Test of the expiry path: a short wait on a barrier that nothing completes. It
      // expires, records DEVERR_TIMEOUT and raises the CTA's abort flag; the CTA winds down.
      if (p.debug_expire) ok = mbar_wait(&sm.never, 0, err, 4096);
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        if (p.skip[p.meta[un.t].b]) continue;
        const int acc = ju & 1;
        ok = mbar_wait(&sm.acc_empty[acc], ((ju >> 1) & 1) ^ 1, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * DEC_NT);
        uint32_t accum = 0;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          const int s = it % DEC_STAGES;
          ok = mbar_wait(&sm.full[s], (it / DEC_STAGES) & 1, err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sm.a[s]), b_addr = smem_u32(sm.b[s]);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma_f16(d_tmem, smem_desc(a_addr + k * 32, 16, 1024), smem_desc(b_addr + k * 32, 16, 1024),
                     idesc, accum);
            accum = 1;
          }
          umma_commit(&sm.empty[s]);
          ++it;
        }
        umma_commit(&sm.acc_full[acc]);
        ++ju;
      }
      umma_commit(&sm.done);
      mbar_drain(&sm.done, 0, err, 1u << 22);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ TMA: M_w in, E_w out
    if (lane == 0) {
      const CUtensorMap* gem = static_cast<const CUtensorMap*>(p.tab.ge_maps);
      const CUtensorMap* ghm = gem + 2 * (size_t)p.B * p.J * p.W;  // G^ maps, one per matrix
      // What each stage holds: (matrix, worker, row0, col0, second 64-column box) for an
      // E tile; worker -1 - g for half g (64 columns, fp32) of the unit's G^ tile.
      int st_t[DEC_MSTAGES] = {}, st_w[DEC_MSTAGES] = {}, st_r[DEC_MSTAGES] = {}, st_c[DEC_MSTAGES] = {},
          st_two[DEC_MSTAGES] = {};
      int64_t st_n[DEC_MSTAGES] = {};
      uint32_t i = 0;
      bool ok = true;
      auto store_tile = [&](uint32_t j) -> bool {
        const int s = (int)(j % DEC_MSTAGES);
        if (!mbar_wait(&sm.mdone[s], (j / DEC_MSTAGES) & 1, err)) return false;
        if (st_w[s] >= 0) {
          const CUtensorMap* em = gem + 2 * ((size_t)st_t[s] * p.W + st_w[s]) + 1;
          tma_store_2d(em, sm.mt[s], st_c[s], st_r[s]);
          if (st_two[s]) tma_store_2d(em, sm.mt[s] + A_BYTES, st_c[s] + 64, st_r[s]);
        } else {  // G^: two boxes of 32 fp32 columns; none starts past the matrix edge
          const CUtensorMap* gm = ghm + st_t[s];
          for (int b = 0; b < 2; ++b)
            if (st_c[s] + 32 * b < st_n[s]) tma_store_2d(gm, sm.mt[s] + b * (DEC_MSTAGE_BYTES / 2), st_c[s] + 32 * b, st_r[s]);
        }
        bulk_commit();
        return true;
      };
      // claim stage i % DEC_MSTAGES: store what it held and wait until the store has read it
      auto claim = [&]() -> bool {
        if (i < DEC_MSTAGES) return true;
        if (!store_tile(i - DEC_MSTAGES)) return false;
        bulk_wait_read_all();
        return true;
      };
      // L2 prefetch of the M tiles kDecPrefetch tiles ahead of their loads
      int pf_u = blockIdx.x, pf_w = 0;
      auto prefetch_next = [&]() {
        while (pf_u < nunits && p.skip[p.meta[units[pf_u].t].b]) pf_u += gridDim.x;
        if (pf_u >= nunits) return;
        const Unit un = units[pf_u];
        const CUtensorMap* mm = maps + (size_t)un.t * NMAPS + MAP_MP;
        tma_prefetch_3d(mm, un.kb0 * DEC_NT, un.tile * BM, pf_w);
        if ((int64_t)un.kb0 * DEC_NT + 64 < p.meta[un.t].n) tma_prefetch_3d(mm, un.kb0 * DEC_NT + 64, un.tile * BM, pf_w);
        if (++pf_w == p.W) { pf_w = 0; pf_u += gridDim.x; }
      };
      for (int k = 0; k < kDecPrefetch; ++k) prefetch_next();
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        const MatMeta& mt = p.meta[un.t];
        const int row0 = un.tile * BM, col0 = un.kb0 * DEC_NT;
        if (!p.skip[mt.b]) {
          const CUtensorMap* mm = maps + (size_t)un.t * NMAPS + MAP_MP;
          const int two = (int64_t)col0 + 64 < mt.n ? 1 : 0;
          for (int w = 0; w < p.W && ok; ++w) {
            const int s = (int)(i % DEC_MSTAGES);
            ok = claim();
            if (!ok) break;
            st_t[s] = un.t; st_w[s] = w; st_r[s] = row0; st_c[s] = col0; st_two[s] = two;
            mbar_arrive_expect_tx(&sm.mfull[s], (uint32_t)(1 + two) * A_BYTES);
            tma_load_3d(sm.mt[s], mm, col0, row0, w, &sm.mfull[s]);
            if (two) tma_load_3d(sm.mt[s] + A_BYTES, mm, col0 + 64, row0, w, &sm.mfull[s]);
            prefetch_next();
            ++i;
          }
        }
        for (int g = 0; g < 2 && ok; ++g) {  // the G^ tile, 64 columns per stage (0 if skipped)
          const int s = (int)(i % DEC_MSTAGES);
          ok = claim();
          if (!ok) break;
          st_t[s] = un.t; st_w[s] = -1 - g; st_r[s] = row0; st_c[s] = col0 + 64 * g; st_n[s] = mt.n;
          mbar_arrive(&sm.mfull[s]);  // the stage is free for the epilogue to fill
          ++i;
        }
      }
      // store the tiles still held by the stages
      for (uint32_t j = (i > DEC_MSTAGES ? i - DEC_MSTAGES : 0); j < i && ok; ++j) ok = store_tile(j);
      if (!ok)  // wait (bounded) for the loads this thread issued before the CTA may exit
        for (uint32_t j = (i > DEC_MSTAGES ? i - DEC_MSTAGES : 0); j < i; ++j)
          mbar_drain(&sm.mfull[j % DEC_MSTAGES], (j / DEC_MSTAGES) & 1, err, 1u << 20);
      bulk_wait_all();
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int quarter = warp & 3;          // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;      // 64-column half of the tile
    const int row_in_tile = quarter * 32 + lane;
    const int sw = row_in_tile & 7;        // 128-byte swizzle phase of this row
    uint32_t ju = 0, i = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const Unit un = units[u];
      const MatMeta& mt = p.meta[un.t];
      const int64_t m = mt.m, n = mt.n;
      const int64_t row = (int64_t)un.tile * BM + row_in_tile;
      const int64_t colh = (int64_t)un.kb0 * DEC_NT + half * 64;
      const bool skipped = p.skip[mt.b] != 0;
      float gv[64];
      if (!skipped) {
        const int acc = ju & 1;
        ok = mbar_wait(&sm.acc_full[acc], (ju >> 1) & 1, err);
        if (!ok) break;
        tc_fence_after();
        // G^ = acc * 2^-(14 + e) as exact power-of-two factors (one rounding at most)
        const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[3]);
        const int tsh = 14 + e;
        const int t1 = tsh > 126 ? 126 : (tsh < -126 ? -126 : tsh);
        const float f1 = __uint_as_float((uint32_t)(127 - t1) << 23);
        const float f2 = __uint_as_float((uint32_t)(127 - (tsh - t1)) << 23);
        const uint32_t t_row = tmem_base + (uint32_t)(acc * DEC_NT + half * 64) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          float v0[16], v1[16];
          tmem_ld16x2(t_row + c, t_row + c + 16, v0, v1);
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            gv[c + i2] = (v0[i2] * f1) * f2;
            gv[c + 16 + i2] = (v1[i2] * f1) * f2;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
        ++ju;
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) gv[c] = 0.f;
      }
      TE* mbase = static_cast<TE*>(mt.mscr);
      // a rescaled bf16 M scratch holds M * 2^sh: undo it exactly, and restore M
      const int msh = reinterpret_cast<const int*>(mt.scal)[SC_MSHIFT];
      const float munscale = __uint_as_float((uint32_t)(127 - msh) << 23);
      for (int w = 0; w < p.W && !skipped; ++w) {
        const int s = (int)(i % DEC_MSTAGES);
        ok = mbar_wait(&sm.mfull[s], (i / DEC_MSTAGES) & 1, err);
        if (!ok) break;
        uint8_t* tile = sm.mt[s] + half * A_BYTES + row_in_tile * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4* cp = reinterpret_cast<uint4*>(tile + ((j ^ sw) << 4));
          const uint4 mv = *cp;
          const TE* mx = reinterpret_cast<const TE*>(&mv);
          __align__(16) TE ev[8], mr[8];
#pragma unroll
          for (int e8 = 0; e8 < 8; ++e8) {
            const float mval = to_f(mx[e8]) * munscale;  // exact: a power of two
            ev[e8] = add_to<TE>(mval, -gv[j * 8 + e8]);
            mr[e8] = from_f<TE>(mval);
          }
          *cp = *reinterpret_cast<const uint4*>(ev);
          if (msh != 0 && row < m && colh + j * 8 < n)
            *reinterpret_cast<uint4*>(mbase + (size_t)w * m * n + row * n + colh + j * 8) =
                *reinterpret_cast<const uint4*>(mr);
        }
        fence_proxy_async_smem();  // E in shared memory, visible to the tensor store
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.mdone[s]);
        ++i;
      }
      if (!ok) break;
      // G^: half g of the tile (this warp's 64 columns when half == g) goes into a stage in
      // the 128-byte-swizzled layout of two 32-column fp32 boxes, which the TMA warp stores.
      // The other half's warps only arrive, but they too wait for the stage first: the TMA
      // warp marks it full only after the stage's previous use is done, and an arrival
      // before that would count toward the previous use (whose store would then start
      // while a slower warp is still writing its tile).
      for (int g = 0; g < 2; ++g) {
        const int s = (int)(i % DEC_MSTAGES);
        ok = mbar_wait(&sm.mfull[s], (i / DEC_MSTAGES) & 1, err);
        if (!ok) break;
        if (half == g) {
          uint8_t* st = sm.mt[s] + row_in_tile * 128;
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(st + b * (DEC_MSTAGE_BYTES / 2) + ((j ^ sw) << 4)) =
                  make_float4(gv[32 * b + 4 * j], gv[32 * b + 4 * j + 1], gv[32 * b + 4 * j + 2], gv[32 * b + 4 * j + 3]);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.mdone[s]);
        ++i;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 256);
}

// ---------------------------------------------------------------- host helpers
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool make_map(CUtensorMap* out, void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
              const uint32_t* box, bool swizzle = true,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_UINT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = fn(out, dtype, (cuuint32_t)rank, base, d, s, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

// B stage bytes and the number of A stages that fit next to two B stages.
// B stage bytes (kps k-blocks' split tiles, each rounded up to 1 KB), the number of A stages
// (kps k-blocks each) that fit next to two B stages, and the kernel's shared memory.
uint32_t gemm_b_stage(int edt, int rp, int kps = 1) {
  const int rows = (edt == DT_BF16 ? 3 : 2) * rp;
  return (uint32_t)kps * (uint32_t)((rows * BK * 2 + 1023) / 1024 * 1024);
}
int gemm_a_stages(uint32_t b_stage, int kps = 1) {
  const size_t budget = kDynSmemCap - 1024 - sizeof(GemmBars) - (size_t)B_STAGES * b_stage;
  return (int)std::min<size_t>(kMaxAStages, budget / ((size_t)kps * A_BYTES));
}
size_t gemm_smem(uint32_t b_stage, int a_stages, int kps = 1) {
  return 1024 + (size_t)a_stages * kps * A_BYTES + (size_t)B_STAGES * b_stage + sizeof(GemmBars);
}
// The Q GEMM stages two k-blocks when three such A stages still fit (fp16 up to r = 128);
// bf16's three split terms make the paired B stages too large, and it stages one.
int qgemm_kps(int edt, int rp) { return gemm_a_stages(gemm_b_stage(edt, rp, 2), 2) >= 3 ? 2 : 1; }
size_t dec_smem() { return sizeof(DecSmem) + 1024; }

struct TcLayout {
  size_t maps = 0, punits = 0, qunits = 0, dunits = 0, total = 0;
  std::vector<size_t> qsplit, psplit, pdec, qdec, ppart;
  int np = 0, nq = 0, nd = 0;
};

TcLayout tc_layout(const psgd_config* c) {
  TcLayout L;
  const int B = c->num_blocks, J = c->mats_per_block;
  const int rp = (c->rank + 15) / 16 * 16, kp = kpad_of(rp);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = (off + bytes + 1023) & ~(size_t)1023; return o; };
  for (int j = 0; j < J; ++j) {
    const int64_t m = c->shapes[j].m, n = c->shapes[j].n;
    const int64_t mt = (m + 127) / 128, nkb = (n + 63) / 64, kch = (nkb + PCHUNK_KB - 1) / PCHUNK_KB;
    const int64_t ntq = (n + 127) / 128, sl = std::max<int64_t>(1, (m + QSLICE_ROWS - 1) / QSLICE_ROWS);
    const int64_t ntd = (n + DEC_NT - 1) / DEC_NT;
    L.np += (int)(mt * kch);
    L.nq += (int)(ntq * sl);
    L.nd += (int)(mt * ntd);
  }
  L.np *= B; L.nq *= B; L.nd *= B;
  L.maps = take(sizeof(CUtensorMap) * NMAPS * (size_t)B * J);
  L.punits = take(sizeof(Unit) * L.np);
  L.qunits = take(sizeof(Unit) * L.nq);
  L.dunits = take(sizeof(Unit) * L.nd);
  for (int t = 0; t < B * J; ++t) {
    const int64_t m = c->shapes[t % J].m, n = c->shapes[t % J].n;
    const int64_t mpad = (m + 127) / 128 * 128, npad = (n + DEC_NT - 1) / DEC_NT * DEC_NT;
    const int64_t kch = ((n + 63) / 64 + PCHUNK_KB - 1) / PCHUNK_KB;
    const int terms = c->err_dtype == PSGD_BF16 ? 3 : 2;
    L.qsplit.push_back(take(2ull * terms * rp * n));
    L.psplit.push_back(take(2ull * terms * rp * mpad));
    L.pdec.push_back(take(2ull * mpad * 3 * kp));
    L.qdec.push_back(take(2ull * npad * 3 * kp));
    L.ppart.push_back(take(4ull * kch * mpad * rp));
  }
  L.total = off;
  return L;
}

}  // namespace

// Rescale the M scratch of bf16 matrices whose max|M| is below 2^-100 by 2^64 (exact:
// bf16 has fp32's exponent range, so even subnormal values scale losslessly), and record
// the shift. The tensor cores flush subnormal bf16 operands, and such matrices have most
// of their mass there. grid = (chunks, B*J*W).
__global__ void k_rescale_tiny(Plan p) {
  const int t = blockIdx.y / p.W, w = blockIdx.y % p.W;
  const MatMeta& mt = p.meta[t];
  const unsigned mx = reinterpret_cast<const unsigned*>(mt.scal)[SC_MAXM];
  if (p.skip[mt.b] || mx == 0u || mx >= 0x0D800000u) return;  // skipped, zero, or max|M| >= 2^-100
  if (blockIdx.x == 0 && threadIdx.x == 0 && w == 0) reinterpret_cast<int*>(mt.scal)[SC_MSHIFT] = 64;
  __nv_bfloat16* mo = static_cast<__nv_bfloat16*>(mt.mscr) + (size_t)w * mt.m * mt.n;
  const int64_t total = mt.m * mt.n;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < total;
       i += (int64_t)gridDim.x * blockDim.x * 8) {
    uint4 v = *reinterpret_cast<const uint4*>(mo + i);
    __nv_bfloat16* x = reinterpret_cast<__nv_bfloat16*>(&v);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = __float2bfloat16_rn(__bfloat162float(x[k]) * 0x1p64f);
    *reinterpret_cast<uint4*>(mo + i) = v;
  }
}

size_t tc_ge_maps_bytes(const psgd_config* cfg) {
  if (cfg->err_dtype == PSGD_F32 || (cfg->flags & PSGD_FLAG_SIMT) || cfg->rank > kRankBlock) return 0;
  const size_t BJ = (size_t)cfg->num_blocks * cfg->mats_per_block;
  return sizeof(CUtensorMap) * (2 * BJ * cfg->num_workers + BJ);
}

// TMA maps of each (matrix, worker) G and E: 2D {n, m}, 128 x 64 boxes, 128-byte swizzle
// (the fused ingest reads G/E tiles through them; the decompression stores E tiles), then
// one per matrix for G^: fp32 {n, m}, 128 x 32 boxes, 128-byte swizzle (decompression).
bool tc_encode_ge_maps(const Handle& h, const void* const* grads, void* const* errs, float* const* ghat,
                       void* out) {
  CUtensorMap* maps = static_cast<CUtensorMap*>(out);
  for (int t = 0; t < h.B * h.J; ++t) {
    const MatMeta& mt = h.meta[t];
    uint64_t d[2] = {(uint64_t)mt.n, (uint64_t)mt.m}, st[1] = {(uint64_t)mt.n * 4};
    uint32_t box[2] = {32, 128};
    if (!make_map(&maps[(size_t)2 * h.B * h.J * h.W + t], ghat[t], 2, d, st, box, true,
                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return false;
  }
  for (int t = 0; t < h.B * h.J; ++t) {
    const MatMeta& mt = h.meta[t];
    uint64_t d[2] = {(uint64_t)mt.n, (uint64_t)mt.m}, st[1] = {(uint64_t)mt.n * 2};
    uint32_t box[2] = {64, 128};
    for (int w = 0; w < h.W; ++w) {
      const size_t slot = (size_t)t * h.W + w;
      if (!make_map(&maps[2 * slot], const_cast<void*>(grads[slot]), 2, d, st, box)) return false;
      if (!make_map(&maps[2 * slot + 1], errs[slot], 2, d, st, box)) return false;
    }
  }
  return true;
}

cudaError_t launch_rescale_tiny(const Handle& h, const Plan& p, cudaStream_t s) {
  k_rescale_tiny<<<dim3(64, p.B * p.J * p.W), 256, 0, s>>>(p);
  h.launches += 1;
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  const int grid = std::min(tp->grid, tp->np);
  const uint32_t bst = gemm_b_stage(h.edt, p.rp);
  const int ast = gemm_a_stages(bst);
  const size_t sm = gemm_smem(bst, ast);
  launch_pdl(k_gemm<false, true>, dim3(grid), dim3(kGemmThreads), sm, s, p, tp->d_maps, tp->d_punits, tp->np, ast, bst, 1, kGemmSegSteps, 1, 0);
  h.launches += 1;
  return cudaGetLastError();
}

size_t tc_workspace_bytes(const psgd_config* cfg) {
  if (cfg->err_dtype == PSGD_F32 || (cfg->flags & PSGD_FLAG_SIMT) || cfg->rank > kRankBlock) return 0;
  return tc_layout(cfg).total;
}

bool tc_supported(const psgd_config* cfg, std::string* why) {
  if (cfg->err_dtype == PSGD_F32) { if (why) *why = "fp32 gradients use the FFMA engine"; return false; }
  if (cfg->rank > kRankBlock) { if (why) *why = "ranks above 128 use the FFMA engine"; return false; }
  int dev = 0, major = 0, minor = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10) { if (why) *why = "tcgen05 needs sm_10x"; return false; }
  if (!encode_fn()) { if (why) *why = "cuTensorMapEncodeTiled unavailable"; return false; }
  return true;
}

cudaError_t tc_plan(Handle& h, char* ws_tc, cudaStream_t s) {
  const TcLayout L = tc_layout(&h.cfg);
  TcPlan* tp = new TcPlan();
  h.tc_plan = tp;
  const int B = h.B, J = h.J, W = h.W, rp = h.rp, kp = kpad_of(rp);
  tp->kp = kp;
  tp->qkps = qgemm_kps(h.edt, rp);
  tp->d_maps = reinterpret_cast<CUtensorMap*>(ws_tc + L.maps);
  tp->d_punits = reinterpret_cast<Unit*>(ws_tc + L.punits);
  tp->d_qunits = reinterpret_cast<Unit*>(ws_tc + L.qunits);
  tp->d_dunits = reinterpret_cast<Unit*>(ws_tc + L.dunits);
  std::vector<CUtensorMap> maps((size_t)B * J * NMAPS);
  std::vector<Unit> pu, qu, du;
  for (int t = 0; t < B * J; ++t) {
    MatMeta& mt = h.meta[t];
    const int64_t m = mt.m, n = mt.n, mpad = (m + 127) / 128 * 128;
    const int64_t npad = (n + DEC_NT - 1) / DEC_NT * DEC_NT;
    mt.qsplit = reinterpret_cast<uint16_t*>(ws_tc + L.qsplit[t]);
    mt.psplit = reinterpret_cast<uint16_t*>(ws_tc + L.psplit[t]);
    mt.pdec = reinterpret_cast<uint16_t*>(ws_tc + L.pdec[t]);
    mt.qdec = reinterpret_cast<uint16_t*>(ws_tc + L.qdec[t]);
    mt.Ppart = reinterpret_cast<float*>(ws_tc + L.ppart[t]);
    const int nkb = (int)((n + 63) / 64);
    mt.kchunks = (nkb + PCHUNK_KB - 1) / PCHUNK_KB;
    CUtensorMap* tm = &maps[(size_t)t * NMAPS];
    bool ok = true;
    {  // M_w as a 3D tensor {n, m, W}
      uint64_t d[3] = {(uint64_t)n, (uint64_t)m, (uint64_t)W};
      uint64_t st[2] = {(uint64_t)n * 2, (uint64_t)m * n * 2};
      uint32_t bp[3] = {64, 128, 1}, bq[3] = {64, (uint32_t)(64 * tp->qkps), 1};
      ok &= make_map(&tm[MAP_MP], mt.mscr, 3, d, st, bp);
      ok &= make_map(&tm[MAP_MQ], mt.mscr, 3, d, st, bq);
    }
    const int nb = (h.edt == DT_BF16 ? 3 : 2) * rp;   // B rows; one or two TMA boxes
    const uint32_t box_rows = (uint32_t)(nb <= 256 ? nb : nb / 2);
    {
      uint64_t d[2] = {(uint64_t)n, (uint64_t)nb}, st[1] = {(uint64_t)n * 2};
      uint32_t b[2] = {64, box_rows};
      ok &= make_map(&tm[MAP_QS], mt.qsplit, 2, d, st, b);
    }
    {
      uint64_t d[2] = {(uint64_t)mpad, (uint64_t)nb}, st[1] = {(uint64_t)mpad * 2};
      uint32_t b[2] = {64, box_rows};
      ok &= make_map(&tm[MAP_PS], mt.psplit, 2, d, st, b);
    }
    {
      uint64_t d[2] = {(uint64_t)(3 * kp), (uint64_t)mpad}, st[1] = {(uint64_t)(3 * kp) * 2};
      uint32_t b[2] = {64, 128};
      ok &= make_map(&tm[MAP_PD], mt.pdec, 2, d, st, b);
    }
    {
      uint64_t d[2] = {(uint64_t)(3 * kp), (uint64_t)npad}, st[1] = {(uint64_t)(3 * kp) * 2};
      uint32_t b[2] = {64, (uint32_t)DEC_NT};
      ok &= make_map(&tm[MAP_QD], mt.qdec, 2, d, st, b);
    }
    if (!ok) return cudaErrorInvalidValue;
    for (int i = 0; i < mt.mtiles; ++i)
      for (int c = 0; c < mt.kchunks; ++c)
        pu.push_back(Unit{t, i, c * PCHUNK_KB, std::min(nkb, (c + 1) * PCHUNK_KB), c, 0});
    // slice-major: the units of one slice of rows come back to back, and each CTA takes a
    // contiguous range of them, so it keeps the slice's B tiles across column tiles
    const int mkb = (int)((m + 63) / 64), skb = QSLICE_ROWS / 64;
    for (int s2 = 0; s2 < mt.S; ++s2)
      for (int i = 0; i < (int)((n + 127) / 128); ++i)
        qu.push_back(Unit{t, i, s2 * skb, std::min(mkb, (s2 + 1) * skb), s2, 0});
    for (int i = 0; i < mt.mtiles; ++i)
      for (int jn = 0; jn < (int)(npad / DEC_NT); ++jn) du.push_back(Unit{t, i, jn, jn + 1, 0, 0});
  }
  // largest units first, so the static round-robin ends with the short ones
  auto by_work = [](const Unit& a, const Unit& b) { return (a.kb1 - a.kb0) > (b.kb1 - b.kb0); };
  std::stable_sort(pu.begin(), pu.end(), by_work);

  tp->np = (int)pu.size(); tp->nq = (int)qu.size(); tp->nd = (int)du.size();
  tp->grid = num_sms();
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_maps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_punits, pu.data(), sizeof(Unit) * pu.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_qunits, qu.data(), sizeof(Unit) * qu.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_dunits, du.data(), sizeof(Unit) * du.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  // The dynamic-size cap leaves room for the kernels' few bytes of static shared memory
  // (the abort flag): static + dynamic must stay within the 227 KB a CTA may use.
  const int gs = kDynSmemCap, ds = (int)dec_smem();
  e = cudaFuncSetAttribute(k_gemm<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_ingest_p<__half, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_ingest_p<__nv_bfloat16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_ingest_p<__half, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_ingest_p<__nv_bfloat16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_decomp_tc<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, ds);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_decomp_tc<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, ds);
  return e;
}

void tc_free(Handle& h) {
  delete static_cast<TcPlan*>(h.tc_plan);
  h.tc_plan = nullptr;
}

// Blocks per matrix of k_qmax: about 2048 blocks in all (a few loads per thread for the
// resblock-shard sizes), at least 8 per matrix.
static unsigned qmax_blocks(int BJ) { return (unsigned)std::min(256, std::max(8, 2048 / std::max(BJ, 1))); }

cudaError_t launch_qmax(const Handle& h, const Plan& p, cudaStream_t s) {
  launch_pdl(k_qmax, dim3(qmax_blocks(p.B * p.J), p.B * p.J), dim3(256), 0, s, p);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_prep_q(const Handle& h, const Plan& p, cudaStream_t s) {
  const int BJ = p.B * p.J;
  launch_pdl(k_qmax, dim3(qmax_blocks(BJ), BJ), dim3(256), 0, s, p);
  dim3 g((unsigned)((h.max_ntiles64 * 64 + 31) / 32), BJ);
  if (h.edt == DT_BF16) launch_pdl(k_qsplit<__nv_bfloat16>, dim3(g), dim3(256), 0, s, p);
  else launch_pdl(k_qsplit<__half>, dim3(g), dim3(256), 0, s, p);
  h.launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_pgemm_tc(const Handle& h, const Plan& p, cudaStream_t s) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  const int grid = std::min(tp->grid, tp->np);
  const uint32_t bst = gemm_b_stage(h.edt, p.rp);
  const int ast = gemm_a_stages(bst);
  const size_t sm = gemm_smem(bst, ast);
  const int seg = kGemmSegSteps;
  if (h.edt == DT_BF16) launch_pdl(k_gemm<false, true>, dim3(grid), dim3(kGemmThreads), sm, s, p, tp->d_maps, tp->d_punits, tp->np, ast, bst, 0, seg, 1, 0);
  else launch_pdl(k_gemm<false, false>, dim3(grid), dim3(kGemmThreads), sm, s, p, tp->d_maps, tp->d_punits, tp->np, ast, bst, 0, seg, 1, 0);
  int64_t per = 0;
  for (int j = 0; j < h.J; ++j) per += (h.meta[j].m * p.rp + 1023) / 1024;
  launch_pdl(k_preduce, dim3((unsigned)(per * p.B)), dim3(256), 0, s, p, PCHUNK_KB);
  h.launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_ingest_p(const Handle& h, const Plan& p, cudaStream_t s) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  const int grid = std::min(tp->grid, tp->np);
  const uint32_t bst = gemm_b_stage(h.edt, p.rp);
  int ast, gst, kps;
  size_t sm;
  ingest_stages(h.edt, bst, &ast, &gst, &kps, &sm);
  const int seg = kIngSegSteps;
  // the mask bitmap (a debug output) has its own instantiation: the ingest warps' issue rate
  // sets this kernel's pace, and the bit assembly would slow every step
  if (h.edt == DT_BF16) {
    if (p.mask) k_ingest_p<__nv_bfloat16, true><<<grid, kIngThreads, sm, s>>>(p, tp->d_maps, tp->d_punits, tp->np, ast, gst, kps, bst, seg);
    else k_ingest_p<__nv_bfloat16, false><<<grid, kIngThreads, sm, s>>>(p, tp->d_maps, tp->d_punits, tp->np, ast, gst, kps, bst, seg);
  } else {
    if (p.mask) k_ingest_p<__half, true><<<grid, kIngThreads, sm, s>>>(p, tp->d_maps, tp->d_punits, tp->np, ast, gst, kps, bst, seg);
    else k_ingest_p<__half, false><<<grid, kIngThreads, sm, s>>>(p, tp->d_maps, tp->d_punits, tp->np, ast, gst, kps, bst, seg);
  }
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_preduce(const Handle& h, const Plan& p, cudaStream_t s) {
  int64_t per = 0;
  for (int j = 0; j < h.J; ++j) per += (h.meta[j].m * p.rp + 1023) / 1024;
  launch_pdl(k_preduce, dim3((unsigned)(per * p.B)), dim3(256), 0, s, p, PCHUNK_KB);
  h.launches += 1;
  return cudaGetLastError();
}

int tc_pchunk_kb() { return PCHUNK_KB; }

int tc_kpad(const Handle& h) { return static_cast<const TcPlan*>(h.tc_plan)->kp; }

cudaError_t launch_qgemm_tc(const Handle& h, const Plan& p, cudaStream_t s, bool psplit_done) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  if (!psplit_done) {
    int64_t per = 0;
    for (int j = 0; j < h.J; ++j) per += (h.meta[j].m + 127) / 128 * 4;
    dim3 g((unsigned)(per * p.B));
    if (h.edt == DT_BF16) launch_pdl(k_psplit<__nv_bfloat16>, dim3(g), dim3(256), 0, s, p, tp->kp);
    else launch_pdl(k_psplit<__half>, dim3(g), dim3(256), 0, s, p, tp->kp);
    h.launches += 1;
  }
  const int grid = std::min(tp->grid, tp->nq);
  const int kps = tp->qkps;
  const uint32_t bst = gemm_b_stage(h.edt, p.rp, kps);
  const int ast = gemm_a_stages(bst, kps);
  const size_t sm = gemm_smem(bst, ast, kps);
  const int seg = kGemmSegSteps;
  if (h.edt == DT_BF16) launch_pdl(k_gemm<true, true>, dim3(grid), dim3(kGemmThreads), sm, s, p, tp->d_maps, tp->d_qunits, tp->nq, ast, bst, 0, seg, kps, 1);
  else launch_pdl(k_gemm<true, false>, dim3(grid), dim3(kGemmThreads), sm, s, p, tp->d_maps, tp->d_qunits, tp->nq, ast, bst, 0, seg, kps, 1);
  h.launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_decomp_tc(const Handle& h, const Plan& p, cudaStream_t s) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  dim3 g((unsigned)h.max_ntiles128 * 4, p.B * p.J);
  launch_pdl(k_qdec, dim3(g), dim3(256), 0, s, p, tp->kp);
  const int grid = std::min(tp->grid, tp->nd);
  if (h.edt == DT_BF16) launch_pdl(k_decomp_tc<__nv_bfloat16>, dim3(grid), dim3(DEC_THREADS), dec_smem(), s, p, tp->d_maps, tp->d_dunits, tp->nd, tp->kp);
  else launch_pdl(k_decomp_tc<__half>, dim3(grid), dim3(DEC_THREADS), dec_smem(), s, p, tp->d_maps, tp->d_dunits, tp->nd, tp->kp);
  h.launches += 2;
  return cudaGetLastError();
}

}  // namespace psgd
