// Tensor-core engine (tcgen05 + TMA, sm_103a) of the step's three matrix products.
//
//   P GEMM   P_part = sum_w M_w[rows, k-chunk] (Q_hi | Q_lo)[k-chunk]     A K-major
//   Q GEMM   Q_part = sum_w M_w[k-slice, cols]^T (P^_hi | P^_lo)[k-slice] A MN-major
//   G^       G^ = (P^_hi | P^_lo | P^_hi) (Q_hi | Q_hi | Q_lo)^T, then E_w = round_E(M_w - G^)
//
// M is exact in its 16-bit type. The fp32 operand (Q or P^) is scaled by a power of two
// and split into 16-bit terms: x*2^e = hi + lo for fp16 (~22 significant bits), and
// hi + mid + lo for bf16 (~24). The terms sit side by side as the N dimension of the
// MMA (N = terms * rp, issued as <= 256-wide pieces), so one pass over M produces every
// partial product in TMEM, and the epilogue adds them. A plain 16-bit product would
// keep 11 (fp16) or 8 (bf16) bits. The decompression
// ("32-bit products for the decompressed gradient", "Zero-Shot Text-to-Image Generation -
// 中文验证版", §证据) uses three products of fp16 splits, so a dropped lo*lo term costs
// ~2^-22.
//
// Persistent kernels, one CTA per SM. Warp 0 issues TMA loads into a ring of
// shared-memory stages. Warp 1 owns TMEM and issues tcgen05.mma from one thread. Four
// (P/Q GEMM) or eight (G^) epilogue warps drain the accumulators, which are double
// buffered in TMEM so the next unit's MMAs overlap the epilogue. Every mbarrier wait is
// bounded. On expiry the kernel records DEVERR_TIMEOUT, waits (bounded) for its own
// TMA loads, releases TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <type_traits>
#include <vector>

#include "handle.h"
#include "tc_ptx.cuh"

namespace psgd {
namespace {

using namespace tc;

constexpr int BM = 128;                // MMA M and A-tile rows (MN extent)
constexpr int BK = 64;                 // K per stage (one 128-byte swizzle span)
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_MAX_ROWS = 3 * kMaxRank;     // split terms x rp
constexpr int B_MAX_BYTES = B_MAX_ROWS * BK * 2;  // 48 KB
constexpr int A_STAGES = 6;
constexpr int B_STAGES = 2;
constexpr int PCHUNK_KB = 4;           // P GEMM: k-blocks of 64 columns per unit
constexpr int QSLICE_ROWS = 512;       // Q GEMM: rows of m per unit (matches Qpart slices)
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
  int grid = 0;
};

__host__ __device__ inline int kpad_of(int rp) { return (rp + 63) / 64 * 64; }

// ---------------------------------------------------------------- small kernels
__device__ __forceinline__ int exp_of_max(unsigned bits) {  // floor(log2 max|x|)
  if (bits == 0u) return 0;
  const int ex = (int)((bits >> 23) & 0xff);
  return (ex == 0 ? -126 : ex - 127);
}

template <typename T> __device__ __forceinline__ uint16_t bits16(T x) {
  return *reinterpret_cast<uint16_t*>(&x);
}

// Split x*2^e into hi + lo in type T (RNE each).
template <typename T>
__device__ __forceinline__ void split2(float xs, uint16_t& hi, uint16_t& lo) {
  const T h = from_f<T>(xs);
  const T l = from_f<T>(__fsub_rn(xs, to_f(h)));
  hi = bits16(h);
  lo = bits16(l);
}

// Split x*2^e into hi + mid + lo in type T (RNE each). Each remainder is exact in fp32.
template <typename T>
__device__ __forceinline__ void split3(float xs, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
  const T h = from_f<T>(xs);
  const float r1 = __fsub_rn(xs, to_f(h));
  const T m = from_f<T>(r1);
  const T l = from_f<T>(__fsub_rn(r1, to_f(m)));
  hi = bits16(h);
  mid = bits16(m);
  lo = bits16(l);
}

// Number of 16-bit terms the fp32 operand of the P and Q GEMMs is split into.
template <typename T> __host__ __device__ constexpr int nterms() { return sizeof(T) == 2 && !std::is_same<T, __half>::value ? 3 : 2; }

// max|Q| of the caller's Q state -> scal[2] (bits). grid = (64, B*J).
__global__ void k_qmax(Plan p) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const float* q = p.tab.q[blockIdx.y];
  const int64_t total = mt.n * p.r;
  unsigned mx = 0u;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
    mx = max(mx, __float_as_uint(fabsf(q[i])));
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((threadIdx.x & 31) == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + 2, mx);
}

// qsplit[terms*rp][n]: rows k*rp + c hold term k of Q[:, c] * 2^e (k = 0 hi, then mid
// for bf16, then lo); e puts max|Q| * 2^e in [2^14, 2^15). Padding rows are 0.
// grid = (ceil(n/256), rp, B*J).
template <typename T>
__global__ void k_qsplit(Plan p) {
  const MatMeta& mt = p.meta[blockIdx.z];
  if (p.skip[mt.b]) return;
  const int c = blockIdx.y, rp = p.rp;
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= mt.n) return;
  const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[2]);
  uint16_t t0 = 0, t1 = 0, t2 = 0;
  if (c < p.r) {
    const float x = ldexpf(p.tab.q[blockIdx.z][j * p.r + c], e);
    if (nterms<T>() == 3) split3<T>(x, t0, t1, t2); else split2<T>(x, t0, t1);
  }
  mt.qsplit[(size_t)c * mt.n + j] = t0;
  mt.qsplit[(size_t)(rp + c) * mt.n + j] = t1;
  if (nterms<T>() == 3) mt.qsplit[(size_t)(2 * rp + c) * mt.n + j] = t2;
}

// P = (sum_c Ppart[c]) * 2^-e / W in chunk order, plus max|P| -> scal[1].
// grid = (ceil(m*rp / 256), B*J).
__global__ void k_preduce(Plan p, int pchunk_kb) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const int rp = p.rp;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t mpad = (mt.m + 127) / 128 * 128;
  unsigned mx = 0u;
  if (i < mt.m * rp) {
    const int kch = (int)(((mt.n + 63) / 64 + pchunk_kb - 1) / pchunk_kb);
    float acc = 0.f;
    for (int c = 0; c < kch; ++c) acc = __fadd_rn(acc, mt.Ppart[(size_t)c * mpad * rp + i]);
    const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[2]);
    const float v = __fdiv_rn(ldexpf(acc, -e), (float)p.W);
    mt.P[i] = v;
    mx = __float_as_uint(fabsf(v));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((threadIdx.x & 31) == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(mt.scal) + 1, mx);
}

// From P^ (m x rp fp32, |entries| <= 1): psplit[terms*rp][mpad] = the terms of
// (P^ * 2^14)^T in type T (the type of M), and pdec[mpad][3 kp] = [hi | lo | hi] in fp16
// for the decompression.
// grid = (ceil(mpad/128), B*J), block 128: thread = row.
template <typename T>
__global__ void k_psplit(Plan p, int kp) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const int64_t mpad = (mt.m + 127) / 128 * 128;
  const int64_t row = (int64_t)blockIdx.x * 128 + threadIdx.x;
  if (row >= mpad) return;
  const int rp = p.rp;
  uint16_t* pd = mt.pdec + (size_t)row * 3 * kp;
  for (int c = 0; c < kp; ++c) {
    const float x = (row < mt.m && c < p.r) ? ldexpf(mt.Phat[row * rp + c], 14) : 0.f;
    uint16_t t0, t1, t2 = 0, hh, hl;
    if (nterms<T>() == 3) split3<T>(x, t0, t1, t2); else split2<T>(x, t0, t1);
    split2<__half>(x, hh, hl);
    if (c < rp) {
      mt.psplit[(size_t)c * mpad + row] = t0;
      mt.psplit[(size_t)(rp + c) * mpad + row] = t1;
      if (nterms<T>() == 3) mt.psplit[(size_t)(2 * rp + c) * mpad + row] = t2;
    }
    pd[c] = hh;
    pd[kp + c] = hl;
    pd[2 * kp + c] = hh;
  }
}

// qdec[npad][3 kp] = [hi | hi | lo] of the new Q * 2^e in fp16 (e from max|Q|, scal[3]).
// grid = (ceil(npad/128), B*J), block 128: thread = row of Q.
__global__ void k_qdec(Plan p, int kp) {
  const MatMeta& mt = p.meta[blockIdx.y];
  if (p.skip[mt.b]) return;
  const int64_t npad = (mt.n + DEC_NT - 1) / DEC_NT * DEC_NT;
  const int64_t row = (int64_t)blockIdx.x * 128 + threadIdx.x;
  if (row >= npad) return;
  const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[3]);
  const float* q = p.tab.q[blockIdx.y];
  uint16_t* qd = mt.qdec + (size_t)row * 3 * kp;
  for (int c = 0; c < kp; ++c) {
    const float x = (row < mt.n && c < p.r) ? ldexpf(q[row * p.r + c], e) : 0.f;
    uint16_t hi, lo;
    split2<__half>(x, hi, lo);
    qd[c] = hi;
    qd[kp + c] = hi;
    qd[2 * kp + c] = lo;
  }
}

// ---------------------------------------------------------------- GEMM kernel
// Shared memory: A ring, B ring, barriers, TMEM address slot.
struct GemmSmem {
  alignas(1024) uint8_t a[A_STAGES][A_BYTES];
  alignas(1024) uint8_t b[B_STAGES][B_MAX_BYTES];
  uint64_t full_a[A_STAGES], empty_a[A_STAGES];
  uint64_t full_b[B_STAGES], empty_b[B_STAGES];
  uint64_t acc_full[2], acc_empty[2], done;
  uint32_t tmem;
};

// MN_A = false: P GEMM (A = M tile K-major, unit = row tile x k-chunk).
// MN_A = true:  Q GEMM (A = M^T tile MN-major, unit = column tile x m-slice).
template <bool MN_A, bool BF16>
__global__ void __launch_bounds__(192, 1)
k_gemm(Plan p, const CUtensorMap* __restrict__ maps, const Unit* __restrict__ units, int nunits) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int TERMS = BF16 ? 3 : 2;
  const int rp = p.rp, N = TERMS * rp;          // B rows = MMA N in total
  const int NACC = N <= 256 ? 2 : 1;            // TMEM accumulators (512 columns)
  const int NBOX = N <= 256 ? 1 : 2;            // TMA boxes per B tile (<= 256 rows each)
  const uint32_t b_bytes = (uint32_t)N * BK * 2;
  int* err = p.err_word;

  if (threadIdx.x == 0) {
    for (int i = 0; i < A_STAGES; ++i) { mbar_init(&sm.full_a[i], 1); mbar_init(&sm.empty_a[i], 1); }
    for (int i = 0; i < B_STAGES; ++i) { mbar_init(&sm.full_b[i], 1); mbar_init(&sm.empty_b[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&sm.acc_full[i], 1); mbar_init(&sm.acc_empty[i], 4); }
    mbar_init(&sm.done, 1);
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
      uint32_t ia = 0, ib = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        const MatMeta& mt = p.meta[un.t];
        if (p.skip[mt.b]) continue;
        const CUtensorMap* mm = maps + (size_t)un.t * NMAPS + (MN_A ? MAP_MQ : MAP_MP);
        const CUtensorMap* mb = maps + (size_t)un.t * NMAPS + (MN_A ? MAP_PS : MAP_QS);
        for (int kb = un.kb0; kb < un.kb1 && ok; ++kb) {
          const int sb = ib % B_STAGES;
          ok = mbar_wait(&sm.empty_b[sb], ((ib / B_STAGES) & 1) ^ 1, err);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.full_b[sb], b_bytes);
          for (int x = 0; x < NBOX; ++x)
            tma_load_2d(sm.b[sb] + x * (N / NBOX) * BK * 2, mb, kb * BK, x * (N / NBOX), &sm.full_b[sb]);
          ++ib;
          for (int w = 0; w < p.W; ++w) {
            const int sa = ia % A_STAGES;
            ok = mbar_wait(&sm.empty_a[sa], ((ia / A_STAGES) & 1) ^ 1, err);
            if (!ok) break;
            mbar_arrive_expect_tx(&sm.full_a[sa], A_BYTES);
            if (!MN_A) {
              tma_load_3d(sm.a[sa], mm, kb * BK, un.tile * BM, w, &sm.full_a[sa]);
            } else {
              tma_load_3d(sm.a[sa], mm, un.tile * BM, kb * BK, w, &sm.full_a[sa]);
              tma_load_3d(sm.a[sa] + A_BYTES / 2, mm, un.tile * BM + 64, kb * BK, w, &sm.full_a[sa]);
            }
            ++ia;
          }
        }
      }
      // wait (bounded) for every load this thread issued before the CTA may exit
      for (uint32_t k = (ia > A_STAGES ? ia - A_STAGES : 0); k < ia; ++k)
        mbar_wait(&sm.full_a[k % A_STAGES], (k / A_STAGES) & 1, err, 1u << 20);
      for (uint32_t k = (ib > B_STAGES ? ib - B_STAGES : 0); k < ib; ++k)
        mbar_wait(&sm.full_b[k % B_STAGES], (k / B_STAGES) & 1, err, 1u << 20);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int n0 = N <= 256 ? N : 256;        // MMA pieces: [0, n0) and [n0, N)
      const uint32_t idesc0 = idesc_f16(BM, n0, BF16, MN_A, false);
      const uint32_t idesc1 = idesc_f16(BM, N > 256 ? N - 256 : 16, BF16, MN_A, false);
      uint32_t ia = 0, ib = 0, ju = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        if (p.skip[p.meta[un.t].b]) continue;
        const int acc = (int)(ju % NACC);
        ok = mbar_wait(&sm.acc_empty[acc], ((ju / NACC) & 1) ^ 1, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
        uint32_t accum = 0;
        for (int kb = un.kb0; kb < un.kb1 && ok; ++kb) {
          const int sb = ib % B_STAGES;
          ok = mbar_wait(&sm.full_b[sb], (ib / B_STAGES) & 1, err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t b_addr = smem_u32(sm.b[sb]);
          for (int w = 0; w < p.W; ++w) {
            const int sa = ia % A_STAGES;
            ok = mbar_wait(&sm.full_a[sa], (ia / A_STAGES) & 1, err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sm.a[sa]);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t adesc = MN_A ? smem_desc(a_addr + k * 2048, A_BYTES / 2, 1024)
                                          : smem_desc(a_addr + k * 32, 16, 1024);
              umma_f16(d_tmem, adesc, smem_desc(b_addr + k * 32, 16, 1024), idesc0, accum);
              if (N > 256)
                umma_f16(d_tmem + 256, adesc, smem_desc(b_addr + 256 * 128 + k * 32, 16, 1024), idesc1, accum);
              accum = 1;
            }
            umma_commit(&sm.empty_a[sa]);
            ++ia;
          }
          umma_commit(&sm.empty_b[sb]);
          ++ib;
        }
        umma_commit(&sm.acc_full[acc]);
        ++ju;
      }
      umma_commit(&sm.done);
      mbar_wait(&sm.done, 0, err, 1u << 22);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint32_t ju = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const Unit un = units[u];
      const MatMeta& mt = p.meta[un.t];
      if (p.skip[mt.b]) continue;
      const int acc = (int)(ju % NACC);
      ok = mbar_wait(&sm.acc_full[acc], (ju / NACC) & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (uint32_t)(acc * 256) + ((uint32_t)(quarter * 32) << 16);
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
      for (int c = 0; c < rp; c += 16) {
        float v[16], t[16];
        tmem_ld16(t_row + c, v);
#pragma unroll
        for (int k = 1; k < TERMS; ++k) {
          tmem_ld16(t_row + k * rp + c, t);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] += t[i];
        }
        if (grow < limit) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(out + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
      ++ju;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------- decompression kernel
struct DecSmem {
  alignas(1024) uint8_t a[A_STAGES][A_BYTES];          // P^ split tiles, 128 x 64
  alignas(1024) uint8_t b[A_STAGES][DEC_NT * BK * 2];  // Q split tiles, 128 x 64
  uint64_t full[A_STAGES], empty[A_STAGES];
  uint64_t acc_full[2], acc_empty[2], done;
  uint32_t tmem;
};

template <typename TE> struct Pack8;
template <> struct Pack8<__half> { using T = uint4; };
template <> struct Pack8<__nv_bfloat16> { using T = uint4; };

// G^ tile 128 x 128 = A B^T over K = 3 kp, then E_w = round_E(M_w - G^) for every w.
// Warps: 0 TMA, 1 MMA, 2..9 epilogue (two warps per TMEM lane quarter, 64 columns each).
template <typename TE>
__global__ void __launch_bounds__(320, 1)
k_decomp_tc(Plan p, const CUtensorMap* __restrict__ maps, const Unit* __restrict__ units, int nunits, int kp) {
  extern __shared__ uint8_t smem_raw[];
  DecSmem& sm = *reinterpret_cast<DecSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = 3 * kp / BK;
  int* err = p.err_word;
  constexpr uint32_t STAGE_TX = A_BYTES + DEC_NT * BK * 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < A_STAGES; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&sm.acc_full[i], 1); mbar_init(&sm.acc_empty[i], 8); }
    mbar_init(&sm.done, 1);
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
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Unit un = units[u];
        if (p.skip[p.meta[un.t].b]) continue;
        const CUtensorMap* ma = maps + (size_t)un.t * NMAPS + MAP_PD;
        const CUtensorMap* mb = maps + (size_t)un.t * NMAPS + MAP_QD;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          const int s = it % A_STAGES;
          ok = mbar_wait(&sm.empty[s], ((it / A_STAGES) & 1) ^ 1, err);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.full[s], STAGE_TX);
          tma_load_2d(sm.a[s], ma, kb * BK, un.tile * BM, &sm.full[s]);
          tma_load_2d(sm.b[s], mb, kb * BK, un.kb0 * DEC_NT, &sm.full[s]);
          ++it;
        }
      }
      for (uint32_t k = (it > A_STAGES ? it - A_STAGES : 0); k < it; ++k)
        mbar_wait(&sm.full[k % A_STAGES], (k / A_STAGES) & 1, err, 1u << 20);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(BM, DEC_NT, false, false, false);
      uint32_t it = 0, ju = 0;
      bool ok = true;
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
          const int s = it % A_STAGES;
          ok = mbar_wait(&sm.full[s], (it / A_STAGES) & 1, err);
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
      mbar_wait(&sm.done, 0, err, 1u << 22);
    }
  } else {
    const int ew = warp - 2;             // 0..7
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int half = ew >> 2;            // column half: 0 -> [0, 64), 1 -> [64, 128)
    const int row_in_tile = quarter * 32 + lane;
    uint32_t ju = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const Unit un = units[u];
      const MatMeta& mt = p.meta[un.t];
      const int64_t m = mt.m, n = mt.n;
      const int64_t row = (int64_t)un.tile * BM + row_in_tile;
      const int64_t col0 = (int64_t)un.kb0 * DEC_NT + half * 64;
      float* gh = p.tab.ghat[un.t];
      if (p.skip[mt.b]) {
        if (row < m)
          for (int c = 0; c < 64; c += 4)
            if (col0 + c < n) *reinterpret_cast<float4*>(gh + row * n + col0 + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int acc = ju & 1;
      ok = mbar_wait(&sm.acc_full[acc], (ju >> 1) & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (uint32_t)(acc * DEC_NT + half * 64) + ((uint32_t)(quarter * 32) << 16);
      // G^ = acc * 2^-(14 + e): P^ was scaled by 2^14 and Q by 2^e. ldexpf keeps
      // results that fall into fp32's subnormal range correctly rounded.
      const int e = 14 - exp_of_max(reinterpret_cast<const unsigned*>(mt.scal)[3]);
      for (int c = 0; c < 64; c += 16) {
        float g[16];
        tmem_ld16(t_row + c, g);
#pragma unroll
        for (int i = 0; i < 16; ++i) g[i] = ldexpf(g[i] * 0x1p-14f, -e);
        const int64_t col = col0 + c;
        if (row < m && col < n) {
          // n is a multiple of 8, so a 16-column group is either fully inside or
          // ends on a multiple of 8 within it.
          const int nv = n - col < 16 ? (int)(n - col) : 16;
          float* gp = gh + row * n + col;
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            if (i < nv) *reinterpret_cast<float4*>(gp + i) = make_float4(g[i], g[i + 1], g[i + 2], g[i + 3]);
          const TE* mbase = static_cast<const TE*>(mt.mscr) + row * n + col;
          for (int w = 0; w < p.W; ++w) {
            const TE* mp = mbase + (size_t)w * m * n;
            TE* ep = static_cast<TE*>(p.tab.e[(size_t)un.t * p.W + w]) + row * n + col;
#pragma unroll
            for (int h = 0; h < 16; h += 8) {
              if (h < nv) {
                uint4 mv = *reinterpret_cast<const uint4*>(mp + h);
                const TE* mx = reinterpret_cast<const TE*>(&mv);
                TE ev[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ev[i] = add_to<TE>(to_f(mx[i]), -g[h + i]);
                *reinterpret_cast<uint4*>(ep + h) = *reinterpret_cast<const uint4*>(ev);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
      ++ju;
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
              const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, (cuuint32_t)rank, base, d, s, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

size_t gemm_smem() { return sizeof(GemmSmem) + 1024; }
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

size_t tc_workspace_bytes(const psgd_config* cfg) {
  if (cfg->err_dtype == PSGD_F32 || (cfg->flags & PSGD_FLAG_SIMT)) return 0;
  return tc_layout(cfg).total;
}

bool tc_supported(const psgd_config* cfg, std::string* why) {
  if (cfg->err_dtype == PSGD_F32) { if (why) *why = "fp32 gradients use the FFMA engine"; return false; }
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
      uint32_t bp[3] = {64, 128, 1}, bq[3] = {64, 64, 1};
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
    const int mkb = (int)((m + 63) / 64), skb = QSLICE_ROWS / 64;
    for (int i = 0; i < (int)((n + 127) / 128); ++i)
      for (int s2 = 0; s2 < mt.S; ++s2)
        qu.push_back(Unit{t, i, s2 * skb, std::min(mkb, (s2 + 1) * skb), s2, 0});
    for (int i = 0; i < mt.mtiles; ++i)
      for (int jn = 0; jn < (int)(npad / DEC_NT); ++jn) du.push_back(Unit{t, i, jn, jn + 1, 0, 0});
  }
  // largest units first, so the static round-robin ends with the short ones
  auto by_work = [](const Unit& a, const Unit& b) { return (a.kb1 - a.kb0) > (b.kb1 - b.kb0); };
  std::stable_sort(pu.begin(), pu.end(), by_work);
  std::stable_sort(qu.begin(), qu.end(), by_work);
  tp->np = (int)pu.size(); tp->nq = (int)qu.size(); tp->nd = (int)du.size();
  tp->grid = num_sms();
  cudaError_t e = cudaMemcpyAsync(tp->d_maps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_punits, pu.data(), sizeof(Unit) * pu.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_qunits, qu.data(), sizeof(Unit) * qu.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(tp->d_dunits, du.data(), sizeof(Unit) * du.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  const int gs = (int)gemm_smem(), ds = (int)dec_smem();
  e = cudaFuncSetAttribute(k_gemm<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_decomp_tc<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, ds);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_decomp_tc<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, ds);
  return e;
}

void tc_free(Handle& h) {
  delete static_cast<TcPlan*>(h.tc_plan);
  h.tc_plan = nullptr;
}

cudaError_t launch_prep_q(const Handle& h, const Plan& p, cudaStream_t s) {
  const int BJ = p.B * p.J;
  k_qmax<<<dim3(64, BJ), 256, 0, s>>>(p);
  dim3 g((unsigned)((h.max_ntiles64 * 64 + 255) / 256), p.rp, BJ);
  if (h.edt == DT_BF16) k_qsplit<__nv_bfloat16><<<g, 256, 0, s>>>(p);
  else k_qsplit<__half><<<g, 256, 0, s>>>(p);
  h.launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_pgemm_tc(const Handle& h, const Plan& p, cudaStream_t s) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  const int grid = std::min(tp->grid, tp->np);
  if (h.edt == DT_BF16) k_gemm<false, true><<<grid, 192, gemm_smem(), s>>>(p, tp->d_maps, tp->d_punits, tp->np);
  else k_gemm<false, false><<<grid, 192, gemm_smem(), s>>>(p, tp->d_maps, tp->d_punits, tp->np);
  int64_t maxe = 0;
  for (const MatMeta& mt : h.meta) maxe = std::max<int64_t>(maxe, mt.m * p.rp);
  k_preduce<<<dim3((unsigned)((maxe + 255) / 256), p.B * p.J), 256, 0, s>>>(p, PCHUNK_KB);
  h.launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_qgemm_tc(const Handle& h, const Plan& p, cudaStream_t s) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  dim3 g((unsigned)h.max_mtiles, p.B * p.J);
  if (h.edt == DT_BF16) k_psplit<__nv_bfloat16><<<g, 128, 0, s>>>(p, tp->kp);
  else k_psplit<__half><<<g, 128, 0, s>>>(p, tp->kp);
  const int grid = std::min(tp->grid, tp->nq);
  if (h.edt == DT_BF16) k_gemm<true, true><<<grid, 192, gemm_smem(), s>>>(p, tp->d_maps, tp->d_qunits, tp->nq);
  else k_gemm<true, false><<<grid, 192, gemm_smem(), s>>>(p, tp->d_maps, tp->d_qunits, tp->nq);
  h.launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_decomp_tc(const Handle& h, const Plan& p, cudaStream_t s) {
  const TcPlan* tp = static_cast<const TcPlan*>(h.tc_plan);
  dim3 g((unsigned)((h.max_ntiles128 * 128 + 127) / 128), p.B * p.J);
  k_qdec<<<g, 128, 0, s>>>(p, tp->kp);
  const int grid = std::min(tp->grid, tp->nd);
  if (h.edt == DT_BF16) k_decomp_tc<__nv_bfloat16><<<grid, 320, dec_smem(), s>>>(p, tp->d_maps, tp->d_dunits, tp->nd, tp->kp);
  else k_decomp_tc<__half><<<grid, 320, dec_smem(), s>>>(p, tp->d_maps, tp->d_dunits, tp->nd, tp->kp);
  h.launches += 2;
  return cudaGetLastError();
}

}  // namespace psgd
