// Split operands of the tensor-core GEMMs: an fp32 value scaled by a power of two, written as
// the sum of two or three 16-bit terms (shared by tc.cu and the cooperative
// orthonormalisation kernel, which writes the Q GEMM's P^ operand at its end).
#pragma once

#include <type_traits>

#include "handle.h"

namespace psgd {
namespace splitdev {

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

// From P^ (m x rp fp32, |entries| <= 1): psplit[terms*rp][mpad] = the terms of
// (P^ * 2^14)^T in type T (the type of M), and pdec[mpad][3 kp] = [hi | lo | hi] in fp16
// for the decompression. A block stages 32 rows of P^ (one contiguous run) in shared
// memory; pdec rows are written 8 columns per 16-byte store, psplit rows 8 rows of P^
// per 16-byte store. Item `blk` covers rows [32 blk, 32 blk + 32); a 256-thread group runs it.
template <typename T, class Bar>
__device__ void psplit_rows(const Plan& p, const MatMeta& mt, int kp, int blk, float (*xs)[kRankBlock + 1],
                            int tid, const Bar& bar) {
  const int64_t mpad = (mt.m + 127) / 128 * 128;
  const int64_t row0 = (int64_t)blk * 32;
  if (row0 >= mpad) return;
  const int r = p.r, rp = p.rp;
  const int64_t left = mt.m - row0;
  const int nrows = left <= 0 ? 0 : (left < 32 ? (int)left : 32);
  const float* src = mt.Phat + row0 * rp;
  {  // stage the rows * 2^14 (exact), warp w rows w, w + 8, ..., lane 16 bytes of a row:
     // every load of a thread before its stores (rp is a multiple of 16, P^ 16-byte aligned)
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = (tid >> 5) + 8 * u, c = (tid & 31) * 4;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rr < nrows && c < rp) v[u] = __ldcg(reinterpret_cast<const float4*>(src + (size_t)rr * rp + c));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = (tid >> 5) + 8 * u, c = (tid & 31) * 4;
      if (c < rp) {
        xs[rr][c] = c < r ? v[u].x * 16384.0f : 0.f;
        xs[rr][c + 1] = c + 1 < r ? v[u].y * 16384.0f : 0.f;
        xs[rr][c + 2] = c + 2 < r ? v[u].z * 16384.0f : 0.f;
        xs[rr][c + 3] = c + 3 < r ? v[u].w * 16384.0f : 0.f;
      }
    }
  }
  bar.sync();
  // pdec rows: [hi | lo | hi], kp / 8 groups of 8 columns per segment (kp / 8 is 8 or 16)
  const int gpr = kp / 8, lg = __ffs(gpr) - 1;
  for (int it = tid; it < 32 * gpr; it += 256) {
    const int rr = it >> lg, c0 = (it & (gpr - 1)) * 8;
    __align__(16) uint16_t hh[8], hl[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) split2<__half>(c0 + i < rp ? xs[rr][c0 + i] : 0.f, hh[i], hl[i]);
    uint16_t* pd = mt.pdec + (size_t)(row0 + rr) * 3 * kp;
    *reinterpret_cast<uint4*>(pd + c0) = *reinterpret_cast<const uint4*>(hh);
    *reinterpret_cast<uint4*>(pd + kp + c0) = *reinterpret_cast<const uint4*>(hl);
    *reinterpret_cast<uint4*>(pd + 2 * kp + c0) = *reinterpret_cast<const uint4*>(hh);
  }
  // psplit rows: term k of column c, rows row0 + 8g .. row0 + 8g + 7
  for (int it = tid; it < rp * 4; it += 256) {
    const int c = it >> 2, g = it & 3;
    __align__(16) uint16_t t0[8], t1[8], t2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      t2[i] = 0;
      if (nterms<T>() == 3) split3<T>(xs[8 * g + i][c], t0[i], t1[i], t2[i]);
      else split2<T>(xs[8 * g + i][c], t0[i], t1[i]);
    }
    const size_t col = (size_t)row0 + 8 * g;
    *reinterpret_cast<uint4*>(mt.psplit + (size_t)c * mpad + col) = *reinterpret_cast<const uint4*>(t0);
    *reinterpret_cast<uint4*>(mt.psplit + (size_t)(rp + c) * mpad + col) = *reinterpret_cast<const uint4*>(t1);
    if (nterms<T>() == 3)
      *reinterpret_cast<uint4*>(mt.psplit + (size_t)(2 * rp + c) * mpad + col) = *reinterpret_cast<const uint4*>(t2);
  }
  bar.sync();  // xs is reused by the group's next item
}

}  // namespace splitdev
}  // namespace psgd
