// Orthonormalisation of one P whose scratch is a fixed device array of the library.
//
// psgd_orthonormalize_static runs, for a single fp32 matrix P (m x r), the same adaptive
// shifted CholeskyQR passes that psgd_step applies to every P of a step (the kernels of
// orth.cu, unchanged). It needs no handle and no workspace, and it allocates nothing:
// not through the CUDA runtime, not through a caching allocator, not on the host.
//
// Who calls it: code that holds one P but no psgd handle (a hook that inspects or
// re-orthonormalises a factor, a consistency check run between steps) and that cannot
// allocate device memory at that point. cudaMalloc and cudaFree synchronise the device,
// which would stall the asynchronous work queued around the call, and a process whose
// device memory is already handed out to a caching allocator or a fixed budget has
// nothing left to give.
//
// Scratch: one file-scope __device__ array, kStaticBytes long (16.1 MiB), in every
// device's copy of this module. It holds the one-matrix plan, the scale and pass-state
// words, R^-1 and the Gram partial sums. The two X buffers of the ping-pong between
// passes alias the caller's output P^: the X <- X R^-1 kernel reads the rows of its own
// tile before its last barrier and writes them after it, and no two tiles share a row,
// so each pass may update its buffer in place.
//
// Limits: 1 <= m <= PSGD_STATIC_MAX_ROWS (16384), 1 <= r <= min(m, 128). The Gram
// partial sums take ceil(m / 64) + 1 slots of r x r floats, as in psgd_step, so both
// entry points add the same terms in the same order.
//
// Order of calls: every call uses the one array, so calls that overlap on the GPU
// (different streams of one device, or host threads that enqueue concurrently on
// different streams) race on it. The caller serialises them, e.g. on one stream.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "handle.h"

namespace psgd {
namespace {

constexpr int64_t kStaticMaxRows = PSGD_STATIC_MAX_ROWS;
constexpr int64_t kStaticMaxChunks = (kStaticMaxRows + kGramRows - 1) / kGramRows;

// Byte offsets inside the array (each 256-byte aligned).
constexpr size_t kOffMeta = 0;                                    // MatMeta
constexpr size_t kOffScal = 512;                                  // kScalWords floats
constexpr size_t kOffState = 768;                                 // kMaxPasses x 4 ints
constexpr size_t kOffSkip = 1024;                                 // one byte (block 0)
constexpr size_t kOffRinv = 1280;                                 // r x r floats
constexpr size_t kOffGpart = kOffRinv + 4 * (size_t)kRankBlock * kRankBlock;
constexpr size_t kStaticBytes =
    kOffGpart + 4 * (size_t)(kStaticMaxChunks + 1) * kRankBlock * kRankBlock;

static_assert(PSGD_STATIC_MAX_COLS == kRankBlock, "column limit = the largest rank");
static_assert(sizeof(MatMeta) <= kOffScal - kOffMeta, "plan slot too small");
static_assert(4 * kScalWords <= kOffState - kOffScal, "scale slot too small");
static_assert(4 * 4 * kMaxPasses <= kOffSkip - kOffState, "pass-state slot too small");
static_assert(kOffGpart % 256 == 0 && kStaticBytes % 256 == 0, "alignment");

__device__ __align__(256) static unsigned char g_scratch[kStaticBytes];

// Device address of g_scratch, looked up with the device current and kept per device,
// together with the ID of the CUDA context it belongs to. A later call in another context
// of that device (after cudaDeviceReset, or when the primary context was released and
// created again, which loads the module anew) looks the address up again instead of
// using one that belonged to the old context.
constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
unsigned char* g_addr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(f);
}

// ID of the calling thread's current context (0 if there is none or it cannot be read).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

psgd_status scratch_address(unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return report_error(PSGD_EUNSUPPORTED, "device index beyond the static scratch table");
  std::lock_guard<std::mutex> lock(g_addr_mu);
  const unsigned long long id = current_ctx_id();
  if (!g_addr[dev] || id == 0 || id != g_ctx_id[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);  // makes the device's context current if needed
    if (e != cudaSuccess) return report_cuda_error(e, "cudaGetSymbolAddress(static scratch)");
    if (!p) return report_error(PSGD_ECUDA, "cudaGetSymbolAddress returned a null address");
    g_addr[dev] = static_cast<unsigned char*>(p);
    g_ctx_id[dev] = current_ctx_id();
  }
  *out = g_addr[dev];
  return PSGD_OK;
}

// Writes the one-matrix plan and clears the words that must start at zero: the max|P|
// word (an atomicMax target; the others are unused here), the skip flag that the passes
// test, and the pass records (not read before they are written; cleared so that a
// record never shows an older call's values). One block of 32 threads.
__global__ void k_static_begin(MatMeta* dst, MatMeta mt, uint8_t* skip) {
  const int t = threadIdx.x;
  if (t == 0) { *dst = mt; *skip = 0; }
  if (t < kScalWords) mt.scal[t] = 0.f;
  if (t < 4 * kMaxPasses) mt.ostate[t] = 0;
}

// max|P| over the m x r entries -> scal[SC_MAXP] as float bits (nonnegative floats
// order like their bit patterns). Grid-stride; one atomic per warp.
__global__ void __launch_bounds__(256) k_static_pmax(const float* P, int64_t count,
                                                     unsigned* word) {
  unsigned mx = 0u;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    mx = max(mx, __float_as_uint(fabsf(P[i])));
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((threadIdx.x & 31) == 0 && mx) atomicMax(word, mx);
}

bool overlaps(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

}  // namespace
}  // namespace psgd

using namespace psgd;

extern "C" psgd_status psgd_orthonormalize_static(const float* p, float* phat, int64_t m,
                                                  int32_t r, void* stream) {
  if (!p || !phat) return report_error(PSGD_EINVAL, "p and phat must be device pointers");
  if (m < 1 || r < 1) return report_error(PSGD_EINVAL, "m and r must be >= 1");
  if (m > kStaticMaxRows) {
    char msg[160];
    snprintf(msg, sizeof msg, "m = %lld exceeds the static scratch limit of %lld rows",
             (long long)m, (long long)kStaticMaxRows);
    return report_error(PSGD_EINVAL, msg);
  }
  if (r > kRankBlock) {
    char msg[160];
    snprintf(msg, sizeof msg, "r = %d exceeds the static scratch limit of %d columns", r,
             kRankBlock);
    return report_error(PSGD_EINVAL, msg);
  }
  if (r > m) return report_error(PSGD_EINVAL, "r must be <= m");
  if ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(phat)) % 4 != 0)
    return report_error(PSGD_EINVAL, "p and phat must be 4-byte aligned");
  const size_t bytes = 4 * (size_t)m * r;
  if (overlaps(p, phat, bytes)) return report_error(PSGD_EINVAL, "p and phat overlap");

  unsigned char* base = nullptr;
  const psgd_status st = scratch_address(&base);
  if (st != PSGD_OK) return st;

  MatMeta mt{};
  mt.m = m;
  mt.n = 0;
  mt.b = 0;
  mt.j = 0;
  mt.C = (int)std::max<int64_t>(1, (m + kGramRows - 1) / kGramRows);
  mt.P = const_cast<float*>(p);  // read only
  mt.Xa = phat;
  mt.Xb = phat;
  mt.Phat = phat;
  mt.ostate = reinterpret_cast<int*>(base + kOffState);
  mt.Gpart = reinterpret_cast<float*>(base + kOffGpart);
  mt.Rinv = reinterpret_cast<float*>(base + kOffRinv);
  mt.scal = reinterpret_cast<float*>(base + kOffScal);

  Plan pl{};
  pl.B = 1; pl.J = 1; pl.W = 1;
  pl.r = r; pl.rp = r;  // dense m x r: the orthonormalisation kernels take any row pitch
  pl.ob_r = r; pl.ob_rp = r; pl.ob_c0 = 0; pl.ob_src0 = 0;
  pl.meta = reinterpret_cast<const MatMeta*>(base + kOffMeta);
  pl.skip = reinterpret_cast<uint8_t*>(base + kOffSkip);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_static_begin<<<1, 32, 0, s>>>(reinterpret_cast<MatMeta*>(base + kOffMeta), mt, pl.skip);
  const int64_t count = m * r;
  const int grid = (int)std::min<int64_t>((count + 255) / 256, 152 * 8);
  k_static_pmax<<<grid, 256, 0, s>>>(p, count,
                                     reinterpret_cast<unsigned*>(mt.scal) + SC_MAXP);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return report_cuda_error(e, "static orthonormalisation set-up");
  e = launch_orth_one(pl, mt.C, (int)((m + 63) / 64), s);
  if (e != cudaSuccess) return report_cuda_error(e, "static orthonormalisation");
  return PSGD_OK;
}
