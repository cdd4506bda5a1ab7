// Host side of the C ABI declared in psgd.h: validation, workspace planning, the
// per-step pointer table, and the launch sequence of one PowerSGD step.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "handle.h"

namespace psgd {
namespace {

thread_local std::string g_last_error;

psgd_status fail(psgd_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

psgd_status cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return PSGD_ECUDA;
}

size_t esize(int dt) { return dt == DT_F32 ? 4 : 2; }
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rows of a Q-GEMM slice (one Q partial sum each): 256 on the tensor engine, where
// finer slices balance its units over the SMs; 512 on the FFMA engine, whose partials
// at large r are large.
constexpr int64_t kSliceRowsTc = 256, kSliceRowsSimt = 512;
int64_t slice_rows(const psgd_config* c) {
  std::string why;
  const bool tc = c->err_dtype != DT_F32 && !(c->flags & PSGD_FLAG_SIMT) && tc_supported(c, &why);
  return tc ? kSliceRowsTc : kSliceRowsSimt;
}

struct Layout {
  size_t total = 0;
  size_t meta = 0, threshold = 0, mask_off = 0, segs = 0, table = 0, err = 0, scal = 0;
  size_t inv_dev = 0, gbar = 0, noskip = 0, xcnt = 0;
  std::vector<size_t> mscr, P, Xa, Xb, Phat, ostate, Qpart, Gpart, Rinv, xp, xq;
  size_t tc = 0;
  size_t table_bytes = 0, maps_bytes = 0, table_stride = 0;
  int64_t nseg = 0;
};

bool valid_dtype(int d) { return d == DT_F32 || d == DT_F16 || d == DT_BF16; }

psgd_status validate_config(const psgd_config* c) {
  if (!c) return fail(PSGD_EINVAL, "config is NULL");
  if (c->num_blocks < 1 || c->mats_per_block < 1 || c->num_workers < 1)
    return fail(PSGD_EINVAL, "num_blocks, mats_per_block and num_workers must be >= 1");
  if (!c->shapes) return fail(PSGD_EINVAL, "shapes is NULL");
  if (!valid_dtype(c->grad_dtype) || !valid_dtype(c->err_dtype))
    return fail(PSGD_EINVAL, "unknown dtype");
  if (c->grad_dtype != c->err_dtype)
    return fail(PSGD_EUNSUPPORTED, "grad_dtype and err_dtype must be equal");
  if (c->rank < 1) return fail(PSGD_EINVAL, "rank must be >= 1");
  if (c->rank > kMaxRank)
    return fail(PSGD_EUNSUPPORTED, "rank above 1024 is not supported");
  if (c->unc_len < 0) return fail(PSGD_EINVAL, "unc_len must be >= 0");
  if ((c->flags & PSGD_FLAG_EXCHANGE) && c->unc_len != 0)
    return fail(PSGD_EUNSUPPORTED, "PSGD_FLAG_EXCHANGE needs unc_len == 0 (reduce gains/biases separately)");
  if ((c->flags & PSGD_FLAG_EXCHANGE) && (c->flags & PSGD_FLAG_STOP_AFTER_INGEST))
    return fail(PSGD_EUNSUPPORTED, "PSGD_FLAG_EXCHANGE and PSGD_FLAG_STOP_AFTER_INGEST do not mix");
  if (!(c->skip_fraction > 0.0 && c->skip_fraction <= 1.0))
    return fail(PSGD_EINVAL, "skip_fraction must be in (0, 1]");
  const size_t es = esize(c->grad_dtype);
  for (int j = 0; j < c->mats_per_block; ++j) {
    const psgd_shape s = c->shapes[j];
    if (s.m < 1 || s.n < 1) return fail(PSGD_EINVAL, "matrix shapes must be positive");
    if ((s.n * (int64_t)es) % 16 != 0)
      return fail(PSGD_EINVAL, "n * element size must be a multiple of 16 bytes");
    if (c->rank > s.m || c->rank > s.n) return fail(PSGD_EINVAL, "rank must be <= min(m, n)");
    if (s.m > (1ll << 31) || s.n > (1ll << 31)) return fail(PSGD_EINVAL, "matrix too large");
  }
  return PSGD_OK;
}

Layout plan_layout(const psgd_config* c) {
  Layout L;
  const int B = c->num_blocks, J = c->mats_per_block, W = c->num_workers;
  const int rp = (c->rank + 15) / 16 * 16;
  const size_t es = esize(c->err_dtype);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = up256(off + bytes); return o; };
  L.meta = take(sizeof(MatMeta) * B * J);
  L.threshold = take(8 * (size_t)B);
  L.mask_off = take(8 * (size_t)B * J * W);
  L.nseg = (int64_t)B * J * W + (c->unc_len > 0 ? (int64_t)B * W : 0);
  L.segs = take(sizeof(IngestSeg) * L.nseg);
  L.table_bytes = 8 * ((size_t)2 * B * J * W + 2 * (size_t)B * J + (size_t)B * W + B) + 4 * (size_t)B;
  L.table_bytes = (L.table_bytes + 127) / 128 * 128;
  L.maps_bytes = tc_ge_maps_bytes(c);
  L.table_stride = up256(L.table_bytes + L.maps_bytes);
  L.table = take(Handle::kTableSlots * L.table_stride);
  L.err = take(16);
  L.scal = take(4 * kScalWords * (size_t)B * J);
  L.inv_dev = take(4 * (size_t)B);
  L.gbar = take(sizeof(GridBarrier));
  L.noskip = take((size_t)B);
  if (c->flags & PSGD_FLAG_EXCHANGE) L.xcnt = take(8 * (size_t)B);
  for (int t = 0; t < B * J; ++t) {
    const psgd_shape s = c->shapes[t % J];
    const int64_t mpad = ceil_div(s.m, 128) * 128;
    const int64_t S = std::max<int64_t>(1, ceil_div(s.m, slice_rows(c)));
    const int64_t C = std::max<int64_t>(1, ceil_div(s.m, kGramRows));
    L.mscr.push_back(take(es * (size_t)W * s.m * s.n));
    L.P.push_back(take(4 * (size_t)mpad * rp));
    L.Xa.push_back(take(4 * (size_t)mpad * rp));
    L.Xb.push_back(take(4 * (size_t)mpad * rp));
    L.Phat.push_back(take(4 * (size_t)mpad * rp));
    L.ostate.push_back(take(4 * 4 * kMaxPasses));
    L.Qpart.push_back(take(4 * (size_t)S * s.n * rp));
    L.Gpart.push_back(take(4 * (size_t)(C + 1) * rp * rp));  // C partials + their sum
    L.Rinv.push_back(take(4 * (size_t)rp * rp));
  }
  if (c->flags & PSGD_FLAG_EXCHANGE) {
    // The exchange buffers of the data-parallel calls: every matrix's P sum back to back
    // in (b, j) order, then every Q sum, so that one all-reduce covers each.
    size_t np = 0, nq = 0;
    for (int t = 0; t < B * J; ++t) {
      np += (size_t)c->shapes[t % J].m * c->rank;
      nq += (size_t)c->shapes[t % J].n * c->rank;
    }
    size_t op = take(4 * np), oq = take(4 * nq);
    for (int t = 0; t < B * J; ++t) {
      L.xp.push_back(op);
      L.xq.push_back(oq);
      op += 4 * (size_t)c->shapes[t % J].m * c->rank;
      oq += 4 * (size_t)c->shapes[t % J].n * c->rank;
    }
  }
  L.tc = take(tc_workspace_bytes(c));
  L.total = off;
  return L;
}

}  // namespace

// Error reporting for the entry points that live in other files.
psgd_status report_error(psgd_status s, const std::string& msg) { return fail(s, msg); }
psgd_status report_cuda_error(cudaError_t e, const char* where) { return cuda_fail(e, where); }

}  // namespace psgd

using namespace psgd;

struct psgd_handle {
  Handle h;
};

extern "C" {

const char* psgd_strerror(psgd_status s) {
  switch (s) {
    case PSGD_OK: return "ok";
    case PSGD_EINVAL: return "invalid argument";
    case PSGD_ECUDA: return "CUDA error";
    case PSGD_EUNSUPPORTED: return "unsupported configuration";
    case PSGD_ETIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* psgd_last_error(void) { return g_last_error.c_str(); }

size_t psgd_workspace_size(const psgd_config* cfg) {
  if (validate_config(cfg) != PSGD_OK) return 0;
  return plan_layout(cfg).total;
}

int64_t psgd_mask_words(const psgd_config* c) {
  if (validate_config(c) != PSGD_OK) return -1;
  int64_t tot = 0;
  for (int j = 0; j < c->mats_per_block; ++j)
    tot += ceil_div(c->shapes[j].m * c->shapes[j].n, 32);
  return tot * c->num_blocks * c->num_workers;
}

int64_t psgd_mask_offset(const psgd_config* c, int32_t b, int32_t j, int32_t w) {
  if (validate_config(c) != PSGD_OK) return -1;
  if (b < 0 || b >= c->num_blocks || j < 0 || j >= c->mats_per_block || w < 0 ||
      w >= c->num_workers)
    return -1;
  int64_t per_block = 0, before_j = 0;
  for (int k = 0; k < c->mats_per_block; ++k) {
    const int64_t words = ceil_div(c->shapes[k].m * c->shapes[k].n, 32);
    if (k < j) before_j += words;
    per_block += words;
  }
  const int64_t wj = ceil_div(c->shapes[j].m * c->shapes[j].n, 32);
  return (int64_t)b * c->num_workers * per_block + before_j * c->num_workers + (int64_t)w * wj;
}

psgd_status psgd_init(const psgd_config* cfg, void* workspace, size_t ws_bytes, void* stream,
                      psgd_handle** out) {
  if (!out) return fail(PSGD_EINVAL, "out is NULL");
  *out = nullptr;
  psgd_status st = validate_config(cfg);
  if (st != PSGD_OK) return st;
  if (!workspace) return fail(PSGD_EINVAL, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(PSGD_EINVAL, "workspace must be 256-byte aligned");
  const Layout L = plan_layout(cfg);
  if (ws_bytes < L.total)
    return fail(PSGD_EINVAL, "workspace too small: need " + std::to_string(L.total) + " bytes");
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  psgd_handle* ph = new (std::nothrow) psgd_handle();
  if (!ph) return fail(PSGD_EINVAL, "out of host memory");
  Handle& h = ph->h;
  h.cfg = *cfg;
  h.shapes.assign(cfg->shapes, cfg->shapes + cfg->mats_per_block);
  h.cfg.shapes = h.shapes.data();
  h.B = cfg->num_blocks; h.J = cfg->mats_per_block; h.W = cfg->num_workers;
  h.r = cfg->rank; h.rp = (cfg->rank + 15) / 16 * 16;
  h.gdt = cfg->grad_dtype; h.edt = cfg->err_dtype;
  h.ws = static_cast<char*>(workspace);
  h.ws_bytes = ws_bytes;
  std::string why;
  h.tc = h.edt != DT_F32 && !(cfg->flags & PSGD_FLAG_SIMT) && tc_supported(cfg, &why);
  if ((cfg->flags & PSGD_FLAG_DEBUG_EXPIRE_WAIT) && !h.tc) {
    delete ph;
    return fail(PSGD_EUNSUPPORTED, "PSGD_FLAG_DEBUG_EXPIRE_WAIT needs the tensor engine");
  }

  const int BJ = h.B * h.J;
  h.d_meta = reinterpret_cast<MatMeta*>(h.ws + L.meta);
  h.d_threshold = reinterpret_cast<int64_t*>(h.ws + L.threshold);
  h.d_mask_off = reinterpret_cast<int64_t*>(h.ws + L.mask_off);
  h.d_segs = reinterpret_cast<IngestSeg*>(h.ws + L.segs);
  h.d_table = h.ws + L.table;
  h.table_bytes = L.table_bytes;
  h.table_stride = L.table_stride;
  h.maps_bytes = h.tc ? L.maps_bytes : 0;
  h.d_err = reinterpret_cast<int*>(h.ws + L.err);
  h.d_scal_all = reinterpret_cast<float*>(h.ws + L.scal);
  h.d_inv_dev = reinterpret_cast<float*>(h.ws + L.inv_dev);
  h.d_gbar = reinterpret_cast<GridBarrier*>(h.ws + L.gbar);
  h.d_noskip = reinterpret_cast<uint8_t*>(h.ws + L.noskip);
  if (cfg->flags & PSGD_FLAG_EXCHANGE) h.d_xcnt = reinterpret_cast<int64_t*>(h.ws + L.xcnt);

  h.meta.resize(BJ);
  for (int t = 0; t < BJ; ++t) {
    const psgd_shape sh = h.shapes[t % h.J];
    MatMeta& mt = h.meta[t];
    std::memset(&mt, 0, sizeof(mt));
    mt.m = sh.m; mt.n = sh.n; mt.b = t / h.J; mt.j = t % h.J;
    mt.S = (int)std::max<int64_t>(1, ceil_div(sh.m, h.tc ? kSliceRowsTc : kSliceRowsSimt));
    mt.C = (int)std::max<int64_t>(1, ceil_div(sh.m, kGramRows));
    mt.mtiles = (int)ceil_div(sh.m, 128);
    mt.mscr = h.ws + L.mscr[t];
    mt.P = reinterpret_cast<float*>(h.ws + L.P[t]);
    mt.Xa = reinterpret_cast<float*>(h.ws + L.Xa[t]);
    mt.Xb = reinterpret_cast<float*>(h.ws + L.Xb[t]);
    mt.Phat = reinterpret_cast<float*>(h.ws + L.Phat[t]);
    mt.ostate = reinterpret_cast<int*>(h.ws + L.ostate[t]);
    mt.Qpart = reinterpret_cast<float*>(h.ws + L.Qpart[t]);
    mt.Gpart = reinterpret_cast<float*>(h.ws + L.Gpart[t]);
    mt.Rinv = reinterpret_cast<float*>(h.ws + L.Rinv[t]);
    mt.scal = h.d_scal_all + kScalWords * t;
    if (cfg->flags & PSGD_FLAG_EXCHANGE) {
      mt.xp = reinterpret_cast<float*>(h.ws + L.xp[t]);
      mt.xq = reinterpret_cast<float*>(h.ws + L.xq[t]);
    }
    h.max_mtiles = std::max(h.max_mtiles, mt.mtiles);
    h.max_S = std::max(h.max_S, mt.S);
    h.max_C = std::max(h.max_C, mt.C);
    h.max_ntiles64 = std::max<int>(h.max_ntiles64, (int)ceil_div(sh.n, 64));
    h.max_mtiles64 = std::max<int>(h.max_mtiles64, (int)ceil_div(sh.m, 64));
    h.max_ntiles128 = std::max<int>(h.max_ntiles128, (int)ceil_div(sh.n, 128));
  }
  // thresholds: ceil(T * W * numel_b) in IEEE double
  int64_t numel_b = cfg->unc_len;
  for (int j = 0; j < h.J; ++j) numel_b += h.shapes[j].m * h.shapes[j].n;
  std::vector<int64_t> thr(h.B, (int64_t)std::ceil(cfg->skip_fraction * (double)(h.W * numel_b)));
  std::vector<int64_t> moff((size_t)BJ * h.W);
  for (int b = 0; b < h.B; ++b)
    for (int j = 0; j < h.J; ++j)
      for (int w = 0; w < h.W; ++w) moff[((size_t)b * h.J + j) * h.W + w] = psgd_mask_offset(cfg, b, j, w);
  // ingest segments
  int64_t cta = 0;
  for (int t = 0; t < BJ; ++t)
    for (int w = 0; w < h.W; ++w) {
      IngestSeg sg{};
      sg.numel = h.meta[t].m * h.meta[t].n;
      sg.cta_start = cta;
      sg.kind = 0; sg.t = t; sg.b = h.meta[t].b; sg.w = w;
      h.segs.push_back(sg);
      cta += ceil_div(sg.numel, kIngestChunk);
    }
  h.unc_cta_start = cta;
  if (cfg->unc_len > 0)
    for (int b = 0; b < h.B; ++b)
      for (int w = 0; w < h.W; ++w) {
        IngestSeg sg{};
        sg.numel = cfg->unc_len;
        sg.cta_start = cta;
        sg.kind = 1; sg.t = -1; sg.b = b; sg.w = w;
        h.segs.push_back(sg);
        cta += ceil_div(sg.numel, kIngestChunk);
      }
  h.ingest_ctas = cta;

  cudaError_t e;
  if (h.tc && (e = tc_plan(h, h.ws + L.tc, s)) != cudaSuccess) {
    tc_free(h);
    delete ph;
    return cuda_fail(e, "tensor-engine plan");
  }
  // Upload the static tables (synchronously: init is not on the hot path).
  e = cudaMemcpyAsync(h.d_meta, h.meta.data(), sizeof(MatMeta) * BJ, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h.d_threshold, thr.data(), 8 * thr.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h.d_mask_off, moff.data(), 8 * moff.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h.d_segs, h.segs.data(), sizeof(IngestSeg) * h.segs.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h.d_err, 0, 16, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h.d_noskip, 0, (size_t)h.B, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void**>(&h.h_stage), Handle::kTableSlots * h.table_stride, cudaHostAllocDefault);
  for (int k = 0; k < Handle::kTableSlots && e == cudaSuccess; ++k)
    e = cudaEventCreateWithFlags(&h.slot_ev[k], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (int k = 0; k < Handle::kTableSlots; ++k)
      if (h.slot_ev[k]) cudaEventDestroy(h.slot_ev[k]);
    if (h.h_stage) cudaFreeHost(h.h_stage);
    tc_free(h);
    delete ph;
    return cuda_fail(e, "psgd_init");
  }
  *out = ph;
  return PSGD_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validation of a step's arguments, the pointer table (uploaded when it changes) and the
// plan of the launches. Every step entry point starts here.
static psgd_status prepare_step(psgd_handle* ph, const psgd_step_args* a, void* stream, Plan& p) {
  if (!ph || !a) return fail(PSGD_EINVAL, "handle or args is NULL");
  Handle& h = ph->h;
  const size_t B = h.B, J = h.J, W = h.W;
  if (!a->grads || !a->errs || !a->q_state || !a->ghat || !a->counts || !a->skip)
    return fail(PSGD_EINVAL, "a required argument array is NULL");
  const bool dev_scales = a->scales_device != nullptr;
  if (!dev_scales && !a->scales) return fail(PSGD_EINVAL, "scales or scales_device is required");
  if (dev_scales && (reinterpret_cast<uintptr_t>(a->scales_device) & 3u))
    return fail(PSGD_EINVAL, "scales_device must be 4-byte aligned");
  if (h.cfg.unc_len > 0 && (!a->unc_in || !a->unc_out))
    return fail(PSGD_EINVAL, "unc_in/unc_out are required when unc_len > 0");
  if ((h.cfg.flags & PSGD_FLAG_MASK) && !a->mask_bits)
    return fail(PSGD_EINVAL, "mask_bits is required with PSGD_FLAG_MASK");
  for (size_t i = 0; i < B * J * W; ++i) {
    if (!a->grads[i] || !a->errs[i]) return fail(PSGD_EINVAL, "NULL gradient or error pointer");
    if (!aligned16(a->grads[i]) || !aligned16(a->errs[i]))
      return fail(PSGD_EINVAL, "gradient and error pointers must be 16-byte aligned");
  }
  for (size_t i = 0; i < B * J; ++i) {
    if (!a->q_state[i] || !a->ghat[i]) return fail(PSGD_EINVAL, "NULL Q or G-hat pointer");
    if (!aligned16(a->ghat[i])) return fail(PSGD_EINVAL, "G-hat pointers must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(a->q_state[i]) & 3u) return fail(PSGD_EINVAL, "Q must be 4-byte aligned");
  }
  for (size_t b = 0; b < B && !dev_scales; ++b) {
    const float s = a->scales[b];
    if (!std::isfinite(s) || !(s > 0.0f)) return fail(PSGD_EINVAL, "scales must be finite and > 0");
  }
  if (h.cfg.unc_len > 0) {
    for (size_t i = 0; i < B * W; ++i)
      if (!a->unc_in[i] || (reinterpret_cast<uintptr_t>(a->unc_in[i]) & 3u))
        return fail(PSGD_EINVAL, "unc_in pointers must be non-NULL and 4-byte aligned");
    for (size_t b = 0; b < B; ++b)
      if (!a->unc_out[b] || (reinterpret_cast<uintptr_t>(a->unc_out[b]) & 3u))
        return fail(PSGD_EINVAL, "unc_out pointers must be non-NULL and 4-byte aligned");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;

  // Pointer table: upload only when it differs from the previous step's.
  std::vector<char> tab(h.table_bytes, 0);
  char* o = tab.data();
  std::memcpy(o, a->grads, 8 * B * J * W); o += 8 * B * J * W;
  std::memcpy(o, a->errs, 8 * B * J * W); o += 8 * B * J * W;
  std::memcpy(o, a->q_state, 8 * B * J); o += 8 * B * J;
  std::memcpy(o, a->ghat, 8 * B * J); o += 8 * B * J;
  if (h.cfg.unc_len > 0) std::memcpy(o, a->unc_in, 8 * B * W);
  o += 8 * B * W;
  if (h.cfg.unc_len > 0) std::memcpy(o, a->unc_out, 8 * B);
  o += 8 * B;
  for (size_t b = 0; b < B; ++b) {  // unused (left 0) when the scales live on the device
    const float inv = dev_scales ? 0.0f : (float)(1.0 / (double)a->scales[b]);
    std::memcpy(o + 4 * b, &inv, 4);
  }
  int slot = -1;
  for (int k = 0; k < Handle::kTableSlots && slot < 0; ++k)
    if (h.slot_used[k] && h.slot_key[k] == tab) slot = k;
  if (slot < 0) {  // a new table: the least recently used slot takes it
    slot = 0;
    for (int k = 1; k < Handle::kTableSlots; ++k)
      if (h.slot_used[k] < h.slot_used[slot]) slot = k;
    char* stage = h.h_stage + (size_t)slot * h.table_stride;
    // The slot's staging buffer may still feed its previous upload (stream order keeps the
    // device copy from overwriting a table that an earlier step still reads).
    if (h.slot_used[slot] && (e = cudaEventSynchronize(h.slot_ev[slot])) != cudaSuccess)
      return cuda_fail(e, "table event");
    std::memcpy(stage, tab.data(), h.table_bytes);
    if (h.maps_bytes && !tc_encode_ge_maps(h, a->grads, a->errs, a->ghat, stage + h.table_bytes))
      return fail(PSGD_ECUDA, "cuTensorMapEncodeTiled failed for a gradient or error buffer");
    if ((e = cudaMemcpyAsync(h.d_table + (size_t)slot * h.table_stride, stage, h.table_bytes + h.maps_bytes,
                             cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail(e, "table upload");
    if ((e = cudaEventRecord(h.slot_ev[slot], s)) != cudaSuccess) return cuda_fail(e, "table event");
    h.slot_key[slot].swap(tab);
    ++h.table_uploads;
  }
  h.slot_used[slot] = ++h.table_clock;

  p = Plan{};
  p.B = h.B; p.J = h.J; p.W = h.W; p.r = h.r; p.rp = h.rp;
  p.ob_r = h.r; p.ob_rp = h.rp; p.ob_c0 = 0; p.ob_src0 = 0;  // the orth driver sets blocks
  p.gdt = h.gdt; p.edt = h.edt;
  p.unc_len = h.cfg.unc_len;
  p.meta = h.d_meta;
  p.threshold = h.d_threshold;
  {
    const char* base = h.d_table + (size_t)slot * h.table_stride;
    p.tab.g = reinterpret_cast<const void* const*>(base);
    p.tab.e = reinterpret_cast<void* const*>(base + 8 * B * J * W);
    p.tab.q = reinterpret_cast<float* const*>(base + 16 * B * J * W);
    p.tab.ghat = reinterpret_cast<float* const*>(base + 16 * B * J * W + 8 * B * J);
    p.tab.unc_in = reinterpret_cast<const float* const*>(base + 16 * B * J * W + 16 * B * J);
    p.tab.unc_out = reinterpret_cast<float* const*>(base + 16 * B * J * W + 16 * B * J + 8 * B * W);
    p.tab.inv_scale = reinterpret_cast<const float*>(base + 16 * B * J * W + 16 * B * J + 8 * B * W + 8 * B);
    p.tab.ge_maps = h.maps_bytes ? base + h.table_bytes : nullptr;
  }
  if (dev_scales) p.tab.inv_scale = h.d_inv_dev;  // formed below, before the ingest
  p.counts = a->counts;
  p.skip = a->skip;
  p.mask = (h.cfg.flags & PSGD_FLAG_MASK) ? a->mask_bits : nullptr;
  p.mask_off = h.d_mask_off;
  p.err_word = h.d_err;
  p.debug_expire = (h.cfg.flags & PSGD_FLAG_DEBUG_EXPIRE_WAIT) ? 1 : 0;
  p.mean_div = (float)h.W;
  p.q_to_exchange = 0;
  return PSGD_OK;
}

// The phases of one step. ex: 0 the whole step (psgd_step); 1 up to the rank's P sum
// (psgd_step_p); 2 skip decision, orthonormalisation and the rank's Q sum (psgd_step_q);
// 3 the new Q state, G^ and E (psgd_step_e).
static psgd_status run_step(psgd_handle* ph, const psgd_step_args* a, Plan& p, void* stream, int ex,
                            const int64_t* block_counts, int w_total) {
  Handle& h = ph->h;
  const size_t B = h.B, J = h.J, W = h.W;
  const bool dev_scales = a->scales_device != nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  cudaEvent_t* ev = nullptr;
  if (ex == 0 && h.prof_used < h.prof_max) ev = &h.prof_events[(size_t)h.prof_used++ * (PSGD_NUM_PHASES + 1)];
  int phase = 0;
  auto mark = [&]() { if (ev) cudaEventRecord(ev[phase++], s); };

  if (ex == 0 || ex == 1) {
    if (ex == 1) {  // the skip decision waits for every rank's counts; P stays a plain sum
      p.skip = h.d_noskip;
      p.mean_div = 1.0f;
    }
    mark();
    if (dev_scales && (e = launch_inv_scale(h.B, a->scales_device, h.d_inv_dev, s)) != cudaSuccess)
      return cuda_fail(e, "inv_scale");
    if (dev_scales) ++h.launches;
    if ((e = cudaMemsetAsync(a->counts, 0, 8 * B * W, s)) != cudaSuccess) return cuda_fail(e, "counts");
    if ((e = cudaMemsetAsync(h.d_scal_all, 0, 4 * kScalWords * B * J, s)) != cudaSuccess) return cuda_fail(e, "scal");
    // The fused path ingests the gradients, writes the mask bitmap when asked, and forms
    // the P partial sums in one sweep; stopping after the ingest (debug) uses the separate
    // ingest kernel.
    const bool fused = h.tc && !(h.cfg.flags & PSGD_FLAG_STOP_AFTER_INGEST);
    if (fused) {
      if ((e = launch_prep_q(h, p, s)) != cudaSuccess) return cuda_fail(e, "prep_q");
      if ((e = launch_ingest_p(h, p, s)) != cudaSuccess) return cuda_fail(e, "ingest_p");
      if ((e = launch_unc_count(h, p, s)) != cudaSuccess) return cuda_fail(e, "unc_count");
    } else if ((e = launch_ingest(h, p, s)) != cudaSuccess) {
      return cuda_fail(e, "ingest");
    }
    mark();
    if (ex == 0 && (e = launch_skip_and_unc(h, p, s)) != cudaSuccess) return cuda_fail(e, "skip");
    mark();
    if (h.cfg.flags & PSGD_FLAG_STOP_AFTER_INGEST) {
      while (ev && phase <= PSGD_NUM_PHASES) mark();
      return PSGD_OK;
    }
    if (fused) {
      if (h.edt == DT_BF16 && (e = launch_rescale_tiny(h, p, s)) != cudaSuccess) return cuda_fail(e, "rescale");
      if ((e = launch_preduce(h, p, s)) != cudaSuccess) return cuda_fail(e, "preduce");
    } else if (h.tc) {
      if ((e = launch_prep_q(h, p, s)) != cudaSuccess) return cuda_fail(e, "prep_q");
      if ((e = launch_pgemm_tc(h, p, s)) != cudaSuccess) return cuda_fail(e, "pgemm_tc");
      if (h.edt == DT_BF16 && (e = launch_rescale_tiny(h, p, s)) != cudaSuccess) return cuda_fail(e, "rescale");
    } else {
      if ((e = launch_qmax(h, p, s)) != cudaSuccess) return cuda_fail(e, "qmax");
      if ((e = launch_pgemm_simt(h, p, s)) != cudaSuccess) return cuda_fail(e, "pgemm");
    }
    if (ex == 1) {
      if ((e = launch_pack_p(h, p, s)) != cudaSuccess) return cuda_fail(e, "exchange P");
      return PSGD_OK;
    }
  }

  if (ex == 0 || ex == 2) {
    if (ex == 2) {  // the summed counts decide; the summed P divides by every rank's workers,
                    // and the Q reduction writes this rank's sum to the exchange buffers
      if ((e = launch_skip_global(h, p, block_counts, w_total, s)) != cudaSuccess) return cuda_fail(e, "skip");
      if ((e = launch_unpack_p(h, p, w_total, s)) != cudaSuccess) return cuda_fail(e, "exchange P");
      p.mean_div = 1.0f;
      p.q_to_exchange = 1;
    }
    mark();
    if (h.r <= kRankBlock) {
      // Pass 0 as separate kernels; the later passes, which a warm-started P rarely needs,
      // in one cooperative launch that leaves at once when none is needed.
      if ((e = launch_orth_passes(h, p, 0, 0, s)) != cudaSuccess) return cuda_fail(e, "orth");
      e = launch_orth_coop(h, p, false, false, 0, tc_pchunk_kb(), 1, s);
      if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();  // nothing was enqueued: separate kernels for the later passes
        e = launch_orth_passes(h, p, 1, kMaxPasses - 1, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "orth");
    } else if ((e = launch_orth(h, p, s)) != cudaSuccess) {
      return cuda_fail(e, "orth");
    }
    mark();
    if (h.tc) {
      if ((e = launch_qgemm_tc(h, p, s, false)) != cudaSuccess) return cuda_fail(e, "qgemm_tc");
    } else if ((e = launch_qgemm_simt(h, p, s)) != cudaSuccess) {
      return cuda_fail(e, "qgemm");
    }
    mark();
    if ((e = launch_qreduce(h, p, s)) != cudaSuccess) return cuda_fail(e, "qreduce");
    if (ex == 2) return PSGD_OK;
  }

  if (ex == 3 && (e = launch_unpack_q(h, p, w_total, s)) != cudaSuccess) return cuda_fail(e, "exchange Q");
  mark();
  if (h.tc) {
    if ((e = launch_decomp_tc(h, p, s)) != cudaSuccess) return cuda_fail(e, "decomp_tc");
  } else if ((e = launch_decomp_simt(h, p, s)) != cudaSuccess) {
    return cuda_fail(e, "decomp");
  }
  mark();
  return PSGD_OK;
}

psgd_status psgd_step(psgd_handle* ph, const psgd_step_args* a, void* stream) {
  Plan p;
  const psgd_status st = prepare_step(ph, a, stream, p);
  if (st != PSGD_OK) return st;
  return run_step(ph, a, p, stream, 0, nullptr, 0);
}

static psgd_status check_exchange(psgd_handle* ph, int w_total) {
  if (!ph) return fail(PSGD_EINVAL, "handle is NULL");
  const Handle& h = ph->h;
  if (!(h.cfg.flags & PSGD_FLAG_EXCHANGE))
    return fail(PSGD_EUNSUPPORTED, "the exchange calls need a handle made with PSGD_FLAG_EXCHANGE");
  if (w_total < h.W) return fail(PSGD_EINVAL, "total_workers must be >= this handle's num_workers");
  return PSGD_OK;
}

psgd_status psgd_step_p(psgd_handle* ph, const psgd_step_args* a, void* stream) {
  psgd_status st = check_exchange(ph, ph ? ph->h.W : 0);
  if (st != PSGD_OK) return st;
  Plan p;
  if ((st = prepare_step(ph, a, stream, p)) != PSGD_OK) return st;
  return run_step(ph, a, p, stream, 1, nullptr, 0);
}

psgd_status psgd_step_q(psgd_handle* ph, const psgd_step_args* a, const int64_t* block_counts,
                        int32_t total_workers, void* stream) {
  psgd_status st = check_exchange(ph, total_workers);
  if (st != PSGD_OK) return st;
  if (!block_counts || (reinterpret_cast<uintptr_t>(block_counts) & 7u))
    return fail(PSGD_EINVAL, "block_counts must be an 8-byte aligned device pointer");
  Plan p;
  if ((st = prepare_step(ph, a, stream, p)) != PSGD_OK) return st;
  return run_step(ph, a, p, stream, 2, block_counts, total_workers);
}

psgd_status psgd_step_e(psgd_handle* ph, const psgd_step_args* a, int32_t total_workers, void* stream) {
  psgd_status st = check_exchange(ph, total_workers);
  if (st != PSGD_OK) return st;
  Plan p;
  if ((st = prepare_step(ph, a, stream, p)) != PSGD_OK) return st;
  return run_step(ph, a, p, stream, 3, nullptr, total_workers);
}

int64_t* psgd_exchange_counts(psgd_handle* ph) { return ph ? ph->h.d_xcnt : nullptr; }

float* psgd_exchange_p(psgd_handle* ph, int32_t b, int32_t j) {
  if (!ph) return nullptr;
  const Handle& h = ph->h;
  if (b < 0 || b >= h.B || j < 0 || j >= h.J) return nullptr;
  return h.meta[(size_t)b * h.J + j].xp;
}

float* psgd_exchange_q(psgd_handle* ph, int32_t b, int32_t j) {
  if (!ph) return nullptr;
  const Handle& h = ph->h;
  if (b < 0 || b >= h.B || j < 0 || j >= h.J) return nullptr;
  return h.meta[(size_t)b * h.J + j].xq;
}

static void destroy_profile(Handle& h) {
  for (cudaEvent_t e : h.prof_events)
    if (e) cudaEventDestroy(e);
  h.prof_events.clear();
  h.prof_max = h.prof_used = 0;
}

psgd_status psgd_profile_begin(psgd_handle* ph, int32_t max_steps) {
  if (!ph || max_steps < 1) return fail(PSGD_EINVAL, "bad handle or max_steps");
  Handle& h = ph->h;
  destroy_profile(h);
  h.prof_events.assign((size_t)max_steps * (PSGD_NUM_PHASES + 1), nullptr);
  for (auto& e : h.prof_events) {
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) { destroy_profile(h); return cuda_fail(err, "profile events"); }
  }
  h.prof_max = max_steps;
  h.prof_used = 0;
  return PSGD_OK;
}

psgd_status psgd_profile_end(psgd_handle* ph, double* phase_ms, int32_t* steps) {
  if (!ph || !phase_ms || !steps) return fail(PSGD_EINVAL, "NULL argument");
  Handle& h = ph->h;
  for (int k = 0; k < PSGD_NUM_PHASES; ++k) phase_ms[k] = 0.0;
  *steps = h.prof_used;
  for (int i = 0; i < h.prof_used; ++i) {
    cudaEvent_t* ev = &h.prof_events[(size_t)i * (PSGD_NUM_PHASES + 1)];
    cudaError_t e = cudaEventSynchronize(ev[PSGD_NUM_PHASES]);
    if (e != cudaSuccess) { destroy_profile(h); return cuda_fail(e, "profile sync"); }
    for (int k = 0; k < PSGD_NUM_PHASES; ++k) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, ev[k], ev[k + 1]);
      if (e != cudaSuccess) { destroy_profile(h); return cuda_fail(e, "profile elapsed"); }
      phase_ms[k] += ms;
    }
  }
  destroy_profile(h);
  return PSGD_OK;
}

int64_t psgd_launch_count(psgd_handle* ph) { return ph ? ph->h.launches : -1; }

psgd_status psgd_check(psgd_handle* ph, void* stream) {
  if (!ph) return fail(PSGD_EINVAL, "handle is NULL");
  Handle& h = ph->h;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "psgd_check");
  int word = 0;
  if ((e = cudaMemcpy(&word, h.d_err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "psgd_check");
  if (word != DEVERR_NONE) {
    cudaMemset(h.d_err, 0, 4);
    if (word == DEVERR_TIMEOUT) return fail(PSGD_ETIMEOUT, "a bounded device-side wait expired");
    return fail(PSGD_ECUDA, "device-side check failed (code " + std::to_string(word) + ")");
  }
  return PSGD_OK;
}

psgd_status psgd_finalize(psgd_handle* ph) {
  if (!ph) return PSGD_OK;
  Handle& h = ph->h;
  for (int k = 0; k < Handle::kTableSlots; ++k)
    if (h.slot_ev[k]) { cudaEventSynchronize(h.slot_ev[k]); cudaEventDestroy(h.slot_ev[k]); }
  if (h.h_stage) cudaFreeHost(h.h_stage);
  destroy_profile(h);
  tc_free(h);
  delete ph;
  return PSGD_OK;
}

const void* psgd_debug_m(psgd_handle* ph, int32_t b, int32_t j, int32_t w) {
  if (!ph) return nullptr;
  Handle& h = ph->h;
  if (b < 0 || b >= h.B || j < 0 || j >= h.J || w < 0 || w >= h.W) return nullptr;
  const MatMeta& mt = h.meta[(size_t)b * h.J + j];
  return static_cast<const char*>(mt.mscr) + (size_t)w * mt.m * mt.n * esize(h.edt);
}

const float* psgd_debug_phat(psgd_handle* ph, int32_t b, int32_t j) {
  if (!ph) return nullptr;
  Handle& h = ph->h;
  if (b < 0 || b >= h.B || j < 0 || j >= h.J) return nullptr;
  return h.meta[(size_t)b * h.J + j].Phat;
}

int32_t psgd_debug_orth(psgd_handle* ph, int32_t b, int32_t j, int32_t* out, void* stream) {
  static_assert(PSGD_MAX_ORTH_PASSES == kMaxPasses, "pass record size");
  if (!ph || !out) return -1;
  Handle& h = ph->h;
  if (b < 0 || b >= h.B || j < 0 || j >= h.J) return -1;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  if (cudaMemcpy(out, h.meta[(size_t)b * h.J + j].ostate, sizeof(int32_t) * 4 * kMaxPasses,
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  for (int p = 0; p < kMaxPasses; ++p)
    if (out[4 * p] != 0) return p + 1;
  return kMaxPasses;
}

const char* psgd_engine(psgd_handle* ph) {
  if (!ph) return "";
  return ph->h.tc ? "tcgen05" : "simt";
}

}  // extern "C"
