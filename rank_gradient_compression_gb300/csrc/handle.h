// Host-side handle of libpsgd.so (shared by the .cu files; not part of the ABI).
#pragma once

#include <string>
#include <vector>

#include "psgd_internal.cuh"

namespace psgd {

// One contiguous range of work for the ingest kernel: matrix (t, w) or gains/biases
// (b, w). CTAs [cta_start, cta_start + ceil(numel / kIngestChunk)) process it.
struct IngestSeg {
  int64_t numel;
  int64_t cta_start;
  int32_t kind;  // 0 = matrix, 1 = gains/biases
  int32_t t;     // matrix index b*J+j (kind 0)
  int32_t b, w;
};

constexpr int kIngestThreads = 256;
constexpr int kIngestVec = 8;     // elements per thread per iteration
constexpr int kIngestIters = 4;   // iterations per CTA
constexpr int64_t kIngestChunk = (int64_t)kIngestThreads * kIngestVec * kIngestIters;

struct Handle {
  psgd_config cfg{};
  std::vector<psgd_shape> shapes;
  int B = 0, J = 0, W = 0, r = 0, rp = 0;
  int gdt = 0, edt = 0;
  bool tc = false;  // tcgen05 engine for the GEMMs
  char* ws = nullptr;
  size_t ws_bytes = 0;

  std::vector<MatMeta> meta;
  MatMeta* d_meta = nullptr;
  int64_t* d_threshold = nullptr;
  int64_t* d_mask_off = nullptr;
  std::vector<IngestSeg> segs;
  IngestSeg* d_segs = nullptr;
  int64_t ingest_ctas = 0;
  int64_t unc_cta_start = 0;  // first CTA of the gains/biases segments

  // Per-step pointer tables (and the TMA maps of G and E), cached in kTableSlots device
  // slots keyed by their host bytes, so that buffer sets used in turn are encoded and
  // uploaded once. Slot k: device bytes at d_table + k * table_stride, pinned staging at
  // h_stage + k * table_stride, upload event, key, last use.
  static constexpr int kTableSlots = 4;
  char* d_table = nullptr;
  size_t table_bytes = 0, table_stride = 0;
  char* h_stage = nullptr;  // pinned, kTableSlots * table_stride
  std::vector<char> slot_key[kTableSlots];
  cudaEvent_t slot_ev[kTableSlots] = {};
  int64_t slot_used[kTableSlots] = {};  // step counter at last use; 0: empty
  int64_t table_clock = 0;
  int64_t table_uploads = 0;            // uploads so far (a test reads it)

  int* d_err = nullptr;
  float* d_scal_all = nullptr;  // [B*J*kScalWords] scaling words, zeroed every step
  float* d_inv_dev = nullptr;   // [B] 1/s_b formed on the device (psgd_step_args.scales_device)
  GridBarrier* d_gbar = nullptr;  // the cooperative orthonormalisation kernel's barrier
  uint8_t* d_noskip = nullptr;    // [B] zeros: the skip flags the exchange's first call runs with
  int64_t* d_xcnt = nullptr;      // [B] exchange: this rank's nonfinite counts per block
  size_t maps_bytes = 0;        // TMA maps of the callers' G and E (tensor engine), after the table
  int max_mtiles = 0, max_S = 0, max_C = 0, max_ntiles64 = 0, max_mtiles64 = 0;
  int max_kchunks = 0, max_ntiles128 = 0;
  void* tc_plan = nullptr;  // tensor-engine work lists (tc.cu)
  mutable int64_t launches = 0;  // kernels enqueued so far
  std::vector<cudaEvent_t> prof_events;  // [max_steps][PSGD_NUM_PHASES + 1]
  int prof_max = 0, prof_used = 0;
};

// Tensor-engine planning and launches (tc.cu).
size_t tc_workspace_bytes(const psgd_config* cfg);
bool tc_supported(const psgd_config* cfg, std::string* why);
cudaError_t tc_plan(Handle& h, char* ws_tc, cudaStream_t s);
cudaError_t launch_prep_q(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_qmax(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_pgemm_tc(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_ingest_p(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_preduce(const Handle& h, const Plan& p, cudaStream_t s);
size_t tc_ge_maps_bytes(const psgd_config* cfg);
bool tc_encode_ge_maps(const Handle& h, const void* const* grads, void* const* errs, float* const* ghat,
                       void* out);
cudaError_t launch_rescale_tiny(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_qgemm_tc(const Handle& h, const Plan& p, cudaStream_t s, bool psplit_done);
int tc_kpad(const Handle& h);
int tc_pchunk_kb();
cudaError_t launch_decomp_tc(const Handle& h, const Plan& p, cudaStream_t s);
void tc_free(Handle& h);

// Per-thread error message of the C ABI (api.cu), for entry points in other files.
psgd_status report_error(psgd_status s, const std::string& msg);
psgd_status report_cuda_error(cudaError_t e, const char* where);

// The orthonormalisation passes for one matrix whose plan, pass state and scratch were
// not laid out by psgd_init (orth.cu). C: Gram row chunks; mtiles64: 64-row tiles.
cudaError_t launch_orth_one(const Plan& p, int C, int mtiles64, cudaStream_t s);

// The orthonormalisation of every matrix (r <= kRankBlock) in one cooperative launch
// (orth_coop.cu): optionally forms P from the tensor engine's partial sums first and
// writes the split P^ operands last. Returns cudaErrorCooperativeLaunchTooLarge, with
// nothing enqueued, when the device cannot hold the grid; the caller then uses the
// separate kernels.
cudaError_t launch_orth_coop(const Handle& h, const Plan& p, bool fused_preduce, bool do_psplit, int kp,
                             int pchunk_kb, int start_pass, cudaStream_t s);
// The orthonormalisation of the step: separate kernels for pass 0, then (r <= kRankBlock)
// the cooperative kernel for the passes after it, or separate kernels for all passes.
cudaError_t launch_orth_passes(const Handle& h, const Plan& p, int first_pass, int last_pass, cudaStream_t s);
int orth_coop_grid();

// Data-parallel exchange points (exchange.cu).
cudaError_t launch_pack_p(const Handle& h, const Plan& p, cudaStream_t s);
cudaError_t launch_skip_global(const Handle& h, const Plan& p, const int64_t* block_counts, int w_total,
                               cudaStream_t s);
cudaError_t launch_unpack_p(const Handle& h, const Plan& p, int w_total, cudaStream_t s);
cudaError_t launch_unpack_q(const Handle& h, const Plan& p, int w_total, cudaStream_t s);
cudaError_t launch_inv_scale(int B, const float* scale, float* inv, cudaStream_t s);

}  // namespace psgd
