// Tensor-core (tcgen05 + TMA) engine of the three matrix products. Planning and launches.
#include "handle.h"

namespace psgd {

size_t tc_workspace_bytes(const psgd_config*) { return 0; }
bool tc_supported(const psgd_config*, std::string* why) {
  if (why) *why = "tensor engine not built";
  return false;
}
cudaError_t tc_plan(Handle&, char*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_prep_q(const Handle&, const Plan&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_pgemm_tc(const Handle&, const Plan&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_qgemm_tc(const Handle&, const Plan&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_decomp_tc(const Handle&, const Plan&, cudaStream_t) { return cudaErrorNotSupported; }
void tc_free(Handle&) {}

}  // namespace psgd
