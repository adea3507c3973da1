// Dispatch of the delta-rule variant (mode VLA_DELTA) to the blocked scan kernel's
// instantiations, one translation unit per head width.
#include "vla_internal.cuh"

namespace vla {

cudaError_t launch_seq_delta_d16(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_seq_delta_d64(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_seq_delta_d128(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);

cudaError_t launch_delta(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built) {
  const bool cluster = ctas == 2;
  switch (d) {
    case 16: return launch_seq_delta_d16(r, bf16, cluster, a, s, built);
    case 64: return launch_seq_delta_d64(r, bf16, cluster, a, s, built);
    case 128: return launch_seq_delta_d128(r, bf16, cluster, a, s, built);
    default: *built = false; return cudaSuccess;
  }
}

}  // namespace vla
