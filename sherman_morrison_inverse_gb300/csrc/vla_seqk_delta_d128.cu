// Instantiations of the blocked scan kernel's delta-rule variant (gist.science summary
// §2.3: the S group writes S with the residual v - S k_hat along alpha_hat) for
// d = d_v = 128: the two-CTA cluster (4 steps per round for r = 1)
// while two CTAs per pair fit on the SMs, else one CTA (2 steps per round, as the
// additive kernel at this width).
#include "vla_seqk.cuh"

namespace vla {

cudaError_t launch_seq_delta_d128(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built) {
  *built = true;
  if (r == 1) {
    if (bf16) return cluster ? launch_seq_cluster_t<128, 1, 4, __nv_bfloat16, true>(a, s)
                             : launch_seq_block_t<128, 1, 2, __nv_bfloat16, false, true>(a, s);
    return cluster ? launch_seq_cluster_t<128, 1, 4, float, true>(a, s)
                   : launch_seq_block_t<128, 1, 2, float, false, true>(a, s);
  }
  if (r == 4) {
    if (bf16) return cluster ? launch_seq_cluster_t<128, 4, 1, __nv_bfloat16, true>(a, s)
                             : launch_seq_block_t<128, 4, 1, __nv_bfloat16, false, true>(a, s);
    return cluster ? launch_seq_cluster_t<128, 4, 1, float, true>(a, s)
                   : launch_seq_block_t<128, 4, 1, float, false, true>(a, s);
  }
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
