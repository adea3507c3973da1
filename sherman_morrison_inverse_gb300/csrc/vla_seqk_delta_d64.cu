// Instantiations of the blocked scan kernel's delta-rule variant (gist.science summary
// §2.3: the S group writes S with the residual v - S k_hat along alpha_hat) for
// d = d_v = 64: one CTA per pair, 4 steps per round for r = 1,
// one step of 4 directions for r = 4.
#include "vla_seqk.cuh"

namespace vla {

cudaError_t launch_seq_delta_d64(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built) {
  *built = true;
  (void)cluster;   // one CTA per pair at this width
  if (r == 1) return bf16 ? launch_seq_block_t<64, 1, 4, __nv_bfloat16, false, true>(a, s)
                          : launch_seq_block_t<64, 1, 4, float, false, true>(a, s);
  if (r == 4) return bf16 ? launch_seq_block_t<64, 4, 1, __nv_bfloat16, false, true>(a, s)
                          : launch_seq_block_t<64, 4, 1, float, false, true>(a, s);
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
