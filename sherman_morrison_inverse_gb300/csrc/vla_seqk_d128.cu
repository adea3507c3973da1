// Instantiations of the blocked sequential scan kernel for d = d_v = 128
// (2 steps per reduction round for r = 1, one step of 4 directions for r = 4).
// cluster: the two-CTA variant (A group and S group on separate SMs).
#include "vla_seqk.cuh"

namespace vla {

cudaError_t launch_seq_block_d128(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s,
                                 bool* built) {
  *built = true;
  if (r == 1) {
    if (bf16) return cluster ? launch_seq_cluster_t<128, 1, 2, __nv_bfloat16>(a, s)
                             : launch_seq_block_t<128, 1, 2, __nv_bfloat16>(a, s);
    return cluster ? launch_seq_cluster_t<128, 1, 2, float>(a, s) : launch_seq_block_t<128, 1, 2, float>(a, s);
  }
  if (r == 4) {
    if (bf16) return cluster ? launch_seq_cluster_t<128, 4, 1, __nv_bfloat16>(a, s)
                             : launch_seq_block_t<128, 4, 1, __nv_bfloat16>(a, s);
    return cluster ? launch_seq_cluster_t<128, 4, 1, float>(a, s) : launch_seq_block_t<128, 4, 1, float>(a, s);
  }
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
