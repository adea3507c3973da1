// Instantiations of the blocked sequential scan kernel for d = d_v = 128.
// r = 1: 2 steps per reduction round on one CTA (512 threads, capped at 128 registers:
// 4-step rounds spill there and run 13 % slower), 4 steps per round on the two-CTA
// cluster (256 threads a CTA, 202 registers, no spills; 11 % faster than 2-step rounds
// on the long-context workload, while 8-step rounds are slower).  r = 4: one step of 4
// directions per round on both.
// cluster: the two-CTA variant (A group and S group on separate SMs).
#include "vla_seqk.cuh"

namespace vla {

cudaError_t launch_seq_block_d128(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s,
                                 bool* built) {
  *built = true;
  if (r == 1) {
    if (bf16) return cluster ? launch_seq_cluster_t<128, 1, 4, __nv_bfloat16>(a, s)
                             : launch_seq_block_t<128, 1, 2, __nv_bfloat16>(a, s);
    return cluster ? launch_seq_cluster_t<128, 1, 4, float>(a, s) : launch_seq_block_t<128, 1, 2, float>(a, s);
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
