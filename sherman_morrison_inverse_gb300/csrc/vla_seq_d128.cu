// Instantiations of the sequential scan kernel for d = d_v = 128.
#include "vla_seq.cuh"

namespace vla {

cudaError_t launch_seq_d128(int r, bool bf16, const ScanArgs& a, cudaStream_t s, bool* built) {
  *built = true;
  if (r == 1) return bf16 ? launch_seq_t<128, 1, __nv_bfloat16>(a, s) : launch_seq_t<128, 1, float>(a, s);
  if (r == 4) return bf16 ? launch_seq_t<128, 4, __nv_bfloat16>(a, s) : launch_seq_t<128, 4, float>(a, s);
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
