// Instantiations of the delta-rule scan kernel: d = d_v in {16, 64, 128}, r in {1, 4},
// float32 or bfloat16 I/O.
#include "vla_delta.cuh"

namespace vla {

cudaError_t launch_delta(int d, int r, bool bf16, const ScanArgs& a, cudaStream_t s, bool* built) {
  *built = true;
  if (d == 16 && r == 1) return bf16 ? launch_delta_t<16, 1, __nv_bfloat16>(a, s) : launch_delta_t<16, 1, float>(a, s);
  if (d == 16 && r == 4) return bf16 ? launch_delta_t<16, 4, __nv_bfloat16>(a, s) : launch_delta_t<16, 4, float>(a, s);
  if (d == 64 && r == 1) return bf16 ? launch_delta_t<64, 1, __nv_bfloat16>(a, s) : launch_delta_t<64, 1, float>(a, s);
  if (d == 64 && r == 4) return bf16 ? launch_delta_t<64, 4, __nv_bfloat16>(a, s) : launch_delta_t<64, 4, float>(a, s);
  if (d == 128 && r == 1) return bf16 ? launch_delta_t<128, 1, __nv_bfloat16>(a, s) : launch_delta_t<128, 1, float>(a, s);
  if (d == 128 && r == 4) return bf16 ? launch_delta_t<128, 4, __nv_bfloat16>(a, s) : launch_delta_t<128, 4, float>(a, s);
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
