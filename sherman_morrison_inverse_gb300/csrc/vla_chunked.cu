// Instantiations of the chunked (Woodbury / LDL^T, tcgen05) scan: d = d_v = 64, bfloat16 or
// float32 I/O, r = 1 (64 steps per chunk) and r = 4 (16 steps per chunk); one CTA per pair
// (ctas = 1) or a cluster of two (ctas = 2: the A side and the S side).
#include "vla_chunk.cuh"

namespace vla {

cudaError_t launch_chunked(int d, int r, bool bf16, int chunk, int ctas, const ScanArgs& a, cudaStream_t s,
                           bool* built) {
  *built = false;
  if (d != 64) return cudaSuccess;
  if (r == 1 && (chunk == 0 || chunk == 64)) {
    *built = true;
    return bf16 ? launch_chunk_t<1, __nv_bfloat16>(a, ctas, s) : launch_chunk_t<1, float>(a, ctas, s);
  }
  if (r == 4 && (chunk == 0 || chunk == 16)) {
    *built = true;
    return bf16 ? launch_chunk_t<4, __nv_bfloat16>(a, ctas, s) : launch_chunk_t<4, float>(a, ctas, s);
  }
  return cudaSuccess;
}

}  // namespace vla
