// Instantiations of the chunked (Woodbury / LDL^T, tcgen05) scan: d = d_v = 64, bfloat16 or
// float32 I/O, r = 1 (64 steps per chunk) and r = 4 (16 steps per chunk); one CTA per pair
// (ctas = 1) or a cluster of two (ctas = 2: the A side and the S side).
#include <atomic>

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

// Two-CTA clusters of the chunked kernel that can be resident at once on the current device
// (0 when the shape is not built or the query fails), cached per device and shape.
int chunked_cluster_capacity(int r, bool bf16) {
  constexpr int kDevices = 64;
  // n + 1 once queried, 0 before; host threads with different handles may query at once and
  // store the same value
  static std::atomic<int> cache[kDevices][2][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices || (r != 1 && r != 4)) {
    cudaGetLastError();
    return 0;
  }
  std::atomic<int>& slot = cache[dev][r == 4][bf16 ? 1 : 0];
  const int known = slot.load(std::memory_order_relaxed);
  if (known > 0) return known - 1;
  int n = 0;
  cudaError_t e = r == 1 ? (bf16 ? cluster_capacity_t<1, __nv_bfloat16>(&n) : cluster_capacity_t<1, float>(&n))
                         : (bf16 ? cluster_capacity_t<4, __nv_bfloat16>(&n) : cluster_capacity_t<4, float>(&n));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  slot.store(n + 1, std::memory_order_relaxed);
  return n;
}

}  // namespace vla
