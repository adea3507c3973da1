// Copy-in of the host-buffer scan: one window of the sequence, gathered from page-locked
// host memory by the SMs.
//
// Each of q, k, v, u is [pairs, T, w] on the host (w = values per step); a window of tj
// steps starting at step `off` is the [pairs, tj, w] block of rows that the scan kernel
// reads.  The copy engines move such strided windows at full link rate for one tensor,
// but at about half of it when the rows of several tensors alternate in 128 KB pieces.
// SM loads through the mapped device address of the host buffer keep the full rate for
// any window, and 1024 threads on each of a few SMs keep enough 16-byte loads in flight
// to cover the link's latency.  So the window is gathered by a small kernel that runs on
// the SMs the scan leaves idle.
#include "vla_internal.cuh"

namespace vla {
namespace {

struct GatherArgs {
  const uint4* src[4];   // device view of host tensor i, [pairs, T, w16[i]] 16-byte vectors
  uint4* dst[4];         // staging window i, [pairs, tj, w16[i]]
  long long w16[4];      // 16-byte vectors per step of tensor i
  long long n[4];        // vectors in window i: pairs * tj * w16[i]
  long long T, off, tj;
};

// The four windows are enumerated as one flat index space (tensor 0's vectors first);
// thread g copies the vectors g, g + stride, g + 2 stride, ... of it.
__global__ void __launch_bounds__(1024) gather_window_kernel(GatherArgs g) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
#pragma unroll 1
  for (int t = 0; t < 4; ++t) {
    const long long n = g.n[t], row = g.tj * g.w16[t], pitch = g.T * g.w16[t], first = g.off * g.w16[t];
    const uint4* __restrict__ src = g.src[t];
    uint4* __restrict__ dst = g.dst[t];
    for (; i < n; i += stride) {
      const long long p = i / row;
      dst[i] = src[p * pitch + first + (i - p * row)];
    }
    i -= n;   // the same thread's next index, counted from the start of tensor t + 1
  }
}

}  // namespace

cudaError_t launch_gather_window(const void* const src[4], void* const dst[4], const long long w_bytes[4],
                                 long long pairs, long long T, long long off, long long tj, int ctas,
                                 cudaStream_t s) {
  GatherArgs g{};
  for (int t = 0; t < 4; ++t) {
    g.src[t] = static_cast<const uint4*>(src[t]);
    g.dst[t] = static_cast<uint4*>(dst[t]);
    g.w16[t] = w_bytes[t] / 16;
    g.n[t] = pairs * tj * g.w16[t];
  }
  g.T = T;
  g.off = off;
  g.tj = tj;
  gather_window_kernel<<<ctas, 1024, 0, s>>>(g);
  return cudaGetLastError();
}

}  // namespace vla
