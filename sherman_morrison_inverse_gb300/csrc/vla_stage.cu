// Copy-in of the host-buffer scan: one window of the sequence, gathered from page-locked
// host memory by the SMs.
//
// Each of q, k, v, u is [pairs, T, w] on the host (w = values per step); a window of tj
// steps starting at step `off` is the [pairs, tj, w] block of rows that the scan kernel
// reads.  The copy engines move such strided windows at full link rate for one tensor,
// but at about half of it when the rows of several tensors alternate in 128 KB pieces.
// SM loads through the mapped device address of the host buffer keep the full rate for
// any window, provided enough 16-byte loads are in flight to cover the link's latency:
// 1024 threads on each of a few SMs, each with up to 8 loads issued before its stores, the
// grid reading consecutive addresses.  So the window is gathered by a small kernel that runs
// on the SMs the scan leaves idle.
#include "vla_internal.cuh"

namespace vla {
namespace {

struct GatherArgs {
  const uint4* src[4];   // device view of host tensor i, [pairs, T, w16[i]] 16-byte vectors
  uint4* dst[4];         // staging window i, [pairs, tj, w16[i]]
  long long w16[4];      // 16-byte vectors per step of tensor i
  long long pairs, T, off, tj;
};

constexpr int kGatherThreads = 1024;
constexpr int kGatherUnroll = 8;   // independent 16-byte loads in flight per thread

// Each tensor's window is one flat index space of pairs * tj * w16 vectors (pair-major, as the
// staging buffer); thread g copies the vectors g, g + G, g + 2 G, ... (G threads in the grid), so
// the grid as a whole streams consecutive host addresses.  Up to kGatherUnroll loads are issued
// before their stores.  Indices fit in 32 bits (the host checks), so the row of an index costs
// one 32-bit division.
__global__ void __launch_bounds__(kGatherThreads) gather_window_kernel(GatherArgs g) {
  const uint32_t G = gridDim.x * (uint32_t)kGatherThreads;
  const uint32_t gtid = blockIdx.x * (uint32_t)kGatherThreads + threadIdx.x;
#pragma unroll 1
  for (int t = 0; t < 4; ++t) {
    // tensor t's fields by a static selection (a run-time index into the parameter block
    // would copy it to local memory)
    const long long w16 = t == 0 ? g.w16[0] : t == 1 ? g.w16[1] : t == 2 ? g.w16[2] : g.w16[3];
    const uint4* __restrict__ src = t == 0 ? g.src[0] : t == 1 ? g.src[1] : t == 2 ? g.src[2] : g.src[3];
    uint4* __restrict__ dst = t == 0 ? g.dst[0] : t == 1 ? g.dst[1] : t == 2 ? g.dst[2] : g.dst[3];
    const uint32_t len = (uint32_t)(g.tj * w16);              // vectors of one pair's window
    const uint32_t n = (uint32_t)(g.pairs * (long long)len);  // vectors of the window
    const long long pitch = g.T * w16, first = g.off * w16;
#pragma unroll 1
    for (uint32_t i0 = gtid; i0 < n; i0 += kGatherUnroll * G) {
      uint4 v[kGatherUnroll];
#pragma unroll
      for (int k = 0; k < kGatherUnroll; ++k) {
        const uint32_t i = i0 + k * G;
        if (i < n) {
          const uint32_t p = i / len;
          v[k] = src[(long long)p * pitch + first + (i - p * len)];
        }
      }
#pragma unroll
      for (int k = 0; k < kGatherUnroll; ++k) {
        const uint32_t i = i0 + k * G;
        if (i < n) dst[i] = v[k];
      }
    }
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
  }
  g.pairs = pairs;
  g.T = T;
  g.off = off;
  g.tj = tj;
  // 32-bit indices: every window of every tensor below 2^31 vectors, with room for the
  // strided indices of the last batch (kGatherUnroll * threads beyond the end)
  const long long limit = (1ll << 31) - (long long)kGatherUnroll * kGatherThreads * ctas;
  for (int t = 0; t < 4; ++t)
    if (pairs * tj * g.w16[t] >= limit) return cudaErrorInvalidValue;
  gather_window_kernel<<<ctas, kGatherThreads, 0, s>>>(g);
  return cudaGetLastError();
}

}  // namespace vla
