// Copy-in of the host-buffer scan: one window of the sequence, gathered from page-locked
// host memory by the SMs.
//
// Each of q, k, v, u is [pairs, T, w] on the host (w = values per step); a window of tj
// steps starting at step `off` is the [pairs, tj, w] block of rows that the scan kernel
// reads.  The copy engines move such strided windows at full link rate for one tensor,
// but at about half of it when the rows of several tensors alternate in 128 KB pieces.
// SM loads through the mapped device address of the host buffer keep the full rate for
// any window, provided enough 16-byte loads are in flight to cover the link's latency:
// 1024 threads on each of a few SMs, each with up to 8 loads issued before its stores.
// So the window is gathered by a small kernel that runs on the SMs the scan leaves idle.
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

// The window of tensor t for pair p is one contiguous run of tj * w16[t] vectors on both
// sides (from step `off` of the pair's [T, w] block into the pair's [tj, w] block).  The
// 4 * pairs runs are taken whole, one per CTA at a time (run = blockIdx.x, + gridDim.x, ...);
// each thread issues up to kGatherUnroll loads before it stores them, so a CTA keeps up to
// 128 KB of host reads in flight.
__global__ void __launch_bounds__(kGatherThreads) gather_window_kernel(GatherArgs g) {
  const long long runs = 4 * g.pairs;
#pragma unroll 1
  for (long long run = blockIdx.x; run < runs; run += gridDim.x) {
    const int t = (int)(run / g.pairs);
    const long long p = run - t * g.pairs;
    // tensor t's fields by a static selection (a run-time index into the parameter block
    // would copy it to local memory)
    const long long w16 = t == 0 ? g.w16[0] : t == 1 ? g.w16[1] : t == 2 ? g.w16[2] : g.w16[3];
    const uint4* s0 = t == 0 ? g.src[0] : t == 1 ? g.src[1] : t == 2 ? g.src[2] : g.src[3];
    uint4* d0 = t == 0 ? g.dst[0] : t == 1 ? g.dst[1] : t == 2 ? g.dst[2] : g.dst[3];
    const long long len = g.tj * w16;
    const uint4* __restrict__ src = s0 + (p * g.T + g.off) * w16;
    uint4* __restrict__ dst = d0 + p * len;
    constexpr long long kBatch = (long long)kGatherUnroll * kGatherThreads;
    long long j0 = threadIdx.x;
#pragma unroll 1
    for (; j0 + (kGatherUnroll - 1) * kGatherThreads < len; j0 += kBatch) {   // whole batches
      uint4 v[kGatherUnroll];
#pragma unroll
      for (int k = 0; k < kGatherUnroll; ++k) v[k] = src[j0 + k * kGatherThreads];
#pragma unroll
      for (int k = 0; k < kGatherUnroll; ++k) dst[j0 + k * kGatherThreads] = v[k];
    }
#pragma unroll 1
    for (; j0 < len; j0 += kGatherThreads) dst[j0] = src[j0];   // the rest of the run
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
  gather_window_kernel<<<ctas, kGatherThreads, 0, s>>>(g);
  return cudaGetLastError();
}

}  // namespace vla
