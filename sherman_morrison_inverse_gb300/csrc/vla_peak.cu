// Measurement helper: the FP32 CUDA-core throughput of this GPU.  Every thread runs
// eight independent chains of packed fp32 fused multiply-adds (FFMA2), enough
// independent work per SM sub-partition to keep the FP32 pipes busy, so the time of
// one launch gives the sustained FP32 peak that the scan's roofline is quoted
// against.  The chains contract towards a fixed point and stay normal numbers.
#include "vla_internal.cuh"

namespace vla {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 8;

__global__ void __launch_bounds__(kProbeThreads) ffma_probe_kernel(long long iters, DevStatus* status) {
  float2 acc[kProbeChains];
#pragma unroll
  for (int j = 0; j < kProbeChains; ++j) acc[j] = make_float2(1e-3f * threadIdx.x + j, 0.5f * j);
  const float2 m = make_float2(0.9999f, 0.9999f), a = make_float2(1e-4f, 2e-4f);
#pragma unroll 1
  for (long long i = 0; i < iters; i += 8) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int j = 0; j < kProbeChains; ++j) acc[j] = __ffma2_rn(acc[j], m, a);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kProbeChains; ++j) s += acc[j].x + acc[j].y;
  if (s == 1.25e30f) atomicOr(&status->reserved, 1u);   // never true: keeps the chains live
}

}  // namespace

cudaError_t launch_ffma_probe(long long iters, int sm_count, DevStatus* status, cudaStream_t s, double* flops) {
  const int grid = (sm_count > 0 ? sm_count : 1) * 4;
  const long long it = (iters + 7) / 8 * 8;
  *flops = (double)grid * kProbeThreads * (double)it * kProbeChains * 4.0;   // FFMA2 = 2 FMA = 4 flops
  ffma_probe_kernel<<<grid, kProbeThreads, 0, s>>>(it, status);
  return cudaGetLastError();
}

}  // namespace vla
