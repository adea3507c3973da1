// Direction projection u_{t,i} = W_u[i] k_t / max(|W_u[i] k_t|_2, 1e-12) for sm_103a: the
// README "VLA v3" item 2 "u_t = normalize(W_u k_t^raw)", computed before the scan (whose u
// input it produces, [n, r, d]).
//
// One thread per token, 128 tokens per tile, tiles taken grid-stride, the ranks one
// after another (W_u[i] in shared memory, d x d float32).  The tile's keys arrive with
// coalesced loads into a padded float32 tile (row stride d + 1: the per-token row
// reads are conflict-free), each thread keeps its key in registers and forms
// x_j = W[j] . k with W's row broadcast from shared memory; x goes to the same padded
// tile, and a second pass writes x_j / max(|x|, 1e-12) with coalesced stores.
// Arithmetic in float32 (float32 or bfloat16 in and out).
#include "vla_internal.cuh"

namespace vla {
namespace prj {

constexpr int TT = 128;   // tokens per tile = threads per CTA

template <int D>
struct Smem {
  static constexpr int W_OFF = 0;                     // [D][D] one rank of W_u
  static constexpr int T_OFF = D * D;                 // [TT][D + 1] keys, then x
  static constexpr int N_OFF = T_OFF + TT * (D + 1);  // [TT] 1 / |x|
  static constexpr size_t bytes = sizeof(float) * (size_t)(N_OFF + TT);
};

template <int D, typename TIO>
__global__ void __launch_bounds__(TT, 1) project_u_kernel(const TIO* __restrict__ k, const float* __restrict__ W,
                                                          TIO* __restrict__ u, long long n, int r) {
  using L = Smem<D>;
  extern __shared__ __align__(16) float sm[];
  float* sW = sm + L::W_OFF;
  float* sT = sm + L::T_OFF;
  float* sN = sm + L::N_OFF;
  const int tid = threadIdx.x;
  const long long ntiles = (n + TT - 1) / TT;
  for (int i = 0; i < r; ++i) {
    __syncthreads();   // the previous rank's tiles are done with sW
    for (int e = tid; e < D * D; e += TT) sW[e] = W[(size_t)i * D * D + e];
    for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const long long t0 = tile * TT;
      const int nt = (int)min((long long)TT, n - t0);
      __syncthreads();   // sW written; the previous tile's stores have read sT and sN
      for (int e = tid; e < TT * D; e += TT) {
        const int tok = e / D, col = e - tok * D;
        sT[tok * (D + 1) + col] = (tok < nt) ? to_f32(k[(t0 + tok) * D + col]) : 0.f;
      }
      __syncthreads();
      float kr[D];
#pragma unroll
      for (int m = 0; m < D; ++m) kr[m] = sT[tid * (D + 1) + m];
      __syncthreads();   // the tile is rewritten with x below
      float nrm = 0.f;
#pragma unroll 4
      for (int j = 0; j < D; ++j) {
        const float4* wr = reinterpret_cast<const float4*>(sW + j * D);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < D / 4; ++m4) {
          const float4 w4 = wr[m4];
          a0 = fmaf(w4.x, kr[4 * m4 + 0], a0);
          a1 = fmaf(w4.y, kr[4 * m4 + 1], a1);
          a2 = fmaf(w4.z, kr[4 * m4 + 2], a2);
          a3 = fmaf(w4.w, kr[4 * m4 + 3], a3);
        }
        const float x = (a0 + a1) + (a2 + a3);
        sT[tid * (D + 1) + j] = x;
        nrm = fmaf(x, x, nrm);
      }
      sN[tid] = 1.f / fmaxf(sqrtf(nrm), 1e-12f);
      __syncthreads();
      for (int e = tid; e < nt * D; e += TT) {
        const int tok = e / D, col = e - tok * D;
        u[((t0 + tok) * r + i) * D + col] = from_f32<TIO>(sT[tok * (D + 1) + col] * sN[tok]);
      }
    }
  }
}

template <int D, typename TIO>
cudaError_t launch_project_t(const void* k, const float* W, void* u, long long n, int r, int sm_count,
                             cudaStream_t s) {
  auto kern = project_u_kernel<D, TIO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem<D>::bytes);
  if (e != cudaSuccess) return e;
  const long long ntiles = (n + TT - 1) / TT;
  const int grid = (int)min(ntiles, (long long)(sm_count > 0 ? sm_count : 1) * 4);
  kern<<<grid, TT, Smem<D>::bytes, s>>>(static_cast<const TIO*>(k), W, static_cast<TIO*>(u), n, r);
  return cudaGetLastError();
}

}  // namespace prj

cudaError_t launch_project_u(int d, bool bf16, const void* k, const float* W, void* u, long long n, int r,
                             int sm_count, cudaStream_t s, bool* built) {
  *built = true;
  if (d == 16) return bf16 ? prj::launch_project_t<16, __nv_bfloat16>(k, W, u, n, r, sm_count, s)
                           : prj::launch_project_t<16, float>(k, W, u, n, r, sm_count, s);
  if (d == 64) return bf16 ? prj::launch_project_t<64, __nv_bfloat16>(k, W, u, n, r, sm_count, s)
                           : prj::launch_project_t<64, float>(k, W, u, n, r, sm_count, s);
  if (d == 128) return bf16 ? prj::launch_project_t<128, __nv_bfloat16>(k, W, u, n, r, sm_count, s)
                            : prj::launch_project_t<128, float>(k, W, u, n, r, sm_count, s);
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
