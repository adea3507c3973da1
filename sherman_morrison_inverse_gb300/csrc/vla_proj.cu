// Direction projection u_{t,i} = W_u[i] k_t / max(|W_u[i] k_t|_2, 1e-12) for sm_103a: the
// README "VLA v3" item 2 "u_t = normalize(W_u k_t^raw)", computed before the scan (whose u
// input it produces, [n, r, d]).
//
// Each thread takes TPT consecutive tokens (4 at d = 16, 2 at d = 64, 1 at d = 128),
// groups taken grid-stride, the ranks one after another (W_u[i] in shared memory, d x d
// float32).  Each thread reads its keys as 16-byte vectors (all independent loads, one
// memory latency per group), forms x_j = W[j] . k for its tokens with W's rows broadcast
// from shared memory, keeps x in its own padded shared-memory rows (stride d + 1,
// conflict-free), and writes x_j / max(|x|, 1e-12) as 16-byte vectors: no barrier
// inside the token loop.  Arithmetic in float32 (float32 or bfloat16 in
// and out).
#include "vla_internal.cuh"

namespace vla {
namespace prj {

constexpr int NTH = 128;   // threads per CTA

// Tokens per thread: each W element read from shared memory feeds TPT tokens' FMAs
// (a broadcast 16-byte read still moves 16 bytes to every lane, so shared-memory
// bandwidth, not the FMA pipe, binds at one token a thread).  Bounded by registers.
template <int D>
constexpr int tpt() { return D <= 16 ? 4 : (D <= 64 ? 2 : 1); }

template <int D>
struct Smem {
  static constexpr int W_OFF = 0;                                  // [D][D] one rank of W_u
  static constexpr int X_OFF = D * D;                              // [NTH * TPT][D + 1] x of each token
  static constexpr size_t bytes = sizeof(float) * (size_t)(X_OFF + NTH * tpt<D>() * (D + 1));
};

// 16-byte vector <-> float32 values of the I/O type
template <typename TIO> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const uint4& w, float* x) {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y); x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
  __device__ static uint4 pack(const float* x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const uint4& w, float* x) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[m]));
      x[2 * m] = f.x;
      x[2 * m + 1] = f.y;
    }
  }
  __device__ static uint4 pack(const float* x) {
    uint32_t ww[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * m], x[2 * m + 1]);   // round to nearest even
      ww[m] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(ww[0], ww[1], ww[2], ww[3]);
  }
};

template <int D, typename TIO>
__global__ void __launch_bounds__(NTH) project_u_kernel(const TIO* __restrict__ k, const float* __restrict__ W,
                                                        TIO* __restrict__ u, long long n, int r) {
  using L = Smem<D>;
  using V = Vec<TIO>;
  constexpr int TP = tpt<D>();
  constexpr int NV = D / V::N;   // 16-byte vectors per row
  extern __shared__ __align__(16) float sm[];
  float* sW = sm + L::W_OFF;
  float* sX = sm + L::X_OFF + threadIdx.x * TP * (D + 1);   // this thread's TP rows of x
  const long long stride = (long long)gridDim.x * NTH * TP;
  for (int i = 0; i < r; ++i) {
    __syncthreads();   // every thread is done with the previous rank's W
    for (int e = threadIdx.x; e < D * D / 4; e += NTH)
      reinterpret_cast<float4*>(sW)[e] = reinterpret_cast<const float4*>(W + (size_t)i * D * D)[e];
    __syncthreads();
    // tokens t0 .. t0 + TP - 1 (those below n)
    for (long long t0 = (blockIdx.x * (long long)NTH + threadIdx.x) * TP; t0 < n; t0 += stride) {
      float kr[TP][D];
#pragma unroll
      for (int p = 0; p < TP; ++p) {
        const bool live = t0 + p < n;
        const uint4* kv = reinterpret_cast<const uint4*>(k + (t0 + p) * D);
#pragma unroll
        for (int v = 0; v < NV; ++v) V::load(live ? __ldg(kv + v) : make_uint4(0u, 0u, 0u, 0u), kr[p] + V::N * v);
      }
      float nrm[TP];
#pragma unroll
      for (int p = 0; p < TP; ++p) nrm[p] = 0.f;
#pragma unroll 2
      for (int j = 0; j < D; ++j) {
        const float4* wr = reinterpret_cast<const float4*>(sW + j * D);
        float a[TP][2];
#pragma unroll
        for (int p = 0; p < TP; ++p) a[p][0] = a[p][1] = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < D / 4; ++m4) {
          const float4 w4 = wr[m4];
#pragma unroll
          for (int p = 0; p < TP; ++p) {
            a[p][0] = fmaf(w4.x, kr[p][4 * m4 + 0], a[p][0]);
            a[p][1] = fmaf(w4.y, kr[p][4 * m4 + 1], a[p][1]);
            a[p][0] = fmaf(w4.z, kr[p][4 * m4 + 2], a[p][0]);
            a[p][1] = fmaf(w4.w, kr[p][4 * m4 + 3], a[p][1]);
          }
        }
#pragma unroll
        for (int p = 0; p < TP; ++p) {
          const float x = a[p][0] + a[p][1];
          sX[p * (D + 1) + j] = x;
          nrm[p] = fmaf(x, x, nrm[p]);
        }
      }
#pragma unroll
      for (int p = 0; p < TP; ++p) {
        if (t0 + p >= n) break;
        const float inv = 1.f / fmaxf(sqrtf(nrm[p]), 1e-12f);
        uint4* uv = reinterpret_cast<uint4*>(u + ((t0 + p) * r + i) * D);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          float y[V::N];
#pragma unroll
          for (int m = 0; m < V::N; ++m) y[m] = sX[p * (D + 1) + V::N * v + m] * inv;
          uv[v] = V::pack(y);
        }
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
  const long long nblk = (n + (long long)NTH * tpt<D>() - 1) / ((long long)NTH * tpt<D>());
  const int grid = (int)min(nblk, (long long)(sm_count > 0 ? sm_count : 1) * 4);
  kern<<<grid, NTH, Smem<D>::bytes, s>>>(static_cast<const TIO*>(k), W, static_cast<TIO*>(u), n, r);
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
