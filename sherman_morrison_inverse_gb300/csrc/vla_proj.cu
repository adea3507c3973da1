// Direction projection u_{t,i} = W_u[i] k_t / max(|W_u[i] k_t|_2, 1e-12) for sm_103a: the
// README "VLA v3" item 2 "u_t = normalize(W_u k_t^raw)", computed before the scan (whose u
// input it produces, [n, r, d]).  Four forms: tensor cores with bf16 operands fed by TMA
// (bfloat16 keys whose r weight sets fit in shared memory; vla_proj_tma.cu), the same
// product with keys through registers (bfloat16 keys otherwise), tensor cores in tf32
// (float32 keys whose operands fit in shared memory) and CUDA cores (d = 128 with float32
// keys).
//
// CUDA-core form: each thread takes TPT consecutive tokens (4 at d = 16, 2 at d = 64, 1 at d = 128),
// groups taken grid-stride, the ranks one after another (W_u[i] in shared memory, d x d
// float32).  Each thread reads its keys as 16-byte vectors (all independent loads, one
// memory latency per group), forms x_j = W[j] . k for its tokens with W's rows broadcast
// from shared memory, keeps x in its own padded shared-memory rows (stride d + 1,
// conflict-free), and writes x_j / max(|x|, 1e-12) as 16-byte vectors: no barrier
// inside the token loop.  Arithmetic in float32 (float32 or bfloat16 in and out).
#include "vla_internal.cuh"
#include "vla_tc.cuh"

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
  extern __shared__ __align__(16) float smc[];
  float* sW = smc + L::W_OFF;
  float* sX = smc + L::X_OFF + threadIdx.x * TP * (D + 1);   // this thread's TP rows of x
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

// ---------------------------------------------------------------------------
// Tensor-core form: x = K W^T for a tile of 128 tokens as one tcgen05 product
// (kind::tf32, M = 128 tokens, N = d outputs, K = d), accumulated in TMEM.  bf16 keys
// are exact in tf32; W is split into tf32 hi + lo parts, so two passes give W to about
// 2^-21 (float32 keys: also k hi + lo, three passes).  Operands sit in shared memory in
// the K-major no-swizzle core-matrix layout (tc::tk_off).  Row t of the result is TMEM
// lane t, which the epilogue thread t reads: it forms |x|, scales, converts and stores
// its token's u row as 16-byte vectors.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

template <int D, typename TIO>
struct TcCfg {
  static constexpr int NP = sizeof(TIO) == 2 ? 2 : 3;        // MMA passes
  static constexpr int F_KH = 0;                              // [128][D] keys (hi)
  static constexpr int F_KL = F_KH + 128 * D;                 // [128][D] keys lo (float32 keys)
  static constexpr int F_WH = F_KL + (NP == 3 ? 128 * D : 0); // [D][D] W hi
  static constexpr int F_WL = F_WH + D * D;                   // [D][D] W lo
  static constexpr int F_END = F_WL + D * D;
  static constexpr size_t bytes = sizeof(float) * (size_t)F_END + 16;   // + mbarrier, TMEM slot
  static constexpr uint32_t TCOLS = D < 32 ? 32 : D;
};

template <int D, typename TIO>
__global__ void __launch_bounds__(NTH) project_u_tc_kernel(const TIO* __restrict__ k, const float* __restrict__ W,
                                                           TIO* __restrict__ u, long long n, int r,
                                                           DevStatus* __restrict__ status) {
  using Cf = TcCfg<D, TIO>;
  using V = Vec<TIO>;
  using tc::tk_off;
  constexpr int NV = D / V::N;
  static_assert(NTH == 128, "one thread per TMEM lane of an M = 128 product");
  extern __shared__ __align__(1024) float sm[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Cf::F_END);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = smem_u32(sm);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(tslot, Cf::TCOLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + ((uint32_t)(32 * warp) << 16);   // this warp's lane quadrant
  uint32_t phase = 0;
  bool failed = false;
  auto st4 = [&](int off, float x0, float x1, float x2, float x3) {
    *reinterpret_cast<float4*>(sm + off) = make_float4(x0, x1, x2, x3);
  };
  const long long ntiles = (n + NTH - 1) / NTH;
  for (int i = 0; i < r && !failed; ++i) {
    // W_u[i] -> hi / lo, K-major (row j = output, K = input m)
    for (int e4 = tid; e4 < D * D / 4; e4 += NTH) {
      const float4 w = reinterpret_cast<const float4*>(W + (size_t)i * D * D)[e4];
      const int j = (4 * e4) / D, m = 4 * e4 - j * D;
      const float h0 = tf32_hi(w.x), h1 = tf32_hi(w.y), h2 = tf32_hi(w.z), h3 = tf32_hi(w.w);
      st4(Cf::F_WH + tk_off(j, m, D), h0, h1, h2, h3);
      st4(Cf::F_WL + tk_off(j, m, D), w.x - h0, w.y - h1, w.z - h2, w.w - h3);
    }
    // this thread's key rows of the next two tiles, loaded two tiles ahead so that the
    // loads overlap the products and epilogues of the tiles before (two register
    // buffers, used alternately by the two halves of the unrolled tile loop)
    auto fetch = [&](long long tile, uint4 (&buf)[NV]) {
      const long long t = tile * NTH + tid;
      const uint4* kv = reinterpret_cast<const uint4*>(k + t * D);
#pragma unroll
      for (int v = 0; v < NV; ++v) buf[v] = (tile < ntiles && t < n) ? __ldg(kv + v) : make_uint4(0u, 0u, 0u, 0u);
    };
    auto process = [&](long long tile, uint4 (&buf)[NV]) -> bool {
      const long long t = tile * NTH + tid;   // this thread's token (row tid of the tile)
      {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          float x[V::N];
          V::load(buf[v], x);
#pragma unroll
          for (int q = 0; q < V::N; q += 4) {
            const int m = V::N * v + q;
            if constexpr (Cf::NP == 3) {
              const float h0 = tf32_hi(x[q]), h1 = tf32_hi(x[q + 1]), h2 = tf32_hi(x[q + 2]), h3 = tf32_hi(x[q + 3]);
              st4(Cf::F_KH + tk_off(tid, m, D), h0, h1, h2, h3);
              st4(Cf::F_KL + tk_off(tid, m, D), x[q] - h0, x[q + 1] - h1, x[q + 2] - h2, x[q + 3] - h3);
            } else {
              st4(Cf::F_KH + tk_off(tid, m, D), x[q], x[q + 1], x[q + 2], x[q + 3]);
            }
          }
        }
      }
      // operands written by the generic proxy -> visible to the tensor core; the previous
      // tile's TMEM reads are done before this tile's product overwrites the accumulator
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) {
        constexpr uint32_t sbo = 32u * D;
        constexpr uint32_t idesc = tc::idesc_tf32(128, D);
        const int xs[3] = {Cf::F_KH, Cf::F_KH, Cf::F_KL}, ys[3] = {Cf::F_WH, Cf::F_WL, Cf::F_WH};
#pragma unroll
        for (int p = 0; p < Cf::NP; ++p)
#pragma unroll
          for (int kk = 0; kk < D / 8; ++kk)
            tc::mma_tf32(tmem, tc::sdesc(sbase + 4u * xs[p] + 256u * kk, sbo),
                         tc::sdesc(sbase + 4u * ys[p] + 256u * kk, sbo), idesc, p > 0 || kk > 0);
        tc::mma_commit(bar);
      }
      fetch(tile + 2 * (long long)gridDim.x, buf);   // the staged keys are consumed; refill two tiles ahead
      if (tid == 0 && !mbar_wait_bounded(bar, phase)) failed = true;
      phase ^= 1u;
      tc::fence_before_sync();
      failed = __syncthreads_or(failed) != 0;
      tc::fence_after_sync();
      if (failed) return false;
      // epilogue: |x| of this thread's row, then the scaled row
      constexpr int CW = D < 32 ? 16 : 32;   // columns per TMEM load
      float nrm = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += CW) {
        float x[CW];
        if constexpr (CW == 32) tc::tmem_ld32(tlane + (uint32_t)c0, x);
        else tc::tmem_ld16(tlane + (uint32_t)c0, x);
#pragma unroll
        for (int j = 0; j < CW; ++j) nrm = fmaf(x[j], x[j], nrm);
      }
      const float inv = 1.f / fmaxf(sqrtf(nrm), 1e-12f);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += CW) {
        float x[CW];
        if constexpr (CW == 32) tc::tmem_ld32(tlane + (uint32_t)c0, x);
        else tc::tmem_ld16(tlane + (uint32_t)c0, x);
        if (t < n) {
          uint4* uv = reinterpret_cast<uint4*>(u + (t * r + i) * D + c0);
#pragma unroll
          for (int v = 0; v < CW / V::N; ++v) {
            float y[V::N];
#pragma unroll
            for (int m = 0; m < V::N; ++m) y[m] = x[V::N * v + m] * inv;
            uv[v] = V::pack(y);
          }
        }
      }
      return true;
    };
    uint4 ka[NV], kb[NV];
    fetch(blockIdx.x, ka);
    fetch(blockIdx.x + (long long)gridDim.x, kb);
    for (long long tile = blockIdx.x; tile < ntiles; tile += 2 * (long long)gridDim.x) {
      if (!process(tile, ka)) break;
      if (tile + gridDim.x < ntiles && !process(tile + gridDim.x, kb)) break;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, Cf::TCOLS);
  if (failed && tid == 0) atomicOr(&status->flags, kStatusTimeout);
}

// ---------------------------------------------------------------------------
// bfloat16 keys: the same product as kind::f16 with bf16 operands.  A key row of d bf16
// values is already a row of operand core matrices, so each 16-byte load is stored as it
// is; W is carried as three bf16 terms w1 + w2 + w3 (w1 = bf16(W), w2 = bf16(W - w1),
// w3 = bf16(W - w1 - w2): about 24 bits), three passes with fp32 accumulation.  The
// operands take 40 KB at d = 64 (the tf32 form 64 KB), so more CTAs share an SM and
// keep more key rows in flight.
template <int D>
struct Bf16Cfg {
  static constexpr int B_K = 0;                                // [128][D] keys, bf16
  static constexpr int B_W = B_K + 128 * D * 2;                // 3 x [D][D] W terms, bf16
  static constexpr int B_END = B_W + 3 * D * D * 2;
  static constexpr size_t bytes = (size_t)B_END + 16;          // + mbarrier, TMEM slot
  static constexpr uint32_t TCOLS = D < 32 ? 32 : D;
};

template <int D>
__global__ void __launch_bounds__(NTH) project_u_bf16_kernel(const __nv_bfloat16* __restrict__ k,
                                                             const float* __restrict__ W,
                                                             __nv_bfloat16* __restrict__ u, long long n, int r,
                                                             DevStatus* __restrict__ status) {
  using Cf = Bf16Cfg<D>;
  using V = Vec<__nv_bfloat16>;
  using tc::tk16_off;
  constexpr int NV = D / 8;   // 16-byte vectors (8 bf16) per row
  static_assert(NTH == 128, "one thread per TMEM lane of an M = 128 product");
  extern __shared__ __align__(1024) unsigned char smb[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smb + Cf::B_END);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = smem_u32(smb);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(tslot, Cf::TCOLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + ((uint32_t)(32 * warp) << 16);
  uint32_t phase = 0;
  bool failed = false;
  auto st16 = [&](int byte_off, const uint4& v) { *reinterpret_cast<uint4*>(smb + byte_off) = v; };
  const long long ntiles = (n + NTH - 1) / NTH;
  for (int i = 0; i < r && !failed; ++i) {
    // W_u[i] -> three bf16 terms, K-major (row j = output, K = input m), 8 values a store
    for (int e8 = tid; e8 < D * D / 8; e8 += NTH) {
      const int j = (8 * e8) / D, m = 8 * e8 - j * D;
      const float4 a = reinterpret_cast<const float4*>(W + (size_t)i * D * D)[2 * e8];
      const float4 b = reinterpret_cast<const float4*>(W + (size_t)i * D * D)[2 * e8 + 1];
      float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int term = 0; term < 3; ++term) {
        float t[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          t[q] = __bfloat162float(__float2bfloat16_rn(x[q]));
          x[q] -= t[q];   // exact: t is x rounded to 8 significant bits
        }
        st16(Cf::B_W + term * D * D * 2 + 2 * tk16_off(j, m, D), V::pack(t));
      }
    }
    auto fetch = [&](long long tile, uint4 (&buf)[NV]) {
      const long long t = tile * NTH + tid;
      const uint4* kv = reinterpret_cast<const uint4*>(k + t * D);
#pragma unroll
      for (int v = 0; v < NV; ++v) buf[v] = (tile < ntiles && t < n) ? __ldg(kv + v) : make_uint4(0u, 0u, 0u, 0u);
    };
    auto process = [&](long long tile, uint4 (&buf)[NV]) -> bool {
      const long long t = tile * NTH + tid;
#pragma unroll
      for (int v = 0; v < NV; ++v) st16(Cf::B_K + 2 * tk16_off(tid, 8 * v, D), buf[v]);
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == 0) {
        constexpr uint32_t sbo = 16u * D;
        constexpr uint32_t idesc = tc::idesc_bf16(128, D);
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc::mma_f16(tmem, tc::sdesc(sbase + Cf::B_K + 256u * kk, sbo),
                        tc::sdesc(sbase + Cf::B_W + p * D * D * 2 + 256u * kk, sbo), idesc, p > 0 || kk > 0);
        tc::mma_commit(bar);
      }
      fetch(tile + 2 * (long long)gridDim.x, buf);   // the staged keys are consumed; refill two tiles ahead
      if (tid == 0 && !mbar_wait_bounded(bar, phase)) failed = true;
      phase ^= 1u;
      tc::fence_before_sync();
      failed = __syncthreads_or(failed) != 0;
      tc::fence_after_sync();
      if (failed) return false;
      constexpr int CW = D < 32 ? 16 : 32;   // columns per TMEM load
      float nrm = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += CW) {
        float x[CW];
        if constexpr (CW == 32) tc::tmem_ld32(tlane + (uint32_t)c0, x);
        else tc::tmem_ld16(tlane + (uint32_t)c0, x);
#pragma unroll
        for (int j = 0; j < CW; ++j) nrm = fmaf(x[j], x[j], nrm);
      }
      const float inv = 1.f / fmaxf(sqrtf(nrm), 1e-12f);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += CW) {
        float x[CW];
        if constexpr (CW == 32) tc::tmem_ld32(tlane + (uint32_t)c0, x);
        else tc::tmem_ld16(tlane + (uint32_t)c0, x);
        if (t < n) {
          uint4* uv = reinterpret_cast<uint4*>(u + (t * r + i) * D + c0);
#pragma unroll
          for (int v = 0; v < CW / 8; ++v) {
            float y[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) y[m] = x[8 * v + m] * inv;
            uv[v] = V::pack(y);
          }
        }
      }
      return true;
    };
    uint4 ka[NV], kb[NV];
    fetch(blockIdx.x, ka);
    fetch(blockIdx.x + (long long)gridDim.x, kb);
    for (long long tile = blockIdx.x; tile < ntiles; tile += 2 * (long long)gridDim.x) {
      if (!process(tile, ka)) break;
      if (tile + gridDim.x < ntiles && !process(tile + gridDim.x, kb)) break;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, Cf::TCOLS);
  if (failed && tid == 0) atomicOr(&status->flags, kStatusTimeout);
}

// The TMA-fed bfloat16 form (vla_proj_tma.cu); *used = false when its operands do not fit.
template <int D>
cudaError_t launch_project_tma(const void* k, const float* W, void* u, long long n, int r, int sm_count,
                               DevStatus* status, cudaStream_t s, bool* used);

template <int D, typename TIO>
cudaError_t launch_project_t(const void* k, const float* W, void* u, long long n, int r, int sm_count,
                             DevStatus* status, cudaStream_t s) {
  const int sms = sm_count > 0 ? sm_count : 1;
  if constexpr (sizeof(TIO) == 2) {   // bfloat16 keys: kind::f16 with bf16 operands
    bool used = false;
    cudaError_t et = launch_project_tma<D>(k, W, u, n, r, sms, status, s, &used);
    if (used || et != cudaSuccess) return et;
    // W's three terms for all r ranks beyond shared memory (d = 128 with r > 1, d = 64 with
    // r > 5): one tile and one rank at a time, keys through registers
    auto kern = project_u_bf16_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Bf16Cfg<D>::bytes);
    if (e != cudaSuccess) return e;
    const long long ntiles = (n + NTH - 1) / NTH;
    const int grid = (int)min(ntiles, (long long)sms * 8);
    kern<<<grid, NTH, Bf16Cfg<D>::bytes, s>>>(static_cast<const __nv_bfloat16*>(k), W,
                                              static_cast<__nv_bfloat16*>(u), n, r, status);
    return cudaGetLastError();
  } else if constexpr (TcCfg<D, TIO>::bytes <= 227 * 1024) {   // float32 keys: kind::tf32
    auto kern = project_u_tc_kernel<D, TIO>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<D, TIO>::bytes);
    if (e != cudaSuccess) return e;
    const long long ntiles = (n + NTH - 1) / NTH;
    const int grid = (int)min(ntiles, (long long)sms * 4);
    kern<<<grid, NTH, TcCfg<D, TIO>::bytes, s>>>(static_cast<const TIO*>(k), W, static_cast<TIO*>(u), n, r,
                                                 status);
    return cudaGetLastError();
  } else {   // d = 128 float32 keys: operands beyond shared memory; CUDA cores
    auto kern = project_u_kernel<D, TIO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem<D>::bytes);
    if (e != cudaSuccess) return e;
    const long long nblk = (n + (long long)NTH * tpt<D>() - 1) / ((long long)NTH * tpt<D>());
    const int grid = (int)min(nblk, (long long)sms * 4);
    kern<<<grid, NTH, Smem<D>::bytes, s>>>(static_cast<const TIO*>(k), W, static_cast<TIO*>(u), n, r);
    return cudaGetLastError();
  }
}

}  // namespace prj

cudaError_t launch_project_u(int d, bool bf16, const void* k, const float* W, void* u, long long n, int r,
                             int sm_count, DevStatus* status, cudaStream_t s, bool* built) {
  *built = true;
  if (d == 16) return bf16 ? prj::launch_project_t<16, __nv_bfloat16>(k, W, u, n, r, sm_count, status, s)
                           : prj::launch_project_t<16, float>(k, W, u, n, r, sm_count, status, s);
  if (d == 64) return bf16 ? prj::launch_project_t<64, __nv_bfloat16>(k, W, u, n, r, sm_count, status, s)
                           : prj::launch_project_t<64, float>(k, W, u, n, r, sm_count, status, s);
  if (d == 128) return bf16 ? prj::launch_project_t<128, __nv_bfloat16>(k, W, u, n, r, sm_count, status, s)
                            : prj::launch_project_t<128, float>(k, W, u, n, r, sm_count, status, s);
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
