// Chunked VLA scan for sm_103a: C steps (M = C r = 64 directions) per chunk in
// exact Woodbury / LDL^T form, with the dense contractions on tcgen05 tensor
// cores (kind::tf32, fp32 accumulation in TMEM).
//
// "Mathematical Primitives" §3 names the Woodbury identity as the closed form of
// r sequential Sherman-Morrison updates, and the gist.science summary §2.4 a
// parallel formulation of the scan; neither writes the chunk algebra out.  For a
// chunk with directions U (rows u_a), s-vectors Sigma (rows s_t) and A_0 = the
// inverse at its start:
//
//   G1  [W^T; Q^T]  = [U; Sigma] A_0                    W = A_0 U, Q = A_0 Sigma
//   G2  [G - I | .] = [W^T; Q^T] [U; Sigma]^T           G = I + U^T A_0 U; rows 64+ give H^T = (U^T Q)^T
//       G = L D L^T (CUDA cores; D_jj are the sequential deltas), Linv = L^{-1}
//   G3  [Z^T | F]   = Linv [W; H^T]^T                   Z = W L^{-T} (the sequential z's), F = Linv H
//       E = D^{-1} F, masked to directions of steps <= t
//   G4  [Z D^{-1} Z^T ; (Z E)^T] = [Z D^{-1}; E^T] Z^T  A_1 = A_0 - Z D^{-1} Z^T,  alpha = Q - Z E
//   G5  [S alpha_t, alpha.alpha ; S phi(q_t), phi(q_t).alpha] = [alpha; Phi_q] [S; alpha]^T
//   G6  [tril(aq) V ; V^T alpha]   = [tril(aq); V^T] [V^T; alpha^T]^T
//       o_t = (S phi(q_t) + sum_{t'<=t} (alpha_t'.phi(q_t)) v_t') / den_t,   S_1 = S + V^T alpha
//
// Renormalisation: ||S_t||^2 = ||S||^2 + 2 sum v_t'^T S alpha_t' + sum (v.v)(alpha.alpha) from the
// products above; the bound ||S|| + sum |v_t||alpha_t| decides that no step can
// exceed tau, otherwise the exact per-step norms give the decisions and the
// per-step scales are folded into tril(aq), alpha^T and the outputs.  When the
// scales of one chunk fall below 2^-64 (tau far below the norm each step adds),
// that chunk's S and outputs are taken step by step from its alpha instead.
// A pivot |D_jj| < 1e-6 means the sequential recurrence takes the singularity
// guard inside the chunk; the chunk is then taken step by step on CUDA cores.
// Chunks end at nudge steps (A += eps_n I is not a rank-1 update).
//
// Operands are fp32 in shared memory, read by the tensor core as tf32; the
// state (A, S) stays fp32.  Built for d = d_v = 64 and bfloat16 I/O.
#pragma once

#include "vla_tc.cuh"

namespace vla {
namespace chk {

constexpr int D = 64;
constexpr int NT = 256;
constexpr int TILE = 64 * 64;         // floats of a TK(64, 64) operand tile
constexpr int GLD = 68;               // leading dimension of the fp32 G staging
constexpr float kGuardEps = 1e-6f;
constexpr float kReadoutEps = 1e-6f;
constexpr float kInvSqrtD = 0.125f;

// High part of a 3xTF32 split: the value with the low 13 mantissa bits cleared
// (exactly representable in tf32); the low part is x - hi.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

template <int R, typename TIO>
struct Cfg {
  static constexpr int C = 64 / R;                        // steps per chunk
  static constexpr int TS = C;                            // steps per input tile
  static constexpr uint32_t QB = TS * D * sizeof(TIO);
  static constexpr uint32_t UB = TS * R * D * sizeof(TIO);
  static constexpr uint32_t STAGE = 3 * QB + UB;
  static constexpr uint32_t STAGE_PAD = (STAGE + 1023) / 1024 * 1024;
  static constexpr int T6T = 64 * C;                      // floats of a TK(64, C) tile
  // float offsets (after the raw stage)
  static constexpr int F_A = 0;                           // A
  static constexpr int F_S = F_A + TILE;                  // S       } [S][alpha][phi(q)] contiguous
  static constexpr int F_AL = F_S + TILE;                 // alpha   }
  static constexpr int F_PQ = F_AL + TILE;                // phi(q)  }
  static constexpr int F_P = F_PQ + TILE;                 // 2 tiles: [U; Sigma] -> G staging -> [Z/D; E^T] -> Y staging
  static constexpr int F_Q = F_P + 2 * TILE;              // 2 tiles: [W^T; Q^T] -> (Z, Q^T) -> alpha Gram
  static constexpr int F_R = F_Q + 2 * TILE;              // 2 tiles: prologue scratch -> [W; H^T] -> T6 (with L)
  static constexpr int F_L = F_R + 2 * TILE;              // 1 tile:  Linv
  static constexpr int F_T6 = F_R;                        // [tril(aq)][V^T][alpha^T], TK(64, C) each
  static constexpr int F_MISC = F_L + TILE;
  // misc block
  static constexpr int M_D = 0, M_ID = 64, M_RDEN = 128, M_VN = 192, M_SL = 256, M_XS = 320, M_AN = 384;
  static constexpr int M_SG = 448, M_IS = 512, M_RED = 576, M_VEC = 640, M_VEC2 = 704, M_SCAL = 768;
  static constexpr int F_VB = F_MISC + 800;               // V of the chunk (TIO) [C][64]
  static constexpr size_t float_bytes = sizeof(float) * (size_t)F_VB + sizeof(TIO) * C * 64;
  static constexpr size_t bar_off = STAGE_PAD + (float_bytes + 15) / 16 * 16;
  static constexpr size_t bytes = bar_off + 64;
  static_assert(3 * T6T <= 3 * TILE, "T6 fits in R and L");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

}  // namespace chk

template <int R, typename TIO>
__global__ void __launch_bounds__(chk::NT, 1) chunk_scan_kernel(ScanArgs a) {
  using namespace chk;
  using Cf = Cfg<R, TIO>;
  constexpr int C = Cf::C, TS = Cf::TS;
  using tc::tk_off;

  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* raw = smem;
  float* sf = reinterpret_cast<float*>(smem + Cf::STAGE_PAD);
  float* misc = sf + Cf::F_MISC;
  TIO* vb = reinterpret_cast<TIO*>(sf + Cf::F_VB);
  uint64_t* in_bar = reinterpret_cast<uint64_t*>(smem + Cf::bar_off);
  uint64_t* mma_bar = in_bar + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(in_bar + 2);
  volatile int* flag = reinterpret_cast<volatile int*>(in_bar + 3);
  const uint32_t sbase = smem_u32(sf);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long pair = blockIdx.x;
  const long long T = a.T;
  const TIO* gq = static_cast<const TIO*>(a.q) + pair * T * D;
  const TIO* gk = static_cast<const TIO*>(a.k) + pair * T * D;
  const TIO* gv = static_cast<const TIO*>(a.v) + pair * T * D;
  const TIO* gu = static_cast<const TIO*>(a.u) + pair * T * R * D;
  TIO* go = static_cast<TIO*>(a.o) + pair * T * D;
  float* gA = a.A + pair * D * D;
  float* gS = a.S + pair * D * D;
  float* gn = a.n + pair * D;

  // ---- state into the operand tiles
  for (int e = tid; e < D * D; e += NT) {
    const int i = e >> 6, j = e & 63;
    sf[Cf::F_A + tk_off(i, j, 64)] = gA[e];
    sf[Cf::F_S + tk_off(i, j, 64)] = gS[e];
  }
  float n_i = (tid < D) ? gn[tid] : 0.f;
  if (tid == 0) {
    mbar_init(in_bar, 1);
    mbar_init(mma_bar, 1);
    fence_mbar_init();
    *flag = 0;
  }
  if (warp == 0) tc::tmem_alloc(tslot, 128);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  const int ntiles = (int)((T + TS - 1) / TS);
  auto issue = [&](int tile) {  // thread 0 only
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const uint32_t qb = (uint32_t)nst * D * sizeof(TIO), ub = (uint32_t)nst * R * D * sizeof(TIO);
    mbar_arrive_expect_tx(in_bar, 3 * qb + ub);
    bulk_g2s(raw, gq + t_start * D, qb, in_bar);
    bulk_g2s(raw + Cf::QB, gk + t_start * D, qb, in_bar);
    bulk_g2s(raw + 2 * Cf::QB, gv + t_start * D, qb, in_bar);
    bulk_g2s(raw + 3 * Cf::QB, gu + t_start * R * D, ub, in_bar);
  };
  if (tid == 0) issue(0);

  uint32_t mma_phase = 0;
  unsigned int flags = 0;
  unsigned long long guard_cnt = 0, renorm_cnt = 0, fallback_cnt = 0;
  bool failed = false;

  // operand tiles written by the generic proxy -> visible to the tensor core;
  // earlier TMEM loads ordered before the next MMA
  auto sync_tc = [&]() {
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  };
  // D = sum over passes of X_p * Y_p^T into TMEM columns 0.. (X_p: M rows, Y_p: N_p rows,
  // both K-major with K columns).  Three passes (hi*hi, lo*hi, hi*lo) give 3xTF32.
  auto gemm_passes = [&](int M, int K, int np, const int* xo, const int* yo, const int* nn) -> bool {
    sync_tc();
    if (tid == 0) {
      const uint32_t sbo = 32u * (uint32_t)K;
      for (int p = 0; p < np; ++p) {
        const uint32_t idesc = tc::idesc_tf32(M, nn[p]);
        for (int kk = 0; kk < K / 8; ++kk)
          tc::mma_tf32(tmem, tc::sdesc(sbase + 4u * xo[p] + 256u * kk, sbo),
                       tc::sdesc(sbase + 4u * yo[p] + 256u * kk, sbo), idesc, p > 0 || kk > 0);
      }
      tc::mma_commit(mma_bar);
      if (!mbar_wait_bounded(mma_bar, mma_phase)) *flag = 1;
    }
    mma_phase ^= 1u;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    return *flag == 0;
  };
  auto gemm = [&](int xoff, int yoff, int M, int N, int K) -> bool {
    const int xo[1] = {xoff}, yo[1] = {yoff}, nn[1] = {N};
    return gemm_passes(M, K, 1, xo, yo, nn);
  };
  // the warp's TMEM lane quadrant and column half
  const int q4 = warp & 3, half = warp >> 2;
  auto tld = [&](int col, float (&v)[16]) { tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)col, v); };

  // block reduction of one float over the CTA (all threads call it)
  auto block_sum = [&](float x) -> float {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    __syncthreads();
    if (lane == 0) misc[Cf::M_RED + warp] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) s += misc[Cf::M_RED + w];
    return s;
  };

  long long pos = 0;
  int loaded = -1;
  while (pos < T && !failed) {
    // ---------------- schedule: chunk [pos, pos + c) inside one input tile, ending at a nudge
    const int tile = (int)(pos / TS);
    const int ts = (int)(pos % TS);
    int c = (int)min((long long)(TS - ts), T - pos);
    bool nudge = false;
    if (a.P > 0) {
      const long long to_nudge = a.P - ((a.t0 + pos) % a.P);
      if (to_nudge <= c) { c = (int)to_nudge; nudge = true; }
    }
    if (tile != loaded) {
      if (tid == 0 && !mbar_wait_bounded(in_bar, (uint32_t)(tile & 1))) *flag = 1;
      __syncthreads();
      if (*flag) { failed = true; break; }
      loaded = tile;
    }
    const TIO* rq = reinterpret_cast<const TIO*>(raw);
    const TIO* rk = reinterpret_cast<const TIO*>(raw + Cf::QB);
    const TIO* rv = reinterpret_cast<const TIO*>(raw + 2 * Cf::QB);
    const TIO* ru = reinterpret_cast<const TIO*>(raw + 3 * Cf::QB);

    // ---------------- prologue: [U; Sigma] -> P, phi(q) -> PQ, V -> vb, phi(k) -> R scratch
    {
      float* prod = sf + Cf::F_R;
      for (int e4 = tid; e4 < 64 * 16; e4 += NT) {   // U rows a (64), 4 columns each
        const int arow = e4 >> 4, col = (e4 & 15) * 4;
        const int t = arow / R, i = arow - t * R;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < c) {
          const TIO* src = ru + ((ts + t) * R + i) * D + col;
          x = make_float4(to_f32(src[0]), to_f32(src[1]), to_f32(src[2]), to_f32(src[3]));
        }
        *reinterpret_cast<float4*>(sf + Cf::F_P + tk_off(arow, col, 64)) = x;
      }
      for (int e4 = tid; e4 < C * 16; e4 += NT) {    // step rows t < C
        const int t = e4 >> 4, col = (e4 & 15) * 4;
        float kx[4] = {0.f, 0.f, 0.f, 0.f}, qx[4] = {0.f, 0.f, 0.f, 0.f};
        TIO vx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) vx[j] = from_f32<TIO>(0.f);
        if (t < c) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            kx[j] = phi_elu1(to_f32(rk[(ts + t) * D + col + j]));
            qx[j] = phi_elu1(to_f32(rq[(ts + t) * D + col + j]));
            vx[j] = rv[(ts + t) * D + col + j];
          }
        }
        *reinterpret_cast<float4*>(sf + Cf::F_P + tk_off(64 + t, col, 64)) =
            make_float4(kx[0] * kInvSqrtD, kx[1] * kInvSqrtD, kx[2] * kInvSqrtD, kx[3] * kInvSqrtD);
        *reinterpret_cast<float4*>(sf + Cf::F_PQ + tk_off(t, col, 64)) = make_float4(qx[0], qx[1], qx[2], qx[3]);
        *reinterpret_cast<float4*>(prod + t * 64 + col) = make_float4(kx[0], kx[1], kx[2], kx[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) vb[t * 64 + col + j] = vx[j];
      }
      for (int e4 = tid; e4 < (64 - C) * 16; e4 += NT) {   // zero rows C..63 of Sigma and phi(q)
        const int t = C + (e4 >> 4), col = (e4 & 15) * 4;
        *reinterpret_cast<float4*>(sf + Cf::F_P + tk_off(64 + t, col, 64)) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(sf + Cf::F_PQ + tk_off(t, col, 64)) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncthreads();
      if (tid < D) {   // n_t = n_{t-1} + phi(k_t); products n_t[i] phi(q_t)[i]
        for (int t = 0; t < c; ++t) {
          n_i += prod[t * 64 + tid];
          prod[t * 64 + tid] = n_i * sf[Cf::F_PQ + tk_off(t, tid, 64)];
        }
        misc[Cf::M_SL + tid] = sf[Cf::F_P + tk_off(64 + c - 1, tid, 64)];   // s of the chunk's last step
      }
      __syncthreads();
      {  // 1/den_t and |v_t|: NT / C threads per step (every lane takes part in the shuffles)
        constexpr int TPS = NT / C;
        constexpr int EPT = 64 / TPS;
        const int t = tid / TPS, part = tid - t * TPS;
        float dn = 0.f, vv = 0.f;
        if (t < c) {
#pragma unroll
          for (int j = 0; j < EPT; ++j) {
            dn += prod[t * 64 + part * EPT + j];
            const float x = to_f32(vb[t * 64 + part * EPT + j]);
            vv = fmaf(x, x, vv);
          }
        }
#pragma unroll
        for (int m = TPS / 2; m >= 1; m >>= 1) {
          dn += __shfl_xor_sync(0xffffffffu, dn, m);
          vv += __shfl_xor_sync(0xffffffffu, vv, m);
        }
        if (t < C && part == 0) {
          misc[Cf::M_RDEN + t] = (t < c) ? __frcp_rn(dn + kReadoutEps) : 0.f;
          misc[Cf::M_VN + t] = (t < c) ? sqrtf(vv) : 0.f;
        }
      }
      __syncthreads();
      // the raw stage is free once the tile's last chunk is converted
      if (tid == 0 && ts + c == TS && tile + 1 < ntiles) {
        fence_proxy_async_smem();
        issue(tile + 1);
      }
    }

    // ---------------- G1: [W^T; Q^T] = [U; Sigma] A_0^T  (M 128, N 64, K 64), A split hi + lo
    // (U is exact in tf32, so two passes make W as accurate as fp32)
    for (int e4 = tid; e4 < TILE / 4; e4 += NT) {
      const float4 x = *reinterpret_cast<const float4*>(sf + Cf::F_A + 4 * e4);
      const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
      *reinterpret_cast<float4*>(sf + Cf::F_R + 4 * e4) = h;
      *reinterpret_cast<float4*>(sf + Cf::F_R + TILE + 4 * e4) = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
    }
    {
      const int xo[2] = {Cf::F_P, Cf::F_P}, yo[2] = {Cf::F_R, Cf::F_R + TILE}, nn[2] = {64, 64};
      if (!gemm_passes(128, 64, 2, xo, yo, nn)) { failed = true; break; }
    }
    {
      float v[16];
      const int row = 32 * q4 + lane;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = 32 * half + 16 * cc;
        tld(col0, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(sf + Cf::F_Q + tk_off(row, col0 + j, 64)) =
              make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        if (row < 64) {   // W (rows i, K = direction) for G3
#pragma unroll
          for (int j = 0; j < 16; ++j) sf[Cf::F_R + tk_off(col0 + j, row, 64)] = v[j];
        }
      }
    }
    // ---------------- G2: [G - I | .] = [W^T; Q^T] [U; Sigma]^T  (M 128, N 128, K 64)
    if (!gemm(Cf::F_Q, Cf::F_P, 128, 128, 64)) { failed = true; break; }
    if (half == 0) {   // columns 0..63 only
      float v[16];
      const int row = 32 * q4 + lane;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int col0 = 16 * cc;
        tld(col0, v);
        if (row < 64) {
#pragma unroll
          for (int j = 0; j < 16; ++j) sf[Cf::F_P + row * GLD + col0 + j] = v[j] + ((row == col0 + j) ? 1.f : 0.f);
        } else {   // H^T rows t for G3 (rows 64.. of [W; H^T])
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(sf + Cf::F_R + tk_off(row, col0 + j, 64)) =
                make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();

    // ---------------- LDL^T of G (fp32, in place in the staging), blocks of 4 columns
    float* Gs = sf + Cf::F_P;
    for (int j0 = 0; j0 < 64; j0 += 4) {
      // the 4 x 4 diagonal block, redundantly in every thread
      float g[4][4], Lb[4][4], Db[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s <= r; ++s) g[r][s] = Gs[(j0 + r) * GLD + j0 + s];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float dj = g[j][j];
#pragma unroll
        for (int k = 0; k < j; ++k) dj = fmaf(-Lb[j][k] * Db[k], Lb[j][k], dj);
        Db[j] = dj;
#pragma unroll
        for (int i = j + 1; i < 4; ++i) {
          float x = g[i][j];
#pragma unroll
          for (int k = 0; k < j; ++k) x = fmaf(-Lb[i][k] * Db[k], Lb[j][k], x);
          Lb[i][j] = x / dj;
        }
      }
      float iDb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) iDb[j] = 1.f / Db[j];
      __syncthreads();   // everyone has read the block before the panel is overwritten
      if (tid < 4) {
        misc[Cf::M_D + j0 + tid] = Db[tid];
        misc[Cf::M_ID + j0 + tid] = iDb[tid];
      }
      if (tid == 0) {
#pragma unroll
        for (int r = 1; r < 4; ++r)
#pragma unroll
          for (int s = 0; s < r; ++s) Gs[(j0 + r) * GLD + j0 + s] = Lb[r][s];
      }
      // panel rows i >= j0 + 4: L[i][j0 + k]
      const int i = j0 + 4 + tid;
      float li[4] = {0.f, 0.f, 0.f, 0.f};
      if (i < 64) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float x = Gs[i * GLD + j0 + k];
#pragma unroll
          for (int kp = 0; kp < k; ++kp) x = fmaf(-li[kp] * Db[kp], Lb[k][kp], x);
          li[k] = x * iDb[k];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) Gs[i * GLD + j0 + k] = li[k];
      }
      __syncthreads();
      // trailing update of the lower triangle: G[i][k] -= sum_k' L[i][k'] D[k'] L[k][k']
      for (int e = tid; e < (64 - j0 - 4) * 16; e += NT) {
        const int ii = j0 + 4 + (e >> 4), kq = (e & 15) * 4;
        float lir[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) lir[k] = Gs[ii * GLD + j0 + k] * Db[k];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kk = kq + j;
          if (kk >= j0 + 4 && kk <= ii) {
            float x = Gs[ii * GLD + kk];
#pragma unroll
            for (int k = 0; k < 4; ++k) x = fmaf(-lir[k], Gs[kk * GLD + j0 + k], x);
            Gs[ii * GLD + kk] = x;
          }
        }
      }
      __syncthreads();
    }
    // pivot check: the guard would fire inside the chunk
    int bad = 0;
    if (tid < 64) {
      const float dj = misc[Cf::M_D + tid];
      bad = !(fabsf(dj) >= kGuardEps) ? 1 : 0;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
      // ============ fallback: the chunk step by step on CUDA cores
      ++fallback_cnt;
      float* vec = misc + Cf::M_VEC;     // u, then s
      float* vec2 = misc + Cf::M_VEC2;   // z, alpha
      const int row = tid >> 2, cq = tid & 3;   // row of A / S and a 16-column quarter
      for (int t = 0; t < c; ++t) {
        const long long st = pos + t;
        for (int i = 0; i < R; ++i) {
          if (tid < 64) vec[tid] = to_f32(gu[(st * R + i) * D + tid]);
          __syncthreads();
          float zp = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) zp = fmaf(sf[Cf::F_A + tk_off(row, 16 * cq + j, 64)], vec[16 * cq + j], zp);
          zp += __shfl_xor_sync(0xffffffffu, zp, 1);
          zp += __shfl_xor_sync(0xffffffffu, zp, 2);
          if (cq == 0) vec2[row] = zp;
          __syncthreads();
          const float dl = 1.f + block_sum(tid < 64 ? vec[tid] * vec2[tid] : 0.f);
          const bool gd = fabsf(dl) < kGuardEps;
          if (tid == 0 && gd) ++guard_cnt;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = 16 * cq + j;
            float& ar = sf[Cf::F_A + tk_off(row, col, 64)];
            if (gd) ar += (row == col) ? kGuardEps : 0.f;
            else ar = fmaf(-vec2[row] / dl, vec2[col], ar);
          }
          __syncthreads();
        }
        const bool nd = nudge && t == c - 1;
        if (nd && cq == (row >> 4)) sf[Cf::F_A + tk_off(row, row, 64)] += a.eps_n;
        if (tid < 64) vec[tid] = phi_elu1(to_f32(gk[st * D + tid])) * kInvSqrtD;
        __syncthreads();
        float ap = 0.f;   // alpha = A s
#pragma unroll
        for (int j = 0; j < 16; ++j) ap = fmaf(sf[Cf::F_A + tk_off(row, 16 * cq + j, 64)], vec[16 * cq + j], ap);
        ap += __shfl_xor_sync(0xffffffffu, ap, 1);
        ap += __shfl_xor_sync(0xffffffffu, ap, 2);
        if (cq == 0) vec2[row] = ap;
        __syncthreads();
        // S += v alpha^T, then the norm
        const float vr = to_f32(vb[t * 64 + row]);   // v of step t
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = 16 * cq + j;
          float& sr = sf[Cf::F_S + tk_off(row, col, 64)];
          sr = fmaf(vr, vec2[col], sr);
          sq = fmaf(sr, sr, sq);
        }
        const float nrm = sqrtf(block_sum(sq));
        if (nrm > a.tau) {
          const float cf = a.tau / nrm;
#pragma unroll
          for (int j = 0; j < 16; ++j) sf[Cf::F_S + tk_off(row, 16 * cq + j, 64)] *= cf;
          if (tid == 0) ++renorm_cnt;
        }
        if (!isfinite(nrm)) flags |= kStatusNonfinite;
        if (tid < 64) vec[tid] = phi_elu1(to_f32(gq[st * D + tid]));
        __syncthreads();
        float op = 0.f;   // o = S phi(q) / den
#pragma unroll
        for (int j = 0; j < 16; ++j) op = fmaf(sf[Cf::F_S + tk_off(row, 16 * cq + j, 64)], vec[16 * cq + j], op);
        op += __shfl_xor_sync(0xffffffffu, op, 1);
        op += __shfl_xor_sync(0xffffffffu, op, 2);
        if (cq == 0) go[st * D + row] = from_f32<TIO>(op * misc[Cf::M_RDEN + t]);
        __syncthreads();
      }
      pos += c;
      continue;
    }
    // ---------------- Linv = L^{-1} (unit lower), 4 threads per column, into the L tile
    {
      const int acol = tid >> 2, sub = tid & 3;   // column a, rows 16 sub .. 16 sub + 15
      float x[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] = (16 * sub + j == acol) ? 1.f : 0.f;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
#pragma unroll
        for (int jb = 0; jb < 16; ++jb) {
          const int b = 16 * bb + jb;
          // x_b (held by the thread with sub == bb) is final: take it out of the rows below
          const float xb = __shfl_sync(0xffffffffu, x[jb], (lane & ~3) | bb);
          if (b >= acol && b < 63) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int l = 16 * sub + j;
              if (l > b) x[j] = fmaf(-Gs[l * GLD + b], xb, x[j]);
            }
          }
        }
      }
      __syncthreads();   // every thread is done with the L factor in P
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int o = tk_off(16 * sub + j, acol, 64);
        const float h = tf32_hi(x[j]);
        sf[Cf::F_L + o] = h;
        sf[Cf::F_P + o] = x[j] - h;   // Linv lo
      }
      // W (rows 0..63 of [W; H^T]) -> hi in place, lo into the second P tile
      for (int e = tid; e < TILE; e += NT) {
        const float w = sf[Cf::F_R + e];
        const float h = tf32_hi(w);
        sf[Cf::F_R + e] = h;
        sf[Cf::F_P + TILE + e] = w - h;
      }
    }
    // ---------------- G3: [Z^T | F] = Linv [W; H^T]^T  (M 64, N 128, K 64), 3xTF32 on Z
    {
      const int xo[3] = {Cf::F_L, Cf::F_P, Cf::F_L}, yo[3] = {Cf::F_R, Cf::F_R, Cf::F_P + TILE}, nn[3] = {128, 128, 64};
      if (!gemm_passes(64, 64, 3, xo, yo, nn)) { failed = true; break; }
    }
    {
      // M = 64 result: rows 16 q .. 16 q + 15 in lanes 0..15 of quadrant q.  The
      // TMEM load is warp-collective: every lane executes it, lanes 16..31 drop it.
      float v[16];
      const int l = 16 * q4 + (lane & 15);
      const float idl = misc[Cf::M_ID + l];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int col0 = 64 * half + 16 * cc;
        tld(col0, v);
        if (lane >= 16) continue;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = col0 + j;
          if (half == 0) {   // Z^T[l][i]: Z (rows i, K = l) and Z D^{-1} (rows i of [Z/D; E^T]), hi + lo
            const int oz = tk_off(col, l, 64);
            const float z = v[j], zh = tf32_hi(z), zd = z * idl, zdh = tf32_hi(zd);
            sf[Cf::F_Q + oz] = zh;
            sf[Cf::F_L + oz] = z - zh;
            sf[Cf::F_P + oz] = zdh;
            sf[Cf::F_R + oz] = zd - zdh;
          } else {           // F[l][t] -> E^T[t][l] (rows 64 + t of [Z/D; E^T]), hi + lo
            const int t = col - 64;
            if (t < C) {
              const float e = (l <= (t + 1) * R - 1) ? v[j] * idl : 0.f, eh = tf32_hi(e);
              const int oe = tk_off(64 + t, l, 64);
              sf[Cf::F_P + oe] = eh;
              sf[Cf::F_R + oe] = e - eh;
            }
          }
        }
      }
    }
    // ---------------- G4: [Z D^{-1} Z^T ; (Z E)^T] = [Z/D; E^T] Z^T  (M 128, N 64, K 64), 3xTF32
    {
      const int xo[3] = {Cf::F_P, Cf::F_R, Cf::F_P}, yo[3] = {Cf::F_Q, Cf::F_Q, Cf::F_L}, nn[3] = {64, 64, 64};
      if (!gemm_passes(128, 64, 3, xo, yo, nn)) { failed = true; break; }
    }
    {
      float v[16];
      const int row = 32 * q4 + lane;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = 32 * half + 16 * cc;
        tld(col0, v);
        if (row < 64) {   // A_1 = A_0 - Z D^{-1} Z^T (+ eps_n I at a nudge)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float& ar = sf[Cf::F_A + tk_off(row, col0 + j, 64)];
            ar = ar - v[j] + ((nudge && row == col0 + j) ? a.eps_n : 0.f);
          }
        } else {          // alpha_t = Q_t - (Z E)_t (+ eps_n s_t at a nudge step)
          const int t = row - 64;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = col0 + j;
            float al = 0.f;
            if (t < c) {
              al = sf[Cf::F_Q + TILE + tk_off(t, col, 64)] - v[j];
              if (nudge && t == c - 1) al = fmaf(a.eps_n, misc[Cf::M_SL + col], al);
            }
            sf[Cf::F_AL + tk_off(t, col, 64)] = al;
            if (t < C) sf[Cf::F_T6 + 2 * Cf::T6T + tk_off(col, t, C)] = al;   // alpha^T (rows j, K = t)
          }
        }
      }
      // V^T (rows i, K = t) for G6
      for (int e = tid; e < 64 * C; e += NT) {
        const int t = e >> 6, i = e & 63;
        sf[Cf::F_T6 + Cf::T6T + tk_off(i, t, C)] = to_f32(vb[t * 64 + i]);
      }
    }
    // ---------------- G5: [S alpha ; S phi(q) | alpha.alpha ; phi(q).alpha] = [alpha; phi(q)] [S; alpha]^T
    if (!gemm(Cf::F_AL, Cf::F_S, 128, 128, 64)) { failed = true; break; }
    {
      float v[16];
      const int row = 32 * q4 + lane;
      float xs = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int col0 = 64 * half + 16 * cc;
        tld(col0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = col0 + j;
          if (row < 64) {
            const int t = row;
            if (half == 0) {          // (S alpha_t)[i] -> v_t . S alpha_t
              if (t < c) xs = fmaf(to_f32(vb[t * 64 + col]), v[j], xs);
            } else {                  // alpha_t . alpha_t'
              const int tp = col - 64;
              if (tp < C && t < C) sf[Cf::F_Q + t * C + tp] = v[j];
              if (tp == t) misc[Cf::M_AN + t] = v[j];
            }
          } else {
            const int t = row - 64;
            if (half == 0) {          // Y_t[i] = (S phi(q_t))[i]
              if (t < C) sf[Cf::F_P + t * 64 + col] = v[j];
            } else {                  // aq[t][t'] = phi(q_t) . alpha_t', t' <= t
              const int tp = col - 64;
              if (t < C && tp < C) sf[Cf::F_T6 + tk_off(t, tp, C)] = (tp <= t && t < c) ? v[j] : 0.f;
            }
          }
        }
      }
      if (row < 64 && half == 0) misc[Cf::M_XS + row] = xs;
    }
    // ||S||^2 and the renormalisation decisions
    {
      float sq = 0.f;
      for (int e = tid; e < D * D; e += NT) {
        const float x = sf[Cf::F_S + e];   // every element of the tile, in tile order
        sq = fmaf(x, x, sq);
      }
      const float ns = block_sum(sq);      // contains __syncthreads: D5 drain writes are visible
      float bound = sqrtf(ns);
      for (int t = 0; t < c; ++t) bound = fmaf(misc[Cf::M_VN + t], sqrtf(fmaxf(misc[Cf::M_AN + t], 0.f)), bound);
      const bool exact = !(bound <= a.tau * (1.f - 0x1p-12f));
      if (!exact) {
        if (tid < 64) {
          misc[Cf::M_SG + tid] = 1.f;   // sigma after step t
          misc[Cf::M_IS + tid] = 1.f;   // 1 / sigma before step t
        }
      } else {
        float* VV = sf + Cf::F_Q + TILE;   // v_t . v_t' for t, t' < c  ([C][C])
        for (int e = tid; e < C * C; e += NT) {
          const int t = e / C, tp = e - t * C;
          float vv = 0.f;
          if (t < c && tp < c) {
            for (int i = 0; i < 64; ++i) vv = fmaf(to_f32(vb[t * 64 + i]), to_f32(vb[tp * 64 + i]), vv);
          }
          VV[e] = vv;
        }
        __syncthreads();
        if (tid == 0) {
          // S_t = sigma_t S_reg,t with S_reg,t = S_0 + sum_{t'<=t} v_t' alpha_t'^T / sigma_{t'-1}.
          // The norms are tracked unscaled (bounded by about tau), the cross terms through
          // the ratios sigma_{t-1} / sigma_{t'-1} <= 1, so nothing overflows however small
          // sigma gets.  Below 2^-64 the folded operands of G6 would grow past 2^64: the
          // chunk's S then goes step by step instead.
          float n2 = ns, sg = 1.f;          // ||S_{t-1}||^2 and sigma_{t-1}
          unsigned int rc = 0;
          int deep_at = 0;
          const float* AA = sf + Cf::F_Q;   // alpha Gram [C][C]
          for (int t = 0; t < c; ++t) {
            misc[Cf::M_IS + t] = 1.f / sg;
            float cross = sg * misc[Cf::M_XS + t];   // sigma_{t-1} v_t^T S_reg,t-1 alpha_t
            for (int tp = 0; tp < t; ++tp)
              cross = fmaf(VV[t * C + tp] * AA[t * C + tp], sg * misc[Cf::M_IS + tp], cross);
            const float vn = misc[Cf::M_VN + t];
            const float npre2 = fmaf(vn * vn, AA[t * C + t], fmaf(2.f, cross, n2));
            const float npre = sqrtf(fmaxf(npre2, 0.f));
            if (npre > a.tau) {
              sg *= a.tau / npre;
              n2 = a.tau * a.tau;
              ++rc;
            } else {
              n2 = npre2;
            }
            if (!isfinite(npre)) flags |= kStatusNonfinite;
            misc[Cf::M_SG + t] = sg;
            if (!(sg >= 0x1p-64f)) { deep_at = 1; break; }
          }
          if (!deep_at) renorm_cnt += rc;
          misc[Cf::M_SCAL] = deep_at ? 1.f : 0.f;
          for (int t = c; t < 64; ++t) {
            misc[Cf::M_SG + t] = sg;
            misc[Cf::M_IS + t] = 1.f / sg;
          }
        }
        __syncthreads();
        if (misc[Cf::M_SCAL] != 0.f) {
          // S and the outputs step by step with the chunk's alpha (A and alpha are final)
          const int row = tid >> 2, cq = tid & 3;
          for (int t = 0; t < c; ++t) {
            const float vr = to_f32(vb[t * 64 + row]);
            float sq = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = 16 * cq + j;
              float& sr = sf[Cf::F_S + tk_off(row, col, 64)];
              sr = fmaf(vr, sf[Cf::F_AL + tk_off(t, col, 64)], sr);
              sq = fmaf(sr, sr, sq);
            }
            const float nrm = sqrtf(block_sum(sq));
            if (nrm > a.tau) {
              const float cf = a.tau / nrm;
#pragma unroll
              for (int j = 0; j < 16; ++j) sf[Cf::F_S + tk_off(row, 16 * cq + j, 64)] *= cf;
              if (tid == 0) ++renorm_cnt;
            }
            if (!isfinite(nrm)) flags |= kStatusNonfinite;
            float op = 0.f;   // o_t = S_t phi(q_t) / den_t (the thread's own S elements)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              op = fmaf(sf[Cf::F_S + tk_off(row, 16 * cq + j, 64)], sf[Cf::F_PQ + tk_off(t, 16 * cq + j, 64)], op);
            op += __shfl_xor_sync(0xffffffffu, op, 1);
            op += __shfl_xor_sync(0xffffffffu, op, 2);
            if (cq == 0) go[(pos + t) * D + row] = from_f32<TIO>(op * misc[Cf::M_RDEN + t]);
          }
          tc::fence_before_sync();
          __syncthreads();
          pos += c;
          continue;
        }
        // fold the per-step scales into tril(aq) (columns t') and alpha^T (columns t)
        for (int e = tid; e < 64 * C; e += NT) {
          const int r = e / C, k = e - r * C;
          const float is = misc[Cf::M_IS + k];
          sf[Cf::F_T6 + tk_off(r, k, C)] *= is;
          sf[Cf::F_T6 + 2 * Cf::T6T + tk_off(r, k, C)] *= is;
        }
      }
    }
    // ---------------- G6: [tril(aq) V ; V^T alpha] = [tril(aq); V^T] [V^T; alpha^T]^T  (M 128, N 128, K C)
    if (!gemm(Cf::F_T6, Cf::F_T6 + Cf::T6T, 128, 128, C)) { failed = true; break; }
    {
      float v[16];
      const int row = 32 * q4 + lane;
      const float sgl = misc[Cf::M_SG + c - 1];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int col0 = 64 * half + 16 * cc;
        if ((row < 64) != (half == 0)) continue;   // only the two useful blocks
        tld(col0, v);
        if (row < 64) {   // outputs of step t
          const int t = row;
          if (t < c) {
            const float sgt = misc[Cf::M_SG + t], rd = misc[Cf::M_RDEN + t];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int i = col0 + j;
              const float o = sgt * (sf[Cf::F_P + t * 64 + i] + v[j]) * rd;
              if (!isfinite(o)) flags |= kStatusNonfinite;
              go[(pos + t) * D + i] = from_f32<TIO>(o);
            }
          }
        } else {          // S_1 = sigma (S + V^T alpha)
          const int i = row - 64;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = col0 - 64 + j;
            float& sr = sf[Cf::F_S + tk_off(i, col, 64)];
            sr = sgl * (sr + v[j]);
          }
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    pos += c;
  }

  // ---- state out, TMEM freed
  tc::fence_before_sync();
  __syncthreads();
  if (!failed) {
    for (int e = tid; e < D * D; e += NT) {
      const int i = e >> 6, j = e & 63;
      gA[e] = sf[Cf::F_A + tk_off(i, j, 64)];
      gS[e] = sf[Cf::F_S + tk_off(i, j, 64)];
    }
    if (tid < D) gn[tid] = n_i;
  } else if (tid == 0) {
    flags |= kStatusTimeout;
    if (loaded + 1 < ntiles) (void)mbar_wait_bounded(in_bar, (uint32_t)((loaded + 1) & 1));
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
  if (flags) atomicOr(&a.status->flags, flags);
  if (tid == 0) {
    if (guard_cnt) atomicAdd(&a.status->guard_count, guard_cnt);
    if (renorm_cnt) atomicAdd(&a.status->renorm_count, renorm_cnt);
    if (fallback_cnt) atomicAdd(&a.status->chunk_fallbacks, fallback_cnt);
  }
}

template <int R, typename TIO>
cudaError_t launch_chunk_t(const ScanArgs& a, cudaStream_t s) {
  using Cf = chk::Cfg<R, TIO>;
  auto kern = chunk_scan_kernel<R, TIO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.pairs, chk::NT, Cf::bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vla
