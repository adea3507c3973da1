// Blocked, warp-specialised sequential VLA scan for sm_103a.
//
// The recurrence ("Mathematical Primitives" §2-§5, README "VLA v3" items 1-5)
// is taken KS steps (M = KS r directions) per reduction round in exact
// Woodbury form ("Mathematical Primitives" §3 names the identity; the
// gist.science summary §2.4 the parallel formulation).  With A_0 the inverse at
// the start of a round and U = [u_1 .. u_M]:
//
//   P = A_0 U,  Q_t = A_0 s_t,  G = I + U^T P = L D L^T   (D_jj = the sequential deltas)
//   A_after  = A_0 - P G^{-1} P^T                            (= the M rank-1 updates)
//   alpha_t  = Q_t - P_{<=e_t} G_{<=e_t}^{-1} (U^T Q_t)_{<=e_t}   (e_t: last direction of step t)
//
// One round needs M + KS products with A_0 (as many as the step-by-step form)
// but one set of reductions instead of M.
//
// One CTA per (batch, head) pair, two warp groups of 2d threads each:
//   A group  owns A in registers; per round: products with A_0 (packed FFMA2),
//            reduce-scatter over the 8 lanes of a row group, Gram scalars
//            (u_a.P_b, u_a.Q_t) as dot products, LDL^T of G in registers,
//            A update, alpha (one writer per element) -> shared memory.
//   S group  owns S in registers and lags one round: S phi(q) products, the
//            scalars alpha_t'.phi(q_t) and |alpha_t|^2, renormalisation, the
//            outputs o_t = (S_0 phi(q_t) + sum_{t'<=t} v_t'(alpha_t'.phi(q_t))) / den_t
//            and S += v alpha^T.
// Each SM sub-partition runs one warp of each group, so one group's reduction
// latency hides behind the other's arithmetic.  alpha is handed over through a
// double-buffered shared array guarded by per-parity named barriers
// (FULL[p]: A arrives, S syncs; EMPTY[p]: S arrives, A syncs), so neither side
// can run two rounds ahead of the other.
//
// Singularity guard: a pivot |D_jj| < 1e-6 means the sequential recurrence would
// take the guard at that direction.  The round then applies nothing and its
// directions are replayed one per round, where the pivot is the sequential
// delta itself and the guard (A += 1e-6 I instead of the update) is taken as the
// pages state it.
//
// Delta-rule variant (DL = true; gist.science summary §2.3): the same A group; the S
// group also forms X_t = S_reg s_t and the scalars alpha_t' . s_t, solves the round's
// residuals w_t = v_t - S_{t-1} k_hat_t row by row, and writes S += w alpha_hat^T.
//
// Renormalisation: S = sigma * S_reg (lazy scale).  Each round reduces ||S_reg||^2
// exactly; with |alpha_t| and |v_t| the bound ||S_t|| <= ||S_0|| + sum |v||alpha| shows
// that no step of the chunk can exceed tau.  Otherwise an extra reduction gives the
// exact per-step norms from ||S_t||^2 = ||S_{t-1}||^2 + 2 v_t^T S_{t-1} alpha_t + |v_t|^2|alpha_t|^2
// and the decisions are taken step by step.
#pragma once

#include <type_traits>

#include "vla_internal.cuh"

namespace vla {

namespace blk {

constexpr float kGuardEps = 1e-6f;
constexpr float kReadoutEps = 1e-6f;
constexpr float kNormEps = 1e-12f;   // floor of |alpha| and |s| in the delta rule's unit vectors
// named barriers (0 is __syncthreads)
constexpr int BAR_A = 1, BAR_S = 2, BAR_FULL0 = 3, BAR_EMPTY0 = 5;

__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__host__ __device__ constexpr int pow2_ceil(int x) { return x <= 1 ? 1 : 2 * pow2_ceil((x + 1) / 2); }
__host__ __device__ constexpr int log2i(int x) { return x <= 1 ? 0 : 1 + log2i(x / 2); }
__host__ __device__ constexpr int up2(int x) { return (x + 1) / 2 * 2; }
__host__ __device__ constexpr int up4(int x) { return (x + 3) / 4 * 4; }

template <int D>
struct Geom {
  static constexpr int RPT = (D == 16) ? 2 : 4;   // rows per thread
  static constexpr int LPR = (D == 16) ? 4 : 8;   // lanes per row group
  static constexpr int CPT = D / LPR;             // columns per thread
  static constexpr int NCH = CPT / 4;             // float4 pieces per vector
  static constexpr int NCP = CPT / 2;             // float2 pairs per row piece
  static constexpr int NG = D / RPT;              // row groups
  static constexpr int GT = NG * LPR;             // threads per warp group (2 d)
  static constexpr int GW = GT / 32;              // warps per group
  static constexpr int NT = 2 * GT;               // threads per CTA
  static constexpr int NSTAGE = 2;
  static_assert(GT == 2 * D && GT % 32 == 0, "two threads per element of a d-vector");
};

template <int D, int R, int KS, typename TIO>
__host__ __device__ constexpr size_t smem_bytes_for(int ts) {
  return (size_t)Geom<D>::NSTAGE * ts * (3 * D + R * D) * sizeof(TIO) +
         sizeof(float) * ((size_t)2 * ts * ((R + 3) * D + 4) + (size_t)ts * D + 4096 + 10 * KS * D * R);
}
template <int D, int R, int KS, typename TIO>
__host__ __device__ constexpr int pick_ts() {
  return smem_bytes_for<D, R, KS, TIO>(32) <= 200 * 1024 ? 32
         : smem_bytes_for<D, R, KS, TIO>(16) <= 200 * 1024 ? 16 : 8;
}

template <int D, int R, int KS, typename TIO, bool DL = false>
struct Cfg {
  using Gm = Geom<D>;
  static constexpr int TS = pick_ts<D, R, KS, TIO>();   // steps per tile
  static constexpr int M = KS * R;                      // directions per round
  static constexpr int NVA = up2(M + KS);               // A-group vectors (P, Q, zero padding)
  static constexpr int NVY = DL ? 2 * KS : KS;          // S-group products: Y (and X = S_reg s_t, delta rule)
  static constexpr int NVS = up2(NVY);                  // S-group vectors (zero padding)
  static constexpr int KVA = Gm::RPT * NVA / Gm::LPR;   // values a lane keeps after the reduce-scatter
  static constexpr int KVS = Gm::RPT * NVS / Gm::LPR;
  static_assert((Gm::RPT * NVA) % Gm::LPR == 0 && (Gm::RPT * NVS) % Gm::LPR == 0, "even split");
  // dot-product jobs
  static constexpr int NJG = M * (M + 1) / 2;           // u_a . P_b, a <= b
  static constexpr int NJH = R * KS * (KS + 1) / 2;     // u_a . Q_t, a <= e_t
  static constexpr int NJA = NJG + NJH;
  static constexpr int NJQ = KS * (KS + 1) / 2;         // alpha_t' . phi(q_t), t' <= t
  static constexpr int NJS = NJQ + KS + (DL ? NJQ : 0); // + alpha_t . alpha_t (+ alpha_t' . s_t, t' <= t)
  static constexpr int NSA = pow2_ceil((NJA + Gm::GW - 1) / Gm::GW);   // job slots per A warp
  static constexpr int NSS = pow2_ceil((NJS + Gm::GW - 1) / Gm::GW);
  static_assert(NSA <= 32 && NSS <= 32, "one pass of job slots");
  // exact-norm scalars.  Additive: v_t^T S alpha_t, alpha_t . alpha_t', v_t . v_t' (t' <= t).
  // Delta rule: v_m^T S alpha_t, X_m^T S alpha_t (all m, t), v_m . X_m' (all), v_m . v_m',
  // X_m . X_m', alpha_t . alpha_t' (m' <= m, t' <= t).
  static constexpr int NTRI = KS * (KS + 1) / 2;
  static constexpr int NMINI = DL ? 3 * KS * KS + 3 * NTRI : KS + KS * (KS + 1);
  static constexpr int MI_VSA = 0, MI_XSA = KS * KS, MI_VX = 2 * KS * KS, MI_VV = 3 * KS * KS,
                       MI_XX = 3 * KS * KS + NTRI, MI_AA = 3 * KS * KS + 2 * NTRI;
  static constexpr int MSTR = up4(NMINI);
  // step record (floats): u[R][D] | s[D] | phi(q)[D] | v[D] | 1/den, |v|, |s|, 0
  static constexpr int OFF_U = 0, OFF_S = R * D, OFF_Q = (R + 1) * D, OFF_V = (R + 2) * D;
  static constexpr int OFF_SC = (R + 3) * D;
  static constexpr int REC = (R + 3) * D + 4;
  static constexpr uint32_t QB = TS * D * sizeof(TIO);
  static constexpr uint32_t UB = TS * R * D * sizeof(TIO);
  static constexpr uint32_t STAGE = 3 * QB + UB;
  // shared memory map (float offsets after the raw ring)
  static constexpr int F_PRE = 0;                          // [2][TS][REC]
  static constexpr int F_ZERO = F_PRE + 2 * TS * REC;      // [REC]   ghost step: zeros, 1/den = 1
  static constexpr int F_PROD = F_ZERO + REC;              // [TS][D] prologue scratch
  static constexpr int F_P = F_PROD + TS * D;              // [2][M][D]
  static constexpr int F_Q = F_P + 2 * M * D;              // [2][KS][D]
  static constexpr int F_Y = F_Q + 2 * KS * D;             // [2][NVY][D]
  static constexpr int F_AL = F_Y + 2 * NVY * D;           // [2][KS][D]
  static constexpr int F_RA = F_AL + 2 * KS * D;           // [NJA]
  static constexpr int F_RS = F_RA + up4(NJA);             // [NJS]
  static constexpr int F_WP = F_RS + up4(NJS);             // [2][GW]
  static constexpr int F_MINI = F_WP + up4(2 * Gm::GW);    // [GW][MSTR]
  static constexpr int F_INFO = F_MINI + Gm::GW * MSTR;    // [2][8] ints
  static constexpr int F_END = F_INFO + 16;
  static constexpr size_t raw_bytes = (size_t)Gm::NSTAGE * STAGE;
  static constexpr size_t bar_off = raw_bytes + sizeof(float) * (size_t)F_END;
  static constexpr size_t bytes = bar_off + 16 * Gm::NSTAGE + 16 + 32;   // + FULL[2], EMPTY[2] (cluster mode)
  static_assert(QB % 16 == 0 && UB % 16 == 0 && REC % 4 == 0, "alignment");
  static_assert(TS % KS == 0, "chunks must tile a tile");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

// Reduce-scatter of N values across the lanes selected by masks LM, LM/2, .., 1:
// afterwards lane position blk (its bits under those masks) holds the full sums
// of slots [blk*N/L, (blk+1)*N/L) in v[0 .. N/L).
template <int N, int LM>
__device__ __forceinline__ void reduce_scatter(float (&v)[N], int lanebits) {
  int n = N;
#pragma unroll
  for (int m = LM; m >= 1; m >>= 1) {
    if (n < 2) break;
    const bool hi = (lanebits & m) != 0;
    const int h = n / 2;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      if (i < h) {
        const float send = hi ? v[i] : v[i + h];
        const float keep = hi ? v[i + h] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
    n = h;
  }
}

}  // namespace blk

// PS = false: status accumulates into a.status (one block per call);
// PS = true:  into a.pair_status[pair] (one record per pair).
// CL = false: one CTA per pair holds both warp groups;
// CL = true:  a cluster of two CTAs per pair: CTA 0 runs the A group, CTA 1 the S
//             group, each on its own SM.  Both CTAs stream and convert the inputs;
//             alpha and the round record go from CTA 0 into CTA 1's shared memory
//             (distributed shared memory), and the FULL / EMPTY hand-off becomes a
//             pair of cluster-scope mbarriers per parity (every thread of the
//             producing group arrives with release semantics; waits are bounded).
template <int D, int R, int KS, typename TIO, bool PS = false, bool CL = false, bool DL = false>
__global__ void __launch_bounds__(CL ? blk::Geom<D>::GT : blk::Geom<D>::NT, 1) seq_block_kernel(ScanArgs a) {
  using namespace blk;
  using Gm = Geom<D>;
  using C = Cfg<D, R, KS, TIO, DL>;
  constexpr int RPT = Gm::RPT, LPR = Gm::LPR, NCH = Gm::NCH, NCP = Gm::NCP, GT = Gm::GT, GW = Gm::GW;
  constexpr int NT = CL ? Gm::GT : Gm::NT, TS = C::TS, NSTAGE = Gm::NSTAGE;
  static_assert(!(PS && CL), "the per-pair status entry point runs one CTA per pair");
  constexpr int M = C::M, REC = C::REC;
  constexpr float kInvSqrtD = (float)(D == 16 ? 0.25 : D == 64 ? 0.125 : 0.08838834764831845);

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* raw = smem;
  float* sf = reinterpret_cast<float*>(smem + C::raw_bytes);
  int* info = reinterpret_cast<int*>(sf + C::F_INFO);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bar_off);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::bar_off + 16 * NSTAGE);
  uint64_t* hb = reinterpret_cast<uint64_t*>(smem + C::bar_off + 16 * NSTAGE + 16);   // FULL[2], EMPTY[2]

  const int tid = threadIdx.x;
  const uint32_t crank = CL ? cluster_ctarank() : 0u;
  const bool isA = CL ? (crank == 0) : (tid < GT);
  const int gid = CL ? tid : (isA ? tid : tid - GT);   // thread index within its group
  const int lane = tid & 31, gw = gid >> 5;      // warp within the group
  const int g = gid / LPR, c = gid % LPR;        // row group, lane within it
  const int row0 = g * RPT;
  const long long pair = CL ? (long long)(blockIdx.x >> 1) : (long long)blockIdx.x;
  const long long T = a.T;

  const TIO* gq = static_cast<const TIO*>(a.q) + pair * T * D;
  const TIO* gk = static_cast<const TIO*>(a.k) + pair * T * D;
  const TIO* gv = static_cast<const TIO*>(a.v) + pair * T * D;
  const TIO* gu = static_cast<const TIO*>(a.u) + pair * T * R * D;
  TIO* go = static_cast<TIO*>(a.o) + pair * T * D;
  float* gA = a.A + pair * D * D;
  float* gS = a.S + pair * D * D;
  float* gn = a.n + pair * D;

  auto colof = [&](int kk, int e) { return 4 * c + 4 * LPR * kk + e; };

  for (int e = tid; e < REC; e += NT) sf[C::F_ZERO + e] = (e == C::OFF_SC) ? 1.f : 0.f;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    if constexpr (CL) {
      for (int p = 0; p < 4; ++p) mbar_init(&hb[p], GT);   // every thread of the producing group arrives
    }
    fence_mbar_init();
    *flag = 0;
  }
  __syncthreads();
  if constexpr (CL) cluster_sync_all();   // the peer's barriers are initialised before any arrival
  // cluster hand-off: FULL[p] lives in CTA 1 (A arrives, S waits), EMPTY[p] in CTA 0
  // (S arrives, A waits); alpha and the round record are stored into CTA 1
  const uint32_t peer = crank ^ 1u;
  auto remote = [&](const void* local) -> uint32_t { return mapa_shared(smem_u32(local), peer); };

  const int ntiles = (int)((T + TS - 1) / TS);
  auto issue = [&](int tile) {  // thread 0 only
    const int stage = tile % NSTAGE;
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const uint32_t qb = (uint32_t)nst * D * sizeof(TIO);
    const uint32_t ub = (uint32_t)nst * R * D * sizeof(TIO);
    unsigned char* base = raw + stage * C::STAGE;
    mbar_arrive_expect_tx(&bars[stage], 3 * qb + ub);
    bulk_g2s(base, gq + t_start * D, qb, &bars[stage]);
    bulk_g2s(base + C::QB, gk + t_start * D, qb, &bars[stage]);
    bulk_g2s(base + 2 * C::QB, gv + t_start * D, qb, &bars[stage]);
    bulk_g2s(base + 3 * C::QB, gu + t_start * R * D, ub, &bars[stage]);
  };
  if (tid == 0) {
    for (int j = 0; j < NSTAGE && j < ntiles; ++j) issue(j);
  }

  // per-tile prologue (the A group's, and in cluster mode also the S group's on its
  // own CTA): float32 records, 1/den_t, |v_t|
  auto prologue = [&](int tile, float& n_i, int gbar) -> bool {
    const int stage = tile % NSTAGE;
    if (gid == 0) {
      if (!mbar_wait_bounded(&bars[stage], (uint32_t)((tile / NSTAGE) & 1))) *flag = 1;
    }
    bar_sync(gbar, GT);
    if (*flag) return false;
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const TIO* rq = reinterpret_cast<const TIO*>(raw + stage * C::STAGE);
    const TIO* rk = reinterpret_cast<const TIO*>(raw + stage * C::STAGE + C::QB);
    const TIO* rv = reinterpret_cast<const TIO*>(raw + stage * C::STAGE + 2 * C::QB);
    const TIO* ru = reinterpret_cast<const TIO*>(raw + stage * C::STAGE + 3 * C::QB);
    float* pre = sf + C::F_PRE + (tile & 1) * TS * REC;
    float* prod = sf + C::F_PROD;
    for (int e4 = gid; e4 < nst * R * D / 4; e4 += GT) {
      const int e = 4 * e4, t = e / (R * D), off = e - t * (R * D);
      const float4 x = make_float4(to_f32(ru[e]), to_f32(ru[e + 1]), to_f32(ru[e + 2]), to_f32(ru[e + 3]));
      *reinterpret_cast<float4*>(pre + t * REC + C::OFF_U + off) = x;
    }
    for (int e4 = gid; e4 < nst * D / 4; e4 += GT) {
      const int e = 4 * e4, t = e / D, i = e - t * D;
      float* rec = pre + t * REC;
      float kx[4], qx[4], vx[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        kx[j] = phi_elu1(to_f32(rk[e + j]));
        qx[j] = phi_elu1(to_f32(rq[e + j]));
        vx[j] = to_f32(rv[e + j]);
      }
      *reinterpret_cast<float4*>(rec + C::OFF_S + i) =
          make_float4(kx[0] * kInvSqrtD, kx[1] * kInvSqrtD, kx[2] * kInvSqrtD, kx[3] * kInvSqrtD);
      *reinterpret_cast<float4*>(rec + C::OFF_Q + i) = make_float4(qx[0], qx[1], qx[2], qx[3]);
      *reinterpret_cast<float4*>(rec + C::OFF_V + i) = make_float4(vx[0], vx[1], vx[2], vx[3]);
      *reinterpret_cast<float4*>(prod + e) = make_float4(kx[0], kx[1], kx[2], kx[3]);
    }
    bar_sync(gbar, GT);
    if (gid < D) {   // n_t = n_{t-1} + phi(k_t); products n_t[i] phi(q_t)[i] in place of phi(k)
      for (int t = 0; t < nst; ++t) {
        n_i += prod[t * D + gid];
        prod[t * D + gid] = n_i * pre[t * REC + C::OFF_Q + gid];
      }
    }
    bar_sync(gbar, GT);
    {  // 1/den_t and |v_t|: TPS threads per step
      constexpr int TPS = GT / TS >= 1 ? GT / TS : 1;
      constexpr int EPT = D / TPS;
      static_assert(EPT % 4 == 0 && TPS <= 32, "den reduction layout");
      const int t = gid / TPS, part = gid - t * TPS;
      float dn = 0.f, vv = 0.f, ss = 0.f;
      if (t < nst) {
#pragma unroll
        for (int j = 0; j < EPT; j += 4) {
          const float4 p = *reinterpret_cast<const float4*>(prod + t * D + part * EPT + j);
          const float4 w = *reinterpret_cast<const float4*>(pre + t * REC + C::OFF_V + part * EPT + j);
          dn += (p.x + p.y) + (p.z + p.w);
          vv = fmaf(w.x, w.x, fmaf(w.y, w.y, fmaf(w.z, w.z, fmaf(w.w, w.w, vv))));
          if constexpr (DL) {
            const float4 k4 = *reinterpret_cast<const float4*>(pre + t * REC + C::OFF_S + part * EPT + j);
            ss = fmaf(k4.x, k4.x, fmaf(k4.y, k4.y, fmaf(k4.z, k4.z, fmaf(k4.w, k4.w, ss))));
          }
        }
      }
      // every lane of the warp takes part in the shuffles (a ragged tile leaves
      // some lanes without a step)
#pragma unroll
      for (int m = TPS / 2; m >= 1; m >>= 1) {
        dn += __shfl_xor_sync(0xffffffffu, dn, m);
        vv += __shfl_xor_sync(0xffffffffu, vv, m);
        if constexpr (DL) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      }
      if (t < nst && part == 0) {
        pre[t * REC + C::OFF_SC] = __frcp_rn(dn + kReadoutEps);
        pre[t * REC + C::OFF_SC + 1] = sqrtf(vv);
        if constexpr (DL) pre[t * REC + C::OFF_SC + 2] = sqrtf(ss);
      }
    }
    bar_sync(gbar, GT);
    if (gid == 0 && tile + NSTAGE < ntiles) {
      fence_proxy_async_smem();
      issue(tile + NSTAGE);
    }
    return true;
  };

  unsigned int flags = 0;

  if (isA) {
    // =====================================================================
    // A group
    // =====================================================================
    float2 A2[RPT][NCP];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
#pragma unroll
      for (int kk = 0; kk < NCH; ++kk) {
        const float4 av = *reinterpret_cast<const float4*>(gA + (row0 + r) * D + colof(kk, 0));
        A2[r][2 * kk] = f2(av.x, av.y);
        A2[r][2 * kk + 1] = f2(av.z, av.w);
      }
    float n_i = (gid < D) ? gn[gid] : 0.f;

    long long pos = 0;
    bool replay = false;
    long long rep_pos = 0;
    int rep_total = 0, rep_col = 0;
    int loaded = -1;
    unsigned long long guard_cnt = 0, replay_cnt = 0;
    int par = 0;
    int rnd = 0;
    while (true) {
      if (rnd >= 2) {   // S is done with round rnd-2
        if constexpr (CL) {
          if (!mbar_wait_cluster_bounded(&hb[2 + (rnd & 1)], (uint32_t)(((rnd - 2) >> 1) & 1))) {
            flags |= kStatusTimeout;
            *flag = 1;
          }
        } else {
          bar_sync(BAR_EMPTY0 + (rnd & 1), NT);
        }
      }
      // ---------------- schedule this round's chunk
      int cA = 0, rep_j = 0;
      bool rep_completes = false, nudgeA = false, haveA = false;
      long long gA0 = 0, a_step = 0;
      if (replay) {
        const long long st = rep_pos + rep_col / R;
        rep_j = rep_col % R;
        rep_completes = (rep_j == R - 1);
        a_step = st;
        gA0 = st;
        cA = rep_completes ? 1 : 0;
        haveA = true;
        if (rep_completes && a.P > 0) nudgeA = ((a.t0 + st + 1) % a.P) == 0;
      } else if (pos < T) {
        long long cmax = min((long long)KS, T - pos);
        cmax = min(cmax, (long long)(TS - (int)(pos % TS)));
        if (a.P > 0) {
          const long long to_nudge = a.P - ((a.t0 + pos) % a.P);
          if (to_nudge <= cmax) { cmax = to_nudge; nudgeA = true; }
        }
        cA = (int)cmax;
        gA0 = pos;
        a_step = pos;
        haveA = true;
      }
      bool stop = !haveA || (CL && *flag != 0);
      if (haveA) {
        const int tile = (int)(a_step / TS);
        if (tile != loaded) {
          if (!prologue(tile, n_i, BAR_A)) {
            stop = true;
            flags |= kStatusTimeout;
          }
          loaded = tile;
        }
      }
      if (stop) {   // publish the end of the sequence to the S group
        if (gid == 0) {
          int* inf = info + (rnd & 1) * 8;
          if constexpr (CL) {
            for (int q = 0; q < 4; ++q) st_cluster_s32(remote(inf + q), 0);
            st_cluster_s32(remote(inf + 4), 1);
          } else {
            inf[0] = 0; inf[1] = 0; inf[2] = 0; inf[3] = 0; inf[4] = 1;
          }
        }
        if constexpr (CL) mbar_arrive_remote(remote(&hb[rnd & 1]));
        else bar_arrive(BAR_FULL0 + (rnd & 1), NT);
        ++rnd;
        break;
      }
      const int baseA = C::F_PRE + ((int)(a_step / TS) & 1) * TS * REC + (int)(a_step % TS) * REC;
      auto offU = [&](int col) -> int {
        if (replay) return (col == 0) ? baseA + C::OFF_U + rep_j * D : C::F_ZERO;
        const int t = col / R;
        return (t < cA) ? baseA + t * REC + C::OFF_U + (col - t * R) * D : C::F_ZERO;
      };
      auto recA = [&](int t) -> int {
        if (replay) return (t == 0 && rep_completes) ? baseA : C::F_ZERO;
        return (t < cA) ? baseA + t * REC : C::F_ZERO;
      };
      const int pbuf = C::F_P + par * M * D, qbuf = C::F_Q + par * KS * D;
      const int abuf = C::F_AL + (rnd & 1) * KS * D;

      // ---------------- phase P: P = A_0 U, Q = A_0 Sigma (row pieces)
      {
        float vals[RPT * C::NVA];
        {
          float2 acc[RPT][C::NVA];
#pragma unroll
          for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int v = 0; v < C::NVA; ++v) acc[r][v] = f2(0.f, 0.f);
#pragma unroll
          for (int v = 0; v < M + KS; ++v) {
            const int base = (v < M) ? offU(v) : recA(v - M) + C::OFF_S;
#pragma unroll
            for (int kk = 0; kk < NCH; ++kk) {
              const float4 x = *reinterpret_cast<const float4*>(sf + base + colof(kk, 0));
              const float2 x0 = f2(x.x, x.y), x1 = f2(x.z, x.w);
#pragma unroll
              for (int r = 0; r < RPT; ++r) {
                acc[r][v] = __ffma2_rn(A2[r][2 * kk], x0, acc[r][v]);
                acc[r][v] = __ffma2_rn(A2[r][2 * kk + 1], x1, acc[r][v]);
              }
            }
          }
#pragma unroll
          for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int v = 0; v < C::NVA; ++v) vals[r * C::NVA + v] = acc[r][v].x + acc[r][v].y;
        }
        reduce_scatter<RPT * C::NVA, LPR / 2>(vals, c);
#pragma unroll
        for (int i = 0; i < C::KVA; ++i) {
          const int slot = c * C::KVA + i;
          const int r = slot / C::NVA, v = slot - r * C::NVA;
          if (v < M) sf[pbuf + v * D + row0 + r] = vals[i];
          else if (v < M + KS) sf[qbuf + (v - M) * D + row0 + r] = vals[i];
        }
      }
      bar_sync(BAR_A, GT);
      // ---------------- phase G: u_a . P_b (a <= b), u_a . Q_t (a <= e_t)
      {
        auto jobs = [&](auto wtag) {
          constexpr int W = decltype(wtag)::value;
          float jv[C::NSA];
#pragma unroll
          for (int s = 0; s < C::NSA; ++s) {
            const int j = s * GW + W;   // compile-time job index
            float acc = 0.f;
            if (j < C::NJA) {
              int oa, ob;
              if (j < C::NJG) {
                int b = 0;
#pragma unroll
                for (int bb = 1; bb < M; ++bb) b += (j >= bb * (bb + 1) / 2) ? 1 : 0;
                oa = offU(j - b * (b + 1) / 2);
                ob = pbuf + b * D;
              } else {
                const int h = j - C::NJG;
                int t = 0;
#pragma unroll
                for (int tt = 1; tt < KS; ++tt) t += (h >= R * tt * (tt + 1) / 2) ? 1 : 0;
                oa = offU(h - R * t * (t + 1) / 2);
                ob = qbuf + t * D;
              }
              if (D >= 32) {
#pragma unroll
                for (int e = 0; e < D / 32; ++e) acc = fmaf(sf[oa + lane + 32 * e], sf[ob + lane + 32 * e], acc);
              } else if (lane < D) {
                acc = sf[oa + lane] * sf[ob + lane];
              }
            }
            jv[s] = acc;
          }
          reduce_scatter<C::NSA, 16>(jv, lane);
          float x = jv[0];
#pragma unroll
          for (int m = 32 / C::NSA / 2; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
          constexpr int SH = 5 - log2i(C::NSA);
          const int j = (lane >> SH) * GW + W;
          if ((lane & ((1 << SH) - 1)) == 0 && j < C::NJA) sf[C::F_RA + j] = x;
        };
        switch (gw) {
          case 0: jobs(std::integral_constant<int, 0>{}); break;
          case 1: if constexpr (GW > 1) jobs(std::integral_constant<int, 1>{}); break;
          case 2: if constexpr (GW > 2) jobs(std::integral_constant<int, 2>{}); break;
          case 3: if constexpr (GW > 3) jobs(std::integral_constant<int, 3>{}); break;
          case 4: if constexpr (GW > 4) jobs(std::integral_constant<int, 4>{}); break;
          case 5: if constexpr (GW > 5) jobs(std::integral_constant<int, 5>{}); break;
          case 6: if constexpr (GW > 6) jobs(std::integral_constant<int, 6>{}); break;
          case 7: if constexpr (GW > 7) jobs(std::integral_constant<int, 7>{}); break;
          default: break;
        }
      }
      bar_sync(BAR_A, GT);
      // ---------------- phase U: LDL^T of G, A update, alpha
      {
        float res[C::NJA];
#pragma unroll
        for (int j = 0; j < C::NJA; ++j) res[j] = sf[C::F_RA + j];
        float Lm[M][M], Dv[M], iD[M];
        bool bad = false;
#pragma unroll
        for (int j = 0; j < M; ++j) {
          float dj = res[j * (j + 1) / 2 + j] + 1.f;
#pragma unroll
          for (int k = 0; k < j; ++k) dj = fmaf(-Lm[j][k] * Dv[k], Lm[j][k], dj);
          Dv[j] = dj;
          bad = bad || !(fabsf(dj) >= kGuardEps);
          iD[j] = __frcp_rn(dj);
#pragma unroll
          for (int i = j + 1; i < M; ++i) {
            float x = res[i * (i + 1) / 2 + j];
#pragma unroll
            for (int k = 0; k < j; ++k) x = fmaf(-Lm[i][k] * Dv[k], Lm[j][k], x);
            Lm[i][j] = x * iD[j];
          }
        }
        if (!isfinite(Dv[0])) flags |= kStatusNonfinite;
        const bool guard = replay && bad;            // replay rounds hold one real direction
        const bool apply = !bad || replay;
        if (bad && !replay) {                        // replay this chunk one direction per round
          replay = true;
          rep_pos = gA0;
          rep_total = cA * R;
          rep_col = 0;
          ++replay_cnt;
        }
        float Li[M][M];
#pragma unroll
        for (int i = 0; i < M; ++i) {
#pragma unroll
          for (int j = 0; j < M; ++j) Li[i][j] = (i == j) ? 1.f : 0.f;
#pragma unroll
          for (int j = 0; j < i; ++j) {
            float x = 0.f;
#pragma unroll
            for (int k = j; k < i; ++k) x = fmaf(-Lm[i][k], Li[k][j], x);
            Li[i][j] = x;
          }
        }
        if (apply) {
          if (!guard) {
            float Gi[M][M];
#pragma unroll
            for (int i = 0; i < M; ++i)
#pragma unroll
              for (int j = i; j < M; ++j) {
                float x = 0.f;
#pragma unroll
                for (int k = j; k < M; ++k) x = fmaf(Li[k][i] * iD[k], Li[k][j], x);
                Gi[i][j] = x;
                Gi[j][i] = x;
              }
            float Pt[RPT][M];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
              float prow[M];
#pragma unroll
              for (int b = 0; b < M; ++b) prow[b] = sf[pbuf + b * D + row0 + r];
#pragma unroll
              for (int aa = 0; aa < M; ++aa) {
                float x = 0.f;
#pragma unroll
                for (int b = 0; b < M; ++b) x = fmaf(prow[b], Gi[b][aa], x);
                Pt[r][aa] = -x;
              }
            }
#pragma unroll
            for (int aa = 0; aa < M; ++aa) {
#pragma unroll
              for (int kk = 0; kk < NCH; ++kk) {
                const float4 pc = *reinterpret_cast<const float4*>(sf + pbuf + aa * D + colof(kk, 0));
                const float2 p0 = f2(pc.x, pc.y), p1 = f2(pc.z, pc.w);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                  const float2 w = f2(Pt[r][aa], Pt[r][aa]);
                  A2[r][2 * kk] = __ffma2_rn(w, p0, A2[r][2 * kk]);
                  A2[r][2 * kk + 1] = __ffma2_rn(w, p1, A2[r][2 * kk + 1]);
                }
              }
            }
          }
          const float dadd = (guard ? kGuardEps : 0.f) + (nudgeA ? a.eps_n : 0.f);
          if (dadd != 0.f) {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
              const int row = row0 + r;
              if (c == ((row >> 2) % LPR)) {
                const int slot = (row / (4 * LPR)) * 4 + (row & 3);
#pragma unroll
                for (int p = 0; p < NCP; ++p) {
                  if (slot == 2 * p) A2[r][p].x += dadd;
                  if (slot == 2 * p + 1) A2[r][p].y += dadd;
                }
              }
            }
          }
          if (guard) ++guard_cnt;
        }
        // alpha of the steps completed this round (zero for ghost steps); one writer per element
        {
          const int h = gid / D, i = gid - (gid / D) * D;
#pragma unroll
          for (int tt = 0; tt < KS; ++tt) {
            if ((tt & 1) != h) continue;
            float al = 0.f;
            const int rs = recA(tt);
            if (apply && rs != C::F_ZERO) {
              al = sf[qbuf + tt * D + i];
              if (!guard) {
                // c_t = G_{<=e}^{-1} (U^T Q_t)_{<=e}: forward and back substitution
                const int e = (tt + 1) * R - 1;
                float y[M];
#pragma unroll
                for (int aa = 0; aa < M; ++aa) {
                  float x = 0.f;
                  if (aa <= e) {
#pragma unroll
                    for (int b = 0; b <= aa; ++b) x = fmaf(Li[aa][b], res[C::NJG + R * tt * (tt + 1) / 2 + b], x);
                  }
                  y[aa] = x * iD[aa];
                }
#pragma unroll
                for (int aa = 0; aa < M; ++aa) {
                  if (aa <= e) {
                    float cfa = 0.f;
#pragma unroll
                    for (int b = aa; b < M; ++b)
                      if (b <= e) cfa = fmaf(Li[b][aa], y[b], cfa);
                    al = fmaf(-sf[pbuf + aa * D + i], cfa, al);
                  }
                }
              }
              const bool last = replay ? rep_completes : (tt == cA - 1);
              const float sadd = (guard ? kGuardEps : 0.f) + ((nudgeA && last) ? a.eps_n : 0.f);
              if (sadd != 0.f) al = fmaf(sadd, sf[rs + C::OFF_S + i], al);
            }
            if constexpr (CL) st_cluster_f32(remote(sf + abuf + tt * D + i), al);
            else sf[abuf + tt * D + i] = al;
          }
        }
        if (gid == 0) {
          int* inf = info + (rnd & 1) * 8;
          const int iv[5] = {apply ? cA : 0, recA(0), (int)(gA0 & 0x7fffffff), (int)(gA0 >> 31), 0};
#pragma unroll
          for (int q = 0; q < 5; ++q) {
            if constexpr (CL) st_cluster_s32(remote(inf + q), iv[q]);
            else inf[q] = iv[q];
          }
        }
        if constexpr (CL) mbar_arrive_remote(remote(&hb[rnd & 1]));
        else bar_arrive(BAR_FULL0 + (rnd & 1), NT);
        // ---------------- bookkeeping
        if (replay && apply) {
          ++rep_col;
          if (rep_col == rep_total) {
            replay = false;
            pos = rep_pos + rep_total / R;
          }
        } else if (!replay) {
          pos += cA;
        }
      }
      par ^= 1;
      ++rnd;
    }
    // rnd rounds were published, the last one the end marker.  S arrived on
    // EMPTY after each real round 0 .. rnd-2; the syncs at the top of the loop
    // matched rounds 0 .. rnd-3, so round rnd-2 is still to be matched.
    if (rnd >= 2) {
      if constexpr (CL) {
        // S's last remote access to this CTA is its EMPTY arrival for round rnd-2
        if (!mbar_wait_cluster_bounded(&hb[2 + ((rnd - 2) & 1)], (uint32_t)(((rnd - 2) >> 1) & 1)))
          flags |= kStatusTimeout;
      } else {
        bar_sync(BAR_EMPTY0 + ((rnd - 2) & 1), NT);
      }
    }
    if (!(flags & kStatusTimeout)) {
#pragma unroll
      for (int r = 0; r < RPT; ++r)
#pragma unroll
        for (int kk = 0; kk < NCH; ++kk) {
          *reinterpret_cast<float4*>(gA + (row0 + r) * D + colof(kk, 0)) =
              make_float4(A2[r][2 * kk].x, A2[r][2 * kk].y, A2[r][2 * kk + 1].x, A2[r][2 * kk + 1].y);
        }
      if (gid < D) gn[gid] = n_i;
    } else if (gid == 0) {
      for (int j = loaded + 1; j < ntiles && j <= loaded + NSTAGE; ++j)
        (void)mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)((j / NSTAGE) & 1));
    }
    if (gid == 0) {
      if constexpr (PS) {
        if (guard_cnt) atomicAdd(&a.pair_status[pair].guard_count, (unsigned int)guard_cnt);
        if (replay_cnt) atomicAdd(&a.pair_status[pair].chunk_fallbacks, (unsigned int)replay_cnt);
      } else {
        if (guard_cnt) atomicAdd(&a.status->guard_count, guard_cnt);
        if (replay_cnt) atomicAdd(&a.status->chunk_fallbacks, replay_cnt);
      }
    }
  } else {
    // =====================================================================
    // S group (one round behind)
    // =====================================================================
    float2 S2[RPT][NCP];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
#pragma unroll
      for (int kk = 0; kk < NCH; ++kk) {
        const float4 sv = *reinterpret_cast<const float4*>(gS + (row0 + r) * D + colof(kk, 0));
        S2[r][2 * kk] = f2(sv.x, sv.y);
        S2[r][2 * kk + 1] = f2(sv.z, sv.w);
      }
    float sigma = 1.f;
    unsigned long long renorm_cnt = 0;
    int par = 0;
    bool timed_out = false;
    [[maybe_unused]] float n_s = (gid < D) ? gn[gid] : 0.f;   // cluster mode: the S CTA's own records
    [[maybe_unused]] int loaded_s = -1;
    for (int rnd = 0;; ++rnd) {
      if constexpr (CL) {
        if (!mbar_wait_cluster_bounded(&hb[rnd & 1], (uint32_t)((rnd >> 1) & 1))) {
          timed_out = true;
          flags |= kStatusTimeout;
          break;
        }
      } else {
        bar_sync(BAR_FULL0 + (rnd & 1), NT);
      }
      const int* inf = info + (rnd & 1) * 8;
      const int cS = inf[0], baseS = inf[1];
      const long long gS0 = (long long)inf[2] | ((long long)inf[3] << 31);
      if (inf[4]) { timed_out = timed_out || (*flag != 0); break; }
      if constexpr (CL) {   // this CTA's copy of the round's tile
        const int tile_s = (int)(gS0 / TS);
        if (cS > 0 && tile_s != loaded_s) {
          if (!prologue(tile_s, n_s, BAR_S)) {
            timed_out = true;
            flags |= kStatusTimeout;
            break;
          }
          loaded_s = tile_s;
        }
      }
      if (cS > 0) {
        auto recS = [&](int t) -> int { return (t < cS) ? baseS + t * REC : C::F_ZERO; };
        const int ybuf = C::F_Y + par * C::NVY * D;   // Y_t at ybuf + t D (delta rule: X_t at ybuf + (KS + t) D)
        const int abuf = C::F_AL + (rnd & 1) * KS * D;
        // ---------------- phase P: Y_t = S_reg phi(q_t) (delta rule: and X_t = S_reg s_t), ||S_reg||^2
        {
          float ns;
          float vals[RPT * C::NVS];
          {
            float2 acc[RPT][C::NVS];
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
              for (int v = 0; v < C::NVS; ++v) acc[r][v] = f2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < C::NVY; ++v) {
              const int base = (v < KS) ? recS(v) + C::OFF_Q : recS(v - KS) + C::OFF_S;
#pragma unroll
              for (int kk = 0; kk < NCH; ++kk) {
                const float4 x = *reinterpret_cast<const float4*>(sf + base + colof(kk, 0));
                const float2 x0 = f2(x.x, x.y), x1 = f2(x.z, x.w);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                  acc[r][v] = __ffma2_rn(S2[r][2 * kk], x0, acc[r][v]);
                  acc[r][v] = __ffma2_rn(S2[r][2 * kk + 1], x1, acc[r][v]);
                }
              }
            }
            float2 n2 = f2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
              for (int p = 0; p < NCP; ++p) n2 = __ffma2_rn(S2[r][p], S2[r][p], n2);
            ns = n2.x + n2.y;
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
              for (int v = 0; v < C::NVS; ++v) vals[r * C::NVS + v] = acc[r][v].x + acc[r][v].y;
          }
          reduce_scatter<RPT * C::NVS, LPR / 2>(vals, c);
#pragma unroll
          for (int i = 0; i < C::KVS; ++i) {
            const int slot = c * C::KVS + i;
            const int r = slot / C::NVS, v = slot - r * C::NVS;
            if (v < C::NVY) sf[ybuf + v * D + row0 + r] = vals[i];
          }
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1) ns += __shfl_xor_sync(0xffffffffu, ns, m);
          if (lane == 0) sf[C::F_WP + par * GW + gw] = ns;
        }
        bar_sync(BAR_S, GT);
        // ---------------- phase G: alpha_t' . phi(q_t) (t' <= t), |alpha_t|^2 (delta rule: alpha_t' . s_t)
        {
          auto jobs = [&](auto wtag) {
            constexpr int W = decltype(wtag)::value;
            float jv[C::NSS];
#pragma unroll
            for (int s = 0; s < C::NSS; ++s) {
              const int j = s * GW + W;
              float acc = 0.f;
              if (j < C::NJS) {
                int oa, ob;
                if (j < C::NJQ) {
                  int t = 0;
#pragma unroll
                  for (int tt = 1; tt < KS; ++tt) t += (j >= tt * (tt + 1) / 2) ? 1 : 0;
                  oa = abuf + (j - t * (t + 1) / 2) * D;
                  ob = recS(t) + C::OFF_Q;
                } else if (j < C::NJQ + KS) {
                  oa = abuf + (j - C::NJQ) * D;
                  ob = oa;
                } else {   // delta rule: alpha_t' . s_t, t' <= t
                  const int jj = j - C::NJQ - KS;
                  int t = 0;
#pragma unroll
                  for (int tt = 1; tt < KS; ++tt) t += (jj >= tt * (tt + 1) / 2) ? 1 : 0;
                  oa = abuf + (jj - t * (t + 1) / 2) * D;
                  ob = recS(t) + C::OFF_S;
                }
                if (D >= 32) {
#pragma unroll
                  for (int e = 0; e < D / 32; ++e)
                    acc = fmaf(sf[oa + lane + 32 * e], sf[ob + lane + 32 * e], acc);
                } else if (lane < D) {
                  acc = sf[oa + lane] * sf[ob + lane];
                }
              }
              jv[s] = acc;
            }
            reduce_scatter<C::NSS, 16>(jv, lane);
            float x = jv[0];
#pragma unroll
            for (int m = 32 / C::NSS / 2; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
            constexpr int SH = 5 - log2i(C::NSS);
            const int j = (lane >> SH) * GW + W;
            if ((lane & ((1 << SH) - 1)) == 0 && j < C::NJS) sf[C::F_RS + j] = x;
          };
          switch (gw) {
            case 0: jobs(std::integral_constant<int, 0>{}); break;
            case 1: if constexpr (GW > 1) jobs(std::integral_constant<int, 1>{}); break;
            case 2: if constexpr (GW > 2) jobs(std::integral_constant<int, 2>{}); break;
            case 3: if constexpr (GW > 3) jobs(std::integral_constant<int, 3>{}); break;
            case 4: if constexpr (GW > 4) jobs(std::integral_constant<int, 4>{}); break;
            case 5: if constexpr (GW > 5) jobs(std::integral_constant<int, 5>{}); break;
            case 6: if constexpr (GW > 6) jobs(std::integral_constant<int, 6>{}); break;
            case 7: if constexpr (GW > 7) jobs(std::integral_constant<int, 7>{}); break;
            default: break;
          }
        }
        bar_sync(BAR_S, GT);
        // ---------------- phase U: renormalisation, outputs, S update
        if constexpr (!DL) {
          float rs_[C::NJS];
#pragma unroll
          for (int j = 0; j < C::NJS; ++j) rs_[j] = sf[C::F_RS + j];
          float ws = 0.f;
#pragma unroll
          for (int w = 0; w < GW; ++w) ws += sf[C::F_WP + par * GW + w];
          const float norm0 = sigma * sqrtf(ws);
          float bound = norm0;
#pragma unroll
          for (int t = 0; t < KS; ++t)
            if (t < cS) bound = fmaf(sf[recS(t) + C::OFF_SC + 1], sqrtf(rs_[C::NJQ + t]), bound);
          if (!isfinite(bound)) flags |= kStatusNonfinite;
          float isg[KS], sg[KS];   // 1/sigma before step t, sigma after it
          const bool exact = !(bound <= a.tau * (1.f - 0x1p-12f));
          if (!exact) {
            const float is = __frcp_rn(sigma);
#pragma unroll
            for (int t = 0; t < KS; ++t) { isg[t] = is; sg[t] = sigma; }
          } else {
            float mv[C::NMINI];
            float vrow[KS][RPT];
#pragma unroll
            for (int t = 0; t < KS; ++t)
#pragma unroll
              for (int r = 0; r < RPT; ++r) vrow[t][r] = sf[recS(t) + C::OFF_V + row0 + r];
#pragma unroll
            for (int t = 0; t < KS; ++t) {   // v_t^T S_reg alpha_t
              float x = 0.f;
#pragma unroll
              for (int kk = 0; kk < NCH; ++kk) {
                const float4 al = *reinterpret_cast<const float4*>(sf + abuf + t * D + colof(kk, 0));
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                  float y = S2[r][2 * kk].x * al.x;
                  y = fmaf(S2[r][2 * kk].y, al.y, y);
                  y = fmaf(S2[r][2 * kk + 1].x, al.z, y);
                  y = fmaf(S2[r][2 * kk + 1].y, al.w, y);
                  x = fmaf(vrow[t][r], y, x);
                }
              }
              mv[t] = x;
            }
#pragma unroll
            for (int t = 0; t < KS; ++t)
#pragma unroll
              for (int tp = 0; tp <= t; ++tp) {
                float xa = 0.f, xv = 0.f;
                if (g == 0) {   // row group 0 covers every column once
#pragma unroll
                  for (int kk = 0; kk < NCH; ++kk)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int col = colof(kk, e);
                      xa = fmaf(sf[abuf + t * D + col], sf[abuf + tp * D + col], xa);
                    }
                }
                if (c == 0) {   // lane 0 of each row group covers its rows once
#pragma unroll
                  for (int r = 0; r < RPT; ++r) xv = fmaf(vrow[t][r], vrow[tp][r], xv);
                }
                mv[KS + t * (t + 1) + 2 * tp] = xa;
                mv[KS + t * (t + 1) + 2 * tp + 1] = xv;
              }
#pragma unroll
            for (int k2 = 0; k2 < C::NMINI; ++k2) {
              float x = mv[k2];
#pragma unroll
              for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
              mv[k2] = x;
            }
            if (lane == 0) {
#pragma unroll
              for (int k2 = 0; k2 < C::NMINI; ++k2) sf[C::F_MINI + gw * C::MSTR + k2] = mv[k2];
            }
            bar_sync(BAR_S, GT);
            float tot[C::NMINI];
#pragma unroll
            for (int k2 = 0; k2 < C::NMINI; ++k2) {
              float x = 0.f;
#pragma unroll
              for (int w = 0; w < GW; ++w) x += sf[C::F_MINI + w * C::MSTR + k2];
              tot[k2] = x;
            }
            float nreg2 = ws, sgc = sigma;
#pragma unroll
            for (int t = 0; t < KS; ++t) {
              isg[t] = __frcp_rn(sgc);
              if (t < cS) {
                float cross = tot[t];
#pragma unroll
                for (int tp = 0; tp < t; ++tp)
                  cross = fmaf(tot[KS + t * (t + 1) + 2 * tp + 1] * tot[KS + t * (t + 1) + 2 * tp], isg[tp], cross);
                const float aa = tot[KS + t * (t + 1) + 2 * t], vv = tot[KS + t * (t + 1) + 2 * t + 1];
                nreg2 = fmaf(2.f * isg[t], cross, nreg2);
                nreg2 = fmaf(vv * aa, isg[t] * isg[t], nreg2);
                const float npre = sgc * sqrtf(fmaxf(nreg2, 0.f));
                if (npre > a.tau) {
                  sgc *= a.tau / npre;
                  ++renorm_cnt;
                }
                if (!isfinite(npre)) flags |= kStatusNonfinite;
              }
              sg[t] = sgc;
            }
          }
          // outputs: o_t = sigma_t (Y_t + sum_{t'<=t} v_t' aq_{t,t'} / sigma_{t'-1}) / den_t
          {
            const int h = gid / D, i = gid - (gid / D) * D;
#pragma unroll
            for (int tt = 0; tt < KS; ++tt) {
              if ((tt & 1) != h || tt >= cS) continue;
              float x = sf[ybuf + tt * D + i];
#pragma unroll
              for (int tp = 0; tp <= tt; ++tp)
                x = fmaf(sf[recS(tp) + C::OFF_V + i] * rs_[tt * (tt + 1) / 2 + tp], isg[tp], x);
              const float o = sg[tt] * x * sf[recS(tt) + C::OFF_SC];
              if (!isfinite(o)) flags |= kStatusNonfinite;
              go[(gS0 + tt) * D + i] = from_f32<TIO>(o);
            }
          }
          // S_reg += sum_t v_t alpha_t^T / sigma_{t-1}
#pragma unroll
          for (int t = 0; t < KS; ++t) {
            if (t < cS) {
              float vr[RPT];
#pragma unroll
              for (int r = 0; r < RPT; ++r) vr[r] = sf[recS(t) + C::OFF_V + row0 + r] * isg[t];
#pragma unroll
              for (int kk = 0; kk < NCH; ++kk) {
                const float4 al = *reinterpret_cast<const float4*>(sf + abuf + t * D + colof(kk, 0));
                const float2 a0 = f2(al.x, al.y), a1 = f2(al.z, al.w);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                  const float2 w = f2(vr[r], vr[r]);
                  S2[r][2 * kk] = __ffma2_rn(w, a0, S2[r][2 * kk]);
                  S2[r][2 * kk + 1] = __ffma2_rn(w, a1, S2[r][2 * kk + 1]);
                }
              }
            }
          }
          sigma = sg[KS - 1];
          if (sigma < 0x1p-16f) {
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
              for (int p = 0; p < NCP; ++p) { S2[r][p].x *= sigma; S2[r][p].y *= sigma; }
            sigma = 1.f;
          }
        }
        else {
          // delta rule (gist.science summary §2.3): S_t = S_{t-1} + w_t alpha_hat_t^T with
          // w_t = v_t - S_{t-1} k_hat_t, k_hat = s / |s|, alpha_hat = alpha / |alpha|.  With the
          // lazy scale S = sigma S_reg and X_t = S_reg,0 s_t from phase P, per row:
          //   w_t = v_t - sigma_{t-1} (X_t / |s_t| + sum_{t'<t} w_t' (alpha_hat_t'.k_hat_t) / sigma_{t'-1}),
          //   S_reg += w_t alpha_hat_t^T / sigma_{t-1},
          //   S_t phi(q_t) = sigma_t (Y_t + sum_{t'<=t} w_t' (alpha_t'.phi(q_t)) / (|alpha_t'| sigma_{t'-1})).
          float rs_[C::NJS];
#pragma unroll
          for (int j = 0; j < C::NJS; ++j) rs_[j] = sf[C::F_RS + j];
          float ws = 0.f;
#pragma unroll
          for (int w = 0; w < GW; ++w) ws += sf[C::F_WP + par * GW + w];
          float ia[KS], isn[KS], ck[KS][KS];   // 1/|alpha_t|, 1/|s_t|, alpha_hat_t' . k_hat_t (t' <= t)
#pragma unroll
          for (int t = 0; t < KS; ++t) {
            ia[t] = 1.f / fmaxf(sqrtf(rs_[C::NJQ + t]), kNormEps);
            isn[t] = 1.f / fmaxf(sf[recS(t) + C::OFF_SC + 2], kNormEps);
          }
#pragma unroll
          for (int t = 0; t < KS; ++t)
#pragma unroll
            for (int tp = 0; tp < KS; ++tp)
              ck[t][tp] = (tp <= t) ? rs_[C::NJQ + KS + t * (t + 1) / 2 + tp] * ia[tp] * isn[t] : 0.f;
          // ||S_t|| <= ||I - k_hat alpha_hat^T||_2 ||S_{t-1}|| + |v_t|, and for unit vectors with
          // c = alpha_hat . k_hat that norm is sqrt((3 - 2c + sqrt(5 - 4c)) / 2): when the bound
          // stays below tau no step of the round renormalises
          float bound = sigma * sqrtf(ws);
#pragma unroll
          for (int t = 0; t < KS; ++t)
            if (t < cS) {
              const float cc = fminf(fmaxf(ck[t][t], -1.f), 1.f);
              const float gr = sqrtf(0.5f * (3.f - 2.f * cc + sqrtf(5.f - 4.f * cc)));
              bound = fmaf(gr, bound, sf[recS(t) + C::OFF_SC + 1]);
            }
          if (!isfinite(bound)) flags |= kStatusNonfinite;
          float isg[KS], sg[KS], sgp[KS];   // 1/sigma before step t, sigma after it, sigma before it
          const bool exact = !(bound <= a.tau * (1.f - 0x1p-12f));
          if (!exact) {
            const float is = __frcp_rn(sigma);
#pragma unroll
            for (int t = 0; t < KS; ++t) { isg[t] = is; sg[t] = sigma; sgp[t] = sigma; }
          } else {
            // the per-step norms from one reduction: w_t = sum_m A_tm v_m + B_tm X_m, so every
            // product they need is a combination of v_m^T S_reg,0 alpha_t, X_m^T S_reg,0 alpha_t,
            // the Gram matrix of {v_m, X_m} and alpha_t . alpha_t'
            float mv[C::NMINI];
#pragma unroll
            for (int k2 = 0; k2 < C::NMINI; ++k2) mv[k2] = 0.f;
            float vrow[KS][RPT], xrow[KS][RPT];
#pragma unroll
            for (int t = 0; t < KS; ++t)
#pragma unroll
              for (int r = 0; r < RPT; ++r) {
                vrow[t][r] = sf[recS(t) + C::OFF_V + row0 + r];
                xrow[t][r] = (t < cS) ? sf[ybuf + (KS + t) * D + row0 + r] : 0.f;
              }
#pragma unroll
            for (int t = 0; t < KS; ++t) {
              float y[RPT];
#pragma unroll
              for (int r = 0; r < RPT; ++r) y[r] = 0.f;
#pragma unroll
              for (int kk = 0; kk < NCH; ++kk) {
                const float4 al = *reinterpret_cast<const float4*>(sf + abuf + t * D + colof(kk, 0));
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                  y[r] = fmaf(S2[r][2 * kk].x, al.x, y[r]);
                  y[r] = fmaf(S2[r][2 * kk].y, al.y, y[r]);
                  y[r] = fmaf(S2[r][2 * kk + 1].x, al.z, y[r]);
                  y[r] = fmaf(S2[r][2 * kk + 1].y, al.w, y[r]);
                }
              }
#pragma unroll
              for (int m = 0; m < KS; ++m)
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                  mv[C::MI_VSA + m * KS + t] = fmaf(vrow[m][r], y[r], mv[C::MI_VSA + m * KS + t]);
                  mv[C::MI_XSA + m * KS + t] = fmaf(xrow[m][r], y[r], mv[C::MI_XSA + m * KS + t]);
                }
            }
            if (c == 0) {   // lane 0 of each row group covers its rows once
#pragma unroll
              for (int m = 0; m < KS; ++m)
#pragma unroll
                for (int mp = 0; mp < KS; ++mp)
#pragma unroll
                  for (int r = 0; r < RPT; ++r) {
                    mv[C::MI_VX + m * KS + mp] = fmaf(vrow[m][r], xrow[mp][r], mv[C::MI_VX + m * KS + mp]);
                    if (mp <= m) {
                      mv[C::MI_VV + m * (m + 1) / 2 + mp] =
                          fmaf(vrow[m][r], vrow[mp][r], mv[C::MI_VV + m * (m + 1) / 2 + mp]);
                      mv[C::MI_XX + m * (m + 1) / 2 + mp] =
                          fmaf(xrow[m][r], xrow[mp][r], mv[C::MI_XX + m * (m + 1) / 2 + mp]);
                    }
                  }
            }
            if (g == 0) {   // row group 0 covers every column once
#pragma unroll
              for (int t = 0; t < KS; ++t)
#pragma unroll
                for (int tp = 0; tp <= t; ++tp)
#pragma unroll
                  for (int kk = 0; kk < NCH; ++kk)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int col = colof(kk, e);
                      mv[C::MI_AA + t * (t + 1) / 2 + tp] =
                          fmaf(sf[abuf + t * D + col], sf[abuf + tp * D + col], mv[C::MI_AA + t * (t + 1) / 2 + tp]);
                    }
            }
#pragma unroll
            for (int k2 = 0; k2 < C::NMINI; ++k2) {
              float x = mv[k2];
#pragma unroll
              for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
              mv[k2] = x;
            }
            if (lane == 0) {
#pragma unroll
              for (int k2 = 0; k2 < C::NMINI; ++k2) sf[C::F_MINI + gw * C::MSTR + k2] = mv[k2];
            }
            bar_sync(BAR_S, GT);
#pragma unroll
            for (int k2 = 0; k2 < C::NMINI; ++k2) {
              float x = 0.f;
#pragma unroll
              for (int w = 0; w < GW; ++w) x += sf[C::F_MINI + w * C::MSTR + k2];
              mv[k2] = x;
            }
            auto vv_ = [&](int m, int mp) { return m >= mp ? mv[C::MI_VV + m * (m + 1) / 2 + mp] : mv[C::MI_VV + mp * (mp + 1) / 2 + m]; };
            auto xx_ = [&](int m, int mp) { return m >= mp ? mv[C::MI_XX + m * (m + 1) / 2 + mp] : mv[C::MI_XX + mp * (mp + 1) / 2 + m]; };
            float cA[KS][KS], cB[KS][KS];
            float nreg2 = ws, sgc = sigma;
#pragma unroll
            for (int t = 0; t < KS; ++t) {
              isg[t] = __frcp_rn(sgc);
              sgp[t] = sgc;
#pragma unroll
              for (int m = 0; m < KS; ++m) {
                cA[t][m] = (m == t) ? 1.f : 0.f;
                cB[t][m] = (m == t) ? -sgc * isn[t] : 0.f;
              }
              if (t < cS) {
#pragma unroll
                for (int tp = 0; tp < t; ++tp) {
                  const float f = sgc * isg[tp] * ck[t][tp];
#pragma unroll
                  for (int m = 0; m < KS; ++m) {
                    cA[t][m] = fmaf(-f, cA[tp][m], cA[t][m]);
                    cB[t][m] = fmaf(-f, cB[tp][m], cB[t][m]);
                  }
                }
                float wsa = 0.f;   // w_t . S_reg,0 alpha_t
#pragma unroll
                for (int m = 0; m < KS; ++m)
                  wsa = fmaf(cA[t][m], mv[C::MI_VSA + m * KS + t], fmaf(cB[t][m], mv[C::MI_XSA + m * KS + t], wsa));
                float ww[KS];      // w_t . w_t'
#pragma unroll
                for (int tp = 0; tp <= t; ++tp) {
                  float x = 0.f;
#pragma unroll
                  for (int m = 0; m < KS; ++m)
#pragma unroll
                    for (int mp = 0; mp < KS; ++mp) {
                      x = fmaf(cA[t][m] * cA[tp][mp], vv_(m, mp), x);
                      x = fmaf(cA[t][m] * cB[tp][mp], mv[C::MI_VX + m * KS + mp], x);
                      x = fmaf(cB[t][m] * cA[tp][mp], mv[C::MI_VX + mp * KS + m], x);
                      x = fmaf(cB[t][m] * cB[tp][mp], xx_(m, mp), x);
                    }
                  ww[tp] = x;
                }
                float cross = wsa;   // w_t . S_reg,t-1 alpha_t, then times 1/|alpha_t|
#pragma unroll
                for (int tp = 0; tp < t; ++tp)
                  cross = fmaf(ww[tp] * mv[C::MI_AA + t * (t + 1) / 2 + tp], ia[tp] * isg[tp], cross);
                cross *= ia[t];
                nreg2 = fmaf(2.f * isg[t], cross, nreg2);
                nreg2 = fmaf(ww[t], isg[t] * isg[t], nreg2);
                const float npre = sgc * sqrtf(fmaxf(nreg2, 0.f));
                if (npre > a.tau) {
                  sgc *= a.tau / npre;
                  ++renorm_cnt;
                }
                if (!isfinite(npre)) flags |= kStatusNonfinite;
              }
              sg[t] = sgc;
            }
          }
          // w_t of row i from v, X and the earlier w's of that row
          auto wrow = [&](int i, float (&w)[KS]) {
#pragma unroll
            for (int t = 0; t < KS; ++t) {
              float x = 0.f;
              if (t < cS) {
                x = fmaf(-sgp[t] * isn[t], sf[ybuf + (KS + t) * D + i], sf[recS(t) + C::OFF_V + i]);
#pragma unroll
                for (int tp = 0; tp < t; ++tp) x = fmaf(-sgp[t] * isg[tp] * ck[t][tp], w[tp], x);
              }
              w[t] = x;
            }
          };
          // outputs: o_t = sigma_t (Y_t + sum_{t'<=t} w_t' (alpha_t'.phi(q_t)) / (|alpha_t'| sigma_{t'-1})) / den_t
          {
            const int h = gid / D, i = gid - (gid / D) * D;
            float wi[KS];
            wrow(i, wi);
#pragma unroll
            for (int tt = 0; tt < KS; ++tt) {
              if ((tt & 1) != h || tt >= cS) continue;
              float x = sf[ybuf + tt * D + i];
#pragma unroll
              for (int tp = 0; tp <= tt; ++tp) x = fmaf(wi[tp] * rs_[tt * (tt + 1) / 2 + tp], ia[tp] * isg[tp], x);
              const float o = sg[tt] * x * sf[recS(tt) + C::OFF_SC];
              if (!isfinite(o)) flags |= kStatusNonfinite;
              go[(gS0 + tt) * D + i] = from_f32<TIO>(o);
            }
          }
          // S_reg += sum_t w_t alpha_t^T / (sigma_{t-1} |alpha_t|)
          {
            float wr[RPT][KS];
#pragma unroll
            for (int r = 0; r < RPT; ++r) wrow(row0 + r, wr[r]);
#pragma unroll
            for (int t = 0; t < KS; ++t) {
              if (t < cS) {
                float vr[RPT];
#pragma unroll
                for (int r = 0; r < RPT; ++r) vr[r] = wr[r][t] * isg[t] * ia[t];
#pragma unroll
                for (int kk = 0; kk < NCH; ++kk) {
                  const float4 al = *reinterpret_cast<const float4*>(sf + abuf + t * D + colof(kk, 0));
                  const float2 a0 = f2(al.x, al.y), a1 = f2(al.z, al.w);
#pragma unroll
                  for (int r = 0; r < RPT; ++r) {
                    const float2 w = f2(vr[r], vr[r]);
                    S2[r][2 * kk] = __ffma2_rn(w, a0, S2[r][2 * kk]);
                    S2[r][2 * kk + 1] = __ffma2_rn(w, a1, S2[r][2 * kk + 1]);
                  }
                }
              }
            }
          }
          sigma = sg[KS - 1];
          if (sigma < 0x1p-16f) {
#pragma unroll
            for (int r = 0; r < RPT; ++r)
#pragma unroll
              for (int p = 0; p < NCP; ++p) { S2[r][p].x *= sigma; S2[r][p].y *= sigma; }
            sigma = 1.f;
          }
        }
      }
      if constexpr (CL) mbar_arrive_remote(remote(&hb[2 + (rnd & 1)]));
      else bar_arrive(BAR_EMPTY0 + (rnd & 1), NT);
      par ^= 1;
    }
    if (!timed_out) {
#pragma unroll
      for (int r = 0; r < RPT; ++r)
#pragma unroll
        for (int kk = 0; kk < NCH; ++kk) {
          *reinterpret_cast<float4*>(gS + (row0 + r) * D + colof(kk, 0)) =
              make_float4(sigma * S2[r][2 * kk].x, sigma * S2[r][2 * kk].y, sigma * S2[r][2 * kk + 1].x,
                          sigma * S2[r][2 * kk + 1].y);
        }
    }
    if constexpr (CL) {
      if (timed_out && gid == 0) {
        for (int j = loaded_s + 1; j < ntiles && j <= loaded_s + NSTAGE; ++j)
          (void)mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)((j / NSTAGE) & 1));
      }
    }
    if (gid == 0 && renorm_cnt) {
      if constexpr (PS) atomicAdd(&a.pair_status[pair].renorm_count, (unsigned int)renorm_cnt);
      else atomicAdd(&a.status->renorm_count, renorm_cnt);
    }
  }
  if (flags) {
    if constexpr (PS) atomicOr(&a.pair_status[pair].flags, flags);
    else atomicOr(&a.status->flags, flags);
  }
}

// DL = true: the delta-rule variant (same A group; the S group writes S with the residual).
template <int D, int R, int KS, typename TIO, bool PS = false, bool DL = false>
cudaError_t launch_seq_block_t(const ScanArgs& a, cudaStream_t s) {
  using C = blk::Cfg<D, R, KS, TIO, DL>;
  auto kern = seq_block_kernel<D, R, KS, TIO, PS, false, DL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.pairs, blk::Geom<D>::NT, C::bytes, s>>>(a);
  return cudaGetLastError();
}

// Cluster mode: two CTAs (A group, S group) per pair.
template <int D, int R, int KS, typename TIO, bool DL = false>
cudaError_t launch_seq_cluster_t(const ScanArgs& a, cudaStream_t s) {
  using C = blk::Cfg<D, R, KS, TIO, DL>;
  auto kern = seq_block_kernel<D, R, KS, TIO, false, true, DL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * (unsigned)a.pairs, 1, 1);
  cfg.blockDim = dim3(blk::Geom<D>::GT, 1, 1);
  cfg.dynamicSmemBytes = C::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace vla
