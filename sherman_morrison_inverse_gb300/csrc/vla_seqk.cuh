// Blocked sequential VLA scan for sm_103a: KS steps per reduction round.
//
// Same recurrence as the step-by-step scan ("Mathematical Primitives" §2-§5,
// README "VLA v3" items 1-5), taken KS steps (M = KS * r directions) per
// reduction round in exact Woodbury form ("Mathematical Primitives" §3 names the
// identity; the gist.science summary §2.4 the parallel formulation).  With
// A_0 the inverse at the start of the round and U = [u_1 .. u_M]:
//
//   P = A_0 U,  Q_t = A_0 s_t,  G = I + U^T P = L D L^T   (D_jj = the sequential deltas)
//   A_after   = A_0 - P G^{-1} P^T                           (= M rank-1 updates)
//   alpha_t   = Q_t - P_{<=e_t} G_{<=e_t}^{-1} (U^T Q_t)_{<=e_t}
//               (e_t = last direction of step t; leading blocks of G)
//
// so one round needs M + KS matrix-vector products with A_0 (the same count as
// the step-by-step form) but one set of reductions instead of M.  The S side
// lags one round: round R applies S += v alpha^T for the steps completed in
// round R-1, whose alpha vectors are then in shared memory, and writes their
// outputs:  o_t = (S_0 phi(q_t) + sum_{t'<=t} v_t' (alpha_t' . phi(q_t))) / den_t.
//
// Round structure (one CTA per (batch, head) pair, NT = 2d threads):
//   phase P  partial products of the thread's 4 x (d/8) pieces of A and S with
//            every vector of the round (packed FFMA2), reduce-scatter across the
//            8 lanes of a row group, rows written to shared memory      -> barrier
//   phase G  the small Gram scalars (u_a.P_b, u_a.Q_t, alpha.phi(q), |alpha|^2)
//            as 64-element dot products spread over the warps           -> barrier
//   phase U  LDL^T of G (every thread, in registers), A update, alpha for
//            this round's steps (one writer per element), and the S side of the
//            previous round's steps.
//
// Singularity guard: a pivot |D_jj| < 1e-6 means the sequential recurrence
// would take the guard at that direction.  The round then applies nothing and
// the same directions are replayed one per round, where the pivot is the
// sequential delta itself and the guard (A += 1e-6 I instead of the update) is
// taken exactly as the pages state it.
//
// Renormalisation: S = sigma * S_reg (lazy scale).  Each round reduces ||S_reg||^2
// exactly; with ||alpha_t|| and ||v_t|| the bound ||S_t|| <= ||S_0|| + sum ||v|| ||alpha||
// decides that no step of the chunk can exceed tau.  Otherwise an extra
// reduction gives the exact per-step norms from
//   ||S_t||^2 = ||S_{t-1}||^2 + 2 v_t^T S_{t-1} alpha_t + |v_t|^2 |alpha_t|^2
// and the decisions are taken step by step.
#pragma once

#include "vla_internal.cuh"

namespace vla {

namespace blk {

constexpr float kGuardEps = 1e-6f;
constexpr float kReadoutEps = 1e-6f;

__host__ __device__ constexpr int pow2_ceil(int x) { return x <= 1 ? 1 : 2 * pow2_ceil((x + 1) / 2); }
__host__ __device__ constexpr int log2i(int x) { return x <= 1 ? 0 : 1 + log2i(x / 2); }

template <int D>
struct Geom {
  static constexpr int RPT = (D == 16) ? 2 : 4;   // rows per thread
  static constexpr int LPR = (D == 16) ? 4 : 8;   // lanes per row group
  static constexpr int CPT = D / LPR;             // columns per thread
  static constexpr int NCH = CPT / 4;             // float4 pieces per vector
  static constexpr int NG = D / RPT;              // row groups
  static constexpr int NT = NG * LPR;             // threads (2 d)
  static constexpr int NW = NT / 32;
  static constexpr int NSTAGE = 2;
  static_assert(NT == 2 * D, "two threads per element of a d-vector");
};

// shared memory bytes for a tile of ts steps (raw ring + records + scratch + buffers)
template <int D, int R, int KS, typename TIO>
__host__ __device__ constexpr size_t smem_bytes_for(int ts) {
  return (size_t)Geom<D>::NSTAGE * ts * (3 * D + R * D) * sizeof(TIO) +
         sizeof(float) * ((size_t)2 * ts * ((R + 3) * D + 4) + (size_t)ts * D + 4096 + 8 * KS * D * 4);
}
template <int D, int R, int KS, typename TIO>
__host__ __device__ constexpr int pick_ts() {
  return smem_bytes_for<D, R, KS, TIO>(32) <= 200 * 1024 ? 32 : smem_bytes_for<D, R, KS, TIO>(16) <= 200 * 1024 ? 16 : 8;
}

template <int D, int R, int KS, typename TIO>
struct Cfg {
  using Gm = Geom<D>;
  static constexpr int TS = pick_ts<D, R, KS, TIO>();         // steps per tile
  static constexpr int M = KS * R;                            // directions per round
  static constexpr int NV = M + 2 * KS;                       // vectors per round: P, Q, Y
  static constexpr int NVAL = Gm::RPT * NV;
  static constexpr int KV = NVAL / Gm::LPR;                   // values a lane keeps after the reduce-scatter
  static_assert(NVAL % Gm::LPR == 0, "reduce-scatter must split evenly");
  // dot-product jobs of phase G
  static constexpr int NJG = M * (M + 1) / 2;                 // u_a . P_b, a <= b
  static constexpr int NJH = R * KS * (KS + 1) / 2;           // u_a . Q_t, a <= e_t
  static constexpr int NJQ = KS * (KS + 1) / 2;               // alpha_t' . phi(q_t), t' <= t
  static constexpr int NJN = KS;                              // alpha_t . alpha_t
  static constexpr int NJOB = NJG + NJH + NJQ + NJN;
  static constexpr int JPW = (NJOB + Gm::NW - 1) / Gm::NW;    // jobs per warp
  static constexpr int NS = pow2_ceil(JPW) < 32 ? pow2_ceil(JPW) : 32;
  static constexpr int NPASS = (JPW + 31) / 32;
  static constexpr int NMINI = KS + KS * (KS + 1);            // exact-norm scalars: v^T S alpha, alpha Gram, v Gram
  // step record (floats): u[R][D] | s[D] | phi(q)[D] | v[D] | den, |v|, 0, 0
  static constexpr int OFF_U = 0, OFF_S = R * D, OFF_Q = (R + 1) * D, OFF_V = (R + 2) * D;
  static constexpr int OFF_SC = (R + 3) * D;
  static constexpr int REC = (R + 3) * D + 4;
  // raw tile bytes (q, k, v: TS x D; u: TS x R x D)
  static constexpr uint32_t QB = TS * D * sizeof(TIO);
  static constexpr uint32_t UB = TS * R * D * sizeof(TIO);
  static constexpr uint32_t STAGE = 3 * QB + UB;
  // shared memory map (float offsets after the raw ring)
  static constexpr int F_PRE = 0;                                    // [2][TS][REC]
  static constexpr int F_ZERO = F_PRE + 2 * TS * REC;                // [REC] zeros
  static constexpr int F_PROD = F_ZERO + REC;                        // [TS][D] scratch
  static constexpr int F_P = F_PROD + TS * D;                        // [2][M][D]
  static constexpr int F_Q = F_P + 2 * M * D;                        // [2][KS][D]
  static constexpr int F_Y = F_Q + 2 * KS * D;                       // [2][KS][D]
  static constexpr int F_AL = F_Y + 2 * KS * D;                      // [2][KS][D]
  static constexpr int F_RES = F_AL + 2 * KS * D;                    // [NJOB] (+pad)
  static constexpr int F_WP = F_RES + ((NJOB + 3) / 4) * 4;          // [2][NW] norm partials (+pad)
  static constexpr int F_MINI = F_WP + ((2 * Gm::NW + 3) / 4) * 4;   // [NW][32]
  static constexpr int F_END = F_MINI + Gm::NW * 32;
  static constexpr size_t raw_bytes = (size_t)Gm::NSTAGE * STAGE;
  static constexpr size_t bar_off = raw_bytes + sizeof(float) * (size_t)F_END;
  static constexpr size_t bytes = bar_off + 16 * Gm::NSTAGE + 16;
  static_assert(QB % 16 == 0 && UB % 16 == 0 && REC % 4 == 0, "alignment");
  static_assert(TS % KS == 0, "chunks must tile a tile");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

}  // namespace blk

template <int D, int R, int KS, typename TIO>
__global__ void __launch_bounds__(blk::Geom<D>::NT, 1) seq_block_kernel(ScanArgs a) {
  using namespace blk;
  using Gm = Geom<D>;
  using C = Cfg<D, R, KS, TIO>;
  constexpr int RPT = Gm::RPT, LPR = Gm::LPR, CPT = Gm::CPT, NCH = Gm::NCH, NT = Gm::NT, NW = Gm::NW;
  constexpr int TS = C::TS, NSTAGE = Gm::NSTAGE;
  constexpr int M = C::M, NV = C::NV, KV = C::KV, REC = C::REC;
  constexpr int NCP = CPT / 2;  // float2 pairs per row piece
  constexpr float kInvSqrtD = (float)(D == 16 ? 0.25 : D == 64 ? 0.125 : 0.08838834764831845);

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* raw = smem;
  float* sf = reinterpret_cast<float*>(smem + C::raw_bytes);   // float-addressed region
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bar_off);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::bar_off + 16 * NSTAGE);

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = tid / LPR, c = tid % LPR;       // row group, lane within the group
  const int row0 = g * RPT;
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

  // column of element (kk, e) of this thread's row piece
  auto colof = [&](int kk, int e) { return 4 * c + 4 * LPR * kk + e; };

  // ---- state into registers: rows row0 .. row0+RPT-1, columns colof(kk, e)
  float2 A2[RPT][NCP], S2[RPT][NCP];
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
#pragma unroll
    for (int kk = 0; kk < NCH; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(gA + (row0 + r) * D + colof(kk, 0));
      const float4 sv = *reinterpret_cast<const float4*>(gS + (row0 + r) * D + colof(kk, 0));
      A2[r][2 * kk] = f2(av.x, av.y);
      A2[r][2 * kk + 1] = f2(av.z, av.w);
      S2[r][2 * kk] = f2(sv.x, sv.y);
      S2[r][2 * kk + 1] = f2(sv.z, sv.w);
    }
  }
  float n_i = (tid < D) ? gn[tid] : 0.f;     // normaliser element tid (prologue prefix sums)

  // zero record, barriers
  for (int e = tid; e < REC; e += NT) sf[C::F_ZERO + e] = (e == C::OFF_SC) ? 1.f : 0.f;  // ghost: den = 1
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    *flag = 0;
  }
  __syncthreads();

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

  // ---- per-tile prologue: float32 records, den_t = n_t . phi(q_t) + 1e-6, |v_t|
  int loaded = -1;
  bool timed_out = false;
  auto prologue = [&](int tile) -> bool {
    const int stage = tile % NSTAGE;
    if (tid == 0) {
      if (!mbar_wait_bounded(&bars[stage], (uint32_t)((tile / NSTAGE) & 1))) *flag = 1;
    }
    __syncthreads();
    if (*flag) return false;
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const TIO* rq = reinterpret_cast<const TIO*>(raw + stage * C::STAGE);
    const TIO* rk = reinterpret_cast<const TIO*>(raw + stage * C::STAGE + C::QB);
    const TIO* rv = reinterpret_cast<const TIO*>(raw + stage * C::STAGE + 2 * C::QB);
    const TIO* ru = reinterpret_cast<const TIO*>(raw + stage * C::STAGE + 3 * C::QB);
    float* pre = sf + C::F_PRE + (tile & 1) * TS * REC;
    for (int e = tid; e < nst * R * D; e += NT) {
      const int t = e / (R * D), off = e - t * (R * D);
      pre[t * REC + C::OFF_U + off] = to_f32(ru[e]);
    }
    for (int e = tid; e < nst * D; e += NT) {
      const int t = e / D, i = e - t * D;
      float* rec = pre + t * REC;
      rec[C::OFF_S + i] = phi_elu1(to_f32(rk[e])) * kInvSqrtD;
      rec[C::OFF_Q + i] = phi_elu1(to_f32(rq[e]));
      rec[C::OFF_V + i] = to_f32(rv[e]);
    }
    __syncthreads();
    float* prod = sf + C::F_PROD;
    if (tid < D) {
      for (int t = 0; t < nst; ++t) {
        n_i += phi_elu1(to_f32(rk[t * D + tid]));
        prod[t * D + tid] = n_i * pre[t * REC + C::OFF_Q + tid];
      }
    }
    __syncthreads();
    // den_t and |v_t|: warp w takes steps w, w + NW, ...
    for (int t = warp; t < nst; t += NW) {
      float dn = 0.f, vv = 0.f;
      for (int i = lane; i < D; i += 32) {
        dn += prod[t * D + i];
        const float x = pre[t * REC + C::OFF_V + i];
        vv = fmaf(x, x, vv);
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        dn += __shfl_xor_sync(0xffffffffu, dn, m);
        vv += __shfl_xor_sync(0xffffffffu, vv, m);
      }
      if (lane == 0) {
        pre[t * REC + C::OFF_SC] = dn + kReadoutEps;
        pre[t * REC + C::OFF_SC + 1] = sqrtf(vv);
      }
    }
    __syncthreads();
    if (tid == 0 && tile + NSTAGE < ntiles) {
      fence_proxy_async_smem();
      issue(tile + NSTAGE);
    }
    return true;
  };

  // ---- round state (uniform across the CTA)
  long long pos = 0;                 // next step to schedule
  bool replay = false;
  long long rep_pos = 0;             // first step of the chunk being replayed
  int rep_total = 0, rep_col = 0;    // its directions, and the next one
  // S-chunk: the steps completed in the previous round
  int cS = 0;                        // real steps (0 .. KS)
  int baseS = 0;                     // float offset of its first record
  long long gS0 = 0;                 // local index of its first step
  float sigma = 1.f;
  int par = 0;
  unsigned long long guard_cnt = 0, renorm_cnt = 0, replay_cnt = 0;
  unsigned int flags = 0;
  const float tau = a.tau;

  while (true) {
    // ================= schedule the A-chunk of this round
    int cA = 0;                      // real steps completed in this round
    int baseA = 0;                   // record offset of the chunk's first step (normal) / the replayed step
    int rep_j = 0;                   // replay: direction within the step
    bool rep_completes = false;
    bool nudgeA = false;
    long long gA0 = 0;
    bool haveA = false;
    long long a_step = -1;           // a step inside the chunk (for the tile check)
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
        const long long to_nudge = a.P - ((a.t0 + pos) % a.P);   // steps up to and including the next nudge
        if (to_nudge <= cmax) { cmax = to_nudge; nudgeA = true; }
      }
      cA = (int)cmax;
      gA0 = pos;
      a_step = pos;
      haveA = true;
    }
    if (!haveA && cS == 0) break;
    if (haveA) {
      const int tile = (int)(a_step / TS);
      if (tile != loaded) {
        if (!prologue(tile)) { timed_out = true; break; }
        loaded = tile;
      }
      baseA = C::F_PRE + (tile & 1) * TS * REC + (int)(a_step % TS) * REC;
    }
    // vector offsets of this round (float offsets into sf)
    auto offU = [&](int col) -> int {        // direction col of the round
      if (!haveA) return C::F_ZERO;
      if (replay) return (col == 0) ? baseA + C::OFF_U + rep_j * D : C::F_ZERO;
      const int t = col / R;
      return (t < cA) ? baseA + t * REC + C::OFF_U + (col - t * R) * D : C::F_ZERO;
    };
    auto recA = [&](int t) -> int {          // record of step slot t (s, phi(q), v)
      if (!haveA) return C::F_ZERO;
      if (replay) return (t == 0 && rep_completes) ? baseA : C::F_ZERO;
      return (t < cA) ? baseA + t * REC : C::F_ZERO;
    };
    auto recS = [&](int t) -> int { return (t < cS) ? baseS + t * REC : C::F_ZERO; };
    const int pbuf = C::F_P + par * M * D, qbuf = C::F_Q + par * KS * D, ybuf = C::F_Y + par * KS * D;
    const int abuf = C::F_AL + par * KS * D, abuf_prev = C::F_AL + (par ^ 1) * KS * D;

    // ================= phase P: partial products
    float vals[RPT * NV];
    {
      float2 acc[RPT][NV];
#pragma unroll
      for (int r = 0; r < RPT; ++r)
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[r][v] = f2(0.f, 0.f);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        int base;
        if (v < M) base = offU(v);
        else if (v < M + KS) base = recA(v - M) + C::OFF_S;
        else base = recS(v - M - KS) + C::OFF_Q;
#pragma unroll
        for (int kk = 0; kk < NCH; ++kk) {
          const float4 x = *reinterpret_cast<const float4*>(sf + base + colof(kk, 0));
          const float2 x0 = f2(x.x, x.y), x1 = f2(x.z, x.w);
#pragma unroll
          for (int r = 0; r < RPT; ++r) {
            if (v < M + KS) {
              acc[r][v] = __ffma2_rn(A2[r][2 * kk], x0, acc[r][v]);
              acc[r][v] = __ffma2_rn(A2[r][2 * kk + 1], x1, acc[r][v]);
            } else {
              acc[r][v] = __ffma2_rn(S2[r][2 * kk], x0, acc[r][v]);
              acc[r][v] = __ffma2_rn(S2[r][2 * kk + 1], x1, acc[r][v]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RPT; ++r)
#pragma unroll
        for (int v = 0; v < NV; ++v) vals[r * NV + v] = acc[r][v].x + acc[r][v].y;
    }
    float ns;  // ||S_reg||^2 partial
    {
      float2 n2 = f2(0.f, 0.f);
#pragma unroll
      for (int r = 0; r < RPT; ++r)
#pragma unroll
        for (int p = 0; p < NCP; ++p) n2 = __ffma2_rn(S2[r][p], S2[r][p], n2);
      ns = n2.x + n2.y;
    }
    // reduce-scatter across the LPR lanes of the row group
    {
      int n = RPT * NV;
#pragma unroll
      for (int m = LPR / 2; m >= 1; m >>= 1) {
        const bool hi = (c & m) != 0;
        const int h = n / 2;
#pragma unroll
        for (int i = 0; i < RPT * NV / 2; ++i) {
          if (i < h) {
            const float send = hi ? vals[i] : vals[i + h];
            const float keep = hi ? vals[i + h] : vals[i];
            vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        n = h;
      }
    }
    // lane c now holds the row sums of slots c*KV .. c*KV + KV - 1 (slot = r*NV + v)
#pragma unroll
    for (int i = 0; i < KV; ++i) {
      const int slot = c * KV + i;
      const int r = slot / NV, v = slot - r * NV;
      const int row = row0 + r;
      int dst;
      if (v < M) dst = pbuf + v * D + row;
      else if (v < M + KS) dst = qbuf + (v - M) * D + row;
      else dst = ybuf + (v - M - KS) * D + row;
      sf[dst] = vals[i];
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ns += __shfl_xor_sync(0xffffffffu, ns, m);
    if (lane == 0) sf[C::F_WP + par * NW + warp] = ns;
    __syncthreads();  // ---------------------------------------------------- BAR1

    // ================= phase G: Gram scalars as dot products over d elements
#pragma unroll
    for (int pass = 0; pass < C::NPASS; ++pass) {
      constexpr int NSL = C::NPASS > 1 ? 32 : C::NS;
      float jv[NSL];
#pragma unroll
      for (int s = 0; s < NSL; ++s) {
        const int j = (pass * 32 + s) * NW + warp;   // job index
        int oa = C::F_ZERO, ob = C::F_ZERO;
        if (j < C::NJG) {
          int b = 0;
#pragma unroll
          for (int bb = 1; bb < M; ++bb) b += (j >= bb * (bb + 1) / 2) ? 1 : 0;
          const int aa = j - b * (b + 1) / 2;
          oa = offU(aa);
          ob = pbuf + b * D;
        } else if (j < C::NJG + C::NJH) {
          const int h = j - C::NJG;
          int t = 0;
#pragma unroll
          for (int tt = 1; tt < KS; ++tt) t += (h >= R * tt * (tt + 1) / 2) ? 1 : 0;
          const int aa = h - R * t * (t + 1) / 2;
          oa = offU(aa);
          ob = qbuf + t * D;
        } else if (j < C::NJG + C::NJH + C::NJQ) {
          const int q = j - C::NJG - C::NJH;
          int t = 0;
#pragma unroll
          for (int tt = 1; tt < KS; ++tt) t += (q >= tt * (tt + 1) / 2) ? 1 : 0;
          const int tp = q - t * (t + 1) / 2;
          oa = abuf_prev + tp * D;
          ob = recS(t) + C::OFF_Q;
        } else if (j < C::NJOB) {
          const int t = j - C::NJG - C::NJH - C::NJQ;
          oa = abuf_prev + t * D;
          ob = oa;
        }
        float acc = 0.f;
        if (D >= 32) {
#pragma unroll
          for (int e = 0; e < D / 32; ++e) {
            const int i = lane + 32 * e;
            acc = fmaf(sf[oa + i], sf[ob + i], acc);
          }
        } else if (lane < D) {
          acc = sf[oa + lane] * sf[ob + lane];
        }
        jv[s] = acc;
      }
      // reduce-scatter over the warp: slot s ends in lanes with (lane >> (5 - log2 NSL)) == s
      {
        int n = NSL;
#pragma unroll
        for (int m = 16; m >= 32 / NSL && m >= 1; m >>= 1) {
          const bool hi = (lane & m) != 0;
          const int h = n / 2;
#pragma unroll
          for (int i = 0; i < NSL / 2; ++i) {
            if (i < h) {
              const float send = hi ? jv[i] : jv[i + h];
              const float keep = hi ? jv[i + h] : jv[i];
              jv[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
          }
          n = h;
        }
#pragma unroll
        for (int m = 32 / NSL / 2; m >= 1; m >>= 1) jv[0] += __shfl_xor_sync(0xffffffffu, jv[0], m);
      }
      constexpr int SH = 5 - log2i(NSL);
      const int s_mine = lane >> SH;
      const int j_mine = (pass * 32 + s_mine) * NW + warp;
      if ((lane & ((1 << SH) - 1)) == 0 && j_mine < C::NJOB) sf[C::F_RES + j_mine] = jv[0];
    }
    __syncthreads();  // ---------------------------------------------------- BAR2

    // ================= phase U
    float res[C::NJOB];
#pragma unroll
    for (int j = 0; j < C::NJOB; ++j) res[j] = sf[C::F_RES + j];

    // ---- A side: LDL^T of G = I + U^T A_0 U
    float Gm_[M][M];
#pragma unroll
    for (int b = 0; b < M; ++b)
#pragma unroll
      for (int aa = 0; aa <= b; ++aa) {
        const float v = res[b * (b + 1) / 2 + aa] + (aa == b ? 1.f : 0.f);
        Gm_[aa][b] = v;
        Gm_[b][aa] = v;
      }
    float Lm[M][M], Dv[M], iD[M];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < M; ++j) {
      float dj = Gm_[j][j];
#pragma unroll
      for (int k = 0; k < j; ++k) dj = fmaf(-Lm[j][k] * Dv[k], Lm[j][k], dj);
      Dv[j] = dj;
      bad = bad || !(fabsf(dj) >= kGuardEps);
      iD[j] = __frcp_rn(dj);
#pragma unroll
      for (int i = j + 1; i < M; ++i) {
        float x = Gm_[i][j];
#pragma unroll
        for (int k = 0; k < j; ++k) x = fmaf(-Lm[i][k] * Dv[k], Lm[j][k], x);
        Lm[i][j] = x * iD[j];
      }
    }
    // in a replay round only direction 0 is real: a bad pivot there is the guard
    const bool guard = replay && bad;
    const bool apply = haveA && (!bad || replay);
    if (haveA && bad && !replay) {   // start replaying this chunk one direction per round
      replay = true;
      rep_pos = gA0;
      rep_total = cA * R;
      rep_col = 0;
      ++replay_cnt;
    }
    // inverse of the unit lower triangle
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
    // per step: coefficients c_t = G_{<=e}^{-1} (U^T Q_t)_{<=e}
    float cf[KS][M];
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      const int e = (t + 1) * R - 1;
      float y[M];
#pragma unroll
      for (int aa = 0; aa < M; ++aa) {
        float x = 0.f;
        if (aa <= e) {
#pragma unroll
          for (int b = 0; b <= aa; ++b) {
            const float h = (b <= e) ? res[C::NJG + R * t * (t + 1) / 2 + b] : 0.f;
            x = fmaf(Li[aa][b], h, x);
          }
        }
        y[aa] = x * iD[aa];
      }
#pragma unroll
      for (int aa = 0; aa < M; ++aa) {
        float x = 0.f;
        if (aa <= e) {
#pragma unroll
          for (int b = aa; b < M; ++b)
            if (b <= e) x = fmaf(Li[b][aa], y[b], x);
        }
        cf[t][aa] = x;
      }
    }
    if (apply) {
      // A -= P G^{-1} P^T   (guard: A += 1e-6 I instead)
      if (!guard) {
        float Gi[M][M];   // G^{-1} = L^{-T} D^{-1} L^{-1}
#pragma unroll
        for (int i = 0; i < M; ++i)
#pragma unroll
          for (int j = 0; j < M; ++j) {
            float x = 0.f;
#pragma unroll
            for (int k = (i > j ? i : j); k < M; ++k) x = fmaf(Li[k][i] * iD[k], Li[k][j], x);
            Gi[i][j] = x;
          }
        float Pt[RPT][M];   // (P G^{-1}) for this thread's rows
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
            const int slot = (row / (4 * LPR)) * 4 + (row & 3);   // element index within the row piece
#pragma unroll
            for (int p = 0; p < NCP; ++p) {
              if (slot == 2 * p) A2[r][p].x += dadd;
              if (slot == 2 * p + 1) A2[r][p].y += dadd;
            }
          }
        }
      }
      // alpha for the steps this round completes: one writer per element
      {
        const int h = tid / D, i = tid - (tid / D) * D;
#pragma unroll
        for (int jj = 0; jj < (KS + 1) / 2; ++jj) {
          const int t = 2 * jj + h;
          if (t < KS) {
            float al = 0.f;
            const int rs = recA(t);
            if (rs != C::F_ZERO) {
              al = sf[qbuf + t * D + i];
              const bool last_step = (replay && rep_completes) ? true : (t == cA - 1);
              float sadd = 0.f;
              if (guard) sadd += kGuardEps;
              if (nudgeA && last_step) sadd += a.eps_n;
              if (!guard) {
#pragma unroll
                for (int tt = 0; tt < KS; ++tt) {
                  if (tt == 2 * jj || tt == 2 * jj + 1) {
                    if (t == tt) {
#pragma unroll
                      for (int b = 0; b < M; ++b)
                        if (b <= (tt + 1) * R - 1) al = fmaf(-sf[pbuf + b * D + i], cf[tt][b], al);
                    }
                  }
                }
              }
              if (sadd != 0.f) al = fmaf(sadd, sf[rs + C::OFF_S + i], al);
            }
            sf[abuf + t * D + i] = al;
          }
        }
      }
      if (guard) ++guard_cnt;
    } else {
      // nothing applied: no alpha is produced this round
#pragma unroll
      for (int jj = 0; jj < (KS + 1) / 2; ++jj) {
        const int t = 2 * jj + tid / D;
        if (t < KS) sf[abuf + t * D + (tid - (tid / D) * D)] = 0.f;
      }
    }

    // ---- S side: the steps completed in the previous round
    if (cS > 0) {
      float ws = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) ws += sf[C::F_WP + par * NW + w];
      const float norm0 = sigma * sqrtf(ws);
      float bound = norm0;
      float an[KS];
#pragma unroll
      for (int t = 0; t < KS; ++t) {
        an[t] = res[C::NJG + C::NJH + C::NJQ + t];
        if (t < cS) bound = fmaf(sf[recS(t) + C::OFF_SC + 1], sqrtf(an[t]), bound);
      }
      if (!isfinite(norm0) || !isfinite(bound)) flags |= kStatusNonfinite;
      // inverse scale before each step (1/sigma_{t-1}) and the scale after it (sigma_t)
      float isg[KS], sg[KS];
      const bool exact = !(bound <= tau * (1.f - 0x1p-12f));
      if (!exact) {
        const float is = __frcp_rn(sigma);
#pragma unroll
        for (int t = 0; t < KS; ++t) { isg[t] = is; sg[t] = sigma; }
      } else {
        // extra reduction: v_t^T S_0 alpha_t, alpha Gram, v Gram
        float mv[C::NMINI];
#pragma unroll
        for (int k = 0; k < C::NMINI; ++k) mv[k] = 0.f;
        float vrow[KS][RPT];
#pragma unroll
        for (int t = 0; t < KS; ++t)
#pragma unroll
          for (int r = 0; r < RPT; ++r) vrow[t][r] = sf[recS(t) + C::OFF_V + row0 + r];
#pragma unroll
        for (int t = 0; t < KS; ++t) {
          float x = 0.f;
#pragma unroll
          for (int kk = 0; kk < NCH; ++kk) {
            const float4 al = *reinterpret_cast<const float4*>(sf + abuf_prev + t * D + colof(kk, 0));
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
        int k = KS;
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
                  xa = fmaf(sf[abuf_prev + t * D + col], sf[abuf_prev + tp * D + col], xa);
                }
            }
            if (c == 0) {   // lane 0 of every row group covers its rows once
#pragma unroll
              for (int r = 0; r < RPT; ++r) xv = fmaf(vrow[t][r], vrow[tp][r], xv);
            }
            mv[k] = xa;
            mv[k + 1] = xv;
            k += 2;
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
          for (int k2 = 0; k2 < C::NMINI; ++k2) sf[C::F_MINI + warp * 32 + k2] = mv[k2];
        }
        __syncthreads();  // ------------------------------------------------ BAR3 (rare)
        float tot[C::NMINI];
#pragma unroll
        for (int k2 = 0; k2 < C::NMINI; ++k2) {
          float x = 0.f;
#pragma unroll
          for (int w = 0; w < NW; ++w) x += sf[C::F_MINI + w * 32 + k2];
          tot[k2] = x;
        }
        // sequential decisions on ||S_reg_t||^2 (S_reg unscaled, scale sigma before step t)
        float nreg2 = ws;
        float sgc = sigma;
#pragma unroll
        for (int t = 0; t < KS; ++t) {
          isg[t] = __frcp_rn(sgc);
          if (t < cS) {
            // v_t^T S_reg_{t-1} alpha_t = v_t^T S_reg_0 alpha_t + sum_{t'<t} (v_t.v_t')(alpha_t'.alpha_t)/sigma_{t'-1}
            float cross = tot[t];
            int kb = KS + t * (t + 1);   // start of (t, 0) pair in the mini list
#pragma unroll
            for (int tp = 0; tp < t; ++tp) cross = fmaf(tot[kb + 2 * tp + 1] * tot[kb + 2 * tp], isg[tp], cross);
            const float aa = tot[kb + 2 * t], vv = tot[kb + 2 * t + 1];
            nreg2 = fmaf(2.f * isg[t], cross, nreg2);
            nreg2 = fmaf(vv * aa, isg[t] * isg[t], nreg2);
            const float npre = sgc * sqrtf(fmaxf(nreg2, 0.f));
            if (npre > tau) {
              sgc *= tau / npre;
              ++renorm_cnt;
            }
            if (!isfinite(npre)) flags |= kStatusNonfinite;
          }
          sg[t] = sgc;
        }
      }
      // outputs o_t = sigma_t (Y_t + sum_{t'<=t} v_t' aq_{t,t'} / sigma_{t'-1}) / den_t
      {
        const int h = tid / D, i = tid - (tid / D) * D;
#pragma unroll
        for (int jj = 0; jj < (KS + 1) / 2; ++jj) {
#pragma unroll
          for (int tt = 2 * jj; tt < 2 * jj + 2 && tt < KS; ++tt) {
            if (tt == 2 * jj + h && tt < cS) {
              const int rs = recS(tt);
              float x = sf[ybuf + tt * D + i];
#pragma unroll
              for (int tp = 0; tp <= tt; ++tp) {
                const float aq = res[C::NJG + C::NJH + tt * (tt + 1) / 2 + tp];
                x = fmaf(sf[recS(tp) + C::OFF_V + i] * aq, isg[tp], x);
              }
              const float o = sg[tt] * x / sf[rs + C::OFF_SC];
              if (!isfinite(o)) flags |= kStatusNonfinite;
              go[(gS0 + tt) * D + i] = from_f32<TIO>(o);
            }
          }
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
            const float4 al = *reinterpret_cast<const float4*>(sf + abuf_prev + t * D + colof(kk, 0));
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
      if (sigma < 0x1p-16f) {   // fold the scale back into S_reg
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
          for (int p = 0; p < NCP; ++p) { S2[r][p].x *= sigma; S2[r][p].y *= sigma; }
        sigma = 1.f;
      }
    }

    // ================= advance
    if (tid == 0) {
      if (haveA && !isfinite(Dv[0])) flags |= kStatusNonfinite;
    }
    if (apply) {
      cS = cA;
      baseS = recA(0);
      gS0 = gA0;
    } else {
      cS = 0;
    }
    if (haveA) {
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
  }

  if (timed_out) {
    if (tid == 0) {
      for (int j = loaded + 1; j < ntiles && j <= loaded + NSTAGE; ++j)
        (void)mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)((j / NSTAGE) & 1));
      atomicOr(&a.status->flags, kStatusTimeout);
    }
    return;
  }

  // ---- state out
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
#pragma unroll
    for (int kk = 0; kk < NCH; ++kk) {
      const float4 av = make_float4(A2[r][2 * kk].x, A2[r][2 * kk].y, A2[r][2 * kk + 1].x, A2[r][2 * kk + 1].y);
      const float4 sv = make_float4(sigma * S2[r][2 * kk].x, sigma * S2[r][2 * kk].y, sigma * S2[r][2 * kk + 1].x,
                                    sigma * S2[r][2 * kk + 1].y);
      *reinterpret_cast<float4*>(gA + (row0 + r) * D + colof(kk, 0)) = av;
      *reinterpret_cast<float4*>(gS + (row0 + r) * D + colof(kk, 0)) = sv;
    }
  }
  if (tid < D) gn[tid] = n_i;
  if (flags) atomicOr(&a.status->flags, flags);   // any thread may have seen a non-finite value
  if (tid == 0) {
    if (guard_cnt) atomicAdd(&a.status->guard_count, guard_cnt);
    if (renorm_cnt) atomicAdd(&a.status->renorm_count, renorm_cnt);
    if (replay_cnt) atomicAdd(&a.status->chunk_fallbacks, replay_cnt);
  }
}

template <int D, int R, int KS, typename TIO>
cudaError_t launch_seq_block_t(const ScanArgs& a, cudaStream_t s) {
  using C = blk::Cfg<D, R, KS, TIO>;
  auto kern = seq_block_kernel<D, R, KS, TIO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.pairs, blk::Geom<D>::NT, C::bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vla
