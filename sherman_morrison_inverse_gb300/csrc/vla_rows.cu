// Row-split sequential VLA scan for sm_103a: one (batch, head) pair on a cluster of NC CTAs,
// for workloads with fewer pairs than SMs.  The recurrence is the step-by-step one
// ("Mathematical Primitives" §2-§5, README "VLA v3" items 1-5, r = 1):
//
//   z = A u, delta = 1 + u.z;  |delta| < 1e-6: A += 1e-6 I,  else A -= z z^T / delta
//   every P-th global step A += eps_n I;  alpha = A s,  s = phi(k) / sqrt(d)
//   S += v alpha^T,  n += phi(k);  ||S||_F > tau: S *= tau / ||S||_F
//   o = S phi(q) / (n.phi(q) + 1e-6)
//
// CTA c of the cluster owns rows R_c = [c RB, (c + 1) RB) of A and the same columns of S
// (RB = d / NC), both in registers, and the matching slice of n.  Per step it forms its slice
// of z and of y = A_old s, and the partial sums u_Rc.z_Rc and z_Rc.s_Rc.  Since
// A_new s = y - z (z.s) / delta (or y + 1e-6 s under the guard, then + eps_n s at a nudge),
// alpha's slice needs no second pass over A.  S's columns R_c take v alpha_Rc^T; the CTA then
// has partial sums of S phi(q) (all d_v rows), of ||S||^2 and of n.phi(q).
//
// One exchange per step through distributed shared memory: every CTA writes, into every
// CTA's slot (double-buffered by step parity), its slice of the next step's z and its two
// scalars, its S phi(q) partials for the outputs that CTA owns (a reduce-scatter: CTA c
// writes o rows [c d/NC, (c + 1) d/NC)), its ||S||^2 and n.phi(q) partials and a failure
// flag; then one hardware cluster barrier (arrive.release / wait.acquire).  Every CTA sums
// the partials in the same order, so delta, the guard, the renormalisation and the exit
// decisions are the same bits in all of them: control flow stays uniform across the
// cluster, and no CTA leaves a barrier that the others wait on.  The renormalisation of
// step t and its outputs are applied after the exchange, before step t + 1 updates S.
//
// Inputs: q, k, v, u of TS steps arrive by 1-D bulk copies (cp.async.bulk) into a two-stage
// ring completing on mbarriers (waits bounded at 2 s; a wait that runs out is carried to
// every CTA of the cluster through the exchange, and all of them stop at the same step with
// VLA_STATUS_TIMEOUT); each tile is converted once into float32 step records (u, s, v, and
// phi(q), phi(k) of the CTA's columns), double-buffered so that conversion needs no extra
// barrier.
#include "vla_internal.cuh"

namespace vla {
namespace rows {

constexpr int NTH = 128;
constexpr float kGuardEps = 1e-6f;
constexpr float kReadoutEps = 1e-6f;

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int D, int NC, typename TIO>
struct Cfg {
  static constexpr int RB = D / NC;             // rows of A / columns of S per CTA
  static constexpr int LA = NTH / RB;           // lanes per row of A
  static constexpr int CA = D / LA;             // columns of A per thread
  static constexpr int LS = NTH / D;            // lanes per row of S (d_v = d)
  static constexpr int CS = RB / LS;            // columns of S per thread
  static constexpr int OB = D / NC;             // outputs per CTA
  static constexpr int TS = D == 128 ? 16 : 32; // steps per input tile
  static constexpr int RAW = TS * 4 * D * (int)sizeof(TIO);   // q, k, v, u of a tile
  static constexpr int REC = TS * (3 * D + 2 * RB);           // floats: U, SG, V [TS][D]; PQ, PK [TS][RB]
  static constexpr int R_U = 0, R_SG = TS * D, R_V = 2 * TS * D, R_PQ = 3 * TS * D, R_PK = 3 * TS * D + TS * RB;
  // exchange slot (floats): z[D] | dp[NC][4] | zsp[NC][4] | p[NC][OB] | nrm[NC][4] | den[NC] | fl[NC]
  static constexpr int X_Z = 0, X_DP = D, X_ZS = X_DP + 4 * NC, X_P = X_ZS + 4 * NC, X_NRM = X_P + NC * OB,
                       X_DEN = X_NRM + 4 * NC, X_FL = X_DEN + NC;
  static constexpr int SLOT = (X_FL + NC + 3) / 4 * 4;
  static constexpr int F_REC = 0;                          // float offsets after the raw ring
  static constexpr int F_SLOT = F_REC + 2 * REC;
  static constexpr int F_AL = F_SLOT + 2 * SLOT;          // alpha's slice [RB]
  static constexpr int F_END = F_AL + (RB + 3) / 4 * 4;
  static constexpr size_t bar_off = (size_t)2 * RAW + sizeof(float) * F_END;
  static constexpr size_t bytes = bar_off + 16;            // two mbarriers
  static_assert(NTH % RB == 0 && LA <= 32 && (LA & (LA - 1)) == 0 && CA % 4 == 0, "A mapping");
  static_assert(NTH % D == 0 || D == 128, "S mapping");
  static_assert(LS >= 1 && CS % 4 == 0 && RB <= 32 && OB <= NTH, "S mapping");
  static_assert(RAW % 16 == 0 && (TS * D * (int)sizeof(TIO)) % 16 == 0, "bulk copy sizes");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

template <int D, int NC, typename TIO>
__global__ void __launch_bounds__(NTH, 1) rows_scan_kernel(ScanArgs a) {
  using Cf = Cfg<D, NC, TIO>;
  constexpr int RB = Cf::RB, LA = Cf::LA, CA = Cf::CA, LS = Cf::LS, CS = Cf::CS, OB = Cf::OB, TS = Cf::TS;
  constexpr float kInvSqrtD = D == 128 ? 0.08838834764831845f : D == 64 ? 0.125f : 0.25f;
  extern __shared__ __align__(128) unsigned char smem[];
  float* sf = reinterpret_cast<float*>(smem + 2 * Cf::RAW);
  uint64_t* in_bar = reinterpret_cast<uint64_t*>(smem + Cf::bar_off);   // [2] input stages

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = (int)cluster_ctarank();
  const long long pair = blockIdx.x / NC;
  const long long T = a.T;
  const TIO* gq = static_cast<const TIO*>(a.q) + pair * T * D;
  const TIO* gk = static_cast<const TIO*>(a.k) + pair * T * D;
  const TIO* gv = static_cast<const TIO*>(a.v) + pair * T * D;
  const TIO* gu = static_cast<const TIO*>(a.u) + pair * T * D;
  TIO* go = static_cast<TIO*>(a.o) + pair * T * D;
  float* gA = a.A + pair * D * D;
  float* gS = a.S + pair * D * D;
  float* gn = a.n + pair * D;

  // A mapping: row ra of this CTA's block (global row gi), columns 4 (pa + LA m') + e
  const int ra = tid / LA, pa = tid % LA, gi = c * RB + ra;
  // S mapping: row rs, local columns 4 (ps + LS m') + e of this CTA's block
  const int rs = tid / LS, ps = tid % LS;
  auto acol = [&](int m) { return 4 * (pa + LA * (m >> 2)) + (m & 3); };
  auto scol = [&](int m) { return 4 * (ps + LS * (m >> 2)) + (m & 3); };
  const int dm = ((gi >> 2) % LA == pa) ? 4 * ((gi >> 2) / LA) + (gi & 3) : -1;   // the diagonal's slot

  float Ar[CA], Sr[CS];
#pragma unroll
  for (int m = 0; m < CA; ++m) Ar[m] = gA[(long long)gi * D + acol(m)];
#pragma unroll
  for (int m = 0; m < CS; ++m) Sr[m] = gS[(long long)rs * D + c * RB + scol(m)];
  float nr = (warp == 0 && lane < RB) ? gn[c * RB + lane] : 0.f;   // n of column c RB + lane
  auto add_diag = [&](float x) {   // A[gi][gi] += x (a static register index, no local memory)
#pragma unroll
    for (int m = 0; m < CA; ++m)
      if (m == dm) Ar[m] += x;
  };

  const int ntiles = (int)((T + TS - 1) / TS);
  auto issue = [&](int tile) {   // one thread
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const uint32_t qb = (uint32_t)nst * D * sizeof(TIO);
    unsigned char* st = smem + (tile & 1) * Cf::RAW;
    uint64_t* bar = in_bar + (tile & 1);
    mbar_arrive_expect_tx(bar, 4 * qb);
    bulk_g2s(st, gq + t_start * D, qb, bar);
    bulk_g2s(st + TS * D * sizeof(TIO), gk + t_start * D, qb, bar);
    bulk_g2s(st + 2 * TS * D * sizeof(TIO), gv + t_start * D, qb, bar);
    bulk_g2s(st + 3 * TS * D * sizeof(TIO), gu + t_start * D, qb, bar);
  };
  if (tid == 0) {
    mbar_init(in_bar, 1);
    mbar_init(in_bar + 1, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    issue(0);
    if (ntiles > 1) issue(1);
  }
  int issued = ntiles > 1 ? 1 : 0;   // the last tile whose copy was issued (thread 0's view)

  bool failed = false;   // this CTA: an input wait ran out
  // wait for tile `tile` and convert it into records buffer (tile & 1); every thread waits
  auto load_tile = [&](int tile) {
    const bool ok = mbar_wait_bounded(in_bar + (tile & 1), (uint32_t)((tile >> 1) & 1));
    failed = __syncthreads_or(!ok) != 0 || failed;
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const TIO* rq = reinterpret_cast<const TIO*>(smem + (tile & 1) * Cf::RAW);
    const TIO* rk = rq + TS * D;
    const TIO* rv = rq + 2 * TS * D;
    const TIO* ru = rq + 3 * TS * D;
    float* rec = sf + Cf::F_REC + (tile & 1) * Cf::REC;
    for (int e = tid; e < nst * D; e += NTH) {
      rec[Cf::R_U + e] = to_f32(ru[e]);
      rec[Cf::R_SG + e] = phi_elu1(to_f32(rk[e])) * kInvSqrtD;
      rec[Cf::R_V + e] = to_f32(rv[e]);
    }
    for (int e = tid; e < nst * RB; e += NTH) {
      const int t = e / RB, jj = e - t * RB;
      rec[Cf::R_PQ + e] = phi_elu1(to_f32(rq[t * D + c * RB + jj]));
      rec[Cf::R_PK + e] = phi_elu1(to_f32(rk[t * D + c * RB + jj]));
    }
    __syncthreads();
    if (tid == 0 && tile + 2 < ntiles) {   // the stage is converted: refill it two tiles ahead
      fence_proxy_async_smem();
      issue(tile + 2);
      issued = tile + 2;
    }
  };

  // z and y = A s for step t (records of its tile), and the warp partials of u.z and z.s
  float zi = 0.f, yi = 0.f;
  auto a_partials = [&](long long t, float& dp, float& zsp) {
    const float* rec = sf + Cf::F_REC + (int)((t / TS) & 1) * Cf::REC;
    const int tl = (int)(t % TS);
    const float* U = rec + Cf::R_U + tl * D;
    const float* SG = rec + Cf::R_SG + tl * D;
    float z0 = 0.f, z1 = 0.f, y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int m4 = 0; m4 < CA / 4; ++m4) {
      const float4 u4 = *reinterpret_cast<const float4*>(U + 4 * (pa + LA * m4));
      const float4 s4 = *reinterpret_cast<const float4*>(SG + 4 * (pa + LA * m4));
      z0 = fmaf(Ar[4 * m4], u4.x, z0);
      z1 = fmaf(Ar[4 * m4 + 1], u4.y, z1);
      z0 = fmaf(Ar[4 * m4 + 2], u4.z, z0);
      z1 = fmaf(Ar[4 * m4 + 3], u4.w, z1);
      y0 = fmaf(Ar[4 * m4], s4.x, y0);
      y1 = fmaf(Ar[4 * m4 + 1], s4.y, y1);
      y0 = fmaf(Ar[4 * m4 + 2], s4.z, y0);
      y1 = fmaf(Ar[4 * m4 + 3], s4.w, y1);
    }
    float z = z0 + z1, y = y0 + y1;
#pragma unroll
    for (int o = 1; o < LA; o <<= 1) {
      z += __shfl_xor_sync(0xffffffffu, z, o);
      y += __shfl_xor_sync(0xffffffffu, y, o);
    }
    zi = z;
    yi = y;
    dp = (pa == 0) ? U[gi] * z : 0.f;
    zsp = (pa == 0) ? z * SG[gi] : 0.f;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      dp += __shfl_xor_sync(0xffffffffu, dp, o);
      zsp += __shfl_xor_sync(0xffffffffu, zsp, o);
    }
  };
  // address of float `off` of slot b in CTA `rank`
  auto remote = [&](int b, int off, int rank) {
    return mapa_shared(smem_u32(sf + Cf::F_SLOT + b * Cf::SLOT + off), (uint32_t)rank);
  };
  auto put_a = [&](int b, float dp, float zsp) {   // z slice, u.z and z.s partials -> every CTA
    if (pa == 0)
      for (int r2 = 0; r2 < NC; ++r2) st_cluster_f32(remote(b, Cf::X_Z + gi, r2), zi);
    if (lane == 0)
      for (int r2 = 0; r2 < NC; ++r2) {
        st_cluster_f32(remote(b, Cf::X_DP + 4 * c + warp, r2), dp);
        st_cluster_f32(remote(b, Cf::X_ZS + 4 * c + warp, r2), zsp);
      }
  };

  unsigned int flags = 0;
  unsigned long long guard_cnt = 0, renorm_cnt = 0;
  const float* slot0 = sf + Cf::F_SLOT;
  float* alpha_s = sf + Cf::F_AL;

  // step 0's A partials; the peers' slots exist once every CTA of the cluster is running
  load_tile(0);
  cluster_barrier();
  {
    float dp, zsp;
    a_partials(0, dp, zsp);
    put_a(0, dp, zsp);
    if (tid == 0)
      for (int r2 = 0; r2 < NC; ++r2) st_cluster_f32(remote(0, Cf::X_FL + c, r2), failed ? 1.f : 0.f);
  }
  cluster_barrier();

  long long to_nudge = (a.P > 0) ? a.P - (a.t0 % a.P) : -1;   // steps until the next nudge (1 = this step)
  bool stop = false;
  long long t = 0;
  // finish step t - 1 from slot b: renormalisation and the outputs this CTA owns
  auto finish = [&](int b, long long tp) {
    const float* sl = slot0 + b * Cf::SLOT;
    float nrm2 = 0.f, den = kReadoutEps;
#pragma unroll
    for (int r2 = 0; r2 < NC; ++r2)
#pragma unroll
      for (int w = 0; w < 4; ++w) nrm2 += sl[Cf::X_NRM + 4 * r2 + w];
    float dsum = 0.f;
#pragma unroll
    for (int r2 = 0; r2 < NC; ++r2) dsum += sl[Cf::X_DEN + r2];
    den += dsum;
    const float nrm = sqrtf(nrm2);
    float cf = 1.f;
    if (nrm > a.tau) {
      cf = a.tau / nrm;
#pragma unroll
      for (int m = 0; m < CS; ++m) Sr[m] *= cf;
      if (c == 0 && tid == 0) ++renorm_cnt;
    }
    if (!isfinite(nrm2) && c == 0 && tid == 0) flags |= kStatusNonfinite;
    if (tid < OB) {
      float p = 0.f;
#pragma unroll
      for (int r2 = 0; r2 < NC; ++r2) p += sl[Cf::X_P + r2 * OB + tid];
      go[tp * D + c * OB + tid] = from_f32<TIO>(p * cf / den);
    }
  };

  for (; t < T; ++t) {
    const int b = (int)(t & 1);
    const float* sl = slot0 + b * Cf::SLOT;
    {
      bool any = false;
#pragma unroll
      for (int r2 = 0; r2 < NC; ++r2) any |= sl[Cf::X_FL + r2] != 0.f;
      if (any) { stop = true; break; }
    }
    if (t > 0) finish(b, t - 1);
    // ---- step t: the update of A's rows and alpha's slice
    float dsum = 0.f, zs = 0.f;
#pragma unroll
    for (int r2 = 0; r2 < NC; ++r2)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        dsum += sl[Cf::X_DP + 4 * r2 + w];
        zs += sl[Cf::X_ZS + 4 * r2 + w];
      }
    const float delta = 1.f + dsum;
    const float* rec = sf + Cf::F_REC + (int)((t / TS) & 1) * Cf::REC;
    const int tl = (int)(t % TS);
    const float s_gi = rec[Cf::R_SG + tl * D + gi];
    float al;
    if (fabsf(delta) < kGuardEps) {
      add_diag(kGuardEps);
      al = yi + kGuardEps * s_gi;
      if (c == 0 && tid == 0) ++guard_cnt;
    } else {
      const float g = zi / delta;
#pragma unroll
      for (int m4 = 0; m4 < CA / 4; ++m4) {
        const float4 z4 = *reinterpret_cast<const float4*>(sl + Cf::X_Z + 4 * (pa + LA * m4));
        Ar[4 * m4] = fmaf(-g, z4.x, Ar[4 * m4]);
        Ar[4 * m4 + 1] = fmaf(-g, z4.y, Ar[4 * m4 + 1]);
        Ar[4 * m4 + 2] = fmaf(-g, z4.z, Ar[4 * m4 + 2]);
        Ar[4 * m4 + 3] = fmaf(-g, z4.w, Ar[4 * m4 + 3]);
      }
      al = yi - zi * (zs / delta);
    }
    if (to_nudge == 1) {
      add_diag(a.eps_n);
      al = fmaf(a.eps_n, s_gi, al);
    }
    if (a.P > 0) to_nudge = (to_nudge == 1) ? a.P : to_nudge - 1;
    if (pa == 0) alpha_s[ra] = al;
    __syncthreads();
    // ---- S's columns, n's slice, the partial sums of the readout and the norm
    const float vv = rec[Cf::R_V + tl * D + rs];
    const float* PQ = rec + Cf::R_PQ + tl * RB;
    float p0 = 0.f, p1 = 0.f, q2 = 0.f;
#pragma unroll
    for (int m4 = 0; m4 < CS / 4; ++m4) {
      const float4 a4 = *reinterpret_cast<const float4*>(alpha_s + 4 * (ps + LS * m4));
      const float4 f4 = *reinterpret_cast<const float4*>(PQ + 4 * (ps + LS * m4));
      Sr[4 * m4] = fmaf(vv, a4.x, Sr[4 * m4]);
      Sr[4 * m4 + 1] = fmaf(vv, a4.y, Sr[4 * m4 + 1]);
      Sr[4 * m4 + 2] = fmaf(vv, a4.z, Sr[4 * m4 + 2]);
      Sr[4 * m4 + 3] = fmaf(vv, a4.w, Sr[4 * m4 + 3]);
      p0 = fmaf(Sr[4 * m4], f4.x, p0);
      p1 = fmaf(Sr[4 * m4 + 1], f4.y, p1);
      p0 = fmaf(Sr[4 * m4 + 2], f4.z, p0);
      p1 = fmaf(Sr[4 * m4 + 3], f4.w, p1);
      q2 = fmaf(Sr[4 * m4], Sr[4 * m4], q2);
      q2 = fmaf(Sr[4 * m4 + 1], Sr[4 * m4 + 1], q2);
      q2 = fmaf(Sr[4 * m4 + 2], Sr[4 * m4 + 2], q2);
      q2 = fmaf(Sr[4 * m4 + 3], Sr[4 * m4 + 3], q2);
    }
    float p = p0 + p1;
#pragma unroll
    for (int o = 1; o < LS; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) q2 += __shfl_xor_sync(0xffffffffu, q2, o);
    float dn = 0.f;
    if (warp == 0) {
      if (lane < RB) {
        nr += rec[Cf::R_PK + tl * RB + lane];
        dn = nr * PQ[lane];
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dn += __shfl_xor_sync(0xffffffffu, dn, o);
    }
    // ---- the next step's A partials (its tile converted first, at a tile boundary)
    const int nb = b ^ 1;
    if (t + 1 < T) {
      if ((t + 1) % TS == 0) load_tile((int)((t + 1) / TS));
      float dp, zsp;
      a_partials(t + 1, dp, zsp);
      put_a(nb, dp, zsp);
    }
    // ---- this step's partials -> the CTAs that own them
    if (ps == 0) st_cluster_f32(remote(nb, Cf::X_P + c * OB + (rs % OB), rs / OB), p);
    if (lane == 0)
      for (int r2 = 0; r2 < NC; ++r2) st_cluster_f32(remote(nb, Cf::X_NRM + 4 * c + warp, r2), q2);
    if (tid == 0)
      for (int r2 = 0; r2 < NC; ++r2) {
        st_cluster_f32(remote(nb, Cf::X_DEN + c, r2), dn);
        st_cluster_f32(remote(nb, Cf::X_FL + c, r2), failed ? 1.f : 0.f);
      }
    cluster_barrier();
  }
  if (!stop) {
    finish((int)(T & 1), T - 1);
#pragma unroll
    for (int m = 0; m < CA; ++m) gA[(long long)gi * D + acol(m)] = Ar[m];
#pragma unroll
    for (int m = 0; m < CS; ++m) gS[(long long)rs * D + c * RB + scol(m)] = Sr[m];
    if (warp == 0 && lane < RB) gn[c * RB + lane] = nr;
  } else {
    flags |= kStatusTimeout;
  }
  // copies still in flight land before the CTA leaves (bounded)
  if (tid == 0)
    for (int j = (issued >= 1 ? issued - 1 : 0); j <= issued; ++j)
      (void)mbar_wait_bounded(in_bar + (j & 1), (uint32_t)((j >> 1) & 1));
  if (c == 0 && tid == 0) {
    if (flags) atomicOr(&a.status->flags, flags);
    if (guard_cnt) atomicAdd(&a.status->guard_count, guard_cnt);
    if (renorm_cnt) atomicAdd(&a.status->renorm_count, renorm_cnt);
  }
  if (failed && tid == 0) atomicOr(&a.status->flags, kStatusTimeout);
}

template <int D, int NC, typename TIO>
cudaError_t launch_rows_t(const ScanArgs& a, cudaStream_t s) {
  using Cf = Cfg<D, NC, TIO>;
  auto kern = rows_scan_kernel<D, NC, TIO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::bytes);
  if (e != cudaSuccess) return e;
  if (NC > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.pairs * NC), 1, 1);
  cfg.blockDim = dim3(NTH, 1, 1);
  cfg.dynamicSmemBytes = Cf::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace rows

// Row-split sequential scan: d in {64, 128}, r = 1, `ctas` CTAs per pair (4 or 8).
cudaError_t launch_rows(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built) {
  *built = true;
  if (r == 1 && d == 64 && ctas == 4) return bf16 ? rows::launch_rows_t<64, 4, __nv_bfloat16>(a, s)
                                                   : rows::launch_rows_t<64, 4, float>(a, s);
  if (r == 1 && d == 64 && ctas == 8) return bf16 ? rows::launch_rows_t<64, 8, __nv_bfloat16>(a, s)
                                                   : rows::launch_rows_t<64, 8, float>(a, s);
  if (r == 1 && d == 128 && ctas == 4) return bf16 ? rows::launch_rows_t<128, 4, __nv_bfloat16>(a, s)
                                                    : rows::launch_rows_t<128, 4, float>(a, s);
  if (r == 1 && d == 128 && ctas == 8) return bf16 ? rows::launch_rows_t<128, 8, __nv_bfloat16>(a, s)
                                                    : rows::launch_rows_t<128, 8, float>(a, s);
  *built = false;
  return cudaSuccess;
}

}  // namespace vla
