// Delta-rule variant of the VLA scan for sm_103a: one CTA per (batch, head) pair,
// one step (one reduction round per direction) at a time.
//
// The gist.science summary §2.3 ("Recursive Update Rule") writes the state with a
// residual and unit-length vectors: A_t is tracked exactly as in the additive
// scan (Sherman-Morrison with the guard, periodic nudging), then
//   alpha_hat_t = A_t k_hat_t / |A_t k_hat_t|,   k_hat_t = phi(k_t) / |phi(k_t)|,
//   S_t = S_{t-1} + (v_t - S_{t-1} k_hat_t) alpha_hat_t^T,
// with the additive scan's normaliser n, renormalisation (||S||_F > tau) and
// readout o_t = S_t phi(q_t) / (n_t . phi(q_t) + 1e-6).  Unit length is x / max(|x|,
// 1e-12).
//
// Layout on chip
//   * A and S (float32) live in registers for the whole scan.  Thread t owns
//     row  i = t / 4  of both, and the 4-column groups {16 kk + 4 c .. +3},
//     c = t % 4, kk = 0 .. d/16 - 1 (so the four lanes of a row read four
//     consecutive 16-byte pieces of every broadcast vector: no bank conflicts).
//   * q, k, v, u stream in through a two-stage ring of bulk asynchronous copies
//     (cp.async.bulk + mbarrier, one copy per array per tile of TS steps); a
//     prologue per tile turns them into float32 phi(q), phi(k), s, u, v records.
//
// One reduction round per direction: every thread forms partial dot products of
// its row piece (A u, A s, S phi(q), S s, ||S||^2); two xor-shuffles finish the row
// sums inside the 4-lane group; the scalars (u.z, s.z, n.phi(q), ||S||^2) reduce
// across the CTA in the same round.  After it, alpha = A_t s = w - z (s.z)/delta
// (+ the guard's and the nudge's eps s) is formed column-wise in every row group,
// and |alpha|, alpha . phi(q) and |s| are summed over the group's four lanes (the
// same numbers in every group, so no second block reduction).  With S = sigma S_reg:
//   S_{t-1} k_hat = sigma (S_reg s) / |s|,   r = v - S_{t-1} k_hat,
//   S_reg += (r / (sigma |alpha|)) alpha^T,  S_t phi(q) = sigma (S_reg phi(q)) + r (alpha . phi(q)) / |alpha|.
// The norm of S_t is reduced in round t+1 and o_t written one step late, as in
// the additive kernels; a final norm-only round settles the last step.
#pragma once

#include "vla_internal.cuh"

namespace vla {

namespace dlt {
constexpr float kGuardEps = 1e-6f;    // singularity threshold and injected diagonal
constexpr float kReadoutEps = 1e-6f;  // readout denominator offset
constexpr float kNormEps = 1e-12f;    // floor of the norms of the unit vectors

template <int D>
struct Cfg {
  static constexpr int NT = 4 * D;       // threads: D rows x 4 column lanes
  static constexpr int NW = NT / 32;     // warps
  static constexpr int CPT = D / 4;      // columns per thread
  static constexpr int NCH = CPT / 4;    // float4 pieces per thread and vector
  static constexpr int TS = D <= 16 ? 64 : (D <= 64 ? 32 : 16);  // steps per tile
  static constexpr int NSTAGE = 2;
};

template <int D, int R, typename TIO>
struct Smem {
  using C = Cfg<D>;
  static constexpr int REC = (R + 4) * D;             // floats per step record
  static constexpr int OFF_U = 0;                     // u_{t,1..R}
  static constexpr int OFF_S = R * D;                 // s = phi(k)/sqrt(d)
  static constexpr int OFF_Q = (R + 1) * D;           // phi(q)
  static constexpr int OFF_K = (R + 2) * D;           // phi(k)
  static constexpr int OFF_V = (R + 3) * D;           // v
  static constexpr uint32_t QB = C::TS * D * sizeof(TIO);       // q, k or v bytes per tile
  static constexpr uint32_t UB = C::TS * R * D * sizeof(TIO);   // u bytes per tile
  static constexpr uint32_t STAGE = 3 * QB + UB;
  static constexpr size_t raw_off = 0;
  static constexpr size_t pre_off = raw_off + C::NSTAGE * STAGE;
  static constexpr size_t zb_off = pre_off + sizeof(float) * C::TS * REC;
  static constexpr size_t wb_off = zb_off + sizeof(float) * 2 * D;
  static constexpr size_t red_off = wb_off + sizeof(float) * 2 * D;
  static constexpr size_t bar_off = (red_off + sizeof(float) * 2 * C::NW * 8 + 15) / 16 * 16;
  static constexpr size_t flag_off = bar_off + sizeof(uint64_t) * C::NSTAGE;
  static constexpr size_t bytes = flag_off + 16;
  static_assert(QB % 16 == 0 && UB % 16 == 0, "tile sizes must be multiples of 16 bytes");
};

}  // namespace dlt

template <int D, int R, typename TIO>
__global__ void __launch_bounds__(dlt::Cfg<D>::NT, 1) delta_scan_kernel(ScanArgs a) {
  using namespace dlt;
  using C = Cfg<D>;
  using L = Smem<D, R, TIO>;
  constexpr int NT = C::NT, NW = C::NW, CPT = C::CPT, NCH = C::NCH, TS = C::TS, NSTAGE = C::NSTAGE;
  constexpr int REC = L::REC;
  constexpr float kInvSqrtD = (float)(D == 16 ? 0.25 : D == 64 ? 0.125 : 0.08838834764831845);
  static_assert(D == 16 || D == 64 || D == 128, "built head widths");

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* raw = smem + L::raw_off;
  float* pre = reinterpret_cast<float*>(smem + L::pre_off);
  float* zbuf = reinterpret_cast<float*>(smem + L::zb_off);
  float* wbuf = reinterpret_cast<float*>(smem + L::wb_off);
  float* red = reinterpret_cast<float*>(smem + L::red_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + L::flag_off);

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int row = tid >> 2, c = tid & 3;
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

  // ---- state into registers
  float Ar[CPT], Sr[CPT];
#pragma unroll
  for (int kk = 0; kk < NCH; ++kk) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = 16 * kk + 4 * c + e;
      Ar[4 * kk + e] = gA[row * D + col];
      Sr[4 * kk + e] = gS[row * D + col];
    }
  }
  float n_row = gn[row];
  // the diagonal entry (row, row) sits in the thread with c == (row % 16) / 4
  const bool own_diag = (c == ((row & 15) >> 2));
  const int diag_slot = 4 * (row >> 4) + (row & 3);

  const int ntiles = (int)((T + TS - 1) / TS);
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    *flag = 0;
  }
  __syncthreads();

  auto issue = [&](int tile) {  // thread 0 only
    const int stage = tile % NSTAGE;
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const uint32_t qb = (uint32_t)nst * D * sizeof(TIO);
    const uint32_t ub = (uint32_t)nst * R * D * sizeof(TIO);
    unsigned char* base = raw + stage * L::STAGE;
    mbar_arrive_expect_tx(&bars[stage], 3 * qb + ub);
    bulk_g2s(base, gq + t_start * D, qb, &bars[stage]);
    bulk_g2s(base + L::QB, gk + t_start * D, qb, &bars[stage]);
    bulk_g2s(base + 2 * L::QB, gv + t_start * D, qb, &bars[stage]);
    bulk_g2s(base + 3 * L::QB, gu + t_start * R * D, ub, &bars[stage]);
  };
  if (tid == 0) {
    for (int j = 0; j < NSTAGE && j < ntiles; ++j) issue(j);
  }

  float sigma = 1.f;                 // S = sigma * S_reg
  float num_prev = 0.f, den_prev = 1.f;
  bool have_prev = false;
  long long t_prev = 0;
  unsigned long long guard_cnt = 0, renorm_cnt = 0;
  unsigned int flags = 0;
  int buf = 0;
  int phase = (a.P > 0) ? (int)(a.t0 % a.P) : 0;   // (t0 + t) mod P before step t+1
  bool timed_out = false;
  int tile = 0;

  for (; tile < ntiles; ++tile) {
    const int stage = tile % NSTAGE;
    const uint32_t parity = (uint32_t)((tile / NSTAGE) & 1);
    if (tid == 0) {
      if (!mbar_wait_bounded(&bars[stage], parity)) *flag = 1;
    }
    __syncthreads();
    if (*flag) { timed_out = true; break; }
    const long long t_base = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_base);

    // ---- prologue: float32 step records
    {
      const TIO* rq = reinterpret_cast<const TIO*>(raw + stage * L::STAGE);
      const TIO* rk = reinterpret_cast<const TIO*>(raw + stage * L::STAGE + L::QB);
      const TIO* rv = reinterpret_cast<const TIO*>(raw + stage * L::STAGE + 2 * L::QB);
      const TIO* ru = reinterpret_cast<const TIO*>(raw + stage * L::STAGE + 3 * L::QB);
      for (int e = tid; e < nst * REC; e += NT) {
        const int tt = e / REC, off = e - tt * REC;
        float val;
        if (off < L::OFF_S) {
          val = to_f32(ru[tt * R * D + off]);
        } else if (off < L::OFF_Q) {
          val = phi_elu1(to_f32(rk[tt * D + off - L::OFF_S])) * kInvSqrtD;
        } else if (off < L::OFF_K) {
          val = phi_elu1(to_f32(rq[tt * D + off - L::OFF_Q]));
        } else if (off < L::OFF_V) {
          val = phi_elu1(to_f32(rk[tt * D + off - L::OFF_K]));
        } else {
          val = to_f32(rv[tt * D + off - L::OFF_V]);
        }
        pre[e] = val;
      }
    }
    __syncthreads();
    if (tid == 0 && tile + NSTAGE < ntiles) {
      fence_proxy_async_smem();
      issue(tile + NSTAGE);
    }

    for (int tt = 0; tt < nst; ++tt) {
      const float* rec = pre + tt * REC;
      float zr = 0.f, wr = 0.f, yr = 0.f, ksr = 0.f, delta = 1.f;
      float tot[8];
      bool guard = false;
      int lb = buf;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const bool last = (i == R - 1);
        const float* uvec = rec + L::OFF_U + i * D;
        float zp[4] = {0.f, 0.f, 0.f, 0.f}, wp[4] = {0.f, 0.f, 0.f, 0.f};
        float yp[4] = {0.f, 0.f, 0.f, 0.f}, sp[4] = {0.f, 0.f, 0.f, 0.f}, ksp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < NCH; ++kk) {
          const int col = 16 * kk + 4 * c;
          const float4 u4 = *reinterpret_cast<const float4*>(uvec + col);
          const float* a4 = &Ar[4 * kk];
          zp[0] = fmaf(a4[0], u4.x, zp[0]);
          zp[1] = fmaf(a4[1], u4.y, zp[1]);
          zp[2] = fmaf(a4[2], u4.z, zp[2]);
          zp[3] = fmaf(a4[3], u4.w, zp[3]);
          if (last) {
            const float4 s4 = *reinterpret_cast<const float4*>(rec + L::OFF_S + col);
            const float4 q4 = *reinterpret_cast<const float4*>(rec + L::OFF_Q + col);
            const float* s_ = &Sr[4 * kk];
            wp[0] = fmaf(a4[0], s4.x, wp[0]);
            wp[1] = fmaf(a4[1], s4.y, wp[1]);
            wp[2] = fmaf(a4[2], s4.z, wp[2]);
            wp[3] = fmaf(a4[3], s4.w, wp[3]);
            yp[0] = fmaf(s_[0], q4.x, yp[0]);
            yp[1] = fmaf(s_[1], q4.y, yp[1]);
            yp[2] = fmaf(s_[2], q4.z, yp[2]);
            yp[3] = fmaf(s_[3], q4.w, yp[3]);
            sp[0] = fmaf(s_[0], s_[0], sp[0]);
            sp[1] = fmaf(s_[1], s_[1], sp[1]);
            sp[2] = fmaf(s_[2], s_[2], sp[2]);
            sp[3] = fmaf(s_[3], s_[3], sp[3]);
            ksp[0] = fmaf(s_[0], s4.x, ksp[0]);   // S_reg s
            ksp[1] = fmaf(s_[1], s4.y, ksp[1]);
            ksp[2] = fmaf(s_[2], s4.z, ksp[2]);
            ksp[3] = fmaf(s_[3], s4.w, ksp[3]);
          }
        }
        float z = (zp[0] + zp[1]) + (zp[2] + zp[3]);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        float w = 0.f, y = 0.f, ns = 0.f, ks = 0.f;
        if (last) {
          w = (wp[0] + wp[1]) + (wp[2] + wp[3]);
          y = (yp[0] + yp[1]) + (yp[2] + yp[3]);
          ns = (sp[0] + sp[1]) + (sp[2] + sp[3]);
          ks = (ksp[0] + ksp[1]) + (ksp[2] + ksp[3]);
          w += __shfl_xor_sync(0xffffffffu, w, 1);
          y += __shfl_xor_sync(0xffffffffu, y, 1);
          ns += __shfl_xor_sync(0xffffffffu, ns, 1);
          ks += __shfl_xor_sync(0xffffffffu, ks, 1);
          w += __shfl_xor_sync(0xffffffffu, w, 2);
          y += __shfl_xor_sync(0xffffffffu, y, 2);
          ns += __shfl_xor_sync(0xffffffffu, ns, 2);
          ks += __shfl_xor_sync(0xffffffffu, ks, 2);
        }
        // scalar partials of this row; lane c carries scalars c and c + 4
        const float u_i = uvec[row];
        float sa, sb;
        if (!last) {
          sa = (c == 0) ? u_i * z : 0.f;
          sb = 0.f;
        } else {
          const float s_i = rec[L::OFF_S + row];
          const float q_i = rec[L::OFF_Q + row];
          const float k_i = rec[L::OFF_K + row];
          sa = (c == 0) ? u_i * z : (c == 1) ? s_i * z : (c == 2) ? q_i * z : q_i * w;
          sb = (c == 0) ? (n_row + k_i) * q_i : (c == 1) ? ns : (c == 2) ? s_i * q_i : 0.f;
        }
        sa += __shfl_xor_sync(0xffffffffu, sa, 4);
        sb += __shfl_xor_sync(0xffffffffu, sb, 4);
        sa += __shfl_xor_sync(0xffffffffu, sa, 8);
        sb += __shfl_xor_sync(0xffffffffu, sb, 8);
        sa += __shfl_xor_sync(0xffffffffu, sa, 16);
        sb += __shfl_xor_sync(0xffffffffu, sb, 16);
        float* rb = red + buf * NW * 8;
        if (lane < 4) {
          rb[warp * 8 + lane] = sa;
          rb[warp * 8 + 4 + lane] = sb;
        }
        if (c == 0) zbuf[buf * D + row] = z;
        if (last && c == 1) wbuf[buf * D + row] = w;
        __syncthreads();
        if (last) {
#pragma unroll
          for (int s = 0; s < 8; ++s) tot[s] = 0.f;
#pragma unroll
          for (int ww = 0; ww < NW; ++ww) {
            const float4 p0 = *reinterpret_cast<const float4*>(rb + ww * 8);
            const float4 p1 = *reinterpret_cast<const float4*>(rb + ww * 8 + 4);
            tot[0] += p0.x; tot[1] += p0.y; tot[2] += p0.z; tot[3] += p0.w;
            tot[4] += p1.x; tot[5] += p1.y; tot[6] += p1.z; tot[7] += p1.w;
          }
        } else {
          tot[0] = 0.f;
#pragma unroll
          for (int ww = 0; ww < NW; ++ww) tot[0] += rb[ww * 8];
        }
        delta = 1.f + tot[0];
        guard = fabsf(delta) < kGuardEps;
        if (!guard) {
          const float zs = z / delta;
#pragma unroll
          for (int kk = 0; kk < NCH; ++kk) {
            const float4 z4 = *reinterpret_cast<const float4*>(zbuf + buf * D + 16 * kk + 4 * c);
            Ar[4 * kk + 0] = fmaf(-zs, z4.x, Ar[4 * kk + 0]);
            Ar[4 * kk + 1] = fmaf(-zs, z4.y, Ar[4 * kk + 1]);
            Ar[4 * kk + 2] = fmaf(-zs, z4.z, Ar[4 * kk + 2]);
            Ar[4 * kk + 3] = fmaf(-zs, z4.w, Ar[4 * kk + 3]);
          }
        } else if (own_diag) {
#pragma unroll
          for (int j = 0; j < CPT; ++j)
            if (j == diag_slot) Ar[j] += kGuardEps;
        }
        if (tid == 0) {
          if (guard) ++guard_cnt;
          if (!isfinite(delta)) flags |= kStatusNonfinite;
        }
        zr = z; wr = w; yr = y; ksr = ks;
        lb = buf;
        buf ^= 1;
      }

      // ---- step tail: nudge, renormalisation of the previous step, alpha, S update
      const float gam = tot[1], nu = tot[4], nS = tot[5];
      bool nudge = false;
      if (a.P > 0) {
        if (++phase == a.P) { nudge = true; phase = 0; }
      }
      if (have_prev) {
        const float nrm = sigma * sqrtf(nS);
        float cf = 1.f;
        if (nrm > a.tau) {
          cf = a.tau / nrm;
          sigma *= cf;
          if (tid == 0) ++renorm_cnt;
        }
        if (tid == 0 && !isfinite(nrm)) flags |= kStatusNonfinite;
        if (c == 0) go[t_prev * D + row] = from_f32<TIO>(cf * num_prev / den_prev);
      }
      const float yv = sigma * yr;                // S_{t-1} phi(q_t) for this row
      const float yk = sigma * ksr;               // S_{t-1} s_t for this row (before the fold below)
      if (sigma < 0x1p-16f) {                     // keep S_reg (and its squared norm) in range
#pragma unroll
        for (int j = 0; j < CPT; ++j) Sr[j] *= sigma;
        sigma = 1.f;
      }
      const float gd = guard ? 0.f : gam / delta;
      const float ga = guard ? kGuardEps : 0.f;
      const float na = nudge ? a.eps_n : 0.f;
      if (nudge && own_diag) {
#pragma unroll
        for (int j = 0; j < CPT; ++j)
          if (j == diag_slot) Ar[j] += a.eps_n;
      }
      // alpha = A_t s on this thread's columns; |alpha|^2, alpha . phi(q), |s|^2 over the row group
      float al[CPT];
      float an = 0.f, aqp = 0.f, ssp = 0.f;
#pragma unroll
      for (int kk = 0; kk < NCH; ++kk) {
        const int col = 16 * kk + 4 * c;
        const float4 w4 = *reinterpret_cast<const float4*>(wbuf + lb * D + col);
        const float4 z4 = *reinterpret_cast<const float4*>(zbuf + lb * D + col);
        const float4 s4 = *reinterpret_cast<const float4*>(rec + L::OFF_S + col);
        const float4 q4 = *reinterpret_cast<const float4*>(rec + L::OFF_Q + col);
        al[4 * kk + 0] = fmaf(-gd, z4.x, fmaf(ga + na, s4.x, w4.x));
        al[4 * kk + 1] = fmaf(-gd, z4.y, fmaf(ga + na, s4.y, w4.y));
        al[4 * kk + 2] = fmaf(-gd, z4.z, fmaf(ga + na, s4.z, w4.z));
        al[4 * kk + 3] = fmaf(-gd, z4.w, fmaf(ga + na, s4.w, w4.w));
        an = fmaf(al[4 * kk + 0], al[4 * kk + 0], fmaf(al[4 * kk + 1], al[4 * kk + 1], an));
        an = fmaf(al[4 * kk + 2], al[4 * kk + 2], fmaf(al[4 * kk + 3], al[4 * kk + 3], an));
        aqp = fmaf(al[4 * kk + 0], q4.x, fmaf(al[4 * kk + 1], q4.y, aqp));
        aqp = fmaf(al[4 * kk + 2], q4.z, fmaf(al[4 * kk + 3], q4.w, aqp));
        ssp = fmaf(s4.x, s4.x, fmaf(s4.y, s4.y, ssp));
        ssp = fmaf(s4.z, s4.z, fmaf(s4.w, s4.w, ssp));
      }
      an += __shfl_xor_sync(0xffffffffu, an, 1);
      aqp += __shfl_xor_sync(0xffffffffu, aqp, 1);
      ssp += __shfl_xor_sync(0xffffffffu, ssp, 1);
      an += __shfl_xor_sync(0xffffffffu, an, 2);
      aqp += __shfl_xor_sync(0xffffffffu, aqp, 2);
      ssp += __shfl_xor_sync(0xffffffffu, ssp, 2);
      // alpha = A_t s is A_t k_hat times |phi(k)| / sqrt(d), so alpha_hat = alpha / |alpha| (the
      // floor applies to |A_t k_hat| = |alpha| sqrt(d) / |phi(k)| in the pages' convention)
      const float inv_a = 1.f / fmaxf(sqrtf(an), kNormEps);
      const float inv_k = 1.f / fmaxf(sqrtf(ssp) * sqrtf((float)D), kNormEps);   // 1 / |phi(k)|
      const float v_i = rec[L::OFF_V + row];
      const float res = v_i - yk * sqrtf((float)D) * inv_k;   // v - S_{t-1} k_hat, k_hat = s sqrt(d) / |phi(k)|
      num_prev = yv + res * aqp * inv_a;          // S_t phi(q_t) before renormalisation
      den_prev = nu + kReadoutEps;                // n_t . phi(q_t) + 1e-6
      have_prev = true;
      t_prev = t_base + tt;
      const float rs = res * inv_a / sigma;
#pragma unroll
      for (int j = 0; j < CPT; ++j) Sr[j] = fmaf(rs, al[j], Sr[j]);
      if (tid == 0 && !(isfinite(nu) && isfinite(aqp) && isfinite(an) && isfinite(yv))) flags |= kStatusNonfinite;
      n_row += rec[L::OFF_K + row];
    }
  }

  if (timed_out) {
    // let copies already in flight land before the CTA's shared memory is released
    if (tid == 0) {
      for (int j = tile; j < ntiles && j < tile + NSTAGE; ++j)
        (void)mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)((j / NSTAGE) & 1));
      atomicOr(&a.status->flags, kStatusTimeout);
    }
    return;
  }

  // ---- settle the last step: one norm-only round
  if (have_prev) {
    float sp = 0.f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) sp = fmaf(Sr[j], Sr[j], sp);
    sp += __shfl_xor_sync(0xffffffffu, sp, 1);
    sp += __shfl_xor_sync(0xffffffffu, sp, 2);
    float sa = (c == 0) ? sp : 0.f;
    sa += __shfl_xor_sync(0xffffffffu, sa, 4);
    sa += __shfl_xor_sync(0xffffffffu, sa, 8);
    sa += __shfl_xor_sync(0xffffffffu, sa, 16);
    float* rb = red + buf * NW * 8;
    if (lane == 0) rb[warp * 8] = sa;
    __syncthreads();
    float nS = 0.f;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) nS += rb[ww * 8];
    const float nrm = sigma * sqrtf(nS);
    float cf = 1.f;
    if (nrm > a.tau) {
      cf = a.tau / nrm;
      sigma *= cf;
      if (tid == 0) ++renorm_cnt;
    }
    if (tid == 0 && !isfinite(nrm)) flags |= kStatusNonfinite;
    if (c == 0) go[t_prev * D + row] = from_f32<TIO>(cf * num_prev / den_prev);
  }

  // ---- state out
#pragma unroll
  for (int kk = 0; kk < NCH; ++kk) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = 16 * kk + 4 * c + e;
      gA[row * D + col] = Ar[4 * kk + e];
      gS[row * D + col] = sigma * Sr[4 * kk + e];
    }
  }
  if (c == 0) gn[row] = n_row;
  if (tid == 0) {
    if (flags) atomicOr(&a.status->flags, flags);
    if (guard_cnt) atomicAdd(&a.status->guard_count, guard_cnt);
    if (renorm_cnt) atomicAdd(&a.status->renorm_count, renorm_cnt);
  }
}

template <int D, int R, typename TIO>
cudaError_t launch_delta_t(const ScanArgs& a, cudaStream_t s) {
  using L = dlt::Smem<D, R, TIO>;
  auto kern = delta_scan_kernel<D, R, TIO>;
  // set on every launch: the attribute belongs to the current device's context
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.pairs, dlt::Cfg<D>::NT, L::bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vla
