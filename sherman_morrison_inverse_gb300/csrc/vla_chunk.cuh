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
//   G1  [W^T; Q^T] = [U; Sigma] A_0^T                    W = A_0 U, Q = A_0 Sigma
//   G2  [G - I; H^T] = [W^T; Q^T] U^T                    G = I + U^T A_0 U, H = U^T Q
//       G = L D L^T (CUDA cores; D_jj are the sequential deltas), Linv = L^{-1}
//   G3  [Z; F^T] = [W; H^T] Linv^T                       Z = W L^{-T} (the sequential z's), F = Linv H
//       E = D^{-1} F, masked to directions of steps <= t
//   G4  [Z D^{-1} Z^T ; (Z E)^T] = [Z D^{-1}; E^T] Z^T   A_1 = A_0 - Z D^{-1} Z^T,  alpha = Q - Z E
//   G5  [S alpha_t, alpha.alpha ; S phi(q_t), phi(q_t).alpha] = [alpha; Phi_q] [S; alpha]^T
//   G6  [. ; tril(aq) V] += [V^T; tril(aq)] (V^T)^T     onto G5's S phi(q_t) rows, still in TMEM
//       [V^T alpha ; .]   = [V^T; tril(aq)] (alpha^T)^T
//       o_t = (S phi(q_t) + sum_{t'<=t} (alpha_t'.phi(q_t)) v_t') / den_t,   S_1 = S + V^T alpha
//
// Every product accumulates in its own range of the 512 TMEM columns, so a result can
// stay there while later products run: G2 takes its X operand straight from G1's
// accumulator, and alpha reads Q from it.  G4's X operand [Z D^{-1}; E^T] is written back
// into tensor memory by G3's drain (tcgen05.st; its rows are the drain threads' lanes), so
// G4 reads only its Y operand from shared memory.  The other drains (lane = row of the result)
// write the next operand row-major: float4 stores into the K-major core-matrix layout,
// free of bank conflicts; the transposed operands (W, alpha^T) are written with a
// per-lane register rotation that spreads the lanes over all banks.  G2 is issued as
// soon as G1 completes, and G5 as soon as alpha is written, so that the rest of the
// previous drain runs beside the product.
//
// LDL^T and L^{-1} run in block columns of 8, right-looking.  Warp 0 walks the chain of
// pivots: it factors each 8 x 8 diagonal block in registers, forms its panel rows and
// applies the column's contribution to the next block column, keeping its rows in
// registers; the seven other warps form L^{-1} block row by block row (the forward
// elimination of the identity) and the trailing updates one step behind, handing over
// through named barriers.  The chain of phases pays for serial work wherever the other
// threads wait, so single-thread jobs go to warps with slack: a helper issues the next
// chunk's input copies at the start of the LDL^T, a thread of an idle warp issues G2.
//
// Renormalisation: ||S_t||^2 = ||S||^2 + 2 sum v_t'^T S alpha_t' + sum (v.v)(alpha.alpha) from the
// products above; the bound ||S|| + sum |v_t||alpha_t| (||S||^2 carried from the previous
// chunk's state update; one warp tests it while G5 runs) decides that no step can exceed
// tau, otherwise the exact per-step norms give the decisions (V V^T on the tensor core; the
// decisions in order on one warp, the cross terms from row prefix sums) and the per-step
// scales are folded into tril(aq), alpha^T and the outputs.  When the scales of one chunk fall below 2^-64 (tau far below the norm
// each step adds), that chunk's S and outputs are taken step by step from its alpha instead.
// A pivot |D_jj| < 1e-6 means the sequential recurrence takes the singularity
// guard inside the chunk; the chunk is then taken step by step on CUDA cores.
// Chunks end at nudge steps (A += eps_n I is not a rank-1 update).
//
// Few pairs (two CTAs per pair fit on the SMs): each pair runs on a cluster of two CTAs,
// one SM each.  CTA 0 carries A (the prologue's [U; Sigma], G1..G4, the LDL^T, the A update
// and alpha), CTA 1 carries S (phi(q), V, n and 1/den, G5, G6, the renormalisation, the
// outputs and S).  The only data that crosses is alpha, 64 x 64 fp32: the threads of CTA 0
// that form it store their rows straight into CTA 1's AL tile with asynchronous stores
// (st.async into distributed shared memory) that count their bytes on an mbarrier there;
// CTA 1 arrives on an mbarrier of CTA 0 once it is done with it.  So the A side, the longer chain, runs up to a chunk ahead
// of the S side (its rows of alpha go out while the other warps update A).  Each side computes what
// the one-CTA form computes, in the same order, so the two forms agree bit for bit, except
// in a chunk where the guard fires: the A side then takes alpha step by step, and the S side
// its chunk path.
//
// Precision: operands are fp32 in shared memory, read by the tensor core as tf32, which
// drops the low 13 mantissa bits (truncation).  The products that carry A forward (G1's
// A_0, G3, G4) are 3xTF32: the fp32 operand x is its own high part, lo = x - hi is stored
// beside it, and hi*hi + lo*hi + hi*lo is accumulated, so A tracks the fp32 recurrence.
// With bfloat16 I/O, G2, G5 and G6 are plain tf32 (U is exact in tf32; the outputs are
// rounded to bf16).  With float32 I/O every product is 3xTF32: [U; Sigma] lo for G1; G2's
// X lo (G1's accumulator minus its tf32 part) stored back into TMEM columns 448..511; the
// low parts of G5's and G6's operands in the P and Q tiles, free by then.  There is no raw
// stage with float32 I/O (it would not fit): bulk copies issued right after a chunk's G6 bring
// the next chunk's q, k, v, u into tiles that G6 and its drain leave alone (PQ, Q tile 1, vb,
// AL), and the prologue converts them there.  The state (A, S) stays fp32.
// Built for d = d_v = 64, r = 1 and 4, bfloat16 and float32 I/O.
#pragma once

#include "vla_tc.cuh"

namespace vla {
namespace chk {

constexpr int D = 64;
constexpr int NT = 256;
constexpr int TILE = 64 * 64;         // floats of a TK(64, 64) operand tile
constexpr int PLD = 68;               // leading dimension of the prologue's phi(k) / phi(q) scratch
constexpr int GLD = 68;               // leading dimension of the fp32 G / L staging (16-byte rows)
constexpr int kHelpers = 224;         // threads of the LDL^T helper warps (warps 1..7)
constexpr int kCopyIssuer = NT - 32;  // warp 7, lane 0 (a helper): issues the next chunk's input copies
constexpr float kGuardEps = 1e-6f;
constexpr float kReadoutEps = 1e-6f;
constexpr float kInvSqrtD = 0.125f;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns of the products' accumulators (lanes = rows of the 128-row results)
constexpr int TC_G1 = 0;      // [W^T; Q^T], read again as G2's X operand and for alpha = Q - Z E
constexpr int TC_G2 = 64;     // [G - I; H^T]
constexpr int TC_G3 = 128;    // [Z; F^T]
constexpr int TC_G4 = 192;    // [Z D^{-1} Z^T; (Z E)^T]
constexpr int TC_G5 = 256;    // 128 columns: [S alpha, alpha.alpha; S phi(q), phi(q).alpha]; G6 adds tril(aq) V
constexpr int TC_G6 = 384;    // V^T alpha
constexpr int TC_XL = 448;    // X low parts: G2's (float32 I/O), then G4's (hi in TC_G2's columns)

// High part of a 3xTF32 split: the value with the low 13 mantissa bits cleared
// (exactly representable in tf32); the low part is x - hi.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// ELU(x) + 1 with the fast exponential intrinsic (a few ulp for the x <= 0 branch;
// the chunked path serves bf16 I/O, whose rounding is far coarser)
__device__ __forceinline__ float phi_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// packed 8 x 8 blocks (row-major, 64 floats, 72 apart) of a 64 x 64 lower-triangular matrix:
// block (bi, bj) with bi >= bj, and the strictly lower blocks (bi > bj) of a second one.  The
// padding puts consecutive blocks two 16-byte bank groups apart, so the blocks that the lanes
// of a helper warp read at once fall in different banks.
constexpr int kBlk = 72;
__host__ __device__ constexpr int pb8(int bi, int bj) { return (bi * (bi + 1) / 2 + bj) * kBlk; }
__host__ __device__ constexpr int pbB(int bi, int bj) { return (bi * (bi - 1) / 2 + bj) * kBlk; }

// 1/x by the SFU's approximate reciprocal (rcp.approx.ftz.f32: about 1 ulp; the pivots of D are >=
// 1 for an SPD A, far from the flushed range; a pivot below the guard threshold is caught anyway)
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// named barriers (ids 1..5; 0 is __syncthreads): `n` threads take part, a multiple of 32
__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int R, typename TIO>
struct Cfg {
  static constexpr bool F32 = sizeof(TIO) == 4;           // float32 I/O: 3xTF32 throughout, no raw stage
  static constexpr int C = 64 / R;                        // steps per chunk
  static constexpr int TS = C;                            // steps per input tile
  static constexpr uint32_t QB = TS * D * sizeof(TIO);
  static constexpr uint32_t UB = TS * R * D * sizeof(TIO);
  // bfloat16: the tile of q, k, v, u lands in a raw stage by bulk copies; float32: the prologue
  // reads it from global memory (prefetched into L2 a tile ahead), the stage would not fit
  static constexpr uint32_t STAGE = F32 ? 0 : 3 * QB + UB;
  static constexpr uint32_t STAGE_PAD = (STAGE + 1023) / 1024 * 1024;
  static constexpr int T6T = 64 * C;                      // floats of a TK(64, C) tile
  // float offsets (after the raw stage); the lifetimes are listed per region
  static constexpr int F_A = 0;                           // A
  static constexpr int F_S = F_A + TILE;                  // S       } [S][alpha][phi(q)] contiguous
  static constexpr int F_AL = F_S + TILE;                 // alpha   }
  static constexpr int F_PQ = F_AL + TILE;                // phi(q)  }
  static constexpr int F_P = F_PQ + TILE;                 // 2 tiles: [U; Sigma] -> G/L staging -> [W; H^T] lo
                                                          //          -> [Z/D; E^T] lo
  static constexpr int F_Q = F_P + 2 * TILE;              // 2 tiles: [W^T; Q^T]; tile 0 -> L^{-1} blocks ->
                                                          //          Linv lo -> Z lo -> alpha Gram; tile 1 -> v Gram
  static constexpr int F_R = F_Q + 2 * TILE;              // 2 tiles: prologue scratch -> A hi/lo -> [W; H^T] (hi)
                                                          //          -> [Z/D; E^T] hi -> T6
  static constexpr int F_L = F_R + 2 * TILE;              // 1 tile:  prologue scratch -> products of the Linv
                                                          //          assembly -> Linv hi -> Z hi -> T6 (alpha^T)
  static constexpr int F_T6 = F_R;                        // [V^T][tril(aq)][alpha^T], TK(64, C) each
  static constexpr int T6_V = 0, T6_Q = T6T, T6_A = 2 * T6T;
  static constexpr int F_MISC = F_L + TILE;
  // misc block
  static constexpr int M_D = 0, M_ID = 64, M_RDEN = 128, M_VN = 192, M_SL = 256, M_XS = 320, M_AN = 384;
  static constexpr int M_SG = 448, M_IS = 512, M_RED = 576, M_VEC = 640, M_VEC2 = 704, M_SCAL = 768;
  static constexpr int M_N = 800, M_NSEG = 864, M_AN2 = 1120;
  static constexpr int M_SS = 1248, M_SSV = 1252, M_EX = 1253;   // ||S||^2 partials, their validity, the bound test
  static constexpr int MISC = 1256;
  static constexpr int F_VB = F_MISC + MISC;              // V of the chunk (TIO) [C][64]
  static constexpr size_t float_bytes = sizeof(float) * (size_t)F_VB + sizeof(TIO) * C * 64;
  static constexpr size_t bar_off = STAGE_PAD + (float_bytes + 15) / 16 * 16;
  static constexpr size_t bytes = bar_off + 64;
  static_assert(3 * T6T <= 3 * TILE, "T6 fits in R and L");
  static_assert(64 * GLD <= 2 * TILE, "staging fits in P");
  static_assert(2 * C * PLD <= 3 * TILE, "prologue scratch fits in R and L");
  static_assert(pb8(7, 7) + 64 <= TILE && pbB(7, 6) + 64 <= TILE, "packed blocks fit in one tile");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

struct MmaPass {
  int x, y, m, n, col;   // operand offsets (floats), shape, TMEM column
  bool acc;              // accumulate into the column's previous value
  int tx = -1;           // >= 0: the X operand is in tensor memory from this column (lanes = rows)
};

}  // namespace chk

// SPLIT: a cluster of two CTAs per pair, CTA 0 the A side and CTA 1 the S side (above).
template <int R, typename TIO, bool SPLIT>
__global__ void __launch_bounds__(chk::NT, 1) chunk_scan_kernel(ScanArgs a) {
  using namespace chk;
  using Cf = Cfg<R, TIO>;
  constexpr int C = Cf::C, TS = Cf::TS;
  using tc::tk_off;
  constexpr bool F32 = Cf::F32;

  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* raw = smem;
  float* sf = reinterpret_cast<float*>(smem + Cf::STAGE_PAD);
  float* misc = sf + Cf::F_MISC;
  TIO* vb = reinterpret_cast<TIO*>(sf + Cf::F_VB);
  uint64_t* in_bar = reinterpret_cast<uint64_t*>(smem + Cf::bar_off);
  uint64_t* mma_bar = in_bar + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(in_bar + 2);
  volatile int* flag = reinterpret_cast<volatile int*>(in_bar + 3);
  volatile int* issued = reinterpret_cast<volatile int*>(in_bar + 4);   // the last tile whose copy was issued
  uint64_t* full_bar = in_bar + 5;    // SPLIT, S side: alpha is in AL
  uint64_t* empty_bar = in_bar + 6;   // SPLIT, A side: the S side is done with the alpha it was sent
  const uint32_t sbase = smem_u32(sf);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = SPLIT ? cluster_ctarank() : 0u;
  const bool doA = !SPLIT || crank == 0;   // this CTA carries A
  const bool doS = !SPLIT || crank == 1;   // this CTA carries S
  const long long pair = SPLIT ? (long long)(blockIdx.x >> 1) : (long long)blockIdx.x;
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
    if (doA) sf[Cf::F_A + tk_off(i, j, 64)] = gA[e];
    if (doS) sf[Cf::F_S + tk_off(i, j, 64)] = gS[e];
  }
  if (doS && tid < D) misc[Cf::M_N + tid] = gn[tid];
  if (tid == 0) misc[Cf::M_SSV] = 0.f;   // ||S||^2 of the initial state: computed by the first chunk
  if (tid == 0) {
    mbar_init(in_bar, 1);
    mbar_init(mma_bar, 1);
    if (SPLIT) {
      mbar_init(full_bar, 1);      // the S side's own arrival with the 16 KB it expects
      mbar_init(empty_bar, 1);     // thread 0 of the S side, remotely, after a CTA barrier
    }
    fence_mbar_init();
    *flag = 0;
  }
  if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if constexpr (SPLIT) cluster_sync_all();   // both CTAs' barriers are initialised before either uses the other's
  const uint32_t tmem = *tslot;
  // SPLIT: alphas sent (A side) and received (S side); the peer's AL tile and barriers
  uint32_t n_sent = 0, n_recv = 0;
  const uint32_t peer_al = SPLIT ? mapa_shared(smem_u32(sf + Cf::F_AL), crank ^ 1u) : 0u;   // bytes
  const uint32_t peer_full = SPLIT ? mapa_shared(smem_u32(full_bar), crank ^ 1u) : 0u;
  const uint32_t peer_empty = SPLIT ? mapa_shared(smem_u32(empty_bar), crank ^ 1u) : 0u;

  const int ntiles = (int)((T + TS - 1) / TS);
  auto issue = [&](int tile) {  // one thread
    *issued = tile;
    const long long t_start = (long long)tile * TS;
    const int nst = (int)min((long long)TS, T - t_start);
    const uint32_t qb = (uint32_t)nst * D * sizeof(TIO), ub = (uint32_t)nst * R * D * sizeof(TIO);
    // each side copies what it reads: k both, u the A side, q and v the S side
    mbar_arrive_expect_tx(in_bar, qb + (doS ? 2 * qb : 0u) + (doA ? ub : 0u));
    if (doS) bulk_g2s(raw, gq + t_start * D, qb, in_bar);
    bulk_g2s(raw + Cf::QB, gk + t_start * D, qb, in_bar);
    if (doS) bulk_g2s(raw + 2 * Cf::QB, gv + t_start * D, qb, in_bar);
    if (doA) bulk_g2s(raw + 3 * Cf::QB, gu + t_start * R * D, ub, in_bar);
  };
  if (!F32 && tid == 0) issue(0);
  // Float32 I/O has no raw stage: a chunk's q, k, v, u are copied into the tiles that are free
  // from the previous chunk's G6 until this chunk's prologue (q -> PQ, k -> Q tile 1, v -> vb,
  // where it stays as it is, u -> AL), issued right after that G6 so that they land beside it.
  // The A side of a cluster has neither G5 nor G6: it takes u into PQ (free there) and issues
  // the next chunk's k and u at the start of its LDL^T.
  constexpr int F_UST = SPLIT ? Cf::F_PQ : Cf::F_AL;   // where a float32 chunk's u is staged
  long long staged_pos = -1;   // the chunk whose inputs were issued last (all threads agree)
  bool stage_pending = false;  // issued and not yet waited for
  uint32_t stage_phase = 0;
  auto stage = [&](long long p0, int cc) {   // one thread
    const uint32_t qb = (uint32_t)cc * D * sizeof(TIO), ub = (uint32_t)cc * R * D * sizeof(TIO);
    mbar_arrive_expect_tx(in_bar, qb + (doS ? 2 * qb : 0u) + (doA ? ub : 0u));
    if (doS) bulk_g2s(sf + Cf::F_PQ, gq + p0 * D, qb, in_bar);
    bulk_g2s(sf + Cf::F_Q + TILE, gk + p0 * D, qb, in_bar);
    if (doS) bulk_g2s(vb, gv + p0 * D, qb, in_bar);
    if (doA) bulk_g2s(sf + F_UST, gu + p0 * R * D, ub, in_bar);
  };

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
  // Issue the passes (each D (+)= X Y^T over K) and commit them to mma_bar (thread 0).
  auto mma_issue = [&](const MmaPass* ps, int np, int K) {
    const uint32_t sbo = 32u * (uint32_t)K;
    for (int p = 0; p < np; ++p) {
      const uint32_t idesc = tc::idesc_tf32(ps[p].m, ps[p].n);
      for (int kk = 0; kk < K / 8; ++kk) {
        if (ps[p].tx >= 0)
          tc::mma_tf32_tx(tmem + (uint32_t)ps[p].col, tmem + (uint32_t)(ps[p].tx + 8 * kk),
                          tc::sdesc(sbase + 4u * ps[p].y + 256u * kk, sbo), idesc, ps[p].acc || kk > 0);
        else
          tc::mma_tf32(tmem + (uint32_t)ps[p].col, tc::sdesc(sbase + 4u * ps[p].x + 256u * kk, sbo),
                       tc::sdesc(sbase + 4u * ps[p].y + 256u * kk, sbo), idesc, ps[p].acc || kk > 0);
      }
    }
    tc::mma_commit(mma_bar);
  };
  // Wait for the committed products; false on a timeout.
  auto mma_wait = [&]() -> bool {
    if (tid == 0 && !mbar_wait_bounded(mma_bar, mma_phase)) *flag = 1;
    mma_phase ^= 1u;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    return *flag == 0;
  };
  // Issue the passes after the operands written so far, wait for them; false on a timeout.
  auto mma_run = [&](const MmaPass* ps, int np, int K) -> bool {
    sync_tc();
    if (tid == 0) mma_issue(ps, np, K);
    return mma_wait();
  };
  // the warp's TMEM lane quadrant and column half
  const int q4 = warp & 3, half = warp >> 2;
  const int row = 32 * q4 + lane;   // row of an M = 128 result held by this thread
  auto tld = [&](int col, float (&v)[16]) { tc::tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)col, v); };
  auto tld32 = [&](int col, float (&v)[32]) { tc::tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)col, v); };
  auto st4 = [&](int off, float x0, float x1, float x2, float x3) {
    *reinterpret_cast<float4*>(sf + off) = make_float4(x0, x1, x2, x3);
  };
  // 3xTF32 operands: the tensor core reads an fp32 operand as tf32 by dropping its low 13
  // mantissa bits, so the fp32 value itself is the high part; the low part x - tf32_hi(x)
  // is stored beside it
  auto st4_lo = [&](int off_lo, const float* x) {
    st4(off_lo, x[0] - tf32_hi(x[0]), x[1] - tf32_hi(x[1]), x[2] - tf32_hi(x[2]), x[3] - tf32_hi(x[3]));
  };
  auto st4_split = [&](int off_hi, int off_lo, const float* x) {
    st4(off_hi, x[0], x[1], x[2], x[3]);
    st4_lo(off_lo, x);
  };

  // x[jj] <- x[(jj + g) & 15]: with g = (lane / 4) % 8, store jj of a transposed write then
  // goes to column (jj + g) & 15 and the 8 lane groups hit 8 different core-matrix rows
  // (32 distinct banks)
  auto rot16 = [](float (&x)[16], int g) {
    if (g & 1) {
      const float f0 = x[0];
#pragma unroll
      for (int m = 0; m < 15; ++m) x[m] = x[m + 1];
      x[15] = f0;
    }
    if (g & 2) {
      const float f0 = x[0], f1 = x[1];
#pragma unroll
      for (int m = 0; m < 14; ++m) x[m] = x[m + 2];
      x[14] = f0;
      x[15] = f1;
    }
    if (g & 4) {
      float f[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) f[m] = x[m];
#pragma unroll
      for (int m = 0; m < 12; ++m) x[m] = x[m + 4];
#pragma unroll
      for (int m = 0; m < 4; ++m) x[12 + m] = f[m];
    }
  };

  // block reduction of two floats over the CTA (all threads call it)
  auto block_sum2 = [&](float& x, float& y) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      x += __shfl_xor_sync(0xffffffffu, x, m);
      y += __shfl_xor_sync(0xffffffffu, y, m);
    }
    __syncthreads();
    if (lane == 0) {
      misc[Cf::M_RED + warp] = x;
      misc[Cf::M_RED + 8 + warp] = y;
    }
    __syncthreads();
    float s = 0.f, s2 = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
      s += misc[Cf::M_RED + w];
      s2 += misc[Cf::M_RED + 8 + w];
    }
    x = s;
    y = s2;
  };
  auto block_sum = [&](float x) -> float {
    float y = 0.f;
    block_sum2(x, y);
    return x;
  };

  // One warp: |alpha_t|^2 -> M_AN and the test ||S|| + sum_t |v_t| |alpha_t| <= tau (with a
  // relative margin for the rounding of the bound) -> M_EX (0: no step of the chunk can renormalise).
  // Reads the chunk length c of the chunk being run.
  int c = 0;
  auto bound_test = [&](float ns) {
    float bsum = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = lane + 32 * h;
      if (t < c) {
        const float an = misc[Cf::M_AN2 + t] + misc[Cf::M_AN2 + 64 + t];
        misc[Cf::M_AN + t] = an;
        bsum = fmaf(misc[Cf::M_VN + t], sqrtf(fmaxf(an, 0.f)), bsum);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, m);
    if (lane == 0) misc[Cf::M_EX] = (sqrtf(ns) + bsum <= a.tau * (1.f - 0x1p-12f)) ? 0.f : 1.f;
  };

  long long pos = 0;
  // steps left until the next nudge (the global step t0 + pos + to_nudge is a multiple of P),
  // carried from chunk to chunk instead of a 64-bit remainder per chunk
  long long to_nudge = (a.P > 0) ? a.P - (a.t0 % a.P) : 0;
  auto advance = [&](int c) {
    pos += c;
    if (a.P > 0) {
      to_nudge -= c;
      if (to_nudge == 0) to_nudge = a.P;
    }
  };
  // float32 I/O: issue the copies of the next chunk's inputs (all threads call it; the tiles
  // they land in must be free, every earlier access to them fenced by a barrier)
  auto stage_next = [&](int issuer) {   // `issuer`: the thread that issues them
    const long long np = pos + c;
    if (np >= T) return;
    long long tn = to_nudge;
    if (a.P > 0) {
      tn -= c;
      if (tn == 0) tn = a.P;
    }
    int nc = (int)min((long long)(TS - np % TS), T - np);
    if (a.P > 0 && tn <= nc) nc = (int)tn;
    if (tid == issuer) stage(np, nc);
    staged_pos = np;
    stage_pending = true;
  };
  // SPLIT, S side: after a CTA barrier that follows every access to the chunk's alpha, thread 0
  // signals the A side (release, cluster scope) that AL may be written again
  auto release_alpha = [&]() {
    if constexpr (SPLIT) {
      if (tid == 0) mbar_arrive_remote(peer_empty);
    }
  };
  // A_1 = A_0 - Z D^{-1} Z^T (+ eps_n I at a nudge): row `row`, columns col0 .. col0 + 15, from
  // the 16 values of G4's result in v
  auto a_update = [&](int row, int col0, const float (&v)[16], bool nudge) {
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      float4* ap = reinterpret_cast<float4*>(sf + Cf::F_A + tk_off(row, col0 + j, 64));
      float4 x = *ap;
      x.x -= v[j];
      x.y -= v[j + 1];
      x.z -= v[j + 2];
      x.w -= v[j + 3];
      if (nudge && (row >> 2) == ((col0 + j) >> 2)) {
        const int dg = row & 3;
        if (dg == 0) x.x += a.eps_n;
        if (dg == 1) x.y += a.eps_n;
        if (dg == 2) x.z += a.eps_n;
        if (dg == 3) x.w += a.eps_n;
      }
      *ap = x;
    }
  };
  // SPLIT, A side, the 128 threads of rows 64 + t: store this thread's half of alpha_t (32
  // values, 128 bytes) into the S side's AL tile, counted on its full_bar; the thread does
  // not wait for them
  auto send_alpha = [&](int t, const float (&al)[32]) {
    if constexpr (SPLIT) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        st_async_v4(peer_al + 4u * (uint32_t)tk_off(t, 32 * half + j, 64), al[j], al[j + 1], al[j + 2], al[j + 3],
                    peer_full);
    }
  };
  int loaded = -1;
  while (pos < T && !failed) {
    // ---------------- schedule: chunk [pos, pos + c) inside one input tile, ending at a nudge
    const int tile = (int)(pos / TS);
    const int ts = (int)(pos % TS);
    c = (int)min((long long)(TS - ts), T - pos);
    bool nudge = false;
    if (a.P > 0) {
      if (to_nudge <= c) { c = (int)to_nudge; nudge = true; }
    }
    if constexpr (F32) {
      if (staged_pos != pos) {   // not issued ahead: the first chunk, or after a step-by-step chunk
        if (tid == 0) stage(pos, c);
        staged_pos = pos;
        stage_pending = true;
      }
      if (tid == 0 && !mbar_wait_bounded(in_bar, stage_phase)) *flag = 1;
      stage_phase ^= 1u;
      __syncthreads();
      if (*flag) { failed = true; break; }
      stage_pending = false;
      loaded = tile;
    } else if (tile != loaded) {
      if (tid == 0 && !mbar_wait_bounded(in_bar, (uint32_t)(tile & 1))) *flag = 1;
      __syncthreads();
      if (*flag) { failed = true; break; }
      loaded = tile;
    }
    const TIO* rq = reinterpret_cast<const TIO*>(raw);
    const TIO* rk = reinterpret_cast<const TIO*>(raw + Cf::QB);
    const TIO* rv = reinterpret_cast<const TIO*>(raw + 2 * Cf::QB);
    const TIO* ru = reinterpret_cast<const TIO*>(raw + 3 * Cf::QB);

    // ---------------- prologue: [U; Sigma] -> P, phi(q) -> PQ, V -> vb, n, 1/den, |v|
    {
      float* pk = sf + Cf::F_R;              // phi(k_t)[i] at t * PLD + i, then n_t[i] phi(q_t)[i]
      float* pq = sf + Cf::F_R + C * PLD;    // phi(q_t)[i]
      // Rows of 8-element pieces: in each group of 8 lanes the rows (row % 8) and the pieces
      // differ, so the 16-byte reads of the bf16 rows and the float4 stores into the
      // core-matrix layout are both free of bank conflicts.
      auto ld8s = [](const float* s, float (&x)[8]) {   // float32 I/O: 8 staged values
        const float4 a0 = *reinterpret_cast<const float4*>(s);
        const float4 a1 = *reinterpret_cast<const float4*>(s + 4);
        x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w; x[4] = a1.x; x[5] = a1.y; x[6] = a1.z; x[7] = a1.w;
      };
      auto unpack8 = [](const uint4& w, float (&x)[8]) {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[m]));
          x[2 * m] = f.x;
          x[2 * m + 1] = f.y;
        }
      };
#pragma unroll
      for (int s8 = 0; s8 < 64 * 8 / NT; ++s8) {   // U rows a (64 x 8 pieces)
        if (!doA) break;
        const int f = tid + NT * s8;
        const int arow = (f >> 6) * 8 + (f & 7), pc = ((f & 7) + (f >> 3)) & 7;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (arow / R < c) {
          if constexpr (F32)
            ld8s(sf + F_UST + arow * D + 8 * pc, x);
          else
            unpack8(*reinterpret_cast<const uint4*>(ru + (ts * R + arow) * D + 8 * pc), x);
        }
        st4(Cf::F_P + tk_off(arow, 8 * pc, 64), x[0], x[1], x[2], x[3]);
        st4(Cf::F_P + tk_off(arow, 8 * pc + 4, 64), x[4], x[5], x[6], x[7]);
        if constexpr (F32) {   // [U; Sigma] low parts -> Q tiles (float32 directions are not tf32-exact)
          st4_lo(Cf::F_Q + tk_off(arow, 8 * pc, 64), x);
          st4_lo(Cf::F_Q + tk_off(arow, 8 * pc + 4, 64), x + 4);
        }
      }
      if constexpr (F32) {
        // step rows t < C; rows c.. are zero (Sigma, phi(q), V)
        constexpr int NSI = (C * 8 + NT - 1) / NT;
        [[maybe_unused]] float kr[NSI][8], qr[NSI][8];
        if constexpr (F32) {
          // the staged k (Q tile 1) and q (PQ) are overwritten by this loop's outputs: every
          // thread reads its pieces first
#pragma unroll
          for (int s = 0; s < NSI; ++s) {
            const int f = tid + NT * s;
            const int t = (f >> 6) * 8 + (f & 7), pc = ((f & 7) + (f >> 3)) & 7;
            if (f < C * 8 && t < c) {
              ld8s(sf + Cf::F_Q + TILE + t * D + 8 * pc, kr[s]);
              if (doS) ld8s(sf + Cf::F_PQ + t * D + 8 * pc, qr[s]);
            }
          }
          __syncthreads();
        }
#pragma unroll
        for (int s = 0; s < NSI; ++s) {
          const int f = tid + NT * s;
          if (f >= C * 8) break;
          const int t = (f >> 6) * 8 + (f & 7), pc = ((f & 7) + (f >> 3)) & 7;
          float kx[8], qx[8];
          uint4 vw = make_uint4(0u, 0u, 0u, 0u);
          if (t < c) {
            if constexpr (F32) {
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                kx[m] = kr[s][m];
                qx[m] = doS ? qr[s][m] : 0.f;
              }
            } else {
              const int off = (ts + t) * D + 8 * pc;
              unpack8(*reinterpret_cast<const uint4*>(rk + off), kx);
              unpack8(*reinterpret_cast<const uint4*>(rq + off), qx);
              vw = *reinterpret_cast<const uint4*>(rv + off);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              kx[m] = phi_fast(kx[m]);
              if (doS) qx[m] = phi_fast(qx[m]);
            }
          } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) kx[m] = qx[m] = 0.f;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = 8 * pc + 4 * h;
            const float* k4 = kx + 4 * h;
            const float* q4p = qx + 4 * h;
            if (doA) {
              st4(Cf::F_P + tk_off(64 + t, col, 64), k4[0] * kInvSqrtD, k4[1] * kInvSqrtD, k4[2] * kInvSqrtD,
                  k4[3] * kInvSqrtD);
              if constexpr (F32) {
                const float s4[4] = {k4[0] * kInvSqrtD, k4[1] * kInvSqrtD, k4[2] * kInvSqrtD, k4[3] * kInvSqrtD};
                st4_lo(Cf::F_Q + tk_off(64 + t, col, 64), s4);
              }
            }
            if (doS) {
              st4(Cf::F_PQ + tk_off(t, col, 64), q4p[0], q4p[1], q4p[2], q4p[3]);
              *reinterpret_cast<float4*>(pk + t * PLD + col) = make_float4(k4[0], k4[1], k4[2], k4[3]);
              *reinterpret_cast<float4*>(pq + t * PLD + col) = make_float4(q4p[0], q4p[1], q4p[2], q4p[3]);
            }
          }
          if constexpr (F32) {   // V was staged into vb as it is; rows past c are zeroed
            if (doS && t >= c) {
              *reinterpret_cast<float4*>(vb + t * 64 + 8 * pc) = make_float4(0.f, 0.f, 0.f, 0.f);
              *reinterpret_cast<float4*>(vb + t * 64 + 8 * pc + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          } else {
            *reinterpret_cast<uint4*>(vb + t * 64 + 8 * pc) = vw;
          }
        }
      } else {
#pragma unroll
        for (int s8 = 0; s8 < (C * 8 + NT - 1) / NT; ++s8) {   // step rows t < C; rows c.. are zero (Sigma, phi(q), V)
          const int f = tid + NT * s8;
          if (C * 8 % NT != 0 && f >= C * 8) break;
          const int t = (f >> 6) * 8 + (f & 7), pc = ((f & 7) + (f >> 3)) & 7;
          float kx[8], qx[8];
          uint4 vw = make_uint4(0u, 0u, 0u, 0u);
          if (t < c) {
            const int off = (ts + t) * D + 8 * pc;
            unpack8(*reinterpret_cast<const uint4*>(rk + off), kx);
            if (doS) {   // the A side's stage holds no q or v
              unpack8(*reinterpret_cast<const uint4*>(rq + off), qx);
              vw = *reinterpret_cast<const uint4*>(rv + off);
            } else {
#pragma unroll
              for (int m = 0; m < 8; ++m) qx[m] = 0.f;
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              kx[m] = phi_fast(kx[m]);
              if (doS) qx[m] = phi_fast(qx[m]);
            }
          } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) kx[m] = qx[m] = 0.f;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = 8 * pc + 4 * h;
            const float* k4 = kx + 4 * h;
            const float* q4p = qx + 4 * h;
            if (doA)
              st4(Cf::F_P + tk_off(64 + t, col, 64), k4[0] * kInvSqrtD, k4[1] * kInvSqrtD, k4[2] * kInvSqrtD,
                  k4[3] * kInvSqrtD);
            if (doS) {
              st4(Cf::F_PQ + tk_off(t, col, 64), q4p[0], q4p[1], q4p[2], q4p[3]);
              *reinterpret_cast<float4*>(pk + t * PLD + col) = make_float4(k4[0], k4[1], k4[2], k4[3]);
              *reinterpret_cast<float4*>(pq + t * PLD + col) = make_float4(q4p[0], q4p[1], q4p[2], q4p[3]);
            }
          }
          if (doS) *reinterpret_cast<uint4*>(vb + t * 64 + 8 * pc) = vw;
        }
      }
      // zero rows C..63 of Sigma and phi(q): the lanes of a warp take 8 rows (8 distinct bank
      // groups of the core-matrix layout) x 4 column groups
      static_assert(C % 8 == 0, "zero rows in groups of 8");
      for (int e4 = tid; e4 < (64 - C) * 16; e4 += NT) {
        const int t = C + 8 * (e4 >> 7) + (e4 & 7), col = ((e4 >> 3) & 15) * 4;
        if (doA) st4(Cf::F_P + tk_off(64 + t, col, 64), 0.f, 0.f, 0.f, 0.f);
        if (doS) st4(Cf::F_PQ + tk_off(t, col, 64), 0.f, 0.f, 0.f, 0.f);
        if (F32 && doA) st4(Cf::F_Q + tk_off(64 + t, col, 64), 0.f, 0.f, 0.f, 0.f);
      }
      __syncthreads();
      if (doA && tid < D) misc[Cf::M_SL + tid] = sf[Cf::F_P + tk_off(64 + c - 1, tid, 64)];   // s of the chunk's last step
      if (doS) {
      // n_t = n_{t-1} + phi(k_t): column i, four segments of C/4 steps (one per thread)
      constexpr int SEG = C / 4;
      const int ci = tid & 63, sg4 = tid >> 6;
      float kseg[SEG], qseg[SEG];   // the segment's phi(k) and phi(q), kept in registers
#pragma unroll
      for (int j = 0; j < SEG; ++j) kseg[j] = pk[(SEG * sg4 + j) * PLD + ci];
      {
        float tot = 0.f;
#pragma unroll
        for (int j = 0; j < SEG; ++j) tot += kseg[j];
        misc[Cf::M_NSEG + sg4 * 64 + ci] = tot;
      }
#pragma unroll
      for (int j = 0; j < SEG; ++j) qseg[j] = pq[(SEG * sg4 + j) * PLD + ci];
      __syncthreads();
      float nrun = misc[Cf::M_N + ci];
#pragma unroll
      for (int s2 = 0; s2 < 3; ++s2)
        if (s2 < sg4) nrun += misc[Cf::M_NSEG + s2 * 64 + ci];
#pragma unroll
      for (int j = 0; j < SEG; ++j) {
        nrun += kseg[j];
        kseg[j] = nrun * qseg[j];
      }
#pragma unroll
      for (int j = 0; j < SEG; ++j) pk[(SEG * sg4 + j) * PLD + ci] = kseg[j];
      __syncthreads();
      if (sg4 == 3) misc[Cf::M_N + ci] = nrun;   // n after the chunk (zero rows past c add nothing)
      {  // 1/den_t and |v_t|: NT / C threads per step (every lane takes part in the shuffles)
        constexpr int TPS = NT / C;
        constexpr int EPT = 64 / TPS;
        const int t = tid / TPS, part = tid - t * TPS;
        float dn = 0.f, vv = 0.f;
        static_assert(EPT % 4 == 0 && (EPT & (EPT - 1)) == 0, "den reduction layout");
        if (t < c) {
#pragma unroll
          for (int j = 0; j < EPT; j += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pk + t * PLD + part * EPT + j);
            // the rows of vb are 128 bytes apart (bf16): each step reads its pieces in its own
            // rotation, so the steps of a warp do not all hit the same banks (|v|^2 only)
            const int jv = (j + 4 * t) & (EPT - 1);
            float2 v01, v23;
            if constexpr (F32) {
              const float4 v4 = *reinterpret_cast<const float4*>(vb + t * 64 + part * EPT + jv);
              v01 = make_float2(v4.x, v4.y);
              v23 = make_float2(v4.z, v4.w);
            } else {
              const uint2 w2 = *reinterpret_cast<const uint2*>(vb + t * 64 + part * EPT + jv);
              v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.x));
              v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.y));
            }
            dn += p4.x;
            dn += p4.y;
            dn += p4.z;
            dn += p4.w;
            vv = fmaf(v01.x, v01.x, vv);
            vv = fmaf(v01.y, v01.y, vv);
            vv = fmaf(v23.x, v23.x, vv);
            vv = fmaf(v23.y, v23.y, vv);
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
      }   // doS
      // the raw stage is free once the tile's last chunk is converted: the S side of a cluster
      // issues the next tile's copies here, the A side (and the one-CTA form) from a helper warp
      // at the start of the LDL^T
      if (!F32 && !doA && tid == 0 && ts + c == TS && tile + 1 < ntiles) {
        fence_proxy_async_smem();
        issue(tile + 1);
      }
      // A's low part -> R tile 1 (A itself is the high part)
      for (int e4 = tid; doA && e4 < TILE / 4; e4 += NT) {
        const float4 x = *reinterpret_cast<const float4*>(sf + Cf::F_A + 4 * e4);
        const float xv[4] = {x.x, x.y, x.z, x.w};
        st4_lo(Cf::F_R + TILE + 4 * e4, xv);
      }
    }

    if (doA) {   // ======== the A side: G1 .. G4, the LDL^T, A and alpha
    // ---------------- G1: [W^T; Q^T] = [U; Sigma] A_0^T  (M 128, N 64, K 64), A_0 hi + lo (and, with
    // float32 I/O, [U; Sigma] lo)
    {
      const MmaPass ps[3] = {{Cf::F_P, Cf::F_A, 128, 64, TC_G1, false},
                             {Cf::F_P, Cf::F_R + TILE, 128, 64, TC_G1, true},
                             {Cf::F_Q, Cf::F_A, 128, 64, TC_G1, true}};
      if (!mma_run(ps, F32 ? 3 : 2, 64)) { failed = true; break; }
    }

    // ---------------- G2: [G - I; H^T] = [W^T; Q^T] U^T  (M 128, N 64, K 64), X read from G1's
    // accumulator in tensor memory; it runs while G1's W is drained.  Q^T stays there for alpha.
    // A thread of warp 3 issues it: the W drain is warps 0, 1, 4 and 5's (rows < 64).
    constexpr int kG2Issuer = 96;
    if constexpr (F32) {
      // 3xTF32 for G2 as well: the low part of G1's accumulator goes to TMEM columns TC_XL.., and
      // G2 takes X hi * U hi + X lo * U hi + X hi * U lo (U lo in the Q tiles)
      float v32[32];
      tld32(TC_G1 + 32 * half, v32);
      float lo[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) lo[j] = v32[j] - tf32_hi(v32[j]);
      tc::tmem_st32(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)(TC_XL + 32 * half), lo);
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (tid == kG2Issuer) {
        MmaPass ps[3] = {{0, Cf::F_P, 128, 64, TC_G2, false}, {0, Cf::F_P, 128, 64, TC_G2, true},
                         {0, Cf::F_Q, 128, 64, TC_G2, true}};
        ps[0].tx = TC_G1;
        ps[1].tx = TC_XL;
        ps[2].tx = TC_G1;
        mma_issue(ps, 3, 64);
      }
      if (row < 64) {   // W[i][a] = W^T[a][i], a = row (warp-uniform): fp32 -> R tile 0
        const int g = (lane >> 2) & 7;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col0 = 32 * half + 16 * cc;
          float (&v)[16] = *reinterpret_cast<float(*)[16]>(v32 + 16 * cc);
          rot16(v, g);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) sf[Cf::F_R + tk_off(col0 + ((jj + g) & 15), row, 64)] = v[jj];
        }
      }
    } else {
    {
      MmaPass ps[1] = {{0, Cf::F_P, 128, 64, TC_G2, false}};
      ps[0].tx = TC_G1;
      if (tid == kG2Issuer) mma_issue(ps, 1, 64);
    }
    if (row < 64) {   // W[i][a] = W^T[a][i], a = row (warp-uniform): fp32 -> R tile 0
      float v32[32];
      const int g = (lane >> 2) & 7;
      tld32(TC_G1 + 32 * half, v32);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = 32 * half + 16 * cc;
        float (&v)[16] = *reinterpret_cast<float(*)[16]>(v32 + 16 * cc);
        rot16(v, g);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sf[Cf::F_R + tk_off(col0 + ((jj + g) & 15), row, 64)] = v[jj];
      }
    }
    }
    if (!mma_wait()) { failed = true; break; }
    float* Gs = sf + Cf::F_P;   // [64][GLD]: G, then L (strict lower) in place
    {
      float v32[32];
      tld32(TC_G2 + 32 * half, v32);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = 32 * half + 16 * cc;
        float (&v)[16] = *reinterpret_cast<float(*)[16]>(v32 + 16 * cc);
        if (row < 64) {
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(Gs + row * GLD + col0 + j) =
                make_float4(v[j] + ((row == col0 + j) ? 1.f : 0.f), v[j + 1] + ((row == col0 + j + 1) ? 1.f : 0.f),
                            v[j + 2] + ((row == col0 + j + 2) ? 1.f : 0.f), v[j + 3] + ((row == col0 + j + 3) ? 1.f : 0.f));
        } else {   // H^T (rows t) fp32 -> R tile 1 (rows 64 + t of [W; H^T])
#pragma unroll
          for (int j = 0; j < 16; j += 4) st4(Cf::F_R + tk_off(row, col0 + j, 64), v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();

    // ---------------- LDL^T of G and X = L^{-1} in 8 x 8 blocks (fp32)
    // Right-looking block LDL^T by block columns of 8.  Warp 0 walks the critical path alone:
    // for block column k it factors the 8 x 8 diagonal block in every lane's registers, turns
    // the rows below it into L (forward substitution against L_kk, then D^{-1}), and applies
    // column k's contribution -L_{.k} D_k L_{k+1,k}^T to block column k+1, so that the next
    // step can start at once.  The seven helper warps follow one step behind: they form block row k
    // of X = L^{-1} (X_kj = L_kk^{-1} B_kj, where B is the identity being eliminated), update
    // B_ij -= L_ik X_kj for i > k, and apply column k's contribution to the block columns
    // beyond k + 1.  Warp 0 and the helpers hand over through named barriers (LB: column k of
    // L is written; UB: the helpers' trailing update for column k is done), used in
    // alternation so that a barrier is never reused before its previous round completed.
    // the A side of a cluster: the next chunk's u (PQ) and k (Q tile 1), free since G1, issued
    // by the thread that issues a bf16 tile's copies (a helper, which waits for warp 0's first
    // column anyway)
    if constexpr (SPLIT && F32) stage_next(kCopyIssuer);
    float* XB = sf + Cf::F_Q;   // X = L^{-1}: 36 lower 8 x 8 blocks
    float* BB = sf + Cf::F_L;   // B: 28 strictly lower 8 x 8 blocks
    if (warp == 0) {
      float* dsc = misc + Cf::M_VEC;   // warp 0's broadcast scratch (64 floats)
      auto ld8 = [](const float* pp, float (&v)[8]) {
        const float4 a0 = *reinterpret_cast<const float4*>(pp), a1 = *reinterpret_cast<const float4*>(pp + 4);
        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w; v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
      };
      auto st8 = [](float* pp, const float (&v)[8]) {
        *reinterpret_cast<float4*>(pp) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(pp + 4) = make_float4(v[4], v[5], v[6], v[7]);
      };
      // lane l owns rows l and 32 + l; ga / gb hold their entries of the current block column
      // (Schur-updated), carried in registers from one step to the next
      float ga[8], gb[8];
      ld8(Gs + lane * GLD, ga);
      ld8(Gs + (32 + lane) * GLD, gb);
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {
        // the diagonal block's rows 8k..8k+7 are lanes 8 (k % 4) .. 8 (k % 4) + 7 of row set k / 4
        const bool owner = (lane >> 3) == (k & 3);
        if (owner) {
          float t[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) t[c] = (k >= 4) ? gb[c] : ga[c];
          st8(dsc + 8 * (lane & 7), t);
        }
        __syncwarp();
        float a8[8][8], d8[8], id8[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) ld8(dsc + 8 * r, a8[r]);   // (entries above the diagonal unused)
        __syncwarp();
        // a8 -> L_kk (strict lower), d8 = D_k, id8 = 1 / D_k
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          d8[j] = a8[j][j];
          id8[j] = rcp_approx(d8[j]);
#pragma unroll
          for (int i = j + 1; i < 8; ++i) {
            const float lij = a8[i][j] * id8[j];
#pragma unroll
            for (int m = j + 1; m <= i; ++m) {
              if (m == i && i == j + 1)   // the next pivot: one rounding step after the reciprocal
                a8[i][m] = fmaf(-(a8[i][j] * a8[i][j]), id8[j], a8[i][m]);
              else
                a8[i][m] = fmaf(-lij, a8[m][j], a8[i][m]);   // a8[m][j] = L_mj D_j
            }
          }
#pragma unroll
          for (int i = j + 1; i < 8; ++i) a8[i][j] *= id8[j];
        }
        // rows -> L: (L D)_r = G'_r L_kk^{-T} by forward substitution, then times D^{-1}.  For the
        // diagonal rows the entries left of the diagonal are L_kk's.  Rows above the block are
        // not stored.
        auto panel = [&](float (&g)[8]) {
#pragma unroll
          for (int c = 1; c < 8; ++c)
#pragma unroll
            for (int m = 0; m < c; ++m) g[c] = fmaf(-a8[c][m], g[m], g[c]);
#pragma unroll
          for (int c = 0; c < 8; ++c) g[c] *= id8[c];
        };
        panel(ga);
        panel(gb);
        if (lane >= 8 * k) st8(Gs + lane * GLD + 8 * k, ga);
        if (32 + lane >= 8 * k) st8(Gs + (32 + lane) * GLD + 8 * k, gb);
        if (lane == 0) {
          st8(misc + Cf::M_D + 8 * k, d8);
          st8(misc + Cf::M_ID + 8 * k, id8);
        }
        bar_arrive(1 + (k & 1), 32 + kHelpers);   // LB: block column k of L and D_k are written
        if (k < 7) {
          // column k's contribution to block column k + 1, -L_{.k} D_k L_{k+1,k}^T: (L D)_{k+1,k}
          // (lanes 8 ((k+1) % 4) .. + 7 of row set (k+1) / 4), transposed, to every lane
          if ((lane >> 3) == ((k + 1) & 3)) {
#pragma unroll
            for (int c = 0; c < 8; ++c) dsc[8 * c + (lane & 7)] = ((k + 1 >= 4) ? gb[c] : ga[c]) * d8[c];
          }
          __syncwarp();
          float2 ldm2[8][4];   // ldm2[c][h] = ((L D)[2h][c], (L D)[2h + 1][c])
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float t[8];
            ld8(dsc + 8 * c, t);
#pragma unroll
            for (int h = 0; h < 4; ++h) ldm2[c][h] = make_float2(t[2 * h], t[2 * h + 1]);
          }
          __syncwarp();
          // the helpers' contributions of columns <= k - 1 to column k + 1 are in the staging
          if (k >= 1) bar_sync(3 + ((k - 1) & 1), 32 + kHelpers);
          auto next = [&](int r, float (&g)[8]) {   // g: this row's L_{r,k}; becomes G'_{r,k+1}
            float cur[8];
            if (r >= 8 * (k + 1)) {
              ld8(Gs + r * GLD + 8 * (k + 1), cur);
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c) cur[c] = 0.f;
            }
            float2 acc[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float2 lc = make_float2(g[c], g[c]);
#pragma unroll
              for (int h = 0; h < 4; ++h) acc[h] = __ffma2_rn(lc, ldm2[c][h], acc[h]);
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              g[2 * h] = cur[2 * h] - acc[h].x;
              g[2 * h + 1] = cur[2 * h + 1] - acc[h].y;
            }
          };
          next(lane, ga);
          next(32 + lane, gb);
        }
      }
        } else {
      const int ot = (warp - 1) * 32 + lane;   // 0 .. kHelpers - 1
      // the next tile's copies, issued here where the helpers wait for warp 0's first column
      if (!F32 && tid == kCopyIssuer && ts + c == TS && tile + 1 < ntiles) {
        fence_proxy_async_smem();
        issue(tile + 1);
      }
      auto ld4 = [](const float* pp) { return *reinterpret_cast<const float4*>(pp); };
      auto ldrow8 = [&](const float* pp, float (&v)[8]) {
        const float4 x0 = ld4(pp), x1 = ld4(pp + 4);
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
      };
#pragma unroll 1
      for (int m = 0; m < 8; ++m) {
        bar_sync(1 + (m & 1), 32 + kHelpers);   // LB: block column m of L is written
        // block row m of X: X_mj = L_mm^{-1} B_mj (j < m), X_mm = L_mm^{-1}; a column per thread
        if (ot < 8 * (m + 1)) {
          const int j = ot >> 3, c = ot & 7;
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = (j == m) ? ((i == c) ? 1.f : 0.f) : BB[pbB(m, j) + 8 * i + c];
          const float* lmm = Gs + 8 * m * GLD + 8 * m;
#pragma unroll
          for (int i = 1; i < 8; ++i) {
            float li[8];
            ldrow8(lmm + i * GLD, li);
#pragma unroll
            for (int pp = 0; pp < i; ++pp) x[i] = fmaf(-li[pp], x[pp], x[i]);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) XB[pb8(m, j) + 8 * i + c] = x[i];
        }
        bar_sync(5, kHelpers);
        if (m < 7) {
          // 2 x 4 tiles of: B_ij -= L_im X_mj (i > m, j <= m; B_im starts at 0), and of the
          // trailing update G'_ic -= L_im D_m L_cm^T (c >= m + 2, i >= c); rows in registers,
          // 16-byte loads
          const int nb = (7 - m) * (m + 1), nt = (6 - m) * (7 - m) / 2;
          for (int q = ot; q < 8 * (nb + nt); q += kHelpers) {
            const int blk = q >> 3, rr = (q >> 1) & 3, cc = q & 1;
            float acc[2][4];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
              for (int b4 = 0; b4 < 4; ++b4) acc[a2][b4] = 0.f;
            if (blk < nb) {
              const int i = m + 1 + blk / (m + 1), j = blk % (m + 1);
              float l0[8], l1[8];
              ldrow8(Gs + (8 * i + 2 * rr) * GLD + 8 * m, l0);
              ldrow8(Gs + (8 * i + 2 * rr + 1) * GLD + 8 * m, l1);
              const float* xc = XB + pb8(m, j) + 4 * cc;
#pragma unroll
              for (int pp = 0; pp < 8; ++pp) {
                const float4 xv = ld4(xc + 8 * pp);
                const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int b4 = 0; b4 < 4; ++b4) {
                  acc[0][b4] = fmaf(l0[pp], xa[b4], acc[0][b4]);
                  acc[1][b4] = fmaf(l1[pp], xa[b4], acc[1][b4]);
                }
              }
              float* dst = BB + pbB(i, j) + 8 * 2 * rr + 4 * cc;
#pragma unroll
              for (int a2 = 0; a2 < 2; ++a2) {
                float4 dv = (j == m) ? make_float4(0.f, 0.f, 0.f, 0.f) : ld4(dst + 8 * a2);
                dv.x -= acc[a2][0];
                dv.y -= acc[a2][1];
                dv.z -= acc[a2][2];
                dv.w -= acc[a2][3];
                *reinterpret_cast<float4*>(dst + 8 * a2) = dv;
              }
            } else {
              int c = m + 2, rem = blk - nb;
              while (rem >= 8 - c) { rem -= 8 - c; ++c; }
              const int i = c + rem;
              float dm[8], l0[8], l1[8], lc[4][8];
              ldrow8(misc + Cf::M_D + 8 * m, dm);
              ldrow8(Gs + (8 * i + 2 * rr) * GLD + 8 * m, l0);
              ldrow8(Gs + (8 * i + 2 * rr + 1) * GLD + 8 * m, l1);
#pragma unroll
              for (int b4 = 0; b4 < 4; ++b4) ldrow8(Gs + (8 * c + 4 * cc + b4) * GLD + 8 * m, lc[b4]);
#pragma unroll
              for (int pp = 0; pp < 8; ++pp) {
                const float a0 = l0[pp] * dm[pp], a1 = l1[pp] * dm[pp];
#pragma unroll
                for (int b4 = 0; b4 < 4; ++b4) {
                  acc[0][b4] = fmaf(a0, lc[b4][pp], acc[0][b4]);
                  acc[1][b4] = fmaf(a1, lc[b4][pp], acc[1][b4]);
                }
              }
              float* dst = Gs + (8 * i + 2 * rr) * GLD + 8 * c + 4 * cc;
#pragma unroll
              for (int a2 = 0; a2 < 2; ++a2) {
                float4 dv = ld4(dst + GLD * a2);
                dv.x -= acc[a2][0];
                dv.y -= acc[a2][1];
                dv.z -= acc[a2][2];
                dv.w -= acc[a2][3];
                *reinterpret_cast<float4*>(dst + GLD * a2) = dv;
              }
            }
          }
          if (m <= 5) bar_arrive(3 + (m & 1), 32 + kHelpers);   // UB: columns >= m + 2 have column m's part
        }
      }
    }
    __syncthreads();
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
      if constexpr (SPLIT) {   // alpha goes into AL step by step: the S side must be done with the last one
        if (tid == 0 && n_sent > 0 && !mbar_wait_cluster_bounded(empty_bar, (n_sent - 1) & 1u)) *flag = 1;
        __syncthreads();
        if (*flag) { failed = true; break; }
      }
      float* vec = misc + Cf::M_VEC;     // u, then s
      float* vec2 = misc + Cf::M_VEC2;   // z, alpha
      const int ar = tid >> 2, cq = tid & 3;   // row of A / S and a 16-column quarter
      for (int t = 0; t < c; ++t) {
        const long long st = pos + t;
        for (int i = 0; i < R; ++i) {
          if (tid < 64) vec[tid] = to_f32(gu[(st * R + i) * D + tid]);
          __syncthreads();
          float zp = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) zp = fmaf(sf[Cf::F_A + tk_off(ar, 16 * cq + j, 64)], vec[16 * cq + j], zp);
          zp += __shfl_xor_sync(0xffffffffu, zp, 1);
          zp += __shfl_xor_sync(0xffffffffu, zp, 2);
          if (cq == 0) vec2[ar] = zp;
          __syncthreads();
          const float dl = 1.f + block_sum(tid < 64 ? vec[tid] * vec2[tid] : 0.f);
          const bool gd = fabsf(dl) < kGuardEps;
          if (tid == 0 && gd) ++guard_cnt;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = 16 * cq + j;
            float& av = sf[Cf::F_A + tk_off(ar, col, 64)];
            if (gd) av += (ar == col) ? kGuardEps : 0.f;
            else av = fmaf(-vec2[ar] / dl, vec2[col], av);
          }
          __syncthreads();
        }
        const bool nd = nudge && t == c - 1;
        if (nd && cq == (ar >> 4)) sf[Cf::F_A + tk_off(ar, ar, 64)] += a.eps_n;
        if (tid < 64) vec[tid] = phi_elu1(to_f32(gk[st * D + tid])) * kInvSqrtD;
        __syncthreads();
        float ap = 0.f;   // alpha = A s
#pragma unroll
        for (int j = 0; j < 16; ++j) ap = fmaf(sf[Cf::F_A + tk_off(ar, 16 * cq + j, 64)], vec[16 * cq + j], ap);
        ap += __shfl_xor_sync(0xffffffffu, ap, 1);
        ap += __shfl_xor_sync(0xffffffffu, ap, 2);
        if (cq == 0) vec2[ar] = ap;
        __syncthreads();
        if constexpr (SPLIT) {   // alpha_t -> AL row t; the S side takes the chunk from there
          if (tid < 64) sf[Cf::F_AL + tk_off(t, tid, 64)] = vec2[tid];
          continue;
        }
        // S += v alpha^T, then the norm
        const float vr = to_f32(vb[t * 64 + ar]);   // v of step t
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = 16 * cq + j;
          float& sr = sf[Cf::F_S + tk_off(ar, col, 64)];
          sr = fmaf(vr, vec2[col], sr);
          sq = fmaf(sr, sr, sq);
        }
        const float nrm = sqrtf(block_sum(sq));
        if (nrm > a.tau) {
          const float cf = a.tau / nrm;
#pragma unroll
          for (int j = 0; j < 16; ++j) sf[Cf::F_S + tk_off(ar, 16 * cq + j, 64)] *= cf;
          if (tid == 0) ++renorm_cnt;
        }
        if (!isfinite(nrm)) flags |= kStatusNonfinite;
        if (tid < 64) vec[tid] = phi_elu1(to_f32(gq[st * D + tid]));
        __syncthreads();
        float op = 0.f;   // o = S phi(q) / den
#pragma unroll
        for (int j = 0; j < 16; ++j) op = fmaf(sf[Cf::F_S + tk_off(ar, 16 * cq + j, 64)], vec[16 * cq + j], op);
        op += __shfl_xor_sync(0xffffffffu, op, 1);
        op += __shfl_xor_sync(0xffffffffu, op, 2);
        if (cq == 0) go[st * D + ar] = from_f32<TIO>(op * misc[Cf::M_RDEN + t]);
        __syncthreads();
      }
      if constexpr (SPLIT) {   // AL (rows c.. zero) -> the S side, by the threads that send it in a normal chunk
        for (int e = tid; e < (64 - c) * 64; e += NT) sf[Cf::F_AL + tk_off(c + (e >> 6), e & 63, 64)] = 0.f;
        __syncthreads();
        if (row >= 64) {
          float al[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) al[j] = sf[Cf::F_AL + tk_off(row - 64, 32 * half + j, 64)];
          send_alpha(row - 64, al);
        }
        ++n_sent;
        __syncthreads();
      } else {
        if (tid == 0) misc[Cf::M_SSV] = 0.f;   // S changed step by step: its norm is recomputed
      }
      advance(c);
      continue;
    }
    // ---------------- Linv -> hi / lo operand tiles
    {
      const float* Xp = XB;
      // Linv (rows l, K = j) -> hi (L tile) + lo (Q tile 0); [W; H^T] -> hi in place + lo (P tiles)
      float lv[4][4];
      int loff[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int f = tid + NT * s;
        const int l = (f >> 7) * 8 + (f & 7), j4 = ((f >> 3) & 15) * 4;
        const int bi = l >> 3, bj = j4 >> 3;
        loff[s] = tk_off(l, j4, 64);
#pragma unroll
        for (int m = 0; m < 4; ++m) lv[s][m] = (bi >= bj) ? Xp[pb8(bi, bj) + (l & 7) * 8 + (j4 & 7) + m] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < 4; ++s) st4_split(Cf::F_L + loff[s], Cf::F_Q + loff[s], lv[s]);
      for (int e4 = tid; e4 < 2 * TILE / 4; e4 += NT) {   // [W; H^T] stays as the high part
        const float4 x = *reinterpret_cast<const float4*>(sf + Cf::F_R + 4 * e4);
        const float xv[4] = {x.x, x.y, x.z, x.w};
        st4_lo(Cf::F_P + 4 * e4, xv);
      }
    }
    // ---------------- G3: [Z; F^T] = [W; H^T] Linv^T  (M 128, N 64, K 64), 3xTF32
    {
      const MmaPass ps[3] = {{Cf::F_R, Cf::F_L, 128, 64, TC_G3, false},
                             {Cf::F_R, Cf::F_Q, 128, 64, TC_G3, true},
                             {Cf::F_P, Cf::F_L, 128, 64, TC_G3, true}};
      if (!mma_run(ps, 3, 64)) { failed = true; break; }
    }
    {
      // G4's X operand [Z D^{-1}; E^T] goes straight back into tensor memory (this thread's lane
      // is its row): hi into G2's columns (drained), lo into TC_XL; Z, G4's Y operand, goes to
      // the L tile (hi) and Q tile 0 (lo)
      float v32[32], xh[32], xl[32];
      tld32(TC_G3 + 32 * half, v32);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const int l = 32 * half + j;
        const float id4[4] = {misc[Cf::M_ID + l], misc[Cf::M_ID + l + 1], misc[Cf::M_ID + l + 2],
                              misc[Cf::M_ID + l + 3]};
        if (row < 64) {   // Z (rows i, K = l); Z D^{-1} rows i
#pragma unroll
          for (int m = 0; m < 4; ++m) xh[j + m] = v32[j + m] * id4[m];
          st4_split(Cf::F_L + tk_off(row, l, 64), Cf::F_Q + tk_off(row, l, 64), v32 + j);
        } else {          // E^T (rows t, K = l), masked to directions of steps <= t
          const int t = row - 64, lim = (t + 1) * R - 1;
#pragma unroll
          for (int m = 0; m < 4; ++m) xh[j + m] = (l + m <= lim) ? v32[j + m] * id4[m] : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) xl[j] = xh[j] - tf32_hi(xh[j]);
      const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);
      tc::tmem_st32(tq + (uint32_t)(TC_G2 + 32 * half), xh);
      tc::tmem_st32(tq + (uint32_t)(TC_XL + 32 * half), xl);
    }
    // ---------------- G4: [Z D^{-1} Z^T ; (Z E)^T] = [Z/D; E^T] Z^T  (M 128, N 64, K 64), 3xTF32, X in TMEM
    {
      MmaPass ps[3] = {{0, Cf::F_L, 128, 64, TC_G4, false},
                       {0, Cf::F_L, 128, 64, TC_G4, true},
                       {0, Cf::F_Q, 128, 64, TC_G4, true}};
      ps[0].tx = TC_G2;
      ps[1].tx = TC_XL;
      ps[2].tx = TC_G2;
      sync_tc();
      if (tid == 0) {
        mma_issue(ps, 3, 64);
        // the A side of a cluster writes alpha into AL next: the S side must be done with the last one
        if (SPLIT && n_sent > 0 && !mbar_wait_cluster_bounded(empty_bar, (n_sent - 1) & 1u)) *flag = 1;
      }
      if (!mma_wait()) { failed = true; break; }
    }
    }   // doA
    {
      float v32[32], al32[32];
      float an = 0.f;
      if (doA) tld32(TC_G4 + 32 * half, v32);
      if constexpr (SPLIT) {
        if (doS) {   // the S side of a cluster: wait for the chunk's alpha in AL
          if (tid == 0) {
            mbar_arrive_expect_tx(full_bar, TILE * sizeof(float));
            if (!mbar_wait_cluster_bounded(full_bar, n_recv & 1u)) *flag = 1;
          }
          ++n_recv;
          __syncthreads();
          if (*flag) { failed = true; break; }
        }
      }
      if (row >= 64) {   // alpha_t = Q_t - (Z E)_t (+ eps_n s_t at a nudge step), rows t (warp-uniform)
        const int t = row - 64;
        if (doA) {
          tld32(TC_G1 + 32 * half, al32);   // Q^T rows, from G1's accumulator
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float x = al32[j] - v32[j];
            if (nudge && t == c - 1) x = fmaf(a.eps_n, misc[Cf::M_SL + 32 * half + j], x);
            if (t >= c) x = 0.f;
            al32[j] = x;
            an = fmaf(x, x, an);
          }
          if (!SPLIT) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              st4(Cf::F_AL + tk_off(t, 32 * half + j, 64), al32[j], al32[j + 1], al32[j + 2], al32[j + 3]);
          }
        } else {   // the S side of a cluster: the same values, from the alpha it was sent
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 x4 = *reinterpret_cast<const float4*>(sf + Cf::F_AL + tk_off(t, 32 * half + j, 64));
            al32[j] = x4.x;
            al32[j + 1] = x4.y;
            al32[j + 2] = x4.z;
            al32[j + 3] = x4.w;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) an = fmaf(al32[j], al32[j], an);
        }
        if (doS) misc[Cf::M_AN2 + 64 * half + t] = an;   // |alpha_t|^2, two halves
      }
      if (SPLIT && doA) {   // the A side of a cluster: alpha to the S side while A is updated
        if (row >= 64) {
          send_alpha(row - 64, al32);
        } else {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            a_update(row, 32 * half + 16 * cc, *reinterpret_cast<float(*)[16]>(v32 + 16 * cc), nudge);
        }
        ++n_sent;
        __syncthreads();
        advance(c);
        continue;
      }
      // ---------------- G5: [S alpha ; S phi(q) | alpha.alpha ; phi(q).alpha] = [alpha; phi(q)] [S; alpha]^T,
      // issued as soon as alpha is written; the rest of G4's drain runs beside it.  With float32
      // I/O it is 3xTF32: [S lo; alpha lo; phi(q) lo] go to the P tiles and Q tile 0 (free once
      // G4 is done), contiguous like [S; alpha; phi(q)]
      if constexpr (F32) {
        if (row >= 64) {
          const int t = row - 64;
#pragma unroll
          for (int j = 0; j < 32; j += 4) st4_lo(Cf::F_P + TILE + tk_off(t, 32 * half + j, 64), al32 + j);
        }
        for (int e4 = tid; e4 < TILE / 4; e4 += NT) {
          const float4 s4 = *reinterpret_cast<const float4*>(sf + Cf::F_S + 4 * e4);
          const float4 q4v = *reinterpret_cast<const float4*>(sf + Cf::F_PQ + 4 * e4);
          const float sv[4] = {s4.x, s4.y, s4.z, s4.w}, qv[4] = {q4v.x, q4v.y, q4v.z, q4v.w};
          st4_lo(Cf::F_P + 4 * e4, sv);
          st4_lo(Cf::F_Q + 4 * e4, qv);
        }
      }
      sync_tc();
      if (tid == 0) {
        const MmaPass ps[3] = {{Cf::F_AL, Cf::F_S, 128, 128, TC_G5, false},
                               {Cf::F_P + TILE, Cf::F_S, 128, 128, TC_G5, true},
                               {Cf::F_AL, Cf::F_P, 128, 128, TC_G5, true}};
        mma_issue(ps, F32 ? 3 : 1, 64);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col0 = 32 * half + 16 * cc;
        float (&v)[16] = *reinterpret_cast<float(*)[16]>(v32 + 16 * cc);
        if (row < 64) {
          if (doA) a_update(row, col0, v, nudge);
        } else if (row - 64 < C) {
          // alpha^T (rows j, K = t): lane group g = lane / 4 writes column col0 + ((jj + g) & 15) in
          // store jj, so the 8 groups hit 8 different core-matrix rows (32 distinct banks)
          const int t = row - 64;
          float (&al)[16] = *reinterpret_cast<float(*)[16]>(al32 + 16 * cc);
          const int g = (lane >> 2) & 7;
          rot16(al, g);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) sf[Cf::F_T6 + Cf::T6_A + tk_off(col0 + ((jj + g) & 15), t, C)] = al[jj];
        }
      }
      // the renormalisation bound ||S|| + sum_t |v_t| |alpha_t| while G5 runs (one warp), when
      // ||S||^2 is carried from the previous chunk's state update; |alpha_t|^2 -> M_AN
      if (warp == 3 && misc[Cf::M_SSV] != 0.f) {
        const float ns = (misc[Cf::M_SS] + misc[Cf::M_SS + 1]) + (misc[Cf::M_SS + 2] + misc[Cf::M_SS + 3]);
        bound_test(ns);
      }
      // V^T (rows i, K = t) for G6: a lane reads column i of four steps (the lanes of a warp
      // read 32 consecutive columns of one step, conflict-free) and stores them as one float4
      for (int e = tid; e < 16 * C; e += NT) {
        const int i = e & 63, t0 = (e >> 6) * 4;
        st4(Cf::F_T6 + Cf::T6_V + tk_off(i, t0, C), to_f32(vb[t0 * 64 + i]), to_f32(vb[(t0 + 1) * 64 + i]),
            to_f32(vb[(t0 + 2) * 64 + i]), to_f32(vb[(t0 + 3) * 64 + i]));
      }
      if (!mma_wait()) { failed = true; break; }
    }
    if (row >= 64) {   // warp-uniform: quadrants 2, 3 (rows 64 + t); S phi(q_t) stays in TMEM for G6
      // aq[t][t'] = phi(q_t) . alpha_t', t' <= t -> tril(aq) rows t of T6 (half h: t' = 32 h .. 32 h + 31)
      const int t = row - 64;
      if (32 * half < C) {
        float v32[32];
        tld32(TC_G5 + 64 + 32 * half, v32);
        if (t < C) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const int tp = 32 * half + j;
            float x[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) x[m] = (tp + m <= t && t < c) ? v32[j + m] : 0.f;
            if (tp < C) st4(Cf::F_T6 + Cf::T6_Q + tk_off(t, tp, C), x[0], x[1], x[2], x[3]);
          }
        }
      }
    }
    // ||S||^2, the bound and the renormalisation decisions
    {
      // ||S||^2: carried from the previous chunk's state update (M_SS; the bound was then tested
      // beside G5), else recomputed here and the bound tested now
      float ns;
      if (misc[Cf::M_SSV] != 0.f) {
        ns = (misc[Cf::M_SS] + misc[Cf::M_SS + 1]) + (misc[Cf::M_SS + 2] + misc[Cf::M_SS + 3]);
      } else {
        float sq = 0.f;
        for (int e4 = tid; e4 < TILE / 4; e4 += NT) {
          const float4 x = *reinterpret_cast<const float4*>(sf + Cf::F_S + 4 * e4);
          sq = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, sq))));
        }
        ns = block_sum(sq);
        if (warp == 0) bound_test(ns);
        __syncthreads();
      }
      const bool exact = misc[Cf::M_EX] != 0.f;
      if (!exact) {
        if (tid < 64) {
          misc[Cf::M_SG + tid] = 1.f;   // sigma after step t
          misc[Cf::M_IS + tid] = 1.f;   // 1 / sigma before step t
        }
      } else {
        // V (rows t, K = i) as an operand tile in P tile 0 (its low part in P tile 1 with float32
        // I/O; both tiles are free since G5), and its Gram V V^T on the tensor core into G1's
        // columns (free since alpha was formed).  Rows C.. of the tile keep stale values: they
        // reach only rows and columns >= C of the product, which are never read.
        for (int f = tid; f < C * 8; f += NT) {
          const int t = (f >> 6) * 8 + (f & 7), pc = ((f & 7) + (f >> 3)) & 7;
          float x[8];
          if constexpr (F32) {
            const float4 a0 = *reinterpret_cast<const float4*>(vb + t * 64 + 8 * pc);
            const float4 a1 = *reinterpret_cast<const float4*>(vb + t * 64 + 8 * pc + 4);
            x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w; x[4] = a1.x; x[5] = a1.y; x[6] = a1.z; x[7] = a1.w;
          } else {
            const uint4 w = *reinterpret_cast<const uint4*>(vb + t * 64 + 8 * pc);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[m]));
              x[2 * m] = f2.x;
              x[2 * m + 1] = f2.y;
            }
          }
          st4(Cf::F_P + tk_off(t, 8 * pc, 64), x[0], x[1], x[2], x[3]);
          st4(Cf::F_P + tk_off(t, 8 * pc + 4, 64), x[4], x[5], x[6], x[7]);
          if constexpr (F32) {
            st4_lo(Cf::F_P + TILE + tk_off(t, 8 * pc, 64), x);
            st4_lo(Cf::F_P + TILE + tk_off(t, 8 * pc + 4, 64), x + 4);
          }
        }
        {
          const MmaPass ps[3] = {{Cf::F_P, Cf::F_P, 128, 64, TC_G1, false},
                                 {Cf::F_P + TILE, Cf::F_P, 128, 64, TC_G1, true},
                                 {Cf::F_P, Cf::F_P + TILE, 128, 64, TC_G1, true}};
          if (!mma_run(ps, F32 ? 3 : 1, 64)) { failed = true; break; }
        }
        // rows t < 64 (lanes of quadrants 0, 1): v_t . S alpha_t from G5's S alpha and the V
        // tile; the products PP[t][t'] = (v_t . v_t') (alpha_t . alpha_t') of row t: their
        // exclusive prefix sums Q[t][m] = sum_{t'<m} PP[t][t'] -> F_Q at m C + t, the diagonal
        // PP[t][t] -> M_VEC
        if (row < 64) {
          float v[16];
          const int t = row;
          if (half == 0) {
            float xs = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              tld(TC_G5 + 16 * cc, v);
#pragma unroll
              for (int j = 0; j < 16; j += 4) {
                const float4 v4 = *reinterpret_cast<const float4*>(sf + Cf::F_P + tk_off(t, 16 * cc + j, 64));
                xs = fmaf(v4.x, v[j], xs);
                xs = fmaf(v4.y, v[j + 1], xs);
                xs = fmaf(v4.z, v[j + 2], xs);
                xs = fmaf(v4.w, v[j + 3], xs);
              }
            }
            misc[Cf::M_XS + t] = (t < c) ? xs : 0.f;
          } else {
            float w[16], q = 0.f;
#pragma unroll
            for (int cc = 0; cc < (C + 15) / 16; ++cc) {
              tld(TC_G5 + 64 + 16 * cc, v);   // alpha_t . alpha_t'
              tld(TC_G1 + 16 * cc, w);        // v_t . v_t'
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int tp = 16 * cc + j;
                const float pp = v[j] * w[j];
                if (tp < C && t < C) {
                  sf[Cf::F_Q + tp * C + t] = q;
                  if (tp == t) misc[Cf::M_VEC + t] = pp;
                  if (tp < t) q += pp;
                }
              }
            }
          }
        }
        __syncthreads();
        if (warp == 0) {
          // S_t = sigma_t S_reg,t with S_reg,t = S_0 + sum_{t'<=t} v_t' alpha_t'^T / sigma_{t'-1}.
          // The norms are tracked unscaled (bounded by about tau), the cross terms through
          // the ratios sigma_{t-1} / sigma_{t'-1} <= 1, so nothing overflows however small
          // sigma gets.  Below 2^-64 the folded operands of G6 would grow past 2^64: the
          // chunk's S then goes step by step instead.
          //   ||S_t||^2 = ||S_{t-1}||^2 + 2 sigma_{t-1} (v_t . S_reg alpha_t + R_t) + PP[t][t],
          //   R_t = sum_{t'<t} PP[t][t'] / sigma_{t'-1}.
          // The decisions are taken in order by one warp.  Lane l keeps, for the steps l and
          // l + 32, x = v . S_reg alpha + R as far as the decisions taken so far go (the scales
          // of the steps not yet decided taken as the current one): at first R_t = Q[t][t].  A
          // renormalisation at step t changes 1/sigma by d for every t' > t, so each later x
          // gains d (Q[t][t] - Q[t][t + 1]) for its own row.
          constexpr int NSL = (C + 31) / 32;
          const float* QB = sf + Cf::F_Q;   // Q[t][m] at m C + t
          float xv[NSL], dg[NSL], qd[NSL];
#pragma unroll
          for (int sl = 0; sl < NSL; ++sl) {
            const int tq = lane + 32 * sl;
            const bool in = tq < c;
            qd[sl] = in ? QB[tq * C + tq] : 0.f;
            xv[sl] = in ? misc[Cf::M_XS + tq] + qd[sl] : 0.f;
            dg[sl] = in ? misc[Cf::M_VEC + tq] : 0.f;
          }
          float n2 = ns, sg = 1.f, isg = 1.f;   // ||S_{t-1}||^2, sigma_{t-1}, 1 / sigma_{t-1}
          unsigned int rc = 0;
          int deep_at = 0;
          // ||S_t|| > tau is decided as ||S_t||^2 > tau^2.  Where a step renormalises, the
          // factor tau / ||S_t|| comes from one reciprocal square root (rsqrt.approx, a few ulp),
          // and 1 / sigma follows by multiplication, keeping the chain of steps short.
          const float tau2 = a.tau * a.tau, itau = 1.f / a.tau;
          float rec_sg[NSL], rec_is[NSL];   // sigma_t and 1 / sigma_{t-1} of this lane's steps
#pragma unroll
          for (int s2 = 0; s2 < NSL; ++s2) rec_sg[s2] = rec_is[s2] = 1.f;
          int t_end = c;
          for (int t = 0; t < c; ++t) {
            const int sl = (NSL > 1 && t >= 32) ? 1 : 0;
            const float x = __shfl_sync(0xffffffffu, NSL > 1 && sl ? xv[NSL - 1] : xv[0], t & 31);
            const float dd = __shfl_sync(0xffffffffu, NSL > 1 && sl ? dg[NSL - 1] : dg[0], t & 31);
            float qn[NSL];   // Q[t'][t + 1] of this lane's later steps, loaded ahead of the decision
            bool later[NSL];
#pragma unroll
            for (int s2 = 0; s2 < NSL; ++s2) {
              const int tq = lane + 32 * s2;
              later[s2] = tq >= t + 2 && tq < c;
              qn[s2] = later[s2] ? QB[(t + 1) * C + tq] : 0.f;
            }
            const float isg_t = isg;
            const float npre2 = fmaf(2.f, sg * x, n2) + dd;
            if (!isfinite(npre2)) flags |= kStatusNonfinite;
            if (npre2 > tau2) {   // the same decision in every lane
              const float rs = rsqrtf(npre2);
              const float sgn = sg * (a.tau * rs);
              const float isn = isg * (npre2 * rs) * itau;
              const float dl = isn - isg;
#pragma unroll
              for (int s2 = 0; s2 < NSL; ++s2) xv[s2] = later[s2] ? fmaf(dl, qd[s2] - qn[s2], xv[s2]) : xv[s2];
              sg = sgn;
              isg = isn;
              n2 = tau2;
              ++rc;
            } else {
              n2 = npre2;
            }
            if (lane == (t & 31)) {   // static register indices
              if (sl == 0) {
                rec_sg[0] = sg;
                rec_is[0] = isg_t;
              } else {
                rec_sg[NSL - 1] = sg;
                rec_is[NSL - 1] = isg_t;
              }
            }
            if (!(sg >= 0x1p-64f)) { deep_at = 1; t_end = t + 1; break; }
          }
#pragma unroll
          for (int s2 = 0; s2 < NSL; ++s2) {
            const int tq = lane + 32 * s2;
            if (tq < t_end) {
              misc[Cf::M_SG + tq] = rec_sg[s2];
              misc[Cf::M_IS + tq] = rec_is[s2];
            }
          }
          if (lane == 0) {
            if (!deep_at) renorm_cnt += rc;
            misc[Cf::M_SCAL] = deep_at ? 1.f : 0.f;
          }
          for (int t = c + lane; t < 64; t += 32) {
            misc[Cf::M_SG + t] = sg;
            misc[Cf::M_IS + t] = isg;
          }
        }
        __syncthreads();
        if (misc[Cf::M_SCAL] != 0.f) {
          // S and the outputs step by step with the chunk's alpha (A and alpha are final)
          const int ar = tid >> 2, cq = tid & 3;
          for (int t = 0; t < c; ++t) {
            const float vr = to_f32(vb[t * 64 + ar]);
            float sq2 = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = 16 * cq + j;
              float& sr = sf[Cf::F_S + tk_off(ar, col, 64)];
              sr = fmaf(vr, sf[Cf::F_AL + tk_off(t, col, 64)], sr);
              sq2 = fmaf(sr, sr, sq2);
            }
            const float nrm = sqrtf(block_sum(sq2));
            if (nrm > a.tau) {
              const float cf = a.tau / nrm;
#pragma unroll
              for (int j = 0; j < 16; ++j) sf[Cf::F_S + tk_off(ar, 16 * cq + j, 64)] *= cf;
              if (tid == 0) ++renorm_cnt;
            }
            if (!isfinite(nrm)) flags |= kStatusNonfinite;
            float op = 0.f;   // o_t = S_t phi(q_t) / den_t (the thread's own S elements)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              op = fmaf(sf[Cf::F_S + tk_off(ar, 16 * cq + j, 64)], sf[Cf::F_PQ + tk_off(t, 16 * cq + j, 64)], op);
            op += __shfl_xor_sync(0xffffffffu, op, 1);
            op += __shfl_xor_sync(0xffffffffu, op, 2);
            if (cq == 0) go[(pos + t) * D + ar] = from_f32<TIO>(op * misc[Cf::M_RDEN + t]);
          }
          if (tid == 0) misc[Cf::M_SSV] = 0.f;   // S changed step by step: its norm is recomputed
          tc::fence_before_sync();
          __syncthreads();
          release_alpha();
          advance(c);
          continue;
        }
        // fold the per-step scales into tril(aq) (columns t') and alpha^T (columns t), in the
        // tiles' memory order: four consecutive floats are one row and columns k0 .. k0 + 3
        for (int e4 = tid; e4 < 16 * C; e4 += NT) {
          const int o = 4 * e4, k0 = ((o % (8 * C)) >> 5) << 2;
          const float4 i4 = *reinterpret_cast<const float4*>(misc + Cf::M_IS + k0);
          float4* pq = reinterpret_cast<float4*>(sf + Cf::F_T6 + Cf::T6_Q + o);
          float4* pa = reinterpret_cast<float4*>(sf + Cf::F_T6 + Cf::T6_A + o);
          float4 xq = *pq, xa = *pa;
          xq.x *= i4.x; xq.y *= i4.y; xq.z *= i4.z; xq.w *= i4.w;
          xa.x *= i4.x; xa.y *= i4.y; xa.z *= i4.z; xa.w *= i4.w;
          *pq = xq;
          *pa = xa;
        }
      }
    }
    // ---------------- G6: X = [V^T; tril(aq)] (M 128, K C); Y = V^T accumulates tril(aq) V onto
    // S phi(q_t) (rows 64 + t, columns 0..63); Y = alpha^T gives V^T alpha (rows i, columns 128..191)
    {
      // float32 I/O: 3xTF32, with the low parts of [V^T; tril(aq); alpha^T] in the P tiles (laid out
      // like T6; G5, their previous user, is done)
      if constexpr (F32) {
        __syncthreads();   // every thread's part of T6 (tril(aq) by rows t, alpha^T, V^T) is written
        for (int e4 = tid; e4 < 3 * Cf::T6T / 4; e4 += NT) {
          const float4 x = *reinterpret_cast<const float4*>(sf + Cf::F_T6 + 4 * e4);
          const float xv[4] = {x.x, x.y, x.z, x.w};
          st4_lo(Cf::F_P + 4 * e4, xv);
        }
      }
      const MmaPass ps[6] = {{Cf::F_T6, Cf::F_T6 + Cf::T6_V, 128, 64, TC_G5, true},
                             {Cf::F_T6, Cf::F_T6 + Cf::T6_A, 128, 64, TC_G6, false},
                             {Cf::F_P, Cf::F_T6 + Cf::T6_V, 128, 64, TC_G5, true},
                             {Cf::F_T6, Cf::F_P + Cf::T6_V, 128, 64, TC_G5, true},
                             {Cf::F_P, Cf::F_T6 + Cf::T6_A, 128, 64, TC_G6, true},
                             {Cf::F_T6, Cf::F_P + Cf::T6_A, 128, 64, TC_G6, true}};
      sync_tc();
      if (tid == 0) mma_issue(ps, F32 ? 6 : 2, C);
      // the next chunk's inputs into AL, PQ, Q tile 1 and vb: G6 and its drain do not touch
      // them, and every earlier access to them is fenced by the barrier above
      if constexpr (F32) stage_next(0);
      if (!mma_wait()) { failed = true; break; }
    }
    {
      float v32[32];
      if (row >= 64) {   // outputs of step t, columns 32 half .. 32 half + 31 (warp-uniform)
        const int t = row - 64;
        const float sgt = misc[Cf::M_SG + t], rd = misc[Cf::M_RDEN + t];
        tld32(TC_G5 + 32 * half, v32);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col0 = 32 * half + 16 * cc;
          float (&v)[16] = *reinterpret_cast<float(*)[16]>(v32 + 16 * cc);
          if (t < c) {
            float ov[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              ov[j] = sgt * v[j] * rd;
              if (!isfinite(ov[j])) flags |= kStatusNonfinite;
            }
            if constexpr (F32) {
              float4* dst = reinterpret_cast<float4*>(go + (pos + t) * D + col0);
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[j] = make_float4(ov[4 * j], ov[4 * j + 1], ov[4 * j + 2], ov[4 * j + 3]);
            } else {
              uint32_t pk[8];
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(ov[j], ov[j + 1]);
                pk[j / 2] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              uint4* dst = reinterpret_cast<uint4*>(go + (pos + t) * D + col0);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
      } else {           // S_1 = sigma (S + V^T alpha), rows i, columns 32 half .. 32 half + 31
        const int i = row;
        const float sgl = misc[Cf::M_SG + c - 1];
        float ss = 0.f;   // this thread's part of ||S_1||^2 for the next chunk's bound
        tld32(TC_G6 + 32 * half, v32);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col0 = 32 * half + 16 * cc;
          float (&v)[16] = *reinterpret_cast<float(*)[16]>(v32 + 16 * cc);
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            float4* sp = reinterpret_cast<float4*>(sf + Cf::F_S + tk_off(i, col0 + j, 64));
            float4 x = *sp;
            x.x = sgl * (x.x + v[j]);
            x.y = sgl * (x.y + v[j + 1]);
            x.z = sgl * (x.z + v[j + 2]);
            x.w = sgl * (x.w + v[j + 3]);
            *sp = x;
            ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, ss))));
          }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (lane == 0) misc[Cf::M_SS + q4 + 2 * half] = ss;   // warps 0, 1, 4, 5
        if (tid == 0) misc[Cf::M_SSV] = 1.f;
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    release_alpha();
    advance(c);
  }

  // ---- state out, TMEM freed
  tc::fence_before_sync();
  __syncthreads();
  if (!failed) {
    for (int e = tid; e < D * D; e += NT) {
      const int i = e >> 6, j = e & 63;
      if (doA) gA[e] = sf[Cf::F_A + tk_off(i, j, 64)];
      if (doS) gS[e] = sf[Cf::F_S + tk_off(i, j, 64)];
    }
    if (doS && tid < D) gn[tid] = misc[Cf::M_N + tid];
  } else if (tid == 0) {
    flags |= kStatusTimeout;
    if (!F32 && *issued > loaded) (void)mbar_wait_bounded(in_bar, (uint32_t)((loaded + 1) & 1));   // a copy in flight
    if (F32 && stage_pending) (void)mbar_wait_bounded(in_bar, stage_phase);                            // staged inputs
  }
  if constexpr (SPLIT) {
    // The asynchronous stores of the last alpha have landed once the S side has taken it (or
    // the wait gives up, long after); then neither CTA touches the other's shared memory again
    if (doA && tid == 0 && n_sent > 0) (void)mbar_wait_cluster_bounded(empty_bar, (n_sent - 1) & 1u);
    cluster_sync_all();
  }
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
  if (flags) atomicOr(&a.status->flags, flags);
  if (tid == 0) {
    if (guard_cnt) atomicAdd(&a.status->guard_count, guard_cnt);
    if (renorm_cnt) atomicAdd(&a.status->renorm_count, renorm_cnt);
    if (fallback_cnt) atomicAdd(&a.status->chunk_fallbacks, fallback_cnt);
  }
}

// How many two-CTA clusters of chunk_scan_kernel<R, TIO, true> fit on the device at once.
template <int R, typename TIO>
cudaError_t cluster_capacity_t(int* n) {
  using Cf = chk::Cfg<R, TIO>;
  auto kern = chunk_scan_kernel<R, TIO, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(chk::NT, 1, 1);
  cfg.dynamicSmemBytes = Cf::bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, kern, &cfg);
}

// ctas = 2: a cluster of two CTAs per pair (the A side and the S side)
template <int R, typename TIO>
cudaError_t launch_chunk_t(const ScanArgs& a, int ctas, cudaStream_t s) {
  using Cf = chk::Cfg<R, TIO>;
  if (ctas != 2) {
    auto kern = chunk_scan_kernel<R, TIO, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::bytes);
    if (e != cudaSuccess) return e;
    kern<<<a.pairs, chk::NT, Cf::bytes, s>>>(a);
    return cudaGetLastError();
  }
  auto kern = chunk_scan_kernel<R, TIO, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * a.pairs), 1, 1);
  cfg.blockDim = dim3(chk::NT, 1, 1);
  cfg.dynamicSmemBytes = Cf::bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace vla
