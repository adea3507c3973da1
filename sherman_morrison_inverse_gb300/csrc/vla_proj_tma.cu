// Direction projection u_{t,i} = W_u[i] k_t / max(|W_u[i] k_t|_2, 1e-12) with bfloat16 keys:
// the README "VLA v3" item 2 "u_t = normalize(W_u k_t^raw)", the form that streams keys and
// directions through the tensor memory accelerator (TMA) on sm_103a.
//
// One persistent CTA per SM walks tiles of 128 tokens (tile = blockIdx.x, + gridDim.x, ...).
// Roles, by warp:
//   warp 0 (one thread)  producer: each key tile [128][d] bf16 arrives with one TMA tensor
//                        load per 64-column slab (128-byte swizzle; 32-byte at d = 16) into a
//                        ring of `ks` stages (as many as shared memory holds beside W and the
//                        staging tiles, up to 8), completing on the stage's `full` mbarrier;
//   warp 1               allocates tensor memory; one thread issues the products: all ranks
//                        of a tile, stacked, as one x = K W^T of N = r d columns (groups of
//                        256 / d ranks when r d > 256), so every key is read from HBM once.  K is
//                        read straight from the swizzled stage, W (three bf16 terms w1 + w2 + w3
//                        of the float32 weights, three passes, fp32 accumulation) from shared
//                        memory.  Jobs alternate between two TMEM accumulators;
//   warps 2..9           two epilogue warpgroups, one per accumulator: thread = token row (its
//                        TMEM lane); per rank it loads the row, forms |x|, scales, rounds to
//                        bf16 and writes the row into a 128-byte-swizzled staging tile (every
//                        8 consecutive lanes hit 8 different 16-byte bank groups); one thread
//                        sends each staging tile out with a TMA tensor store.
// Handshakes: key stage full (TMA bytes) -> MMA; MMA commit -> accumulator full -> epilogue;
// epilogue arrivals -> accumulator empty -> next MMA into it; MMA commit after a tile's last
// product -> key stage empty -> producer.  Staging tiles are reused after the bulk-async group
// that read them has finished reading.  Every wait is bounded (2 s): a wait that runs out
// sets VLA_STATUS_TIMEOUT, and the CTA drains what it started and returns.
#include <cuda.h>   // CUtensorMap and the encode entry point's types (resolved at run time)

#include "vla_internal.cuh"
#include "vla_tc.cuh"

namespace vla {
namespace prj {

constexpr int kTmaThreads = 320;   // 10 warps
constexpr int kRows = 128;         // tokens per tile = TMEM lanes of an M = 128 product

template <int D>
struct TmaCfg {
  static constexpr int BX = D < 64 ? D : 64;                // columns of a slab (box width)
  static constexpr int NSLAB = D / BX;                      // slabs per row: 1, or 2 at d = 128
  static constexpr int SLAB = kRows * BX * 2;               // bytes of one [128][BX] bf16 slab
  static constexpr int KEY = NSLAB * SLAB;                  // bytes of one key tile
  static constexpr int KMAX = 8;                            // key stages at most
  static constexpr int NSU = 2;                             // staging slabs per epilogue group
  static constexpr int GMAX = 256 / D;                      // ranks per product (N <= 256)
  static constexpr uint32_t SW_MODE = BX == 64 ? 2u : 6u;   // descriptor swizzle: 128 B / 32 B
  static constexpr uint32_t SW_SBO = 8u * BX * 2u;          // bytes between 8-row groups
  // shared memory: the key ring (ks stages) | staging (2 groups x NSU slabs) | three W terms
  // ([r d][d] bf16 each) | mbarriers (2 ks + 5) | TMEM slot and failure flag
  __host__ __device__ static size_t off_stg(int ks) { return (size_t)ks * KEY; }
  __host__ __device__ static size_t off_w(int ks) { return off_stg(ks) + (size_t)2 * NSU * SLAB; }
  __host__ __device__ static size_t w_bytes(int r) { return (size_t)3 * r * D * D * 2; }
  __host__ __device__ static size_t bar_off(int r, int ks) { return (off_w(ks) + w_bytes(r) + 15) / 16 * 16; }
  __host__ __device__ static size_t bytes(int r, int ks) { return bar_off(r, ks) + 8 * (2 * ks + 5) + 16; }
  // the most key stages (<= KMAX) that fit in `limit` bytes beside the rest; 0 if fewer than 2
  static int stages(int r, size_t limit) {
    for (int ks = KMAX; ks >= 2; --ks)
      if (bytes(r, ks) <= limit) return ks;
    return 0;
  }
};

// K-major operand of 16-bit elements in the swizzled layout a TMA tiled load writes: rows of
// BX elements (BX * 2 bytes), 8-row groups SBO bytes apart, 16-byte chunks permuted within
// each swizzle atom by the address bits above them (the atom starts on a 1024-byte boundary).
__device__ __forceinline__ uint64_t sdesc_sw(uint32_t saddr, uint32_t sbo_bytes, uint32_t mode) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                               // leading-dimension offset (unused here)
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;                                // descriptor version (fixed field)
  d |= (uint64_t)mode << 61;                             // swizzle mode
  return d;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// Named barrier over n threads that also ORs a flag across them.
__device__ __forceinline__ bool named_or(int id, int n, bool x) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)x), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// N consecutive fp32 columns of this warp's 32 TMEM lanes; the wait is inside the same asm
// statement, so no use of the values can be scheduled before it.
template <int N>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float* v);
template <>
__device__ __forceinline__ void tmem_row<16>(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
template <>
__device__ __forceinline__ void tmem_row<32>(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // round to nearest even
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D>
__global__ void __launch_bounds__(kTmaThreads, 1)
    project_u_tma_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_u,
                         const float* __restrict__ W, long long n, int r, int ks, uint32_t tmem_cols,
                         DevStatus* __restrict__ status) {
  using Cf = TmaCfg<D>;
  constexpr int BX = Cf::BX, NSLAB = Cf::NSLAB;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the swizzled stages need 1024-byte alignment; report rather than run misaligned
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicOr(&status->flags, kStatusTimeout);
    return;
  }
  const size_t boff = Cf::bar_off(r, ks);
  const size_t off_w = Cf::off_w(ks), off_stg = Cf::off_stg(ks);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + boff);   // [ks] key stage loaded
  uint64_t* empty = full + ks;                                  // [ks] key stage consumed
  uint64_t* tfull = empty + ks;                                 // [2] accumulator written
  uint64_t* tempty = tfull + 2;                                 // [2] accumulator drained
  uint64_t* done = tempty + 2;                                  // every product issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* fail = reinterpret_cast<volatile int*>(tslot + 1);

  const int ngroups = (r + Cf::GMAX - 1) / Cf::GMAX;          // products per tile
  const int G = r < Cf::GMAX ? r : Cf::GMAX;                   // ranks per product
  const long long ntiles = (n + kRows - 1) / kRows;
  const long long nlt = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;   // this CTA's tiles
  const long long njobs = nlt * ngroups;

  // W_u -> three bf16 terms, K-major no-swizzle, rows i d + j (output j of rank i), K = input m
  {
    const int rows = r * D;
    for (int e8 = tid; e8 < rows * D / 8; e8 += kTmaThreads) {
      const int row = (8 * e8) / D, m = 8 * e8 - row * D;
      const float4 a = reinterpret_cast<const float4*>(W)[2 * e8];
      const float4 b = reinterpret_cast<const float4*>(W)[2 * e8 + 1];
      float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int term = 0; term < 3; ++term) {
        uint32_t p[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float t0 = __bfloat162float(__float2bfloat16_rn(x[2 * q]));
          const float t1 = __bfloat162float(__float2bfloat16_rn(x[2 * q + 1]));
          p[q] = pack_bf16x2(t0, t1);
          x[2 * q] -= t0;       // exact: t is x rounded to 8 significant bits
          x[2 * q + 1] -= t1;
        }
        *reinterpret_cast<uint4*>(smem + off_w + (size_t)term * rows * D * 2 + 2 * tc::tk16_off(row, m, D)) =
            make_uint4(p[0], p[1], p[2], p[3]);
      }
    }
  }
  if (tid == 0) {
    for (int s = 0; s < ks; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 128);
    }
    mbar_init(done, 1);
    *fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(tslot, tmem_cols);
  fence_proxy_async_smem();   // W, written by the generic proxy, is read by the tensor core
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t bufcols = tmem_cols / 2;

  if (warp == 0) {
    // ---------------- producer
    if (lane == 0) {
      long long lt = 0;
      int s = 0;          // stage of tile lt
      uint32_t k = 0;     // use of that stage
      for (; lt < nlt && !*fail; ++lt) {
        if (k > 0 && !mbar_wait_bounded(empty + s, (k - 1) & 1u)) { *fail = 1; break; }
        const int y = (int)((blockIdx.x + lt * gridDim.x) * kRows);
        mbar_arrive_expect_tx(full + s, (uint32_t)Cf::KEY);
#pragma unroll
        for (int sl = 0; sl < NSLAB; ++sl) tma_load_2d(smem + s * Cf::KEY + sl * Cf::SLAB, &map_k, sl * BX, y, full + s);
        if (++s == ks) { s = 0; ++k; }
      }
      // the last load of each stage has landed before the CTA can leave (bounded)
      for (long long j = (lt > ks ? lt - ks : 0); j < lt; ++j)
        if (!mbar_wait_bounded(full + (int)(j % ks), (uint32_t)((j / ks) & 1))) *fail = 1;
    }
  } else if (warp == 1) {
    // ---------------- products
    if (lane == 0) {
      const uint32_t idesc_full = tc::idesc_bf16(128, G * D);
      const uint32_t sbase = smem_u32(smem);
      const size_t term_bytes = (size_t)r * D * D * 2;
      int s = 0, g = 0;   // stage of the current tile, rank group of the current job
      uint32_t k = 0;     // use of that stage
      for (long long jl = 0; jl < njobs && !*fail; ++jl) {
        if (g == 0 && !mbar_wait_bounded(full + s, k & 1u)) { *fail = 1; break; }
        const int b = (int)(jl & 1);
        const long long use = jl >> 1;
        if (use > 0 && !mbar_wait_bounded(tempty + b, (uint32_t)((use - 1) & 1))) { *fail = 1; break; }
        tc::fence_after_sync();
        const int i0 = g * G, ng = (r - i0) < G ? (r - i0) : G;
        const uint32_t idesc = ng == G ? idesc_full : tc::idesc_bf16(128, ng * D);
        const uint32_t d_tmem = tmem + (uint32_t)b * bufcols;
        const uint32_t kbase = sbase + (uint32_t)(s * Cf::KEY);
        const uint32_t wbase = sbase + (uint32_t)off_w + (uint32_t)(i0 * D * D * 2);
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = kbase + (uint32_t)((kk * 16) / BX) * Cf::SLAB + (uint32_t)(((kk * 16) % BX) * 2);
            tc::mma_f16(d_tmem, sdesc_sw(ka, Cf::SW_SBO, Cf::SW_MODE),
                        tc::sdesc(wbase + (uint32_t)(p * term_bytes) + 256u * kk, 16u * D), idesc, p > 0 || kk > 0);
          }
        tc::mma_commit(tfull + b);
        if (g == ngroups - 1) {
          tc::mma_commit(empty + s);   // the stage's last reader
          g = 0;
          if (++s == ks) { s = 0; ++k; }
        } else {
          ++g;
        }
      }
      tc::mma_commit(done);
      if (!mbar_wait_bounded(done, 0)) *fail = 1;
    }
  } else {
    // ---------------- epilogue: group eg takes the jobs jl = eg, eg + 2, ...
    const int eg = (warp - 2) >> 2;
    const int q = warp & 3;                           // TMEM lane quadrant of this warp
    const int row = 32 * q + lane;                    // token row of the tile
    const bool issuer = (warp == 2 + 4 * eg) && lane == 0;
    const int bar_id = 1 + eg;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)eg * bufcols;
    unsigned char* stg0 = smem + off_stg + eg * Cf::NSU * Cf::SLAB;
    const int swz = BX == 64 ? (row & 7) : ((row >> 2) & 1);
    long long unit = 0;
    for (long long jl = eg; jl < njobs; jl += 2) {
      const long long use = jl >> 1;
      const bool ok = mbar_wait_bounded(tfull + eg, (uint32_t)(use & 1));
      if (named_or(bar_id, 128, !ok || *fail)) { *fail = 1; break; }
      tc::fence_after_sync();
      const long long lt = jl / ngroups;
      const int g = (int)(jl - lt * ngroups);
      const int i0 = g * G, ng = (r - i0) < G ? (r - i0) : G;
      const int y = (int)((blockIdx.x + lt * gridDim.x) * kRows);
      for (int ii = 0; ii < ng; ++ii) {
        float x[D];
        if constexpr (D == 16) {
          tmem_row<16>(tl + (uint32_t)(ii * D), x);
        } else {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) tmem_row<32>(tl + (uint32_t)(ii * D + c0), x + c0);
        }
        if (ii == ng - 1) {   // the accumulator is drained: the next product may overwrite it
          tc::fence_before_sync();
          mbar_arrive1(tempty + eg);
        }
        float nrm = 0.f;
#pragma unroll
        for (int j = 0; j < D; ++j) nrm = fmaf(x[j], x[j], nrm);
        const float inv = 1.f / fmaxf(sqrtf(nrm), 1e-12f);
#pragma unroll
        for (int sl = 0; sl < NSLAB; ++sl, ++unit) {
          unsigned char* stg = stg0 + (int)(unit % Cf::NSU) * Cf::SLAB;
#pragma unroll
          for (int c = 0; c < BX / 8; ++c) {
            const float* xs = x + sl * BX + 8 * c;
            const uint4 v = make_uint4(pack_bf16x2(xs[0] * inv, xs[1] * inv), pack_bf16x2(xs[2] * inv, xs[3] * inv),
                                       pack_bf16x2(xs[4] * inv, xs[5] * inv), pack_bf16x2(xs[6] * inv, xs[7] * inv));
            *reinterpret_cast<uint4*>(stg + row * (BX * 2) + 16 * (c ^ swz)) = v;
          }
          fence_proxy_async_smem();
          // the store that read the other staging slab has finished reading it before anyone
          // moves on to write that slab
          if (issuer) bulk_wait_read0();
          named_sync(bar_id, 128);
          if (issuer) {
            tma_store_2d(&map_u, (i0 + ii) * D + sl * BX, y, stg);
            bulk_commit();
          }
        }
      }
    }
    if (issuer) bulk_wait0();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, tmem_cols);
  if (tid == 0 && *fail) atomicOr(&status->flags, kStatusTimeout);
}

// ---------------------------------------------------------------------------
// host side

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encode_fn() {
  static EncodeTiled fn = []() -> EncodeTiled {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// [rows][cols] bf16 row-major at `base`, tiles of [128][box_cols]; false if it cannot be encoded
static bool encode_2d(CUtensorMap* m, const void* base, long long rows, long long cols, int box_cols, bool sw128) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)kRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch the TMA form when its operands fit (shared memory for W's three terms of all r ranks,
// n below 2^31 tokens, tensor maps encodable); *used = false leaves the call to the other form.
template <int D>
cudaError_t launch_project_tma(const void* k, const float* W, void* u, long long n, int r, int sm_count,
                               DevStatus* status, cudaStream_t s, bool* used) {
  using Cf = TmaCfg<D>;
  *used = false;
  const int ks = Cf::stages(r, 227 * 1024);
  if (ks < 2 || n <= 0 || n >= (1ll << 31) - kRows) return cudaSuccess;
  const size_t bytes = Cf::bytes(r, ks);
  CUtensorMap mk, mu;
  if (!encode_2d(&mk, k, n, D, Cf::BX, Cf::BX == 64) || !encode_2d(&mu, u, n, (long long)r * D, Cf::BX, Cf::BX == 64))
    return cudaSuccess;
  const int G = r < Cf::GMAX ? r : Cf::GMAX;
  uint32_t cols = 32;
  while (cols < 2u * (uint32_t)(G * D)) cols <<= 1;
  auto kern = project_u_tma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const long long ntiles = (n + kRows - 1) / kRows;
  const int grid = (int)(ntiles < sm_count ? ntiles : (sm_count > 0 ? sm_count : 1));
  *used = true;
  kern<<<grid, kTmaThreads, bytes, s>>>(mk, mu, W, n, r, ks, cols, status);
  return cudaGetLastError();
}

template cudaError_t launch_project_tma<16>(const void*, const float*, void*, long long, int, int, DevStatus*,
                                            cudaStream_t, bool*);
template cudaError_t launch_project_tma<64>(const void*, const float*, void*, long long, int, int, DevStatus*,
                                            cudaStream_t, bool*);
template cudaError_t launch_project_tma<128>(const void*, const float*, void*, long long, int, int, DevStatus*,
                                             cudaStream_t, bool*);

}  // namespace prj
}  // namespace vla
