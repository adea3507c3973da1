// Internal declarations shared by the scan kernels and the C ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace vla {

// Device-side status block, accumulated with atomics by every CTA at its end.
struct DevStatus {
  unsigned int flags;
  unsigned int reserved;
  unsigned long long guard_count;
  unsigned long long renorm_count;
  unsigned long long chunk_fallbacks;
};

// Per-pair status record (used by the entry point that allocates nothing).
struct PairStatus {
  unsigned int flags;
  unsigned int guard_count;
  unsigned int renorm_count;
  unsigned int chunk_fallbacks;
};

constexpr unsigned int kStatusNonfinite = 1u;
constexpr unsigned int kStatusTimeout = 2u;

// Arguments of one scan launch (plain pointers; the pair index p = b*H + h is
// blockIdx.x).
struct ScanArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* u;
  float* A;
  float* S;
  float* n;
  void* o;
  long long T;
  long long t0;
  int P;
  float eps_n;
  float tau;
  int pairs;
  DevStatus* status;          // accumulated status (handle entry point)
  PairStatus* pair_status;    // per-pair status (no-allocation entry point)
};

// Host-side launchers; each returns cudaSuccess or the launch error.
cudaError_t launch_seq(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_chunked(int d, int r, bool bf16, int chunk, int ctas, const ScanArgs& a, cudaStream_t s,
                           bool* built);
cudaError_t launch_delta(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_project_u(int d, bool bf16, const void* k, const float* W, void* u, long long n, int r,
                             int sm_count, DevStatus* status, cudaStream_t s, bool* built);
// Gather the window [off, off + tj) of four [pairs, T, w_bytes[i]] host tensors (read
// through the device addresses src[i] of page-locked host memory) into dense
// [pairs, tj, w_bytes[i]] device buffers dst[i]; w_bytes[i] and all pointers 16-byte
// aligned.  `ctas` CTAs of 1024 threads.
cudaError_t launch_gather_window(const void* const src[4], void* const dst[4], const long long w_bytes[4],
                                 long long pairs, long long T, long long off, long long tj, int ctas,
                                 cudaStream_t s);

// One CTA whose thread 0 waits limit_ns on an mbarrier that nothing completes and then
// sets kStatusTimeout in *status (the path every bounded wait of the scans takes).
cudaError_t launch_wait_selftest(DevStatus* status, unsigned long long limit_ns, cudaStream_t s);

// Message returned by vla_last_error(NULL) on the calling thread.
void set_thread_error(const char* msg);

// --------------------------------------------------------------------------
// device helpers (inline PTX: mbarrier, bulk asynchronous copies, timers)
// --------------------------------------------------------------------------

// Upper bound on any wait for an input copy.  A copy of a few tens of KB lands
// in microseconds; after this long the CTA gives up and reports a timeout.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed, false after limit_ns (kWaitLimitNs).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t_start = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t_start > limit_ns) return false;
  }
}

// ---- thread-block clusters: distributed shared memory and cluster-scope mbarriers

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs arrives and waits (both CTAs of a cluster are
// resident together, so this completes).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Asynchronous store of four floats into another CTA of the cluster (addr and bar are that
// CTA's shared-memory addresses, from mapa_shared): 16 bytes of complete_tx on its mbarrier
// bar, which makes them visible to the threads that see the phase complete.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float x, float y, float z, float w, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(x), "f"(y), "f"(z), "f"(w), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Arrive (release, cluster scope) on an mbarrier in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire: true when the phase completed, false
// after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t_start = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer_ns() - t_start > kWaitLimitNs) return false;
  }
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float phi_elu1(float x) {
  // ELU(x) + 1 with alpha = 1: x + 1 for x > 0, exp(x) otherwise.
  return x > 0.f ? x + 1.f : expf(x);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace vla
