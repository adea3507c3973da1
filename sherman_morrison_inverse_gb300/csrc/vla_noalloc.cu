// Scan entry point that allocates nothing (see vla_scan_fwd_noalloc in vla.h).
//
// Its scratch -- one status record per (batch, head) pair, which the kernel
// accumulates into -- lives in a file-scope __device__ array instead of memory
// that a handle would allocate.  In host code the array's name only stands in
// for the symbol; the device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernel.
#include <cmath>
#include <mutex>

#include "vla.h"
#include "vla_seqk.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The scratch: VLA_NOALLOC_MAX_PAIRS records of 16 bytes (256 KB), held by
// every GPU that loads the library until the process exits.
static __device__ __align__(256) vla::PairStatus g_pair_scratch[VLA_NOALLOC_MAX_PAIRS];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on `device` (which must be current).
cudaError_t scratch_on(int device, vla::PairStatus** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_pair_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = p;
  }
  *out = static_cast<vla::PairStatus*>(g_scratch_ptr[device]);
  return cudaSuccess;
}

vla_err_t fail(vla_err_t code, const char* msg) {
  vla::set_thread_error(msg);
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" vla_err_t vla_scan_fwd_noalloc(const void* q, const void* k, const void* v, const void* u,
                                          float* A, float* S, float* n, void* o, int B, int H, long long T,
                                          int d, int dv, int r, int P, float eps_n, float tau, long long t0,
                                          vla_dtype_t io_dtype, vla_pair_status_t* pair_status, void* stream) {
  vla::set_thread_error("");
  if (B < 0 || H < 0 || T < 0 || d <= 0 || dv <= 0 || r <= 0)
    return fail(VLA_ERR_INVALID_ARG, "vla_scan_fwd_noalloc: negative size or non-positive d/dv/r");
  if (P < 0 || t0 < 0 || !(tau > 0.f) || !std::isfinite(eps_n))
    return fail(VLA_ERR_INVALID_ARG, "vla_scan_fwd_noalloc: bad P, t0, tau or eps_n");
  if (io_dtype != VLA_F32 && io_dtype != VLA_BF16)
    return fail(VLA_ERR_INVALID_ARG, "vla_scan_fwd_noalloc: unknown io_dtype");
  const long long pairs = (long long)B * H;
  if (pairs > VLA_NOALLOC_MAX_PAIRS)
    return fail(VLA_ERR_INVALID_ARG,
                "vla_scan_fwd_noalloc: B*H exceeds VLA_NOALLOC_MAX_PAIRS (16384), the size of its static scratch");
  if (pairs == 0 || T == 0) return VLA_OK;
  if (!A || !S || !n || !q || !k || !v || !u || !o)
    return fail(VLA_ERR_INVALID_ARG, "vla_scan_fwd_noalloc: NULL pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(u) || !aligned16(A) || !aligned16(S))
    return fail(VLA_ERR_INVALID_ARG, "vla_scan_fwd_noalloc: q, k, v, u, A and S must be 16-byte aligned");
  if (d != 64 || dv != 64 || (r != 1 && r != 4))
    return fail(VLA_ERR_UNSUPPORTED, "vla_scan_fwd_noalloc: built for d = dv = 64 and r in {1, 4}");

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess || device < 0 || device >= kMaxDevices)
    return fail(VLA_ERR_CUDA, "vla_scan_fwd_noalloc: no usable current device");
  vla::PairStatus* scratch = nullptr;
  e = scratch_on(device, &scratch);
  if (e != cudaSuccess) return fail(VLA_ERR_CUDA, "vla_scan_fwd_noalloc: cudaGetSymbolAddress failed");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = sizeof(vla::PairStatus) * (size_t)pairs;
  e = cudaMemsetAsync(scratch, 0, bytes, s);   // the records accumulate: start this call at zero
  if (e != cudaSuccess) return fail(VLA_ERR_CUDA, "vla_scan_fwd_noalloc: clearing the scratch failed");

  vla::ScanArgs a{};
  a.q = q; a.k = k; a.v = v; a.u = u;
  a.A = A; a.S = S; a.n = n; a.o = o;
  a.T = T; a.t0 = t0; a.P = P; a.eps_n = eps_n; a.tau = tau;
  a.pairs = (int)pairs;
  a.status = nullptr;
  a.pair_status = scratch;
  const bool bf16 = io_dtype == VLA_BF16;
  if (r == 1)
    e = bf16 ? vla::launch_seq_block_t<64, 1, 4, __nv_bfloat16, true>(a, s)
             : vla::launch_seq_block_t<64, 1, 4, float, true>(a, s);
  else
    e = bf16 ? vla::launch_seq_block_t<64, 4, 1, __nv_bfloat16, true>(a, s)
             : vla::launch_seq_block_t<64, 4, 1, float, true>(a, s);
  if (e != cudaSuccess) return fail(VLA_ERR_CUDA, "vla_scan_fwd_noalloc: launch failed");
  if (pair_status) {
    e = cudaMemcpyAsync(pair_status, scratch, bytes, cudaMemcpyDefault, s);
    if (e != cudaSuccess) return fail(VLA_ERR_CUDA, "vla_scan_fwd_noalloc: copying the status failed");
  }
  return VLA_OK;
}
