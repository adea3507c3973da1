// C ABI of the VLA scan: argument checks, handle, status block, dispatch.
#include "vla.h"
#include "vla_internal.cuh"

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

namespace vla {
cudaError_t launch_seq_block_d16(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_seq_block_d64(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_seq_block_d128(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);

cudaError_t launch_seq(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built) {
  const bool cluster = ctas == 2;
  switch (d) {
    case 16: return launch_seq_block_d16(r, bf16, cluster, a, s, built);
    case 64: return launch_seq_block_d64(r, bf16, cluster, a, s, built);
    case 128: return launch_seq_block_d128(r, bf16, cluster, a, s, built);
    default: *built = false; return cudaSuccess;
  }
}
}  // namespace vla

namespace {
thread_local std::string g_create_error;
}

void vla::set_thread_error(const char* msg) { g_create_error = msg ? msg : ""; }

struct vla_handle_s {
  int device = 0;
  int sm_count = 0;
  vla::DevStatus* status = nullptr;
  std::string last_error;
};

namespace {

vla_err_t fail(vla_handle_t h, vla_err_t code, const std::string& msg) {
  if (h) h->last_error = msg; else g_create_error = msg;
  return code;
}

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

// Runs `fn` with `device` current and restores the caller's device.
template <typename F>
cudaError_t on_device(int device, F fn) {
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return e;
  if (prev != device) {
    e = cudaSetDevice(device);
    if (e != cudaSuccess) return e;
  }
  cudaError_t r = fn();
  if (prev != device) {
    cudaError_t e2 = cudaSetDevice(prev);
    if (r == cudaSuccess) r = e2;
  }
  return r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

vla_err_t vla_create(vla_handle_t* h, int device) {
  if (!h) return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_create: h is NULL");
  *h = nullptr;
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return fail(nullptr, VLA_ERR_CUDA, cuda_msg("vla_create: cudaGetDeviceCount", e));
  if (device < 0 || device >= count)
    return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_create: no CUDA device " + std::to_string(device));
  vla_handle_s* hh = new (std::nothrow) vla_handle_s();
  if (!hh) return fail(nullptr, VLA_ERR_NOMEM, "vla_create: out of host memory");
  hh->device = device;
  e = on_device(device, [&]() -> cudaError_t {
    cudaError_t r = cudaDeviceGetAttribute(&hh->sm_count, cudaDevAttrMultiProcessorCount, device);
    if (r != cudaSuccess) return r;
    r = cudaMalloc(&hh->status, sizeof(vla::DevStatus));
    if (r != cudaSuccess) return r;
    return cudaMemset(hh->status, 0, sizeof(vla::DevStatus));
  });
  if (e != cudaSuccess) {
    if (hh->status) on_device(device, [&]() { return cudaFree(hh->status); });
    delete hh;
    return fail(nullptr, e == cudaErrorMemoryAllocation ? VLA_ERR_NOMEM : VLA_ERR_CUDA,
                cuda_msg("vla_create: status block", e));
  }
  *h = hh;
  g_create_error.clear();
  return VLA_OK;
}

vla_err_t vla_scan_fwd(vla_handle_t h, const void* q, const void* k, const void* v, const void* u,
                       float* A, float* S, float* n, void* o, int B, int H, long long T, int d, int dv,
                       int r, int P, float eps_n, float tau, long long t0, vla_dtype_t io_dtype,
                       vla_mode_t mode, int chunk, void* stream) {
  if (!h) return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_scan_fwd: handle is NULL");
  h->last_error.clear();
  if (B < 0 || H < 0 || T < 0 || d <= 0 || dv <= 0 || r <= 0)
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: negative size or non-positive d/dv/r");
  if (P < 0) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: P < 0");
  if (t0 < 0) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: t0 < 0");
  if (!(tau > 0.f)) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: tau must be > 0 (NaN rejected)");
  if (!std::isfinite(eps_n)) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: eps_n must be finite");
  if (io_dtype != VLA_F32 && io_dtype != VLA_BF16)
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: unknown io_dtype");
  if (mode != VLA_SEQUENTIAL && mode != VLA_CHUNKED && mode != VLA_DELTA)
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: unknown mode");
  const long long pairs = (long long)B * H;
  if (pairs > 0x7fffffffLL) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: B*H too large");
  if (pairs == 0) return VLA_OK;
  if (!A || !S || !n) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: NULL state pointer");
  if (T == 0) return VLA_OK;
  if (!q || !k || !v || !u || !o) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: NULL stream pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(u) || !aligned16(A) || !aligned16(S))
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: q, k, v, u, A and S must be 16-byte aligned");
  if (mode == VLA_CHUNKED && !aligned16(o))
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: VLA_CHUNKED needs o 16-byte aligned");
  if (d != dv) return fail(h, VLA_ERR_UNSUPPORTED, "vla_scan_fwd: built only for d == dv");

  vla::ScanArgs a{};
  a.q = q; a.k = k; a.v = v; a.u = u;
  a.A = A; a.S = S; a.n = n; a.o = o;
  a.T = T; a.t0 = t0; a.P = P; a.eps_n = eps_n; a.tau = tau;
  a.pairs = (int)pairs;
  a.status = h->status;
  const bool bf16 = io_dtype == VLA_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool built = false;
  // sequential mode: CTAs per pair.  By default a cluster of two for d = 128 while 2 B H
  // CTAs fit on the SMs (one CTA of 4 d threads would be capped at 128 registers a thread
  // and spill); one otherwise (at d <= 64 the hand-off between two SMs costs more than
  // the issue slots it frees).
  const int ctas = (mode != VLA_SEQUENTIAL) ? 0
                   : (chunk != 0 ? chunk : ((d == 128 && 2 * pairs <= h->sm_count) ? 2 : 1));
  cudaError_t e = cudaSuccess;
  if ((mode == VLA_SEQUENTIAL && ctas != 1 && ctas != 2) || (mode == VLA_DELTA && chunk != 0)) {
    built = false;
  } else {
    e = on_device(h->device, [&]() -> cudaError_t {
      if (mode == VLA_SEQUENTIAL) return vla::launch_seq(d, r, bf16, ctas, a, s, &built);
      if (mode == VLA_DELTA) return vla::launch_delta(d, r, bf16, a, s, &built);
      return vla::launch_chunked(d, r, bf16, chunk, a, s, &built);
    });
  }
  if (!built) {
    char buf[384];
    std::snprintf(buf, sizeof buf,
                  "vla_scan_fwd: not built for d=%d dv=%d r=%d dtype=%s mode=%s chunk=%d "
                  "(sequential: d=dv in {16,64,128}, r in {1,4}, chunk = CTAs per pair 1 or 2, 0 = default; "
                  "chunked: d=dv=64, bf16, r=1 chunk 64 or r=4 chunk 16, 0 = default; "
                  "delta: d=dv in {16,64,128}, r in {1,4}, chunk 0)",
                  d, dv, r, bf16 ? "bf16" : "f32", mode == VLA_SEQUENTIAL ? "sequential" : mode == VLA_DELTA ? "delta" : "chunked", chunk);
    return fail(h, VLA_ERR_UNSUPPORTED, buf);
  }
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_scan_fwd: launch", e));
  return VLA_OK;
}

vla_err_t vla_project_u(vla_handle_t h, const void* k_raw, const float* W_u, void* u, long long n_tokens,
                        int d, int r, vla_dtype_t io_dtype, void* stream) {
  if (!h) return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_project_u: handle is NULL");
  h->last_error.clear();
  if (n_tokens < 0) return fail(h, VLA_ERR_INVALID_ARG, "vla_project_u: n_tokens < 0");
  if (r < 1 || r > 8) return fail(h, VLA_ERR_INVALID_ARG, "vla_project_u: r must be 1..8");
  if (io_dtype != VLA_F32 && io_dtype != VLA_BF16)
    return fail(h, VLA_ERR_INVALID_ARG, "vla_project_u: unknown io_dtype");
  if (n_tokens == 0) return VLA_OK;
  if (!k_raw || !W_u || !u) return fail(h, VLA_ERR_INVALID_ARG, "vla_project_u: NULL pointer");
  bool built = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = on_device(h->device, [&]() -> cudaError_t {
    return vla::launch_project_u(d, io_dtype == VLA_BF16, k_raw, W_u, u, n_tokens, r, h->sm_count, s, &built);
  });
  if (!built) return fail(h, VLA_ERR_UNSUPPORTED, "vla_project_u: built for d in {16, 64, 128}");
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_project_u: launch", e));
  return VLA_OK;
}

vla_err_t vla_status(vla_handle_t h, void* stream, vla_status_t* out) {
  if (!h || !out) return fail(h, VLA_ERR_INVALID_ARG, "vla_status: NULL argument");
  vla::DevStatus st{};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = on_device(h->device, [&]() -> cudaError_t {
    cudaError_t r = cudaMemcpyAsync(&st, h->status, sizeof st, cudaMemcpyDeviceToHost, s);
    if (r != cudaSuccess) return r;
    r = cudaMemsetAsync(h->status, 0, sizeof st, s);
    if (r != cudaSuccess) return r;
    return cudaStreamSynchronize(s);
  });
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_status", e));
  out->flags = st.flags;
  out->reserved = 0;
  out->guard_count = st.guard_count;
  out->renorm_count = st.renorm_count;
  out->chunk_fallbacks = st.chunk_fallbacks;
  return VLA_OK;
}

const char* vla_last_error(vla_handle_t h) {
  return h ? h->last_error.c_str() : g_create_error.c_str();
}

vla_err_t vla_destroy(vla_handle_t h) {
  if (!h) return VLA_OK;
  cudaError_t e = on_device(h->device, [&]() -> cudaError_t {
    cudaError_t r = cudaDeviceSynchronize();
    cudaError_t r2 = cudaFree(h->status);
    return r != cudaSuccess ? r : r2;
  });
  delete h;
  if (e != cudaSuccess) return fail(nullptr, VLA_ERR_CUDA, cuda_msg("vla_destroy", e));
  return VLA_OK;
}

}  // extern "C"
