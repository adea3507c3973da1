// C ABI of the VLA scan: argument checks, handle, status block, dispatch.
#include "vla.h"
#include "vla_internal.cuh"

#include <cuda.h>   // driver types for the pointer-attribute query (resolved at run time)

#include <cmath>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>

namespace vla {
cudaError_t launch_seq_block_d16(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_seq_block_d64(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);
cudaError_t launch_seq_block_d128(int r, bool bf16, bool cluster, const ScanArgs& a, cudaStream_t s, bool* built);

// the row-split scan on a cluster of `ctas` (4 or 8) CTAs per pair (vla_rows.cu)
cudaError_t launch_rows(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built);
// two-CTA clusters of the chunked kernel resident at once (vla_chunked.cu)
int chunked_cluster_capacity(int r, bool bf16);

cudaError_t launch_seq(int d, int r, bool bf16, int ctas, const ScanArgs& a, cudaStream_t s, bool* built) {
  if (ctas == 4 || ctas == 8) return launch_rows(d, r, bf16, ctas, a, s, built);
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

namespace {
constexpr int kHostSlots = 3;   // staging slots of the host-buffer path (copy in / scan / copy out)
}

struct vla_handle_s {
  int device = 0;
  int sm_count = 0;
  vla::DevStatus* status = nullptr;
  std::string last_error;
  // Host-buffer path (vla_scan_fwd_host), made on its first use: a device workspace with
  // the state and kHostSlots staging slots, a copy-in and a copy-out stream, and events.
  bool host_ready = false;
  int last_gathered = -1;       // copy-in path and window of the last vla_scan_fwd_host call
  long long last_seg = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr;
  cudaEvent_t ev_in[kHostSlots] = {}, ev_run[kHostSlots] = {}, ev_out[kHostSlots] = {};
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

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Shapes with a kernel (the list in the UNSUPPORTED message below).
bool shape_built(int d, int dv, int r, bool bf16, vla_mode_t mode, int chunk, int ctas) {
  if (d != dv || (d != 16 && d != 64 && d != 128) || (r != 1 && r != 4)) return false;
  switch (mode) {
    case VLA_SEQUENTIAL:
      return ctas == 1 || ctas == 2 || ((ctas == 4 || ctas == 8) && r == 1 && (d == 64 || d == 128));
    case VLA_DELTA: return chunk == 0;
    case VLA_CHUNKED:
      return d == 64 && ((r == 1 && (chunk == 0 || chunk == 64)) || (r == 4 && (chunk == 0 || chunk == 16)));
  }
  return false;
}

// Argument checks shared by the device and host entry points; sets *ctas (CTAs per pair).
// Sequential and delta modes: by default a cluster of two for d = 128 while 2 B H CTAs fit
// on the SMs (one CTA of 4 d threads would be capped at 128 registers a thread and spill);
// one otherwise (at d <= 64 the hand-off between two SMs costs more than the issue slots it
// frees).  Chunked mode: a cluster of two (the A side and the S side of each chunk on two
// SMs) while 2 B H CTAs fit on the SMs and B H such clusters can be resident at once (the
// occupancy query), else one: clusters in two waves would take longer than one CTA each.
vla_err_t check_scan(vla_handle_t h, const char* fn, int B, int H, long long T, int d, int dv, int r, int P,
                     float eps_n, float tau, long long t0, vla_dtype_t io_dtype, vla_mode_t mode, int chunk,
                     int* ctas) {
  const std::string f(fn);
  if (B < 0 || H < 0 || T < 0 || d <= 0 || dv <= 0 || r <= 0)
    return fail(h, VLA_ERR_INVALID_ARG, f + ": negative size or non-positive d/dv/r");
  if (P < 0) return fail(h, VLA_ERR_INVALID_ARG, f + ": P < 0");
  if (t0 < 0) return fail(h, VLA_ERR_INVALID_ARG, f + ": t0 < 0");
  if (!(tau > 0.f)) return fail(h, VLA_ERR_INVALID_ARG, f + ": tau must be > 0 (NaN rejected)");
  if (!std::isfinite(eps_n)) return fail(h, VLA_ERR_INVALID_ARG, f + ": eps_n must be finite");
  if (io_dtype != VLA_F32 && io_dtype != VLA_BF16) return fail(h, VLA_ERR_INVALID_ARG, f + ": unknown io_dtype");
  if (mode != VLA_SEQUENTIAL && mode != VLA_CHUNKED && mode != VLA_DELTA)
    return fail(h, VLA_ERR_INVALID_ARG, f + ": unknown mode");
  const long long pairs = (long long)B * H;
  if (pairs > 0x7fffffffLL) return fail(h, VLA_ERR_INVALID_ARG, f + ": B*H too large");
  if (d != dv) return fail(h, VLA_ERR_UNSUPPORTED, f + ": built only for d == dv");
  const int auto_ctas = (d == 128 && 2 * pairs <= h->sm_count) ? 2 : 1;
  const bool bf16 = io_dtype == VLA_BF16;
  const int chunk_ctas =
      (mode == VLA_CHUNKED && 2 * pairs <= h->sm_count && pairs <= vla::chunked_cluster_capacity(r, bf16)) ? 2 : 1;
  *ctas = mode == VLA_SEQUENTIAL ? (chunk != 0 ? chunk : auto_ctas) : mode == VLA_DELTA ? auto_ctas : chunk_ctas;
  if (!shape_built(d, dv, r, bf16, mode, chunk, *ctas)) {
    char buf[400];
    std::snprintf(buf, sizeof buf,
                  "%s: not built for d=%d dv=%d r=%d dtype=%s mode=%s chunk=%d "
                  "(sequential: d=dv in {16,64,128}, r in {1,4}, chunk = CTAs per pair 1 or 2, 0 = default, "
                  "or 4 / 8 (rows of A split) at d in {64,128} with r = 1; "
                  "chunked: d=dv=64, bf16 or f32, r=1 chunk 64 or r=4 chunk 16, 0 = default; "
                  "delta: d=dv in {16,64,128}, r in {1,4}, chunk 0)",
                  fn, d, dv, r, bf16 ? "bf16" : "f32",
                  mode == VLA_SEQUENTIAL ? "sequential" : mode == VLA_DELTA ? "delta" : "chunked", chunk);
    return fail(h, VLA_ERR_UNSUPPORTED, buf);
  }
  return VLA_OK;
}

// Launch the kernel of (mode, d, r, dtype) on `s`; the shape was checked by check_scan.
cudaError_t dispatch(const vla::ScanArgs& a, int d, int r, bool bf16, vla_mode_t mode, int chunk, int ctas,
                     cudaStream_t s) {
  bool built = false;
  cudaError_t e = mode == VLA_SEQUENTIAL ? vla::launch_seq(d, r, bf16, ctas, a, s, &built)
                  : mode == VLA_DELTA    ? vla::launch_delta(d, r, bf16, ctas, a, s, &built)
                                         : vla::launch_chunked(d, r, bf16, chunk, ctas, a, s, &built);
  return built ? e : cudaErrorNotSupported;
}

// Steps per window of the host-buffer path, a multiple of 64 (whole chunks in VLA_CHUNKED
// mode).  Gathered by the SMs: the whole sequence up to 2048 steps, else about 32 windows
// of at least 512 steps, so that the copy-in of one window overlaps the scan of the one
// before and the pipeline fills and drains in a thirty-second of the sequence (windows of
// 384 to 768 steps give the same end-to-end time at T = 16384, 1024 steps 2 % more).
// Copied by the copy engines: rows of at least 512 KB (`step_bytes` = bytes a step of the
// narrowest input takes), below which the engines lose rate when rows of four tensors
// alternate.
long long default_segment(long long T, bool gathered, long long step_bytes) {
  if (T <= 2048) return T;
  long long seg = ((T + 31) / 32 + 63) / 64 * 64;
  if (seg < 512) seg = 512;
  if (!gathered) {
    const long long rows = ((512 * 1024 + step_bytes - 1) / step_bytes + 63) / 64 * 64;
    if (seg < rows) seg = rows;
  }
  return seg < T ? seg : T;
}

// Device address through which a kernel may read the host buffer [p, p + bytes), or
// NULL when that range is not inside one page-locked host allocation mapped into the
// current device's address space (pageable memory, a range that runs past its
// allocation, no mapping) or p is not 16-byte aligned.  Both ends must be CUDA host
// memory whose device addresses are bytes - 1 apart and that belong to the same
// allocation (the driver's buffer id), so the whole range is one mapped allocation.
const void* mapped_host_range(const void* p, size_t bytes) {
  if (!p || bytes == 0 || !aligned16(p)) return nullptr;
  using GetAttr = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);
  static GetAttr get_attr = []() -> GetAttr {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<GetAttr>(fn);
  }();
  if (!get_attr) return nullptr;
  const char* last = static_cast<const char*>(p) + bytes - 1;
  cudaPointerAttributes a0{}, a1{};
  if (cudaPointerGetAttributes(&a0, p) != cudaSuccess || cudaPointerGetAttributes(&a1, last) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a0.type != cudaMemoryTypeHost || a1.type != cudaMemoryTypeHost || !a0.devicePointer || !a1.devicePointer)
    return nullptr;
  if (static_cast<const char*>(a1.devicePointer) - static_cast<const char*>(a0.devicePointer) !=
      static_cast<ptrdiff_t>(bytes - 1))
    return nullptr;
  unsigned long long id0 = 0, id1 = 0;
  if (get_attr(&id0, CU_POINTER_ATTRIBUTE_BUFFER_ID, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS ||
      get_attr(&id1, CU_POINTER_ATTRIBUTE_BUFFER_ID, reinterpret_cast<CUdeviceptr>(last)) != CUDA_SUCCESS ||
      id0 != id1 || id0 == 0)
    return nullptr;
  return a0.devicePointer;
}

void host_path_free(vla_handle_t h);

cudaError_t host_path_init(vla_handle_t h) {
  if (h->host_ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking);
  cudaEvent_t* evs[] = {&h->ev_start, &h->ev_end};
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < kHostSlots && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_run[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) h->host_ready = true;
  else host_path_free(h);
  return e;
}

void host_path_free(vla_handle_t h) {
  if (h->ws) cudaFree(h->ws);
  if (h->s_in) cudaStreamDestroy(h->s_in);
  if (h->s_out) cudaStreamDestroy(h->s_out);
  for (cudaEvent_t* ev : {&h->ev_start, &h->ev_end}) {
    if (*ev) cudaEventDestroy(*ev);
    *ev = nullptr;
  }
  for (int i = 0; i < kHostSlots; ++i)
    for (cudaEvent_t* ev : {&h->ev_in[i], &h->ev_run[i], &h->ev_out[i]}) {
      if (*ev) cudaEventDestroy(*ev);
      *ev = nullptr;
    }
  h->ws = nullptr;
  h->ws_bytes = 0;
  h->s_in = h->s_out = nullptr;
  h->host_ready = false;
}

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
  const char* fn = "vla_scan_fwd";
  if (!h) return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_scan_fwd: handle is NULL");
  h->last_error.clear();
  int ctas = 0;
  vla_err_t err = check_scan(h, fn, B, H, T, d, dv, r, P, eps_n, tau, t0, io_dtype, mode, chunk, &ctas);
  if (err != VLA_OK) return err;
  const long long pairs = (long long)B * H;
  if (pairs == 0) return VLA_OK;
  if (!A || !S || !n) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: NULL state pointer");
  if (T == 0) return VLA_OK;
  if (!q || !k || !v || !u || !o) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: NULL stream pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(u) || !aligned16(A) || !aligned16(S))
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: q, k, v, u, A and S must be 16-byte aligned");
  if (mode == VLA_CHUNKED && !aligned16(o))
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd: VLA_CHUNKED needs o 16-byte aligned");

  vla::ScanArgs a{};
  a.q = q; a.k = k; a.v = v; a.u = u;
  a.A = A; a.S = S; a.n = n; a.o = o;
  a.T = T; a.t0 = t0; a.P = P; a.eps_n = eps_n; a.tau = tau;
  a.pairs = (int)pairs;
  a.status = h->status;
  cudaError_t e = on_device(h->device, [&]() {
    return dispatch(a, d, r, io_dtype == VLA_BF16, mode, chunk, ctas, static_cast<cudaStream_t>(stream));
  });
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_scan_fwd: launch", e));
  return VLA_OK;
}

vla_err_t vla_scan_fwd_host(vla_handle_t h, const void* q, const void* k, const void* v, const void* u,
                            float* A, float* S, float* n, void* o, int B, int H, long long T, int d,
                            int dv, int r, int P, float eps_n, float tau, long long t0,
                            vla_dtype_t io_dtype, vla_mode_t mode, int chunk, long long seg,
                            void* stream) {
  const char* fn = "vla_scan_fwd_host";
  if (!h) return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_scan_fwd_host: handle is NULL");
  h->last_error.clear();
  int ctas = 0;
  vla_err_t err = check_scan(h, fn, B, H, T, d, dv, r, P, eps_n, tau, t0, io_dtype, mode, chunk, &ctas);
  if (err != VLA_OK) return err;
  if (seg < 0) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd_host: seg < 0");
  const long long pairs = (long long)B * H;
  if (pairs == 0) return VLA_OK;
  if (!A || !S || !n) return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd_host: NULL state pointer");
  if (T == 0) return VLA_OK;
  if (!q || !k || !v || !u || !o)
    return fail(h, VLA_ERR_INVALID_ARG, "vla_scan_fwd_host: NULL stream pointer");

  const bool bf16 = io_dtype == VLA_BF16;
  const size_t es = bf16 ? 2 : 4;
  const size_t P_ = (size_t)pairs;
  const long long w_bytes[4] = {(long long)(d * es), (long long)(d * es), (long long)(dv * es),
                                (long long)(r * d * es)};
  const void* host_in[4] = {q, k, v, u};
  // copy-in path: the SM gather when every input is one mapped page-locked allocation
  const void* mapped[4] = {};
  bool gathered = true;
  std::string what;
  cudaError_t e = on_device(h->device, [&]() -> cudaError_t {
    for (int t = 0; t < 4 && gathered; ++t) {
      mapped[t] = mapped_host_range(host_in[t], P_ * (size_t)T * (size_t)w_bytes[t]);
      gathered = mapped[t] != nullptr;
    }
    return cudaSuccess;
  });
  if (seg == 0) seg = default_segment(T, gathered, std::min(w_bytes[0], w_bytes[2]));
  if (seg > T) seg = T;
  h->last_gathered = gathered ? 1 : 0;
  h->last_seg = seg;
  // workspace: state, then kHostSlots slots of [q | k | v | u | o], each piece [pairs, seg, .]
  const size_t sg = (size_t)seg;
  const size_t bA = align256(P_ * d * d * 4), bS = align256(P_ * dv * d * 4), bn = align256(P_ * d * 4);
  const size_t bq = align256(P_ * sg * d * es), bv = align256(P_ * sg * dv * es);
  const size_t bu = align256(P_ * sg * r * d * es);
  const size_t slot = 2 * bq + bv + bu + bv;
  const size_t need = bA + bS + bn + kHostSlots * slot;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // CTAs of the gather: the SMs the scan leaves idle (one scan CTA per pair, two in the
  // two-CTA cluster variants), at least 8 and at most 32.
  const long long scan_sms = std::min<long long>(pairs * (ctas == 2 ? 2 : 1), h->sm_count);
  const int gather_ctas = (int)std::max<long long>(8, std::min<long long>(32, h->sm_count - scan_sms));
  e = on_device(h->device, [&]() -> cudaError_t {
    cudaError_t r_ = host_path_init(h);
    if (r_ != cudaSuccess) { what = "stream/event creation"; return r_; }
    if (h->ws_bytes < need) {
      what = "workspace allocation";
      if (h->ws) {
        r_ = cudaEventSynchronize(h->ev_end);   // the last host-path call no longer uses it
        if (r_ != cudaSuccess) return r_;
        r_ = cudaFree(h->ws);
        h->ws = nullptr;
        h->ws_bytes = 0;
        if (r_ != cudaSuccess) return r_;
      }
      r_ = cudaMalloc(&h->ws, need);
      if (r_ != cudaSuccess) { h->ws = nullptr; return r_; }
      h->ws_bytes = need;
    }
    what = "enqueue";
    char* base = static_cast<char*>(h->ws);
    float* dA = reinterpret_cast<float*>(base);
    float* dS = reinterpret_cast<float*>(base + bA);
    float* dn = reinterpret_cast<float*>(base + bA + bS);
    char* slots = base + bA + bS + bn;
#define VLA_TRY(x) do { cudaError_t r2 = (x); if (r2 != cudaSuccess) return r2; } while (0)
    // start after the caller's earlier work on `stream` and after the previous host-path call
    VLA_TRY(cudaEventRecord(h->ev_start, s));
    for (cudaStream_t t : {h->s_in, h->s_out}) {
      VLA_TRY(cudaStreamWaitEvent(t, h->ev_start, 0));
      VLA_TRY(cudaStreamWaitEvent(t, h->ev_end, 0));
    }
    VLA_TRY(cudaStreamWaitEvent(s, h->ev_end, 0));
    VLA_TRY(cudaMemcpyAsync(dA, A, P_ * d * d * 4, cudaMemcpyHostToDevice, h->s_in));
    VLA_TRY(cudaMemcpyAsync(dS, S, P_ * dv * d * 4, cudaMemcpyHostToDevice, h->s_in));
    VLA_TRY(cudaMemcpyAsync(dn, n, P_ * d * 4, cudaMemcpyHostToDevice, h->s_in));
    const long long nseg = (T + seg - 1) / seg;
    for (long long j = 0; j < nseg; ++j) {
      const int sl = (int)(j % kHostSlots);
      const long long off = j * seg;
      const size_t tj = (size_t)std::min(seg, T - off);
      char* sq = slots + sl * slot;
      char* sk = sq + bq;
      char* sv = sk + bq;
      char* su = sv + bv;
      char* so = su + bu;
      // copy in: a [pairs, tj, w] window of each [pairs, T, w] host tensor
      if (j >= kHostSlots) VLA_TRY(cudaStreamWaitEvent(h->s_in, h->ev_run[sl], 0));
      void* const dst_in[4] = {sq, sk, sv, su};
      if (gathered) {
        VLA_TRY(vla::launch_gather_window(mapped, dst_in, w_bytes, pairs, T, off, (long long)tj, gather_ctas,
                                          h->s_in));
      } else {
        for (int t = 0; t < 4; ++t) {
          const size_t w = (size_t)w_bytes[t];
          VLA_TRY(cudaMemcpy2DAsync(dst_in[t], tj * w, static_cast<const char*>(host_in[t]) + off * w,
                                    (size_t)T * w, tj * w, P_, cudaMemcpyHostToDevice, h->s_in));
        }
      }
      VLA_TRY(cudaEventRecord(h->ev_in[sl], h->s_in));
      // scan the window on the caller's stream
      VLA_TRY(cudaStreamWaitEvent(s, h->ev_in[sl], 0));
      if (j >= kHostSlots) VLA_TRY(cudaStreamWaitEvent(s, h->ev_out[sl], 0));
      vla::ScanArgs a{};
      a.q = sq; a.k = sk; a.v = sv; a.u = su;
      a.A = dA; a.S = dS; a.n = dn; a.o = so;
      a.T = (long long)tj; a.t0 = t0 + off; a.P = P; a.eps_n = eps_n; a.tau = tau;
      a.pairs = (int)pairs;
      a.status = h->status;
      VLA_TRY(dispatch(a, d, r, bf16, mode, chunk, ctas, s));
      VLA_TRY(cudaEventRecord(h->ev_run[sl], s));
      // copy out the window of o
      VLA_TRY(cudaStreamWaitEvent(h->s_out, h->ev_run[sl], 0));
      VLA_TRY(cudaMemcpy2DAsync(static_cast<char*>(o) + off * dv * es, (size_t)T * dv * es, so, tj * dv * es,
                                tj * dv * es, P_, cudaMemcpyDeviceToHost, h->s_out));
      VLA_TRY(cudaEventRecord(h->ev_out[sl], h->s_out));
    }
    // the final state, after the last window's scan (s_out already waits for it)
    VLA_TRY(cudaMemcpyAsync(A, dA, P_ * d * d * 4, cudaMemcpyDeviceToHost, h->s_out));
    VLA_TRY(cudaMemcpyAsync(S, dS, P_ * dv * d * 4, cudaMemcpyDeviceToHost, h->s_out));
    VLA_TRY(cudaMemcpyAsync(n, dn, P_ * d * 4, cudaMemcpyDeviceToHost, h->s_out));
    VLA_TRY(cudaEventRecord(h->ev_end, h->s_out));
    VLA_TRY(cudaStreamWaitEvent(s, h->ev_end, 0));
#undef VLA_TRY
    return cudaSuccess;
  });
  if (e != cudaSuccess) {
    const vla_err_t code = e == cudaErrorMemoryAllocation ? VLA_ERR_NOMEM : VLA_ERR_CUDA;
    return fail(h, code, cuda_msg(("vla_scan_fwd_host: " + what).c_str(), e));
  }
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
  if (!aligned16(k_raw) || !aligned16(W_u) || !aligned16(u))
    return fail(h, VLA_ERR_INVALID_ARG, "vla_project_u: k_raw, W_u and u must be 16-byte aligned");
  bool built = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = on_device(h->device, [&]() -> cudaError_t {
    return vla::launch_project_u(d, io_dtype == VLA_BF16, k_raw, W_u, u, n_tokens, r, h->sm_count, h->status, s,
                                 &built);
  });
  if (!built) return fail(h, VLA_ERR_UNSUPPORTED, "vla_project_u: built for d in {16, 64, 128}");
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_project_u: launch", e));
  return VLA_OK;
}

vla_err_t vla_selftest_wait(vla_handle_t h, unsigned int limit_ms, void* stream) {
  if (!h) return fail(nullptr, VLA_ERR_INVALID_ARG, "vla_selftest_wait: handle is NULL");
  h->last_error.clear();
  if (limit_ms < 1 || limit_ms > 5000) return fail(h, VLA_ERR_INVALID_ARG, "vla_selftest_wait: limit_ms must be 1..5000");
  cudaError_t e = on_device(h->device, [&]() {
    return vla::launch_wait_selftest(h->status, 1000000ull * limit_ms, static_cast<cudaStream_t>(stream));
  });
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_selftest_wait: launch", e));
  return VLA_OK;
}

}  // extern "C"

namespace vla {
// The FP32 throughput probe (vla_peak.cu): 4 CTAs of 256 threads per SM, `iters` (rounded
// up to a multiple of 8) packed FMAs on 8 chains per thread; *flops = the launch's flops.
cudaError_t launch_ffma_probe(long long iters, int sm_count, DevStatus* status, cudaStream_t s, double* flops);
}  // namespace vla

extern "C" {

vla_err_t vla_ffma_probe(vla_handle_t h, long long iters, double* flops, void* stream) {
  if (!h || !flops) return fail(h, VLA_ERR_INVALID_ARG, "vla_ffma_probe: NULL argument");
  h->last_error.clear();
  if (iters < 8 || iters > (1ll << 30)) return fail(h, VLA_ERR_INVALID_ARG, "vla_ffma_probe: iters must be 8..2^30");
  cudaError_t e = on_device(h->device, [&]() {
    return vla::launch_ffma_probe(iters, h->sm_count, h->status, static_cast<cudaStream_t>(stream), flops);
  });
  if (e != cudaSuccess) return fail(h, VLA_ERR_CUDA, cuda_msg("vla_ffma_probe: launch", e));
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

vla_err_t vla_host_path_info(vla_handle_t h, int* gathered, long long* seg) {
  if (!h || !gathered || !seg) return fail(h, VLA_ERR_INVALID_ARG, "vla_host_path_info: NULL argument");
  *gathered = h->last_gathered;
  *seg = h->last_seg;
  return VLA_OK;
}

const char* vla_last_error(vla_handle_t h) {
  return h ? h->last_error.c_str() : g_create_error.c_str();
}

vla_err_t vla_destroy(vla_handle_t h) {
  if (!h) return VLA_OK;
  cudaError_t e = on_device(h->device, [&]() -> cudaError_t {
    cudaError_t r = cudaDeviceSynchronize();
    host_path_free(h);
    cudaError_t r2 = cudaFree(h->status);
    return r != cudaSuccess ? r : r2;
  });
  delete h;
  if (e != cudaSuccess) return fail(nullptr, VLA_ERR_CUDA, cuda_msg("vla_destroy", e));
  return VLA_OK;
}

}  // extern "C"
