// abi.cu -- the exported C entry points of libtrellis.so (declared in
// include/trellis.h): argument validation on the host, then one kernel
// launch on the caller's stream.  Nothing here allocates device memory.
//
// The checks follow the pages' TrellisGeometry rules ("trellis-linear.ts":
// trellisGeometry throws unless the words hold whole k-bit symbols and the
// columns are whole blocks; fusedGateUpSwiglu throws for M > 4) and add the
// GPU kernels' own supported set (k in {2,3,4}, L in {12,16}, T = 256,
// 16-byte aligned pointers).  Every failed check returns before any CUDA call.
#include <cstdint>
#include <cuda_runtime.h>

#include "devcache.h"
#include "launch.h"
#include "trellis.h"

namespace {

constexpr int kAbiVersion = 101;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int geom_ok(const trellis_geom_t* g) {
  if (!g) return TRELLIS_ENULL;
  if (g->k < 2 || g->k > 4) return TRELLIS_EGEOM;
  if (g->L != 16 && g->L != 12) return TRELLIS_EGEOM;
  if (g->T != trellis::kT_host) return TRELLIS_EGEOM;
  if (g->axis != 0 && g->axis != 1) return TRELLIS_EGEOM;
  if (g->rows < 1 || g->cols < 1 || g->cols % g->T != 0) return TRELLIS_EGEOM;
  if (((int64_t)g->T * g->k) % 32 != 0) return TRELLIS_EGEOM;
  if (g->rows > INT32_MAX || g->cols > INT32_MAX || g->rows * g->cols > ((int64_t)1 << 40))
    return TRELLIS_EGEOM;
  if (g->reserved != 0) return TRELLIS_EGEOM;
  if (g->interleave != 0) {  // the pages' interleaved layout exists for k = 3, T = 256, axis 0 only
    if (g->interleave != 2 || g->k != 3 || g->axis != 0 || g->cols % (2 * g->T) != 0) return TRELLIS_EGEOM;
  }
  return TRELLIS_OK;
}

// The current device must be compute capability 10.3 (the library holds
// sm_103a code only).  Cached per device.
int device_ok() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return TRELLIS_EDEVICE;
  }
  static trellis::PerDevice<int> ok_of;
  const auto probe = [dev] {
    int major = 0, minor = 0;
    const bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                    major == 10 && minor == 3;
    if (!ok) cudaGetLastError();
    return ok ? TRELLIS_OK : TRELLIS_EDEVICE;
  };
  return dev < trellis::kMaxDevices ? ok_of.get(dev, probe, TRELLIS_EDEVICE) : probe();
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? TRELLIS_OK : TRELLIS_ECUDA; }

}  // namespace

extern "C" {

int trellis_abi_version(void) { return kAbiVersion; }

const char* trellis_status_string(int status) {
  switch (status) {
    case TRELLIS_OK: return "ok";
    case TRELLIS_EGEOM: return "unsupported or inconsistent trellis geometry";
    case TRELLIS_EM: return "M outside the range this call supports";
    case TRELLIS_EALIGN: return "a pointer is not 16-byte aligned";
    case TRELLIS_EAXIS: return "the geometry's axis does not fit this call";
    case TRELLIS_EWORKSPACE: return "workspace missing, misaligned or too small";
    case TRELLIS_ECUDA: return "CUDA error at launch";
    case TRELLIS_ENULL: return "a required pointer is NULL";
    case TRELLIS_EDEVICE: return "no usable sm_103 CUDA device is current";
    default: return "unknown status";
  }
}

int trellis_check_geom(const trellis_geom_t* g) { return geom_ok(g); }

int trellis_expand_bf16(const uint32_t* codes, const uint16_t* scales, uint16_t* out, const trellis_geom_t* g,
                        trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (!codes || !scales || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(out)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_expand_bf16(codes, scales, out, g->k, g->L, g->rows, g->cols, g->interleave,
                                                 static_cast<cudaStream_t>(stream)));
}

int trellis_matvec_axis1(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                         const trellis_geom_t* g, trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->axis != 1) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!codes || !scales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(out)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_matvec_axis1(codes, scales, x, out, M, g->k, g->L, g->rows, g->cols,
                                                  static_cast<cudaStream_t>(stream)));
}

int trellis_matvec_axis1_host(const uint32_t* codes, const uint16_t* scales, const uint16_t* x_host,
                              uint16_t* out_host, int M, const trellis_geom_t* g, uint16_t* x_dev, uint16_t* out_dev,
                              trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->axis != 1) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!codes || !scales || !x_host || !out_host || !x_dev || !out_dev) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x_dev) || !aligned16(out_dev)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)M * (size_t)g->cols * sizeof(uint16_t), ob = (size_t)M * (size_t)g->rows * sizeof(uint16_t);
  // Pinned, 16-byte aligned host buffers are reached through their device mapping: x by a fetch kernel, the
  // output by the matvec's own stores.  Anything else goes through the copy engines.
  const void* xv = aligned16(x_host) ? trellis::mapped_host_view(x_host) : nullptr;
  void* ov = aligned16(out_host) ? const_cast<void*>(trellis::mapped_host_view(out_host)) : nullptr;
  if (xv && !aligned16(xv)) xv = nullptr;
  if (ov && !aligned16(ov)) ov = nullptr;
  const cudaError_t ex = xv ? trellis::launch_fetch16(x_dev, xv, xb, s)
                            : cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s);
  if (ex != cudaSuccess) return TRELLIS_ECUDA;
  uint16_t* o = ov ? static_cast<uint16_t*>(ov) : out_dev;
  if (trellis::launch_matvec_axis1(codes, scales, x_dev, o, M, g->k, g->L, g->rows, g->cols, s) != cudaSuccess)
    return TRELLIS_ECUDA;
  return ov ? TRELLIS_OK : cuda_status(cudaMemcpyAsync(out_host, out_dev, ob, cudaMemcpyDeviceToHost, s));
}

int trellis_matvec_axis1_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                               int M, const trellis_geom_t* g, trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->axis != 1) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!codes || !scales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(out)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_matvec_axis1_bf16w(codes, scales, x, out, M, g->k, g->L, g->rows, g->cols,
                                                        static_cast<cudaStream_t>(stream)));
}

int trellis_matvec_axis0_bf16w(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out,
                               int M, const trellis_geom_t* g, void* workspace, size_t workspace_bytes,
                               trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->axis != 0) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!codes || !scales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(out)) return TRELLIS_EALIGN;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < trellis::axis0_workspace_bytes(M, g->rows, g->cols))
    return TRELLIS_EWORKSPACE;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_matvec_axis0_bf16w(codes, scales, x, out, M, g->k, g->L, g->rows, g->cols,
                                                        g->interleave, workspace, static_cast<cudaStream_t>(stream)));
}

size_t trellis_workspace_bytes(int M, const trellis_geom_t* g) {
  if (geom_ok(g) != TRELLIS_OK || M < 1 || M > 4) return 0;
  return trellis::axis0_workspace_bytes(M, g->rows, g->cols);
}

int trellis_matvec_axis0(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                         const trellis_geom_t* g, void* workspace, size_t workspace_bytes,
                         trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->axis != 0) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!codes || !scales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(out)) return TRELLIS_EALIGN;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < trellis::axis0_workspace_bytes(M, g->rows, g->cols))
    return TRELLIS_EWORKSPACE;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_matvec_axis0(codes, scales, x, out, M, g->k, g->L, g->rows, g->cols,
                                                  g->interleave, workspace, static_cast<cudaStream_t>(stream)));
}

int trellis_gateup_swiglu(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                          const uint16_t* uscales, const uint16_t* x, uint16_t* out, int M, const trellis_geom_t* g,
                          trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->axis != 1) return TRELLIS_EAXIS;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!gcodes || !gscales || !ucodes || !uscales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(gcodes) || !aligned16(gscales) || !aligned16(ucodes) || !aligned16(uscales) || !aligned16(x) ||
      !aligned16(out))
    return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_gateup_swiglu(gcodes, gscales, ucodes, uscales, x, out, M, g->k, g->L,
                                                   g->rows, g->cols, static_cast<cudaStream_t>(stream)));
}

int trellis_mlp_decode(const uint32_t* gcodes, const uint16_t* gscales, const uint32_t* ucodes,
                       const uint16_t* uscales, const uint32_t* dcodes, const uint16_t* dscales, const uint16_t* x,
                       uint16_t* hidden, uint16_t* out, int M, const trellis_geom_t* g_up,
                       const trellis_geom_t* g_down, void* workspace, size_t workspace_bytes,
                       trellis_stream_t stream) {
  int st = geom_ok(g_up);
  if (st) return st;
  if ((st = geom_ok(g_down))) return st;
  if (g_up->axis != 1 || g_down->axis != 0) return TRELLIS_EAXIS;
  if (g_up->rows != g_down->rows || g_up->cols != g_down->cols) return TRELLIS_EGEOM;
  if (M < 1 || M > 4) return TRELLIS_EM;
  if (!gcodes || !gscales || !ucodes || !uscales || !dcodes || !dscales || !x || !hidden || !out)
    return TRELLIS_ENULL;
  if (!aligned16(gcodes) || !aligned16(gscales) || !aligned16(ucodes) || !aligned16(uscales) ||
      !aligned16(dcodes) || !aligned16(dscales) || !aligned16(x) || !aligned16(hidden) || !aligned16(out))
    return TRELLIS_EALIGN;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < trellis::axis0_workspace_bytes(M, g_down->rows, g_down->cols))
    return TRELLIS_EWORKSPACE;
  if ((st = device_ok())) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = trellis::launch_gateup_swiglu(gcodes, gscales, ucodes, uscales, x, hidden, M, g_up->k, g_up->L,
                                                g_up->rows, g_up->cols, s);
  if (e != cudaSuccess) return TRELLIS_ECUDA;
  e = trellis::launch_matvec_axis0(dcodes, dscales, hidden, out, M, g_down->k, g_down->L, g_down->rows,
                                   g_down->cols, g_down->interleave, workspace, s);
  return cuda_status(e);
}

int trellis_gemm_prefill(const uint32_t* codes, const uint16_t* scales, const uint16_t* x, uint16_t* out, int M,
                         const trellis_geom_t* g, trellis_stream_t stream) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->interleave) return TRELLIS_EGEOM;
  if (g->axis == 0 && g->rows % 8 != 0) return TRELLIS_EGEOM;  // x rows of axis 0 must be 16-byte multiples
  if (M < 1 || M > (1 << 24)) return TRELLIS_EM;
  if (!codes || !scales || !x || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(out)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(trellis::launch_gemm_prefill(codes, scales, x, out, M, g->k, g->L, g->axis, g->rows, g->cols,
                                                  static_cast<cudaStream_t>(stream)));
}

int trellis_prefill_plan(int M, const trellis_geom_t* g, int sms, int* tokens_per_tile, int* launches) {
  int st = geom_ok(g);
  if (st) return st;
  if (g->interleave) return TRELLIS_EGEOM;
  if (g->axis == 0 && g->rows % 8 != 0) return TRELLIS_EGEOM;
  if (M < 1 || M > (1 << 24)) return TRELLIS_EM;
  if (!tokens_per_tile || !launches) return TRELLIS_ENULL;
  if (sms < 1) {  // the current device's SM count
    if ((st = device_ok())) return st;
    sms = trellis::device_sm_count();
  }
  trellis::PrefillLaunch plan[2];
  const int n = trellis::prefill_plan(M, g->axis, g->axis == 1 ? g->rows : g->cols, g->axis == 1 ? g->cols : g->rows,
                                      sms, tokens_per_tile, plan);
  for (int i = 0; i < n; ++i) {
    launches[3 * i] = plan[i].t0;
    launches[3 * i + 1] = plan[i].count;
    launches[3 * i + 2] = plan[i].S;
  }
  return n;
}

int trellis_load_floor(const uint32_t* codes, uint32_t* out, const trellis_geom_t* g, trellis_stream_t stream) {
  int st = trellis_check_geom(g);
  if (st) return st;
  if (g->axis != 1) return TRELLIS_EAXIS;
  if (g->interleave) return TRELLIS_EGEOM;
  if (!codes || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(out)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(
      trellis::launch_load_floor(codes, out, g->k, g->rows, g->cols, static_cast<cudaStream_t>(stream)));
}

int trellis_load_floor_rows(const uint32_t* codes, uint32_t* out, const trellis_geom_t* g, trellis_stream_t stream) {
  int st = trellis_check_geom(g);
  if (st) return st;
  if (g->axis != 1) return TRELLIS_EAXIS;
  if (g->interleave) return TRELLIS_EGEOM;
  if (!codes || !out) return TRELLIS_ENULL;
  if (!aligned16(codes) || !aligned16(out)) return TRELLIS_EALIGN;
  if ((st = device_ok())) return st;
  return cuda_status(
      trellis::launch_load_floor_rows(codes, out, g->k, g->rows, g->cols, static_cast<cudaStream_t>(stream)));
}

int trellis_set_wait_limit(uint64_t nanoseconds) {
  trellis::set_wait_limit_ns(nanoseconds);
  return TRELLIS_OK;
}

int trellis_device_error(int reset) {
  int st = device_ok();
  if (st) return st;
  const int v = trellis::read_device_error(reset);
  return v < 0 ? TRELLIS_ECUDA : v;
}

}  // extern "C"
