// gsi_api.cu -- the C ABI declared in include/gsi.h: argument checks, handle
// and workspace lifetime, and dispatch to the decode (T = 1) and batched
// (T > 1) paths.  Page: "Technical summary: Gated Subspace Inference for
// transformer acceleration", sections 2.1-2.2.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "gsi_device.cuh"
#include "gsi_internal.h"
#include "gsi_tc_gemm.h"

namespace {

constexpr int64_t kDefaultMaxT = 512;

bool valid_k(int64_t k) {
  return k == 16 || k == 32 || k == 64 || k == 128 || k == 256 || k == 512;
}

gsi_status_t check_shape(int64_t d_out, int64_t d, int64_t k) {
  if (d_out <= 0 || d <= 0 || k <= 0) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (d % 8 != 0 || d_out % 8 != 0 || !valid_k(k) || k > d) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (d_out > (int64_t(1) << 30) || d > (int64_t(1) << 24)) return GSI_ERR_UNSUPPORTED_SHAPE;
  return GSI_OK;
}

gsi_status_t grow_batched(gsi_handle* h, int64_t max_T) {
  if (max_T <= h->max_T) return GSI_OK;
  const size_t bytes = gsi::batched_workspace_bytes(max_T, h->d, h->k);
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) return GSI_ERR_NOMEM;
  if (cudaMemset(p, 0, bytes) != cudaSuccess) {
    cudaFree(p);
    return GSI_ERR_CUDA;
  }
  if (h->bws) {
    cudaDeviceSynchronize();
    cudaFree(h->bws);
  }
  h->bws = p;
  h->bws_bytes = bytes;
  gsi::batched_bind_workspace(h, p, max_T);
  gsi_status_t st = gsi::batched_prepare(h);
  if (st != GSI_OK) return st;
  return gsi::tc_gemm_prepare(h);
}

gsi_status_t grow_staging(gsi_handle* h, int64_t T) {
  if (T <= h->st_T) return GSI_OK;
  const size_t bytes = size_t(T) * (h->d * 2 + h->d_out * 4 + 4 + 1) + 1024;
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) return GSI_ERR_NOMEM;
  if (h->st_dev) {
    cudaDeviceSynchronize();
    cudaFree(h->st_dev);
  }
  h->st_dev = p;
  h->st_bytes = bytes;
  h->st_T = T;
  return GSI_OK;
}

}  // namespace

extern "C" {

const char* gsi_status_string(gsi_status_t s) {
  switch (s) {
    case GSI_OK: return "GSI_OK";
    case GSI_ERR_INVALID_ARG: return "GSI_ERR_INVALID_ARG: null or misaligned pointer, NaN eps, or T < 0";
    case GSI_ERR_UNSUPPORTED_SHAPE:
      return "GSI_ERR_UNSUPPORTED_SHAPE: need d % 8 == 0, d_out % 8 == 0, k in {16,32,64,128,256,512}, k <= d";
    case GSI_ERR_NOMEM: return "GSI_ERR_NOMEM: allocation failed";
    case GSI_ERR_CUDA: return "GSI_ERR_CUDA: a CUDA call or kernel launch failed";
    case GSI_ERR_WORKSPACE: return "GSI_ERR_WORKSPACE: T exceeds the reserved workspace (call gsi_reserve)";
    case GSI_ERR_TIMEOUT: return "GSI_ERR_TIMEOUT: a bounded device-side wait ran out";
    case GSI_ERR_LAUNCH:
      return "GSI_ERR_LAUNCH: a kernel found its launch configuration inconsistent and did nothing";
    case GSI_ERR_RANK:
      return "GSI_ERR_RANK: calibration lost a column of its block (zero or non-finite) or its factorisation broke down";
  }
  return "unknown gsi_status_t";
}

gsi_status_t gsi_create(const void* W, const void* V_k, const void* M, int64_t d_out, int64_t d,
                        int64_t k, float eps, gsi_handle_t* out) {
  if (!out) return GSI_ERR_INVALID_ARG;
  *out = nullptr;
  if (!W || !V_k || !M || std::isnan(eps)) return GSI_ERR_INVALID_ARG;
  if (!gsi::aligned16(W) || !gsi::aligned16(V_k) || !gsi::aligned16(M)) return GSI_ERR_INVALID_ARG;
  gsi_status_t st = check_shape(d_out, d, k);
  if (st != GSI_OK) return st;

  gsi_handle* h = new (std::nothrow) gsi_handle();
  if (!h) return GSI_ERR_NOMEM;
  h->W = static_cast<const __nv_bfloat16*>(W);
  h->V = static_cast<const __nv_bfloat16*>(V_k);
  h->M = static_cast<const __nv_bfloat16*>(M);
  h->d_out = d_out;
  h->d = d;
  h->k = k;
  h->eps = eps;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return GSI_ERR_CUDA;
  }
  // fixed workspace: Gram matrix, decode accumulators, the packed correction
  // tiles and accumulators of the one-barrier kernel, barrier words, status
  h->dec_acc_stride = int(k + 4);
  const bool want3 = k >= 64 && k <= 256;
  const size_t gram_b = size_t(k) * k * 4;
  const size_t acc_b = size_t(2) * h->dec_acc_stride * 4;
  const size_t F_b = want3 ? gsi::corr_tiles_elems(int(k)) * 2 : 0;
  const size_t acc3_b = want3 ? gsi::decode_cr_acc_floats(k) * 4 : 0;
  auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t ws = r256(gram_b) + r256(acc_b) + r256(F_b) + r256(acc3_b) + 256;
  if (cudaMalloc(&h->ws, ws) != cudaSuccess) {
    delete h;
    return GSI_ERR_NOMEM;
  }
  h->ws_bytes = ws;
  char* p = static_cast<char*>(h->ws);
  h->gram = reinterpret_cast<float*>(p);
  p += r256(gram_b);
  h->dec_acc = reinterpret_cast<float*>(p);
  p += r256(acc_b);
  if (want3) {
    h->cr_F = reinterpret_cast<__nv_bfloat16*>(p);
    p += r256(F_b);
    h->cr_acc = reinterpret_cast<float*>(p);
    p += r256(acc3_b);
  }
  h->dec_bar = reinterpret_cast<uint32_t*>(p);
  h->status = reinterpret_cast<uint32_t*>(p + 64);
  h->cr_bar = reinterpret_cast<uint32_t*>(p + 128);
  st = GSI_OK;
  if (cudaMemset(h->ws, 0, ws) != cudaSuccess) st = GSI_ERR_CUDA;
  if (st == GSI_OK) st = gsi::decode_configure(h);
  if (st == GSI_OK) st = gsi::gram_launch(h->V, d, k, h->gram, h->cr_F, nullptr);
  // the one-exchange kernel serves T = 1 whenever its shape fits; it needs the
  // largest column norm of V_k and a bound of ||E||_2, both from the Gram step
  if (st == GSI_OK && want3) {
    std::vector<float> gram(size_t(k) * k);
    std::vector<uint16_t> tiles(gsi::corr_tiles_elems(int(k)));
    if (cudaMemcpy(gram.data(), h->gram, gram.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(tiles.data(), h->cr_F, tiles.size() * 2, cudaMemcpyDeviceToHost) != cudaSuccess) {
      st = GSI_ERR_CUDA;
    } else {
      double vmax2 = 0.0;
      for (int64_t j = 0; j < k; ++j) vmax2 = std::max(vmax2, double(gram[size_t(j) * k + j]));
      h->cr_vmax = float(std::sqrt(vmax2) * (1.0 + 1e-6));
      const double nb = gsi::corr_norm_bound(tiles.data(), int(k));
      float f = float(nb);
      if (double(f) < nb) f = std::nextafter(f, INFINITY);
      h->cr_normE = f;
      h->cr_ok = std::isfinite(f) && gsi::decode_cr_configure(h) == GSI_OK;
    }
  }
  if (st == GSI_OK) st = grow_batched(h, kDefaultMaxT);
  if (st == GSI_OK) st = grow_staging(h, kDefaultMaxT);
  if (st == GSI_OK && cudaDeviceSynchronize() != cudaSuccess) st = GSI_ERR_CUDA;
  if (st != GSI_OK) {
    gsi_destroy(h);
    return st;
  }
  *out = h;
  return GSI_OK;
}

gsi_status_t gsi_forward(gsi_handle_t h, const void* x, int64_t T, float* y, uint8_t* gate,
                         float* rho, cudaStream_t stream) {
  if (!h || T < 0) return GSI_ERR_INVALID_ARG;
  if (T == 0) return GSI_OK;
  if (!x || !y || !gsi::aligned16(x) || !gsi::aligned16(y)) return GSI_ERR_INVALID_ARG;
  if (rho && (reinterpret_cast<uintptr_t>(rho) & 3u)) return GSI_ERR_INVALID_ARG;  // fp32 stores
  if (T == 1)
    return h->cr_ok ? gsi::decode_cr_launch(h, x, y, gate, rho, stream)
                    : gsi::decode_launch(h, x, y, gate, rho, stream);
  if (T > h->max_T) return GSI_ERR_WORKSPACE;
  return gsi::batched_launch(h, x, T, y, gate, rho, stream);
}

namespace {

// One token's x from page-locked host memory into the handle's device
// staging, by one CTA (16-byte loads, all in flight at once): the one-token
// kernel reads x from every CTA, which is cheap from device memory (L2) and
// dear over the host link.  Launched with programmatic dependent launch, so
// the next kernel's CTAs stage their weights while it runs.
__device__ __forceinline__ void stage_copy(const uint4* src, uint4* dst,
                                           int n16) {
  constexpr int kPer = 16;
  uint4 v[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = int(threadIdx.x) + j * 256;
    if (i < n16) v[j] = src[i];
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = int(threadIdx.x) + j * 256;
    if (i < n16) dst[i] = v[j];
  }
  for (int i = int(threadIdx.x) + kPer * 256; i < n16; i += 256) dst[i] = src[i];
}

__global__ void __launch_bounds__(256) stage_x_kernel(const uint4* src,
                                                      uint4* dst, int n16) {
  gsi::pdl_launch_dependents();
  gsi::pdl_wait();  // x may have been written by the previous kernel
  stage_copy(src, dst, n16);
}

// The same for the members of a group, one CTA per member.
struct StageJobs {
  const uint4* src[gsi::kMaxGroup];
  uint4* dst[gsi::kMaxGroup];
  int n16[gsi::kMaxGroup];
};
__global__ void __launch_bounds__(256) stage_x_group_kernel(const __grid_constant__ StageJobs j) {
  gsi::pdl_launch_dependents();
  gsi::pdl_wait();
  const int m = blockIdx.x;
  stage_copy(j.src[m], j.dst[m], j.n16[m]);
}

// True if the device can address p directly at the same address: page-locked
// host memory (cudaHostAlloc, cudaMallocHost, cudaHostRegister) under unified
// addressing, or managed memory.
bool device_addressable(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error of an unknown pointer
    return false;
  }
  return (at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged ||
          at.type == cudaMemoryTypeDevice) &&
         at.devicePointer == p;
}

}  // namespace

gsi_status_t gsi_forward_host(gsi_handle_t h, const void* x_host, int64_t T, float* y_host,
                              uint8_t* gate_host, float* rho_host, cudaStream_t stream) {
  if (!h || T < 0) return GSI_ERR_INVALID_ARG;
  if (T == 0) return GSI_OK;
  if (!x_host || !y_host) return GSI_ERR_INVALID_ARG;
  // One token in page-locked memory: a one-CTA kernel brings x into the
  // device staging, and the map writes y, gate and rho in place over the host
  // link (no copy nodes: consecutive calls chain like device calls)
  if (T == 1 && gsi::aligned16(x_host) && device_addressable(x_host) &&
      device_addressable(y_host) && (!gate_host || device_addressable(gate_host)) &&
      (!rho_host || device_addressable(rho_host))) {
    uint4* xd = static_cast<uint4*>(h->st_dev);
    if (gsi::launch_pdl(stage_x_kernel, dim3(1), dim3(256), 0, stream,
                        static_cast<const uint4*>(x_host), xd, int(h->d / 8)) != cudaSuccess)
      return GSI_ERR_CUDA;
    return gsi_forward(h, xd, 1, y_host, gate_host, rho_host, stream);
  }
  if (T > h->st_T || (T > 1 && T > h->max_T)) return GSI_ERR_WORKSPACE;
  char* p = static_cast<char*>(h->st_dev);
  void* xd = p;
  // Many tokens in page-locked memory: x is copied in once, and the kernels
  // write y, gate and rho in place over the host link while the GEMMs run
  // (no copy of y back)
  if (gsi::aligned16(y_host) && device_addressable(y_host) &&
      (!gate_host || device_addressable(gate_host)) && (!rho_host || device_addressable(rho_host)) &&
      (!rho_host || (reinterpret_cast<uintptr_t>(rho_host) & 3u) == 0)) {
    if (cudaMemcpyAsync(xd, x_host, size_t(T) * h->d * 2, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
      return GSI_ERR_CUDA;
    return gsi_forward(h, xd, T, y_host, gate_host, rho_host, stream);
  }
  // staging: x, then y, rho and gate back to back for this T (one copy
  // returns all three when the caller's buffers are laid out the same way)
  p += (size_t(h->st_T) * h->d * 2 + 255) / 256 * 256;
  const size_t y_bytes = size_t(T) * h->d_out * 4;
  float* yd = reinterpret_cast<float*>(p);
  float* rd = reinterpret_cast<float*>(p + y_bytes);
  uint8_t* gd = reinterpret_cast<uint8_t*>(p + y_bytes + size_t(T) * 4);
  if (cudaMemcpyAsync(xd, x_host, size_t(T) * h->d * 2, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return GSI_ERR_CUDA;
  gsi_status_t st = gsi_forward(h, xd, T, yd, gd, rd, stream);
  if (st != GSI_OK) return st;
  const bool packed = rho_host == reinterpret_cast<float*>(reinterpret_cast<char*>(y_host) + y_bytes) &&
                      gate_host == reinterpret_cast<uint8_t*>(rho_host + T);
  if (packed) {
    if (cudaMemcpyAsync(y_host, yd, y_bytes + size_t(T) * 5, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return GSI_ERR_CUDA;
    return GSI_OK;
  }
  if (cudaMemcpyAsync(y_host, yd, y_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return GSI_ERR_CUDA;
  if (gate_host && cudaMemcpyAsync(gate_host, gd, size_t(T), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return GSI_ERR_CUDA;
  if (rho_host && cudaMemcpyAsync(rho_host, rd, size_t(T) * 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return GSI_ERR_CUDA;
  return GSI_OK;
}

gsi_status_t gsi_precompute_M(const void* W, const void* V_k, void* M, int64_t d_out, int64_t d,
                              int64_t k, cudaStream_t stream) {
  if (!W || !V_k || !M) return GSI_ERR_INVALID_ARG;
  if (!gsi::aligned16(W) || !gsi::aligned16(V_k) || !gsi::aligned16(M)) return GSI_ERR_INVALID_ARG;
  gsi_status_t st = check_shape(d_out, d, k);
  if (st != GSI_OK) return st;
  return gsi::precompute_M_launch(static_cast<const __nv_bfloat16*>(W),
                                  static_cast<const __nv_bfloat16*>(V_k),
                                  static_cast<__nv_bfloat16*>(M), d_out, d, k, stream);
}

gsi_status_t gsi_reserve(gsi_handle_t h, int64_t max_T) {
  if (!h || max_T < 0 || max_T > (int64_t(1) << 24)) return GSI_ERR_INVALID_ARG;
  gsi_status_t st = grow_batched(h, max_T);
  if (st != GSI_OK) return st;
  st = grow_staging(h, std::max<int64_t>(max_T, 1));
  if (st != GSI_OK) return st;
  return cudaDeviceSynchronize() == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

gsi_status_t gsi_device_status(gsi_handle_t h, cudaStream_t stream) {
  if (!h) return GSI_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GSI_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, h->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GSI_ERR_CUDA;
  if (word) {
    const uint32_t zero = 0;
    if (cudaMemcpy(h->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return GSI_ERR_CUDA;
  }
  if (word & gsi::kStatusBadLaunch) return GSI_ERR_LAUNCH;
  return (word & gsi::kStatusTimeout) ? GSI_ERR_TIMEOUT : GSI_OK;
}

}  // extern "C"

namespace {

template <typename T>
void erase_value(std::vector<T*>& v, T* x) {
  v.erase(std::remove(v.begin(), v.end(), x), v.end());
}

// Remove h's prefetch target (a handle or a group), both directions.
void unlink_target(gsi_handle* h) {
  if (h->pf_next) erase_value(h->pf_next->pf_from, h);
  if (h->pf_group) erase_value(h->pf_group->pf_from, h);
  h->pf_next = nullptr;
  h->pf_group = nullptr;
}

}  // namespace

extern "C" {

gsi_status_t gsi_set_prefetch(gsi_handle_t h, gsi_handle_t next) {
  if (!h) return GSI_ERR_INVALID_ARG;
  if (next && next->device != h->device) return GSI_ERR_INVALID_ARG;
  unlink_target(h);
  h->pf_next = next;
  if (next) next->pf_from.push_back(h);
  return GSI_OK;
}

gsi_status_t gsi_set_prefetch_group(gsi_handle_t h, gsi_group_t next) {
  if (!h) return GSI_ERR_INVALID_ARG;
  if (next && next->device != h->device) return GSI_ERR_INVALID_ARG;
  unlink_target(h);
  h->pf_group = next;
  if (next) next->pf_from.push_back(h);
  return GSI_OK;
}

gsi_status_t gsi_group_create(int n, const gsi_handle_t* handles, gsi_group_t* out) {
  if (!out) return GSI_ERR_INVALID_ARG;
  *out = nullptr;
  if (!handles || n < 1 || n > gsi::kMaxGroup) return GSI_ERR_INVALID_ARG;
  for (int m = 0; m < n; ++m) {
    if (!handles[m]) return GSI_ERR_INVALID_ARG;
    for (int j = 0; j < m; ++j)
      if (handles[j] == handles[m]) return GSI_ERR_INVALID_ARG;  // one workspace, one call
  }
  for (int m = 0; m < n; ++m)
    if (!handles[m]->cr_ok || handles[m]->k != handles[0]->k ||
        handles[m]->device != handles[0]->device)
      return GSI_ERR_UNSUPPORTED_SHAPE;
  gsi_group* g = new (std::nothrow) gsi_group();
  if (!g) return GSI_ERR_NOMEM;
  g->n = n;
  g->k = int(handles[0]->k);
  g->device = handles[0]->device;
  for (int m = 0; m < n; ++m) g->h[m] = handles[m];
  const gsi_status_t st = gsi::group_configure(g);
  if (st != GSI_OK) {
    delete g;
    return st;
  }
  *out = g;
  return GSI_OK;
}

gsi_status_t gsi_group_forward(gsi_group_t g, const void* const* x, float* const* y,
                               uint8_t* const* gate, float* const* rho, cudaStream_t stream) {
  if (!g || !x || !y) return GSI_ERR_INVALID_ARG;
  for (int m = 0; m < g->n; ++m)
    if (!x[m] || !y[m] || !gsi::aligned16(x[m]) || !gsi::aligned16(y[m]) ||
        (rho && rho[m] && (reinterpret_cast<uintptr_t>(rho[m]) & 3u)))
      return GSI_ERR_INVALID_ARG;
  return gsi::group_launch(g, x, y, gate, rho, stream);
}

gsi_status_t gsi_group_forward_host(gsi_group_t g, const void* const* x_host,
                                    float* const* y_host, uint8_t* const* gate_host,
                                    float* const* rho_host, cudaStream_t stream) {
  if (!g || !x_host || !y_host) return GSI_ERR_INVALID_ARG;
  bool direct = true;
  for (int m = 0; m < g->n; ++m) {
    const uint8_t* gm = gate_host ? gate_host[m] : nullptr;
    const float* rm = rho_host ? rho_host[m] : nullptr;
    if (!x_host[m] || !y_host[m] || !gsi::aligned16(x_host[m]) ||
        (rm && (reinterpret_cast<uintptr_t>(rm) & 3u)))
      return GSI_ERR_INVALID_ARG;
    direct = direct && gsi::aligned16(y_host[m]) && device_addressable(x_host[m]) &&
             device_addressable(y_host[m]) && (!gm || device_addressable(gm)) &&
             (!rm || device_addressable(rm));
  }
  const void* xd[gsi::kMaxGroup] = {};
  for (int m = 0; m < g->n; ++m) xd[m] = g->h[m]->st_dev;
  if (direct) {
    StageJobs j;
    std::memset(&j, 0, sizeof j);
    for (int m = 0; m < g->n; ++m) {
      j.src[m] = static_cast<const uint4*>(x_host[m]);
      j.dst[m] = static_cast<uint4*>(g->h[m]->st_dev);
      j.n16[m] = int(g->h[m]->d / 8);
    }
    if (gsi::launch_pdl(stage_x_group_kernel, dim3(unsigned(g->n)), dim3(256), 0, stream, j) !=
        cudaSuccess)
      return GSI_ERR_CUDA;
    return gsi::group_launch(g, xd, y_host, gate_host, rho_host, stream);
  }
  // through each member's staging: x, then y, rho and gate for one token
  float* yd[gsi::kMaxGroup] = {};
  float* rd[gsi::kMaxGroup] = {};
  uint8_t* gd[gsi::kMaxGroup] = {};
  for (int m = 0; m < g->n; ++m) {
    gsi_handle* h = g->h[m];
    char* p = static_cast<char*>(h->st_dev) + (size_t(h->st_T) * h->d * 2 + 255) / 256 * 256;
    yd[m] = reinterpret_cast<float*>(p);
    rd[m] = reinterpret_cast<float*>(p + size_t(h->d_out) * 4);
    gd[m] = reinterpret_cast<uint8_t*>(p + size_t(h->d_out) * 4 + 4);
    if (cudaMemcpyAsync(h->st_dev, x_host[m], size_t(h->d) * 2, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
      return GSI_ERR_CUDA;
  }
  const gsi_status_t st = gsi::group_launch(g, xd, yd, gd, rd, stream);
  if (st != GSI_OK) return st;
  for (int m = 0; m < g->n; ++m) {
    gsi_handle* h = g->h[m];
    if (cudaMemcpyAsync(y_host[m], yd[m], size_t(h->d_out) * 4, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
      return GSI_ERR_CUDA;
    if (gate_host && gate_host[m] &&
        cudaMemcpyAsync(gate_host[m], gd[m], 1, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return GSI_ERR_CUDA;
    if (rho_host && rho_host[m] &&
        cudaMemcpyAsync(rho_host[m], rd[m], 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return GSI_ERR_CUDA;
  }
  return GSI_OK;
}

gsi_status_t gsi_group_set_prefetch(gsi_group_t g, gsi_handle_t next) {
  if (!g) return GSI_ERR_INVALID_ARG;
  if (next && next->device != g->device) return GSI_ERR_INVALID_ARG;
  if (g->pf_next) erase_value(g->pf_next->pf_from_groups, g);
  g->pf_next = next;
  if (next) next->pf_from_groups.push_back(g);
  return GSI_OK;
}

void gsi_group_destroy(gsi_group_t g) {
  if (!g) return;
  cudaDeviceSynchronize();
  for (gsi_handle* p : g->pf_from)
    if (p->pf_group == g) p->pf_group = nullptr;
  if (g->pf_next) erase_value(g->pf_next->pf_from_groups, g);
  delete g;
}

void gsi_destroy(gsi_handle_t h) {
  if (!h) return;
  cudaDeviceSynchronize();
  // unlink prefetch links in both directions before the memory goes away
  for (gsi_handle* p : h->pf_from)
    if (p->pf_next == h) p->pf_next = nullptr;
  for (gsi_group* g : h->pf_from_groups)
    if (g->pf_next == h) g->pf_next = nullptr;
  if (h->pf_next && h->pf_next != h) erase_value(h->pf_next->pf_from, h);
  if (h->pf_group) erase_value(h->pf_group->pf_from, h);
  if (h->ws) cudaFree(h->ws);
  if (h->bws) cudaFree(h->bws);
  if (h->st_dev) cudaFree(h->st_dev);
  delete h;
}

int gsi_forward_launch_count(gsi_handle_t h, int64_t T) {
  // (gsi_forward; gsi_forward_host on page-locked memory adds one launch)
  if (!h || T <= 0) return 0;
  if (T == 1) return 1;
  return gsi::batched_launch_count(h, T);
}

}  // extern "C"

namespace gsi {

// Upper bound of ||A||_2 for the symmetric matrix A whose quadratic form the
// correction tiles compute: g^T A g = sum over tiles I <= J of g_I^T F_IJ g_J,
// i.e. A_II = sym(F_II), A_IJ = F_IJ / 2, A_JI = F_IJ^T / 2.  For symmetric A,
// ||A^(2^p)||_F^(1 / 2^p) = (sum_i lambda_i^(2^(p+1)))^(1 / 2^(p+1)) is at
// least max |lambda_i| = ||A||_2 and at most k^(1 / 2^(p+1)) times it; four
// squarings (p = 4) give a bound within a factor 256^(1/32) = 1.19 at k = 256.
// fp64 throughout, with each power renormalised to unit Frobenius norm.
double corr_norm_bound(const uint16_t* tiles, int k) {
  const int t16 = k / 16;
  std::vector<double> A(size_t(k) * k, 0.0), B(size_t(k) * k, 0.0);
  auto bf = [](uint16_t b) {
    uint32_t u = uint32_t(b) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return double(f);
  };
  for (int I = 0; I < t16; ++I)
    for (int J = I; J < t16; ++J) {
      const uint16_t* t = tiles + size_t(corr_tile_index(I, J, t16)) * 256;
      for (int r = 0; r < 16; ++r)
        for (int c = 0; c < 16; ++c) {
          const double v = 0.5 * bf(t[corr_tile_pos(r, c)]);
          A[size_t(16 * I + r) * k + 16 * J + c] += v;
          A[size_t(16 * J + c) * k + 16 * I + r] += v;
        }
    }
  auto fro = [k](const std::vector<double>& M) {
    double s = 0.0;
    for (size_t i = 0; i < size_t(k) * k; ++i) s += M[i] * M[i];
    return std::sqrt(s);
  };
  double f = fro(A);
  if (!(f > 0.0)) return 0.0;
  if (!std::isfinite(f)) return f;
  for (double& v : A) v /= f;
  double log_norm = std::log(f);  // log ||A^(2^j)||_F
  for (int p = 1; p <= 4; ++p) {
    std::fill(B.begin(), B.end(), 0.0);
    for (int i = 0; i < k; ++i)
      for (int l = 0; l < k; ++l) {
        const double a = A[size_t(i) * k + l];
        if (a == 0.0) continue;
        const double* row = &A[size_t(l) * k];
        double* out = &B[size_t(i) * k];
        for (int j = 0; j < k; ++j) out[j] += a * row[j];
      }
    const double n = fro(B);
    if (!(n > 0.0)) return 0.0;
    for (double& v : B) v /= n;
    log_norm = 2.0 * log_norm + std::log(n);
    A.swap(B);
  }
  return std::exp(log_norm / 16.0) * (1.0 + 1e-9);
}

}  // namespace gsi
