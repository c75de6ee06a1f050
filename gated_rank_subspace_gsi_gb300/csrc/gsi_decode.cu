// gsi_decode.cu -- the T = 1 (decode) path of the GSI gated linear map as ONE
// persistent kernel per call.
//
// Page: "Technical summary: Gated Subspace Inference for transformer
// acceleration" [GSI].  Per token x (section 2.1 eq. 1-2, section 2.2):
//   g = V_k^T x,  r = x - V_k g,  rho = ||r|| / ||x||,
//   y = M g if rho < eps (fast path, reads M: d_out x k)
//   y = W x otherwise    (slow path, reads W: d_out x d).
//
// Work split.  The grid has G co-resident CTAs (at most one per SM).  CTA c
// owns a contiguous slice of V_k rows (d / G rows) and a contiguous slice of
// output rows (d_out / G rows of M and of W).  Before it waits on the
// previous kernel (programmatic dependent launch), each CTA starts 1-D bulk
// copies of its V_k slice and its M slice into shared memory: these weights
// do not depend on x, so their HBM reads overlap the previous kernel's tail.
//   phase 1  partial g_c = V_c^T x_c and partial ||x_c||^2, reduced into a
//            global accumulator with vector red.add; grid barrier 1
//   phase 2  every CTA reads the full g; partial ||r||^2 = sum over its rows
//            of (x_i - V_i . g)^2 (the explicit residual of eq. 1, computed
//            from the V_k slice still in shared memory); grid barrier 2
//   phase 3  every CTA forms rho and the gate from the same sums (so all
//            CTAs take the same branch) and computes its rows of y: M_c g
//            from shared memory, or W_c x streamed from HBM.
// Accumulators are double-buffered by a launch epoch kept on the device, so
// the kernel needs no memset and can be replayed in a CUDA graph.
#include <algorithm>
#include <cfloat>

#include "gsi_device.cuh"
#include "gsi_internal.h"

namespace gsi {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;

struct DecodeArgs {
  const __nv_bfloat16* W;
  const __nv_bfloat16* V;
  const __nv_bfloat16* M;
  const __nv_bfloat16* x;
  float* y;
  uint8_t* gate;
  float* rho;
  int d_out, d;
  float eps;
  int rows_M, rows_V;
  int stage_M, stage_V;
  float* acc;
  int acc_stride;
  uint32_t* bar;
  uint32_t* status;
};

// Lane geometry for rows of K bf16 values read as 16-byte chunks.
template <int K>
struct RowLanes {
  static constexpr int CPR = K / 8;                 // chunks per row
  static constexpr int LPR = CPR < 32 ? CPR : 32;   // lanes per row
  static constexpr int CPL = CPR / LPR;             // chunks per lane
  static constexpr int RPI = 32 / LPR;              // rows per warp step
};

// Dynamic shared-memory layout (byte offsets), identical on host and device.
struct DecodeSmem {
  size_t sx, sg, sred, sM, sV, total;
};
__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline DecodeSmem decode_smem(int d, int K, int rows_M, int rows_V,
                                                  bool stage_M, bool stage_V) {
  DecodeSmem s;
  s.sx = 0;
  s.sg = align_up(s.sx + size_t(d) * 2, 128);
  s.sred = align_up(s.sg + size_t(K) * 4, 128);
  s.sM = align_up(s.sred + size_t(kDecWarps) * K * 4, 128);
  s.sV = align_up(s.sM + (stage_M ? size_t(rows_M) * K * 2 : 0), 128);
  s.total = align_up(s.sV + (stage_V ? size_t(rows_V) * K * 2 : 0), 128);
  return s;
}

__device__ __forceinline__ float block_sum(float v, float* s_red) {
  v = warp_sum_xor<32>(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kDecWarps; ++w) t += s_red[w];
  return t;  // valid in thread 0
}

template <int K>
__global__ void __launch_bounds__(kDecThreads, 1) gsi_decode_kernel(DecodeArgs a) {
  using L = RowLanes<K>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t s_bar;
  __shared__ int s_ok;
  __shared__ float s_red[kDecWarps];
  __shared__ uint32_t s_epoch;
  __shared__ float s_sums[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, G = gridDim.x;
  const int m0 = cta * a.rows_M;
  const int nM = max(0, min(a.d_out, m0 + a.rows_M) - m0);
  const int v0 = cta * a.rows_V;
  const int nV = max(0, min(a.d, v0 + a.rows_V) - v0);

  const DecodeSmem lay = decode_smem(a.d, K, a.rows_M, a.rows_V, a.stage_M, a.stage_V);
  __nv_bfloat16* sx = reinterpret_cast<__nv_bfloat16*>(smem + lay.sx);
  float* sg = reinterpret_cast<float*>(smem + lay.sg);
  float* sred = reinterpret_cast<float*>(smem + lay.sred);
  __nv_bfloat16* sM = reinterpret_cast<__nv_bfloat16*>(smem + lay.sM);
  __nv_bfloat16* sV = reinterpret_cast<__nv_bfloat16*>(smem + lay.sV);

  // ---- prologue: stage this CTA's weights (independent of x) ------------
  const uint32_t bytes_M = a.stage_M ? uint32_t(nM) * K * 2 : 0u;
  const uint32_t bytes_V = a.stage_V ? uint32_t(nV) * K * 2 : 0u;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&s_bar, bytes_M + bytes_V);
    constexpr uint32_t kChunk = 32768;
    const char* gV = reinterpret_cast<const char*>(a.V + size_t(v0) * K);
    for (uint32_t off = 0; off < bytes_V; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sV) + off, gV + off, min(kChunk, bytes_V - off), &s_bar);
    const char* gM = reinterpret_cast<const char*>(a.M + size_t(m0) * K);
    for (uint32_t off = 0; off < bytes_M; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sM) + off, gM + off, min(kChunk, bytes_M - off), &s_bar);
  }
  pdl_launch_dependents();
  pdl_wait();  // x and this handle's workspace are now safe to touch

  if (tid == 0) s_epoch = ld_cg_u32(a.bar + 1);
  // x (d bf16) into shared memory: phase 1 needs its slice, the slow path all.
  for (int i = tid; i < a.d / 8; i += kDecThreads)
    reinterpret_cast<uint4*>(sx)[i] = reinterpret_cast<const uint4*>(a.x)[i];
  __syncthreads();
  const uint32_t e = s_epoch;
  float* acc = a.acc + size_t(e & 1u) * a.acc_stride;
  if (cta == 0) {  // clear the buffer the next launch accumulates into
    float* nxt = a.acc + size_t((e + 1u) & 1u) * a.acc_stride;
    for (int i = tid; i < a.acc_stride; i += kDecThreads) nxt[i] = 0.f;
  }
  bool ok = mbar_wait_bounded(&s_bar, 0, a.status);
  ok = __syncthreads_and(ok) != 0;
  const int nVw = ok ? nV : 0;
  const int nMw = ok ? nM : 0;

  const __nv_bfloat16* Vs = a.stage_V ? sV : a.V + size_t(v0) * K;
  const __nv_bfloat16* Ms = a.stage_M ? sM : a.M + size_t(m0) * K;
  const int slot = lane / L::LPR, li = lane % L::LPR;

  // ---- phase 1: partial g and ||x||^2 -----------------------------------
  {
    float accg[L::CPL][8];
#pragma unroll
    for (int c = 0; c < L::CPL; ++c)
#pragma unroll
      for (int j = 0; j < 8; ++j) accg[c][j] = 0.f;
    for (int r = warp * L::RPI + slot; r < nVw; r += kDecWarps * L::RPI) {
      const float xi = bf16_to_f32(sx[v0 + r]);
#pragma unroll
      for (int c = 0; c < L::CPL; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(Vs + size_t(r) * K + (li + c * L::LPR) * 8);
        float f[8];
        bf16x8_to_f32(v, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) accg[c][j] = fmaf(f[j], xi, accg[c][j]);
      }
    }
#pragma unroll
    for (int o = L::LPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < L::CPL; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) accg[c][j] += __shfl_xor_sync(0xFFFFFFFFu, accg[c][j], o);
    if (slot == 0) {
#pragma unroll
      for (int c = 0; c < L::CPL; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) sred[warp * K + (li + c * L::LPR) * 8 + j] = accg[c][j];
    }
    float sxp = 0.f;
    for (int i = tid; i < nVw; i += kDecThreads) {
      const float xv = bf16_to_f32(sx[v0 + i]);
      sxp = fmaf(xv, xv, sxp);
    }
    const float sx_tot = block_sum(sxp, s_red);  // contains __syncthreads
    if (nVw > 0) {
      for (int t = tid; t < K / 4; t += kDecThreads) {
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kDecWarps; ++w)
#pragma unroll
          for (int q = 0; q < 4; ++q) s4[q] += sred[w * K + t * 4 + q];
        red_add_v4_f32(acc + t * 4, s4[0], s4[1], s4[2], s4[3]);
      }
      if (tid == 0) red_add_f32(acc + K, sx_tot);
    }
  }
  ok = grid_barrier(a.bar, (2u * e + 1u) * uint32_t(G), a.status, &s_ok) && ok;

  // ---- phase 2: partial ||r||^2 with r = x - V_k g ----------------------
  for (int t = tid; t < K; t += kDecThreads) sg[t] = ld_cg_f32(acc + t);
  __syncthreads();
  float gl[L::CPL][8];
#pragma unroll
  for (int c = 0; c < L::CPL; ++c)
#pragma unroll
    for (int j = 0; j < 8; ++j) gl[c][j] = sg[(li + c * L::LPR) * 8 + j];
  {
    float srp = 0.f;
    const int nR = ok ? nVw : 0;
    for (int r0 = warp * L::RPI; r0 < nR; r0 += kDecWarps * L::RPI) {
      const int r = r0 + slot;
      float dot = 0.f;
      if (r < nR) {
#pragma unroll
        for (int c = 0; c < L::CPL; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(Vs + size_t(r) * K + (li + c * L::LPR) * 8);
          float f[8];
          bf16x8_to_f32(v, f);
#pragma unroll
          for (int j = 0; j < 8; ++j) dot = fmaf(f[j], gl[c][j], dot);
        }
      }
      dot = warp_sum_xor<L::LPR>(dot);
      if (li == 0 && r < nR) {
        const float ri = bf16_to_f32(sx[v0 + r]) - dot;
        srp = fmaf(ri, ri, srp);
      }
    }
    const float sr_tot = block_sum(srp, s_red);
    if (tid == 0 && nR > 0) red_add_f32(acc + K + 1, sr_tot);
  }
  ok = grid_barrier(a.bar, (2u * e + 2u) * uint32_t(G), a.status, &s_ok) && ok;

  // ---- phase 3: gate and the branch it picks ----------------------------
  if (tid == 0) {
    s_sums[0] = ld_cg_f32(acc + K);
    s_sums[1] = ld_cg_f32(acc + K + 1);
  }
  __syncthreads();
  const float sxv = s_sums[0];
  float srv = s_sums[1];
  float rho;
  if (!(fabsf(sxv) <= FLT_MAX)) {
    rho = __int_as_float(0x7FC00000);  // non-finite x: NaN, slow path
  } else if (sxv == 0.f) {
    rho = 0.f;
  } else {
    if (!(srv >= 0.f)) srv = (srv == srv) ? 0.f : srv;
    rho = sqrtf(srv / sxv);
  }
  const bool slow = !(rho < a.eps);
  if (cta == 0 && tid == 0) {
    // a CTA whose bounded wait ran out reports NaN (rho, and its rows of y
    // below), so that a caller without a status word can still see it
    if (a.gate) a.gate[0] = (slow || !ok) ? 1 : 0;
    if (a.rho) a.rho[0] = ok ? rho : __int_as_float(0x7FC00000);
  }

  if (ok) {
    if (!slow) {
      // y rows of this CTA = M_c g
      for (int r0 = warp * L::RPI; r0 < nMw; r0 += kDecWarps * L::RPI) {
        const int r = r0 + slot;
        float dot = 0.f;
        if (r < nMw) {
#pragma unroll
          for (int c = 0; c < L::CPL; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(Ms + size_t(r) * K + (li + c * L::LPR) * 8);
            float f[8];
            bf16x8_to_f32(v, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) dot = fmaf(f[j], gl[c][j], dot);
          }
        }
        dot = warp_sum_xor<L::LPR>(dot);
        if (li == 0 && r < nMw) a.y[m0 + r] = dot;
      }
    } else {
      // y rows of this CTA = W_c x, W streamed from HBM, 4 rows per warp
      const int nch = a.d / 8;
      const uint4* sx4 = reinterpret_cast<const uint4*>(sx);
      const int nMs = nM;  // the slow path does not depend on the M staging
      for (int rb = warp * 4; rb < nMs; rb += kDecWarps * 4) {
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4* wr[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = min(rb + q, nMs - 1);
          wr[q] = reinterpret_cast<const uint4*>(a.W + size_t(m0 + r) * a.d);
        }
        int j = lane;
        for (; j + 32 < nch; j += 64) {
          uint4 w0[4], w1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) { w0[q] = ld_stream_v4(wr[q] + j); w1[q] = ld_stream_v4(wr[q] + j + 32); }
          float xa[8], xb[8];
          bf16x8_to_f32(sx4[j], xa);
          bf16x8_to_f32(sx4[j + 32], xb);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float f[8];
            bf16x8_to_f32(w0[q], f);
#pragma unroll
            for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xa[t], acc4[q]);
            bf16x8_to_f32(w1[q], f);
#pragma unroll
            for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xb[t], acc4[q]);
          }
        }
        for (; j < nch; j += 32) {
          float xa[8];
          bf16x8_to_f32(sx4[j], xa);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float f[8];
            bf16x8_to_f32(ld_stream_v4(wr[q] + j), f);
#pragma unroll
            for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xa[t], acc4[q]);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) acc4[q] = warp_sum_xor<32>(acc4[q]);
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (rb + q < nMs) a.y[m0 + rb + q] = acc4[q];
        }
      }
    }
  } else {
    for (int r = tid; r < nM; r += kDecThreads) a.y[m0 + r] = __int_as_float(0x7FC00000);
  }
  if (cta == 0 && tid == 0) {
    __threadfence();
    a.bar[1] = e + 1u;  // every CTA read the epoch before barrier 1
  }
}

template <int K>
const void* decode_kernel_ptr() {
  return reinterpret_cast<const void*>(&gsi_decode_kernel<K>);
}

const void* decode_kernel_for(int64_t k) {
  switch (k) {
    case 16: return decode_kernel_ptr<16>();
    case 32: return decode_kernel_ptr<32>();
    case 64: return decode_kernel_ptr<64>();
    case 128: return decode_kernel_ptr<128>();
    case 256: return decode_kernel_ptr<256>();
    case 512: return decode_kernel_ptr<512>();
    default: return nullptr;
  }
}

}  // namespace

gsi_status_t decode_configure(gsi_handle* h) {
  const void* fn = decode_kernel_for(h->k);
  if (!fn) return GSI_ERR_UNSUPPORTED_SHAPE;
  int max_optin = 0;
  if (cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess)
    return GSI_ERR_CUDA;
  const int64_t rows_hint = (std::max(h->d_out, h->d) + 7) / 8;
  const int G = int(std::max<int64_t>(1, std::min<int64_t>(h->num_sms, rows_hint)));
  const int rows_M = int((h->d_out + G - 1) / G);
  const int rows_V = int((h->d + G - 1) / G);
  const size_t static_smem = 1024;  // mbarrier, reduction scratch, margins
  bool stage_M = true, stage_V = true;
  DecodeSmem lay = decode_smem(int(h->d), int(h->k), rows_M, rows_V, stage_M, stage_V);
  if (lay.total + static_smem > size_t(max_optin)) {
    stage_M = false;
    lay = decode_smem(int(h->d), int(h->k), rows_M, rows_V, stage_M, stage_V);
  }
  if (lay.total + static_smem > size_t(max_optin)) {
    stage_V = false;
    lay = decode_smem(int(h->d), int(h->k), rows_M, rows_V, stage_M, stage_V);
  }
  if (lay.total + static_smem > size_t(max_optin)) return GSI_ERR_UNSUPPORTED_SHAPE;
  // The limit is a property of the kernel function, shared by every handle
  // with this k: raise it to the device maximum once, never per handle.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return GSI_ERR_CUDA;
  const int fn_limit = max_optin - int(fa.sharedSizeBytes);
  if (int(lay.total) > fn_limit) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (fa.maxDynamicSharedSizeBytes < fn_limit &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, fn_limit) != cudaSuccess)
    return GSI_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kDecThreads, lay.total) != cudaSuccess)
    return GSI_ERR_CUDA;
  // The kernel's CTAs wait on one another: all of them must fit at once.
  if (per_sm < 1 || int64_t(per_sm) * h->num_sms < G) return GSI_ERR_UNSUPPORTED_SHAPE;
  h->dec_grid = G;
  h->dec_rows_M = rows_M;
  h->dec_rows_V = rows_V;
  h->dec_stage_M = stage_M;
  h->dec_stage_V = stage_V;
  h->dec_smem = lay.total;
  return GSI_OK;
}

gsi_status_t decode_launch(gsi_handle* h, const void* x, float* y, uint8_t* gate, float* rho,
                           cudaStream_t s) {
  DecodeArgs a;
  a.W = h->W;
  a.V = h->V;
  a.M = h->M;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.y = y;
  a.gate = gate;
  a.rho = rho;
  a.d_out = int(h->d_out);
  a.d = int(h->d);
  a.eps = h->eps;
  a.rows_M = h->dec_rows_M;
  a.rows_V = h->dec_rows_V;
  a.stage_M = h->dec_stage_M ? 1 : 0;
  a.stage_V = h->dec_stage_V ? 1 : 0;
  a.acc = h->dec_acc;
  a.acc_stride = h->dec_acc_stride;
  a.bar = h->dec_bar;
  a.status = h->status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h->dec_grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = h->dec_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (h->use_pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t err;
  switch (h->k) {
    case 16: err = cudaLaunchKernelEx(&cfg, gsi_decode_kernel<16>, a); break;
    case 32: err = cudaLaunchKernelEx(&cfg, gsi_decode_kernel<32>, a); break;
    case 64: err = cudaLaunchKernelEx(&cfg, gsi_decode_kernel<64>, a); break;
    case 128: err = cudaLaunchKernelEx(&cfg, gsi_decode_kernel<128>, a); break;
    case 256: err = cudaLaunchKernelEx(&cfg, gsi_decode_kernel<256>, a); break;
    case 512: err = cudaLaunchKernelEx(&cfg, gsi_decode_kernel<512>, a); break;
    default: return GSI_ERR_UNSUPPORTED_SHAPE;
  }
  return err == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

}  // namespace gsi

// ---------------------------------------------------------------------------
// gsi_forward_noalloc: the decode kernel above, run without a handle and with
// its scratch (reduction buffers, arrival counter, launch epoch, status word)
// in a fixed file-scope device array instead of handle-owned memory.
// ---------------------------------------------------------------------------
#include <mutex>

namespace gsi {
namespace {

constexpr int kNoAllocMaxK = 512;                      // largest k the scratch holds
constexpr int kNoAllocAccStride = kNoAllocMaxK + 4;    // floats per accumulator buffer
constexpr size_t kNoAllocAccBytes = size_t(2) * kNoAllocAccStride * sizeof(float);
constexpr size_t kNoAllocBarOffset = (kNoAllocAccBytes + 127) / 128 * 128;
constexpr size_t kNoAllocBytes = kNoAllocBarOffset + 128;  // + counter, epoch, status

// 4.4 KB per GPU that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
// the largest k of the one-token path fits the fixed scratch
static_assert(kNoAllocMaxK >= 512, "scratch must hold the largest supported k");

std::mutex g_noalloc_mutex;
unsigned char* g_noalloc_ptr[kMaxDevices] = {};
int g_noalloc_sms[kMaxDevices] = {};

// Launch plans of earlier calls, by device and shape, so that a repeated shape
// skips the attribute and occupancy queries of decode_configure.
struct NoAllocPlan {
  int device = -1;
  int64_t d_out = 0, d = 0, k = 0;
  int grid = 0, rows_M = 0, rows_V = 0;
  bool stage_M = false, stage_V = false;
  size_t smem = 0;
};
constexpr int kNoAllocPlans = 32;
NoAllocPlan g_noalloc_plans[kNoAllocPlans];
int g_noalloc_next_plan = 0;

// Device address of the scratch array on device `dev` (current), looked up
// once per device (the host-side symbol is only a stand-in, never a device
// address), and the device's SM count.
gsi_status_t noalloc_scratch(int dev, unsigned char** out, int* num_sms) {
  if (dev < 0 || dev >= kMaxDevices) return GSI_ERR_CUDA;
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GSI_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GSI_ERR_CUDA;
    g_noalloc_sms[dev] = sms;
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_noalloc_ptr[dev];
  *num_sms = g_noalloc_sms[dev];
  return GSI_OK;
}

// decode_configure for h, or the plan an earlier call on the same device and
// shape computed.
gsi_status_t noalloc_configure(gsi_handle* h) {
  for (const NoAllocPlan& p : g_noalloc_plans) {
    if (p.device == h->device && p.d_out == h->d_out && p.d == h->d && p.k == h->k) {
      h->dec_grid = p.grid;
      h->dec_rows_M = p.rows_M;
      h->dec_rows_V = p.rows_V;
      h->dec_stage_M = p.stage_M;
      h->dec_stage_V = p.stage_V;
      h->dec_smem = p.smem;
      return GSI_OK;
    }
  }
  const gsi_status_t st = decode_configure(h);
  if (st != GSI_OK) return st;
  NoAllocPlan& p = g_noalloc_plans[g_noalloc_next_plan];
  g_noalloc_next_plan = (g_noalloc_next_plan + 1) % kNoAllocPlans;
  p.device = h->device;
  p.d_out = h->d_out;
  p.d = h->d;
  p.k = h->k;
  p.grid = h->dec_grid;
  p.rows_M = h->dec_rows_M;
  p.rows_V = h->dec_rows_V;
  p.stage_M = h->dec_stage_M;
  p.stage_V = h->dec_stage_V;
  p.smem = h->dec_smem;
  return GSI_OK;
}

}  // namespace
}  // namespace gsi

extern "C" gsi_status_t gsi_forward_noalloc(const void* W, const void* V_k, const void* M,
                                            int64_t d_out, int64_t d, int64_t k, float eps,
                                            const void* x, float* y, uint8_t* gate, float* rho,
                                            cudaStream_t stream) {
  using namespace gsi;
  if (!W || !V_k || !M || !x || !y || eps != eps) return GSI_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(V_k) || !aligned16(M) || !aligned16(x) || !aligned16(y))
    return GSI_ERR_INVALID_ARG;
  if (rho && (reinterpret_cast<uintptr_t>(rho) & 3u)) return GSI_ERR_INVALID_ARG;  // fp32 store
  // k above 512 fails this shape check, before any use of the scratch
  if (d_out <= 0 || d <= 0 || d % 8 != 0 || d_out % 8 != 0 || k > d ||
      (k != 16 && k != 32 && k != 64 && k != 128 && k != 256 && k != 512) ||
      d_out > (int64_t(1) << 30) || d > (int64_t(1) << 24))
    return GSI_ERR_UNSUPPORTED_SHAPE;
  gsi_handle h;  // configuration only: no memory is allocated for it
  h.W = static_cast<const __nv_bfloat16*>(W);
  h.V = static_cast<const __nv_bfloat16*>(V_k);
  h.M = static_cast<const __nv_bfloat16*>(M);
  h.d_out = d_out;
  h.d = d;
  h.k = k;
  h.eps = eps;
  if (cudaGetDevice(&h.device) != cudaSuccess) return GSI_ERR_CUDA;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    gsi_status_t st = noalloc_scratch(h.device, &scratch, &h.num_sms);
    if (st != GSI_OK) return st;
    st = noalloc_configure(&h);
    if (st != GSI_OK) return st;
  }
  h.dec_acc = reinterpret_cast<float*>(scratch);
  h.dec_acc_stride = kNoAllocAccStride;
  h.dec_bar = reinterpret_cast<uint32_t*>(scratch + kNoAllocBarOffset);
  h.status = reinterpret_cast<uint32_t*>(scratch + kNoAllocBarOffset + 64);
  h.use_pdl = false;
  // Every call starts from zeroed accumulators, counter and epoch, whatever
  // shape the previous call on this device had.
  if (cudaMemsetAsync(scratch, 0, kNoAllocBytes, stream) != cudaSuccess) return GSI_ERR_CUDA;
  return decode_launch(&h, x, y, gate, rho, stream);
}
