// gsi_decode3.cu -- the T = 1 (decode) path of the GSI gated linear map as one
// persistent kernel per call with ONE grid-wide exchange (k <= 256).
//
// Page: "Technical summary: Gated Subspace Inference for transformer
// acceleration" [GSI].  Per token x (section 2.1 eq. 1-2, section 2.2):
//   g = V_k^T x,  rho = ||x - V_k g|| / ||x||,
//   y = M g if rho < eps (fast path), y = W x otherwise (slow path).
//
// The residual norm comes from the identity
//   ||x - V_k g||^2 = ||x||^2 - g.g + g^T E g,   E = V_k^T V_k - I,
// which holds for any V_k (expand the square and use V_k^T x = g).  The
// correction g^T E g is a k x k quadratic form on data every CTA already has
// once g is known, so unlike the explicit residual it needs no second pass
// over V_k and no second exchange between CTAs.  E is stored once per handle
// (made in fp64) as its upper 16 x 16 bf16 tiles in MMA operand order
// (gsi_internal.h); the form is evaluated with warp-level bf16 MMAs against
// g split into bf16 high and low parts (g = hi + lo to ~2^-17), accumulated
// in fp32.
//
// Work split.  G co-resident CTAs (at most one per SM); CTA c owns d / G rows
// of V_k and d_out / G output rows (of M and of W).  Before it waits on the
// previous kernel (programmatic dependent launch) each CTA starts 1-D bulk
// copies of its V_k slice, its M slice and F into shared memory: none depends
// on x, so these reads overlap the previous kernel's tail.
//   phase 1   partial g_c = V_c^T x_c and ||x_c||^2, added with vector
//             red.add into one of kCopies accumulator copies (copy c % 8),
//             which spreads the atomic traffic over 8 addresses per word;
//             then the grid barrier (release add / acquire poll)
//   phase 2   every CTA sums the copies in a fixed order (the same g, bit for
//             bit, in every CTA, hence the same gate); half of the warps form
//             g^T E g and g.g (MMA over the correction tiles) while the others
//             form the speculative fast-path rows M_c g, 8 rows per warp step
//             (group_dot)
//   phase 3   thread 0 forms rho and the gate; the CTA stores M_c g, or, on
//             the rare slow token, streams its rows of W from HBM for W_c x.
// With a prefetch link (gsi_set_prefetch) the last warp also issues, right
// after the barrier, L2 prefetches of its 1 / G share of the next call's
// V_k, M and correction tiles, so the next call stages them from L2.
// The accumulators are double-buffered by a launch epoch kept on the device:
// CTA 0 zeroes the buffer the next launch uses, so no memset is needed and
// the kernel replays in a CUDA graph.
#include <algorithm>
#include <cfloat>

#include "gsi_device.cuh"
#include "gsi_internal.h"

namespace gsi {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCopies = 8;  // accumulator copies of (g, ||x||^2)

struct Decode3Args {
  const __nv_bfloat16* W;
  const __nv_bfloat16* V;
  const __nv_bfloat16* M;
  const __nv_bfloat16* F;
  const __nv_bfloat16* x;
  float* y;
  uint8_t* gate;
  float* rho;
  int d_out, d;
  float eps;
  int rows_M, rows_V;
  int stage_M;     // M slice staged in shared memory (V_k slice and F always are)
  float* acc;      // [2][kCopies][acc_stride]
  int acc_stride;  // >= k + 1, multiple of 4
  uint32_t* bar;   // [0] arrival counter, [1] launch epoch
  uint32_t* status;
  // operands of the next call to prefetch into L2 (bytes 0: none), each CTA
  // its 1 / G share
  const char* pf[3];
  uint32_t pf_bytes[3];
};

// Lane geometry: a row of K bf16 values is K / 8 16-byte chunks, one per lane
// of a row group of LPR = K / 8 lanes (K <= 256, so LPR <= 32).
template <int K>
struct Lanes3 {
  static_assert(K >= 16 && K <= 256 && (K & (K - 1)) == 0, "k in {16, ..., 256}");
  static constexpr int LPR = K / 8;             // lanes per row
  static constexpr int RPI = 32 / LPR;          // row groups per warp
  static constexpr int NB = LPR < 8 ? LPR : 8;  // rows per row group per step
  static constexpr int RS = RPI * NB;           // rows per warp step
};

__device__ __forceinline__ void red_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Prefetch [p, p + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t v;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
  return v;
}

// Dot products of NB rows at once.  Lane li of a row group of LPR lanes holds
// v[i], its 8-column partial of row i (i < NB).  A butterfly over sub-groups
// of NB lanes (offsets NB/2 .. 1; each step a lane keeps one half of its rows
// and sends the other half) leaves lane li the sub-group sum of row li % NB;
// xor steps over offsets NB .. LPR/2 then add the sub-groups.  Cost:
// NB - 1 + log2(LPR / NB) shuffles for NB rows.
template <int LPR, int NB>
__device__ __forceinline__ float group_dot(float (&v)[NB], int li) {
#pragma unroll
  for (int o = NB / 2; o >= 1; o >>= 1) {
    const bool up = (li & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = NB; o < LPR; o <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
  return r;
}

// D += A B for one 16 x 16 (A, row-major) by 16 x 8 (B, column-major) bf16
// product with fp32 accumulation (registers in the PTX fragment layout).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint4& a, const uint2& b) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__device__ __forceinline__ float warp_sum_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Dynamic shared-memory layout (byte offsets), identical on host and device.
struct Smem3 {
  size_t sM, sV, sF, wpart, xs, g, ys, bfrag, total;
};
__host__ __device__ inline size_t al3(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline Smem3 smem3_layout(int K, int rows_M, int rows_V, bool stage_M) {
  Smem3 s;
  size_t o = 0;
  s.sM = o;    o = al3(o + (stage_M ? size_t(rows_M) * K * 2 : 0), 128);
  s.sV = o;    o = al3(o + size_t(rows_V) * K * 2, 128);
  s.sF = o;    o = al3(o + corr_tiles_elems(K) * 2, 128);
  s.wpart = o; o = al3(o + size_t(kWarps) * K * 4, 16);
  s.xs = o;    o = al3(o + size_t(rows_V) * 4, 16);
  s.g = o;     o = al3(o + size_t(K) * 4, 16);
  s.ys = o;    o = al3(o + size_t(rows_M) * 4, 16);
  s.bfrag = o; o = al3(o + size_t(K / 16) * 32 * 8, 128);
  s.total = o;
  return s;
}

template <int K, bool kStageM>
__global__ void __launch_bounds__(kThreads, 1) gsi_decode3_kernel(Decode3Args a) {
  using L = Lanes3<K>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_epoch;
  __shared__ int s_ok;
  __shared__ float s_sx;
  __shared__ float s_qw[kWarps], s_ggw[kWarps];
  __shared__ float s_rho;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, G = gridDim.x;
  const Smem3 lay = smem3_layout(K, a.rows_M, a.rows_V, kStageM);
  // Launch self-check (uniform over the grid, before any wait): a launch that
  // does not cover d and d_out, or got less shared memory than its layout,
  // does nothing and reports it.
  if (blockDim.x != kThreads || int64_t(G) * a.rows_M < a.d_out || int64_t(G) * a.rows_V < a.d ||
      dynamic_smem_bytes() < lay.total || (a.stage_M != 0) != kStageM) {
    if (cta == 0 && tid == 0) atomicOr(a.status, kStatusBadLaunch);
    return;
  }
  const int m0 = cta * a.rows_M;
  const int nM = max(0, min(a.d_out, m0 + a.rows_M) - m0);
  const int v0 = cta * a.rows_V;
  const int nV = max(0, min(a.d, v0 + a.rows_V) - v0);
  const int slot = lane / L::LPR, li = lane % L::LPR;

  __nv_bfloat16* sM = reinterpret_cast<__nv_bfloat16*>(smem + lay.sM);
  __nv_bfloat16* sV = reinterpret_cast<__nv_bfloat16*>(smem + lay.sV);
  __nv_bfloat16* sF = reinterpret_cast<__nv_bfloat16*>(smem + lay.sF);
  float* s_wpart = reinterpret_cast<float*>(smem + lay.wpart);  // [warps][K]
  float* s_xs = reinterpret_cast<float*>(smem + lay.xs);        // [rows_V]
  float* s_g = reinterpret_cast<float*>(smem + lay.g);          // [K]
  float* s_ys = reinterpret_cast<float*>(smem + lay.ys);        // [rows_M]
  uint2* s_bfrag = reinterpret_cast<uint2*>(smem + lay.bfrag);  // [K / 16][32]

  // ---- prologue: stage this CTA's weights (independent of x) ------------
  const uint32_t bytes_M = kStageM ? uint32_t(nM) * K * 2 : 0u;
  const uint32_t bytes_V = uint32_t(nV) * K * 2;
  const uint32_t bytes_F = uint32_t(corr_tiles_elems(K)) * 2;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&s_bar, bytes_M + bytes_V + bytes_F);
    constexpr uint32_t kChunk = 32768;
    const char* gV = reinterpret_cast<const char*>(a.V + size_t(v0) * K);
    for (uint32_t off = 0; off < bytes_V; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sV) + off, gV + off, min(kChunk, bytes_V - off), &s_bar);
    const char* gF = reinterpret_cast<const char*>(a.F);
    for (uint32_t off = 0; off < bytes_F; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sF) + off, gF + off, min(kChunk, bytes_F - off), &s_bar);
    const char* gM = reinterpret_cast<const char*>(a.M + size_t(m0) * K);
    for (uint32_t off = 0; off < bytes_M; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sM) + off, gM + off, min(kChunk, bytes_M - off), &s_bar);
  }
  pdl_launch_dependents();
  pdl_wait();  // x and this handle's workspace are now safe to touch

  // ---- phase 1: x slice, partial g and ||x_c||^2 ---------------------------
  if (tid == 0) s_epoch = ld_cg_u32(a.bar + 1);
  for (int i = tid; i < nV; i += kThreads) s_xs[i] = bf16_to_f32(a.x[v0 + i]);
  bool ok = mbar_wait_bounded(&s_bar, 0, a.status);
  ok = __syncthreads_and(ok) != 0;
  const uint32_t e = s_epoch;
  float* acc = a.acc + size_t(e & 1u) * kCopies * a.acc_stride;
  if (cta == 0) {  // clear the buffers the next launch accumulates into
    float* nxt = a.acc + size_t((e + 1u) & 1u) * kCopies * a.acc_stride;
    for (int i = tid; i < kCopies * a.acc_stride; i += kThreads) nxt[i] = 0.f;
  }
  const int nVw = ok ? nV : 0;
  const int nMw = ok ? nM : 0;
  const __nv_bfloat16* Vs = sV;
  const __nv_bfloat16* Ms = kStageM ? sM : a.M + size_t(m0) * K;
  const __nv_bfloat16* Fs = sF;
  // B operands of the correction MMAs (filled after the barrier): for column
  // block J, lane l holds rows 2 (l % 4) + {0, 1, 8, 9} of the 16 x 8 block
  // whose column 0 is the bf16 high part of g_J, column 1 its remainder and
  // the other columns zero; the zero part is written here
  constexpr int T16 = K / 16;
  for (int t = tid; t < T16 * 24; t += kThreads) s_bfrag[(t / 24) * 32 + 8 + t % 24] = make_uint2(0u, 0u);
  if (warp == kWarps - 1) {  // ||x_c||^2 (x_i^2 is exact in fp32 for bf16 x_i)
    float sx = 0.f;
    for (int i = lane; i < nVw; i += 32) sx = fmaf(s_xs[i], s_xs[i], sx);
    sx = warp_sum_all(sx);
    if (lane == 0) s_sx = sx;
  }
  {
    float accg[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) accg[j] = 0.f;
    for (int r = warp * L::RPI + slot; r < nVw; r += kWarps * L::RPI) {
      const float xi = s_xs[r];
      const uint4 v = *reinterpret_cast<const uint4*>(Vs + size_t(r) * K + li * 8);
      float f[8];
      bf16x8_to_f32(v, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) accg[j] = fmaf(f[j], xi, accg[j]);
    }
#pragma unroll
    for (int o = L::LPR; o < 32; o <<= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j) accg[j] += __shfl_xor_sync(0xFFFFFFFFu, accg[j], o);
    if (slot == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) s_wpart[warp * K + li * 8 + j] = accg[j];
    }
  }
  __syncthreads();
  float* my_copy = acc + size_t(cta % kCopies) * a.acc_stride;
  if (nVw > 0) {
    for (int t = tid; t < K / 4; t += kThreads) {
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
#pragma unroll
        for (int q = 0; q < 4; ++q) s4[q] += s_wpart[w * K + t * 4 + q];
      red_add_v4_f32(my_copy + t * 4, s4[0], s4[1], s4[2], s4[3]);
    }
    if (tid == 0) red_add_f32(my_copy + K, s_sx);
  }

  // ---- the grid barrier ---------------------------------------------------
  __syncthreads();
  if (tid == 0) {
    const uint32_t target = (e + 1u) * uint32_t(G);
    red_release_u32(a.bar, 1u);
    int good = 1;
    if (static_cast<int32_t>(ld_acquire_gpu(a.bar) - target) < 0) {
      const uint64_t t0 = globaltimer_ns();
      while (static_cast<int32_t>(ld_acquire_gpu(a.bar) - target) < 0) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.status, kStatusTimeout);
          good = 0;
          break;
        }
      }
    }
    s_ok = good;
  }
  __syncthreads();
  ok = ok && s_ok;
  if (warp == kWarps - 1) {
    // this CTA's share of the next call's operands, into L2.  Issued after
    // the barrier, when the rest of this call works from shared memory: the
    // stream then does not delay this call's x read, atomics or barrier.
#pragma unroll
    for (int o = 0; o < 3; ++o) {
      const uint32_t bytes = a.pf_bytes[o];
      const uint32_t share = (bytes / 16 + G - 1) / G * 16;
      const uint32_t lo = min(bytes, uint32_t(cta) * share), hi = min(bytes, lo + share);
      constexpr uint32_t kPiece = 16384;
      for (uint32_t off = lo + uint32_t(lane) * kPiece; off < hi; off += 32u * kPiece)
        prefetch_l2(a.pf[o] + off, min(kPiece, hi - off));
    }
  }

  // ---- phase 2: g (same order in every CTA), g^T E g, g.g, speculative M g --
  for (int t = tid; t < K; t += kThreads) {
    float gsum = 0.f;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) gsum += ld_cg_f32(acc + size_t(c) * a.acc_stride + t);
    s_g[t] = gsum;
    // g_t is row kk = t % 16 of column block J = t / 16: register kk / 8,
    // lane pair (kk % 8) / 2, half kk % 2 of lanes pair (high) and 4 + pair (low)
    const __nv_bfloat16 hi = __float2bfloat16_rn(gsum);
    const __nv_bfloat16 lo = __float2bfloat16_rn(gsum - __bfloat162float(hi));
    const int kk = t & 15, pos = (kk >> 3) * 2 + (kk & 1), pr = (kk & 7) >> 1;
    __nv_bfloat16* bf = reinterpret_cast<__nv_bfloat16*>(s_bfrag + (t >> 4) * 32);
    bf[pr * 4 + pos] = hi;
    bf[(4 + pr) * 4 + pos] = lo;
  }
  if (tid == 0) {
    float sx = 0.f;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) sx += ld_cg_f32(acc + size_t(c) * a.acc_stride + K);
    s_sx = sx;
  }
  __syncthreads();
  constexpr int kQuadWarps = T16 > 1 ? T16 / 2 : 1;
  if (warp < kQuadWarps) {
    // g^T E g = sum over tiles I <= J of g_I . (F_IJ g_J); this warp takes
    // row blocks I1 = warp (T16 - warp tiles) and I2 = T16 - 1 - warp
    // (warp + 1 tiles), T16 + 1 independent MMAs in all
    constexpr int kSteps = T16 > 1 ? T16 + 1 : 1;
    const uint4* tiles = reinterpret_cast<const uint4*>(Fs);
    const int grp = lane >> 2;
    const int I1 = warp, I2 = T16 - 1 - warp, n1 = T16 - warp;
    const float g10 = s_g[I1 * 16 + grp], g11 = s_g[I1 * 16 + grp + 8];
    const float g20 = s_g[I2 * 16 + grp], g21 = s_g[I2 * 16 + grp + 8];
    float qsum = 0.f;
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      const bool first = st < n1;
      const int I = first ? I1 : I2;
      const int J = first ? I1 + st : I2 + (st - n1);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(d, tiles[corr_tile_index(I, J, T16) * 32 + lane], s_bfrag[J * 32 + lane]);
      // columns 0 (high) and 1 (low) of rows grp and grp + 8 (lanes with
      // lane % 4 == 0; the other lanes hold the zero columns)
      qsum = fmaf(first ? g10 : g20, d[0] + d[1], qsum);
      qsum = fmaf(first ? g11 : g21, d[2] + d[3], qsum);
    }
    float ggsum = fmaf(g10, g10, g11 * g11);
    if (I2 != I1) ggsum = fmaf(g20, g20, fmaf(g21, g21, ggsum));
    if ((lane & 3) != 0) qsum = ggsum = 0.f;
    qsum = warp_sum_all(qsum);
    ggsum = warp_sum_all(ggsum);
    if (lane == 0) {
      s_qw[warp] = qsum;
      s_ggw[warp] = ggsum;
    }
  } else {
    // speculative fast path: this CTA's rows of M g
    float gl[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) gl[j] = s_g[li * 8 + j];
    constexpr int kYWarps = kWarps - kQuadWarps;
    for (int rb = (warp - kQuadWarps) * L::RS; rb < nMw; rb += kYWarps * L::RS) {
      float v[L::NB];
#pragma unroll
      for (int i = 0; i < L::NB; ++i) {
        const int r = rb + slot * L::NB + i;
        float dot = 0.f;
        if (r < nMw) {
          const uint4 mv = *reinterpret_cast<const uint4*>(Ms + size_t(r) * K + li * 8);
          float f[8];
          bf16x8_to_f32(mv, f);
#pragma unroll
          for (int j = 0; j < 8; ++j) dot = fmaf(f[j], gl[j], dot);
        }
        v[i] = dot;
      }
      const float yr = group_dot<L::LPR, L::NB>(v, li);
      const int r = rb + slot * L::NB + li % L::NB;
      if (li < L::NB && r < nMw) s_ys[r] = yr;
    }
  }
  __syncthreads();

  // ---- gate ------------------------------------------------------------------
  if (tid == 0) {
    // fp32 throughout: the sums' relative error (~1e-7 of ||x||^2) moves rho by
    // ~1e-6 near any practical eps, and fp64 is slow on this part
    float quad = 0.f, gg = 0.f;
    for (int w = 0; w < kQuadWarps; ++w) {
      quad += s_qw[w];
      gg += s_ggw[w];
    }
    const float sx = s_sx;
    float rho;
    if (!(fabsf(sx) <= FLT_MAX)) {
      rho = __int_as_float(0x7FC00000);  // non-finite x: NaN, slow path
    } else if (sx == 0.f) {
      rho = 0.f;
    } else {
      float sr = (sx - gg) + quad;
      if (!(sr >= 0.f)) sr = (sr == sr) ? 0.f : sr;
      rho = sqrtf(sr / sx);
    }
    s_rho = rho;
    if (cta == 0) {
      if (a.gate) a.gate[0] = (rho < a.eps) ? 0 : 1;
      if (a.rho) a.rho[0] = rho;
    }
  }
  __syncthreads();
  const bool slow = !(s_rho < a.eps);

  // ---- phase 3: the branch the gate picked ---------------------------------
  if (ok) {
    if (!slow) {
      for (int r = tid; r < nMw; r += kThreads) a.y[m0 + r] = s_ys[r];
    } else {
      // W_c x, W streamed from HBM, 4 rows per warp
      const int nch = a.d / 8;
      const uint4* x4 = reinterpret_cast<const uint4*>(a.x);
      for (int rb = warp * 4; rb < nM; rb += kWarps * 4) {
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4* wr[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = min(rb + q, nM - 1);
          wr[q] = reinterpret_cast<const uint4*>(a.W + size_t(m0 + r) * a.d);
        }
        int j = lane;
        for (; j + 32 < nch; j += 64) {
          uint4 w0[4], w1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            w0[q] = ld_stream_v4(wr[q] + j);
            w1[q] = ld_stream_v4(wr[q] + j + 32);
          }
          float xa[8], xb[8];
          bf16x8_to_f32(x4[j], xa);
          bf16x8_to_f32(x4[j + 32], xb);
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
          bf16x8_to_f32(x4[j], xa);
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
            if (rb + q < nM) a.y[m0 + rb + q] = acc4[q];
        }
      }
    }
  }
  if (cta == 0 && tid == 0) {
    __threadfence();
    a.bar[1] = e + 1u;  // every CTA read the epoch before the barrier
  }
}

template <int K>
const void* kernel3_ptr(bool stage_M) {
  return stage_M ? reinterpret_cast<const void*>(&gsi_decode3_kernel<K, true>)
                 : reinterpret_cast<const void*>(&gsi_decode3_kernel<K, false>);
}

const void* decode3_kernel_for(int64_t k, bool stage_M) {
  switch (k) {
    case 16: return kernel3_ptr<16>(stage_M);
    case 32: return kernel3_ptr<32>(stage_M);
    case 64: return kernel3_ptr<64>(stage_M);
    case 128: return kernel3_ptr<128>(stage_M);
    case 256: return kernel3_ptr<256>(stage_M);
    default: return nullptr;
  }
}

int acc3_stride(int64_t k) { return int((k + 1 + 3) / 4 * 4); }

}  // namespace

size_t decode3_acc_floats(int64_t k) { return size_t(2) * kCopies * acc3_stride(k); }

gsi_status_t decode3_configure(gsi_handle* h) {
  if (!decode3_kernel_for(h->k, true)) return GSI_ERR_UNSUPPORTED_SHAPE;
  int max_optin = 0;
  if (cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess)
    return GSI_ERR_CUDA;
  const int64_t rows_hint = (std::max(h->d_out, h->d) + 7) / 8;
  const int G = int(std::max<int64_t>(1, std::min<int64_t>(h->num_sms, rows_hint)));
  const int rows_M = int((h->d_out + G - 1) / G);
  const int rows_V = int((h->d + G - 1) / G);
  const int K = int(h->k);
  // Both variants of a k have the same static shared memory.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, decode3_kernel_for(h->k, true)) != cudaSuccess) return GSI_ERR_CUDA;
  const int fn_limit = max_optin - int(fa.sharedSizeBytes);
  // V_k slice and F are always staged; the M slice too when it fits (else it
  // is read from global memory after the barrier).
  const bool stage_M = smem3_layout(K, rows_M, rows_V, true).total <= size_t(fn_limit);
  const size_t smem = smem3_layout(K, rows_M, rows_V, stage_M).total;
  if (smem > size_t(fn_limit)) return GSI_ERR_UNSUPPORTED_SHAPE;
  const void* fn = decode3_kernel_for(h->k, stage_M);
  // The limit belongs to the kernel function, shared by every handle with
  // this k: raise it to the device maximum once, never per handle.
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return GSI_ERR_CUDA;
  if (fa.maxDynamicSharedSizeBytes < fn_limit &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, fn_limit) != cudaSuccess)
    return GSI_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem) != cudaSuccess)
    return GSI_ERR_CUDA;
  // The CTAs wait on one another: all of them must fit at once.
  if (per_sm < 1 || int64_t(per_sm) * h->num_sms < G) return GSI_ERR_UNSUPPORTED_SHAPE;
  h->dec3_grid = G;
  h->dec3_rows_M = rows_M;
  h->dec3_rows_V = rows_V;
  h->dec3_stage_M = stage_M;
  h->dec3_smem = smem;
  return GSI_OK;
}

gsi_status_t decode3_launch(gsi_handle* h, const void* x, float* y, uint8_t* gate, float* rho,
                            cudaStream_t s) {
  Decode3Args a;
  a.W = h->W;
  a.V = h->V;
  a.M = h->M;
  a.F = h->dec3_F;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.y = y;
  a.gate = gate;
  a.rho = rho;
  a.d_out = int(h->d_out);
  a.d = int(h->d);
  a.eps = h->eps;
  a.rows_M = h->dec3_rows_M;
  a.rows_V = h->dec3_rows_V;
  a.stage_M = h->dec3_stage_M ? 1 : 0;
  a.acc = h->dec3_acc;
  a.acc_stride = acc3_stride(h->k);
  a.bar = h->dec3_bar;
  a.status = h->status;
  // operands above 64 MiB are not prefetched (a large share of L2)
  const gsi_handle* n = h->pf_next;
  const int64_t kMaxPrefetch = int64_t(64) << 20;
  const int64_t pf_b[3] = {n ? n->d * n->k * 2 : 0, n ? n->d_out * n->k * 2 : 0,
                           (n && n->dec3_F) ? int64_t(corr_tiles_elems(int(n->k))) * 2 : 0};
  const void* pf_p[3] = {n ? n->V : nullptr, n ? n->M : nullptr, n ? n->dec3_F : nullptr};
  for (int o = 0; o < 3; ++o) {
    const bool on = pf_b[o] > 0 && pf_b[o] <= kMaxPrefetch;
    a.pf[o] = on ? static_cast<const char*>(pf_p[o]) : nullptr;
    a.pf_bytes[o] = on ? uint32_t(pf_b[o]) : 0u;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h->dec3_grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = h->dec3_smem;
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
  const void* fn = decode3_kernel_for(h->k, h->dec3_stage_M);
  if (!fn) return GSI_ERR_UNSUPPORTED_SHAPE;
  void* args[] = {&a};
  return cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

}  // namespace gsi
