// gsi_batched.cu -- the T > 1 path of the GSI gated linear map.
//
// Page: "Technical summary: Gated Subspace Inference for transformer
// acceleration" [GSI], sections 2.1-2.2.  For T tokens at once:
//   1. projection   G = X V_k (T x k) and ||x_t||^2            (section 2.1)
//   2. gate         ||r_t||^2 = ||x_t||^2 - 2 g_t.g_t + g_t^T Gm g_t with
//                   Gm = V_k^T V_k (exact identity for r = x - V_k g),
//                   rho_t = ||r_t|| / ||x_t||, gate_t = !(rho_t < eps)
//   3. partition    stable partition of 0..T-1 by gate into index lists, and
//      + gather     fast tokens' g_t (as bf16 hi + lo pairs) and slow tokens'
//                   x_t into dense operand blocks, in one launch
//   4. GEMMs        Y_fast = G_fast M^T and Y_slow = X_slow W^T on the
//                   tcgen05 tensor cores (gsi_tc_gemm.cu), each output row
//                   scattered back to its token's row of y.
// Counts of fast and slow tokens stay on the device; GEMM CTAs whose token
// tile lies past the count exit before reading weights.
#include <algorithm>
#include <cfloat>

#include "gsi_device.cuh"
#include "gsi_internal.h"
#include "gsi_tc_gemm.h"

namespace gsi {
namespace {

constexpr int kProjRows = 64;    // V_k rows per CTA
constexpr int kProjTok = 16;     // tokens per CTA
constexpr int kGateTok = 8;      // tokens per CTA in the gate kernel

// G[t][a] += sum_{i in chunk} x[t][i] V[i][a]; sx[t] += sum_{i in chunk} x[t][i]^2.
template <int K>
__global__ void __launch_bounds__(256) proj_kernel(const __nv_bfloat16* __restrict__ x,
                                                   const __nv_bfloat16* __restrict__ V,
                                                   int T, int d, float* __restrict__ G,
                                                   float* __restrict__ sx) {
  __shared__ float sxv[kProjTok][kProjRows + 1];
  const int i0 = blockIdx.x * kProjRows, t0 = blockIdx.y * kProjTok;
  const int nrow = min(kProjRows, d - i0), ntok = min(kProjTok, T - t0);
  for (int q = threadIdx.x; q < kProjTok * kProjRows; q += blockDim.x) {
    const int t = q / kProjRows, i = q % kProjRows;
    sxv[t][i] = (t < ntok && i < nrow) ? __bfloat162float(x[size_t(t0 + t) * d + i0 + i]) : 0.f;
  }
  __syncthreads();
  for (int a = threadIdx.x; a < K; a += blockDim.x) {
    float acc[kProjTok];
#pragma unroll
    for (int t = 0; t < kProjTok; ++t) acc[t] = 0.f;
    for (int i = 0; i < nrow; ++i) {
      const float v = __bfloat162float(V[size_t(i0 + i) * K + a]);
#pragma unroll
      for (int t = 0; t < kProjTok; ++t) acc[t] = fmaf(v, sxv[t][i], acc[t]);
    }
    for (int t = 0; t < ntok; ++t) red_add_f32(G + size_t(t0 + t) * K + a, acc[t]);
  }
  if (threadIdx.x < ntok) {
    float s = 0.f;
    for (int i = 0; i < nrow; ++i) s = fmaf(sxv[threadIdx.x][i], sxv[threadIdx.x][i], s);
    red_add_f32(sx + t0 + threadIdx.x, s);
  }
}

// rho and gate of kGateTok tokens per CTA.
template <int K>
__global__ void __launch_bounds__(256) gate_kernel(const float* __restrict__ G,
                                                   const float* __restrict__ sx,
                                                   const float* __restrict__ gram, int T,
                                                   float eps, uint8_t* __restrict__ gate_int,
                                                   uint8_t* __restrict__ gate_out,
                                                   float* __restrict__ rho_out) {
  __shared__ float sg[kGateTok][K];
  __shared__ float sred[kGateTok][2][8];
  const int t0 = blockIdx.x * kGateTok;
  const int ntok = min(kGateTok, T - t0);
  for (int q = threadIdx.x; q < kGateTok * K; q += blockDim.x) {
    const int t = q / K, a = q % K;
    sg[t][a] = t < ntok ? G[size_t(t0 + t) * K + a] : 0.f;
  }
  __syncthreads();
  float quad[kGateTok], gg[kGateTok];
#pragma unroll
  for (int t = 0; t < kGateTok; ++t) quad[t] = gg[t] = 0.f;
  for (int a = threadIdx.x; a < K; a += blockDim.x) {
    float hg[kGateTok];
#pragma unroll
    for (int t = 0; t < kGateTok; ++t) hg[t] = 0.f;
    for (int b = 0; b < K; ++b) {
      const float gm = gram[size_t(b) * K + a];  // Gm is symmetric: row b, column a
#pragma unroll
      for (int t = 0; t < kGateTok; ++t) hg[t] = fmaf(gm, sg[t][b], hg[t]);
    }
#pragma unroll
    for (int t = 0; t < kGateTok; ++t) {
      quad[t] = fmaf(sg[t][a], hg[t], quad[t]);
      gg[t] = fmaf(sg[t][a], sg[t][a], gg[t]);
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int t = 0; t < kGateTok; ++t) {
    const float q = warp_sum_xor<32>(quad[t]);
    const float g2 = warp_sum_xor<32>(gg[t]);
    if (lane == 0) {
      sred[t][0][warp] = q;
      sred[t][1][warp] = g2;
    }
  }
  __syncthreads();
  if (threadIdx.x < ntok) {
    const int t = threadIdx.x;
    float q = 0.f, g2 = 0.f;
    for (int w = 0; w < int(blockDim.x / 32); ++w) {
      q += sred[t][0][w];
      g2 += sred[t][1][w];
    }
    const float sxv = sx[t0 + t];
    float rho;
    if (!(fabsf(sxv) <= FLT_MAX)) {
      rho = __int_as_float(0x7FC00000);
    } else if (sxv == 0.f) {
      rho = 0.f;
    } else {
      float sr = sxv - 2.f * g2 + q;
      if (!(sr >= 0.f)) sr = (sr == sr) ? 0.f : sr;
      rho = sqrtf(sr / sxv);
    }
    const uint8_t slow = (rho < eps) ? 0 : 1;
    gate_int[t0 + t] = slow;
    if (gate_out) gate_out[t0 + t] = slow;
    if (rho_out) rho_out[t0 + t] = rho;
  }
}

// rho and gate of 8 tokens per CTA from the Gram identity in the form
// ||x - V g||^2 = ||x||^2 - g.g + g^T E g, E = V^T V - I (the one-token
// kernel's form), with g^T E g on warp-level bf16 MMAs over the handle's
// correction tiles (upper 16 x 16 tiles of E, MMA operand order, see
// gsi_internal.h).  All 8 warps load (the projection partials and the x rows
// are read with many independent loads in flight).  The correction then runs
// on all 8 warps: warp w takes tokens 4 (w % 2) .. 4 (w % 2) + 3 and every
// fourth tile (tile index = w / 2 mod 4); the B operand's 8 columns are those
// tokens' g as bf16 high part and remainder (column 2j + part for token j),
// so lane (grp, tig) accumulates token tig.  The four warps' partial sums of a
// token are added in warp order.
constexpr int kGateMmaTok = 8;
constexpr int kGateMmaThreads = 256;
constexpr int kGatePad = 8;  // floats of padding per staged g row (no bank conflicts)

// One warp's share of g^T E g: the correction tiles (I, J), I <= J, whose
// storage index is TS mod 4, in (I, J) order.  Tile (I, J) contributes
// g_I . (F_IJ g_J); lane (grp, tig) holds columns 2 tig (high part) and
// 2 tig + 1 (low part) of token tig, rows grp and grp + 8.
template <int T16, int TS>
__device__ __forceinline__ float gate_corr_subset(const uint4* sF, const float* gq,
                                                  const uint2 (&bfr)[T16], int lane, int grp) {
  float q = 0.f;
#pragma unroll
  for (int I = 0; I < T16; ++I) {
#pragma unroll
    for (int J = I; J < T16; ++J) {
      if ((corr_tile_index(I, J, T16) & 3) != TS) continue;
      float dd[4] = {0.f, 0.f, 0.f, 0.f};
      const uint4 A = sF[corr_tile_index(I, J, T16) * 32 + lane];
      asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
          "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
          : "+f"(dd[0]), "+f"(dd[1]), "+f"(dd[2]), "+f"(dd[3])
          : "r"(A.x), "r"(A.y), "r"(A.z), "r"(A.w), "r"(bfr[J].x), "r"(bfr[J].y));
      q = fmaf(gq[I * 16 + grp], dd[0] + dd[1], q);
      q = fmaf(gq[I * 16 + grp + 8], dd[2] + dd[3], q);
    }
  }
  return q;
}

// With S > 0, g is the sum (in slice order) of the S projection partials P[s]
// and is also written to G for the gather; with S = 0 it is read from G.
template <int K>
__global__ void __launch_bounds__(kGateMmaThreads) gate_mma_kernel(
    float* G, const float* P, int S, size_t split_stride,
    const __nv_bfloat16* x, const __nv_bfloat16* F, int T, int d,
    float eps, uint8_t* gate_int, uint8_t* gate_out,
    float* rho_out, uint32_t* status, const float* sxp,
    size_t sxp_stride) {
  constexpr int T16 = K / 16;
  constexpr int kTiles = T16 * (T16 + 1) / 2;
  constexpr int kRow = K + kGatePad;
  extern __shared__ __align__(128) unsigned char smem[];
  uint4* sF = reinterpret_cast<uint4*>(smem);                          // [kTiles][32]
  float* sg = reinterpret_cast<float*>(smem + size_t(kTiles) * 512);   // [8][kRow]
  uint2* sB = reinterpret_cast<uint2*>(smem + size_t(kTiles) * 512 +
                                       size_t(kGateMmaTok) * kRow * 4);  // [2][T16][32]
  __shared__ float s_sx[kGateMmaTok], s_gg[kGateMmaTok];
  __shared__ float s_q[4][kGateMmaTok];
  __shared__ uint64_t s_bar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int t0 = blockIdx.x * kGateMmaTok;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = uint32_t(kTiles) * 512;
    mbar_arrive_expect_tx(&s_bar, bytes);
    constexpr uint32_t kChunk = 32768;
    for (uint32_t off = 0; off < bytes; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sF) + off, reinterpret_cast<const char*>(F) + off,
               min(kChunk, bytes - off), &s_bar);
  }
  pdl_launch_dependents();
  pdl_wait();  // the projection's output and x are now visible
  // Every load of the CTA is issued before the first add: the S projection
  // partials of the 8 tokens' g (float4 units, kGU per thread) and the x rows
  // (warp w takes token w, kXU 16-byte chunks per lane and pass).
  constexpr int kGU = (kGateMmaTok * K / 4 + kGateMmaThreads - 1) / kGateMmaThreads;
  constexpr int kXU = 16;
  float4 part[kGU][tc_proj_max_splits()];
  float4 gv[kGU];
#pragma unroll
  for (int u = 0; u < kGU; ++u) {
    const int q = tid + u * kGateMmaThreads;
    const int t = q / (K / 4), a4 = q % (K / 4);
    const bool live = q < kGateMmaTok * K / 4 && t0 + t < T;
    const size_t o = size_t(t0 + t) * K + size_t(a4) * 4;
    gv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sl = 0; sl < tc_proj_max_splits(); ++sl)
      part[u][sl] = (live && sl < S) ? *reinterpret_cast<const float4*>(P + size_t(sl) * split_stride + o)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    if (live && S == 0) gv[u] = *reinterpret_cast<const float4*>(G + o);
  }
  // ||x_t||^2 (x_i^2 is exact in fp32; four partial sums per lane): from the
  // tensor-core projection's per-slice sums when it made them, else from x
  const int tx = t0 + warp;
  const bool x_from_slices = S > 0 && sxp != nullptr;
  const float sx_slice = (x_from_slices && lane < S && tx < T) ? sxp[size_t(lane) * sxp_stride + tx] : 0.f;
  const uint4* xr = reinterpret_cast<const uint4*>(x + size_t(tx) * d);
  const int nch = x_from_slices ? 0 : d / 8;
  float acc4[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint4 ch[kXU];
#pragma unroll
    for (int u = 0; u < kXU; ++u) {
      const int c = lane + u * 32;
      ch[u] = (tx < T && c < nch) ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kGU; ++u) {
      const int q = tid + u * kGateMmaThreads;
      if (q >= kGateMmaTok * K / 4) continue;
      const int t = q / (K / 4), a4 = q % (K / 4);
      if (S > 0) {
#pragma unroll
        for (int sl = 0; sl < tc_proj_max_splits(); ++sl) {
          gv[u].x += part[u][sl].x;
          gv[u].y += part[u][sl].y;
          gv[u].z += part[u][sl].z;
          gv[u].w += part[u][sl].w;
        }
        if (t0 + t < T) *reinterpret_cast<float4*>(G + size_t(t0 + t) * K + size_t(a4) * 4) = gv[u];
      }
      *reinterpret_cast<float4*>(sg + t * kRow + a4 * 4) = gv[u];
    }
#pragma unroll
    for (int u = 0; u < kXU; ++u) {
      float f[8];
      bf16x8_to_f32(ch[u], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc4[e & 3] = fmaf(f[e], f[e], acc4[e & 3]);
    }
  }
  // rows longer than 32 * kXU chunks (d > 4096): further passes
  for (int c0 = lane + 32 * kXU; tx < T && c0 < nch; c0 += 32 * kXU) {
    uint4 ch[kXU];
#pragma unroll
    for (int u = 0; u < kXU; ++u) {
      const int c = c0 + u * 32;
      ch[u] = c < nch ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kXU; ++u) {
      float f[8];
      bf16x8_to_f32(ch[u], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc4[e & 3] = fmaf(f[e], f[e], acc4[e & 3]);
    }
  }
  {
    float sxv = x_from_slices ? sx_slice : (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
    sxv = warp_sum_xor<32>(sxv);
    if (lane == 0) s_sx[warp] = sxv;
  }
  __syncthreads();
  {
    const float* gr = sg + warp * kRow;
    float v = 0.f;
    for (int a = lane; a < K; a += 32) v = fmaf(gr[a], gr[a], v);
    v = warp_sum_xor<32>(v);
    if (lane == 0) s_gg[warp] = v;
  }
  // B operands of both token groups (4 tokens each), one per column block J
  // and lane, built once for the CTA while the correction tiles land: lane
  // (grp, tig) holds rows 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 of token
  // grp / 2, as the bf16 high part (grp even) or remainder (grp odd)
  for (int e = tid; e < 2 * T16 * 32; e += kGateMmaThreads) {
    const int ln = e & 31, J = (e >> 5) % T16, tgi = e / (32 * T16);
    const int gp = ln >> 2, tg4 = ln & 3;
    const float* gb = sg + (tgi * 4 + gp / 2) * kRow;
    const int a = J * 16 + 2 * tg4;
    const float v[4] = {gb[a], gb[a + 1], gb[a + 8], gb[a + 9]};
    uint32_t p[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v[q]);
      const __nv_bfloat16 part = (gp & 1) ? __float2bfloat16_rn(v[q] - __bfloat162float(hi)) : hi;
      p[q] = __bfloat16_as_ushort(part);
    }
    sB[e] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
  const bool ok = mbar_wait_bounded(&s_bar, 0, status);
  __syncthreads();
  const int tg = warp & 1, ts = warp >> 1;  // token group, tile subset
  uint2 bfr[T16];
#pragma unroll
  for (int J = 0; J < T16; ++J) bfr[J] = sB[(tg * T16 + J) * 32 + lane];
  // g^T E g over this warp's tile subset
  const float* gq = sg + (tg * 4 + tig) * kRow;
  float q = 0.f;
  if (ok) {
    // the subset is a template argument, so that each warp's tiles unroll to
    // straight-line code whose shared-memory loads and MMAs overlap
    switch (ts) {
      case 0: q = gate_corr_subset<T16, 0>(sF, gq, bfr, lane, grp); break;
      case 1: q = gate_corr_subset<T16, 1>(sF, gq, bfr, lane, grp); break;
      case 2: q = gate_corr_subset<T16, 2>(sF, gq, bfr, lane, grp); break;
      default: q = gate_corr_subset<T16, 3>(sF, gq, bfr, lane, grp); break;
    }
  }
  // sum over grp (lanes of equal tig), then over the four tile subsets
  q += __shfl_xor_sync(0xFFFFFFFFu, q, 4);
  q += __shfl_xor_sync(0xFFFFFFFFu, q, 8);
  q += __shfl_xor_sync(0xFFFFFFFFu, q, 16);
  if (lane < 4) s_q[ts][tg * 4 + lane] = q;
  __syncthreads();
  if (tid < kGateMmaTok) {
    const int tl = tid, t = t0 + tl;
    q = ((s_q[0][tl] + s_q[1][tl]) + s_q[2][tl]) + s_q[3][tl];
    if (t < T) {
      const float sxv = s_sx[tl];
      float rho;
      if (!ok) {
        rho = __int_as_float(0x7FC00000);
      } else if (!(fabsf(sxv) <= FLT_MAX)) {
        rho = __int_as_float(0x7FC00000);  // non-finite x: NaN, slow path
      } else if (sxv == 0.f) {
        rho = 0.f;
      } else {
        float sr = (sxv - s_gg[tl]) + q;
        if (!(sr >= 0.f)) sr = (sr == sr) ? 0.f : sr;
        rho = sqrtf(sr / sxv);
      }
      const uint8_t slow = (rho < eps) ? 0 : 1;
      gate_int[t] = slow;
      if (gate_out) gate_out[t] = slow;
      if (rho_out) rho_out[t] = rho;
    }
  }
}

template <int K>
size_t gate_mma_smem() {
  constexpr int T16 = K / 16;
  return size_t(T16) * (T16 + 1) / 2 * 512 + size_t(kGateMmaTok) * (K + kGatePad) * 4 +
         size_t(2) * T16 * 32 * 8;
}

// V_k (d x k) -> V_k^T (k x d), 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_kernel(const __nv_bfloat16* __restrict__ V, int d,
                                                        int k, __nv_bfloat16* __restrict__ VT) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int a0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
  for (int q = threadIdx.x; q < 32 * 32; q += blockDim.x) {
    const int r = q / 32, c = q % 32;
    if (i0 + r < d && a0 + c < k) tile[r][c] = V[size_t(i0 + r) * k + a0 + c];
  }
  __syncthreads();
  for (int q = threadIdx.x; q < 32 * 32; q += blockDim.x) {
    const int r = q / 32, c = q % 32;  // VT row a0 + r, column i0 + c
    if (a0 + r < k && i0 + c < d) VT[size_t(a0 + r) * d + i0 + c] = tile[c][r];
  }
}

// Partition and gather in one launch, one CTA per token t.  The CTA counts
// the slow gates before t (every CTA reads the T gate bytes), which places t
// in the stable partition [fast tokens | slow tokens]:
//   fast: row pos = t - (slow before t) of the G_fast planes, hi = bf16(g) in
//         plane 0 and lo = bf16(g - hi) in plane 1 (hi + lo carries g to
//         ~2^-16 relative), and idx_fast[pos] = t;
//   slow: row pos = (slow before t) of X_slow (a bf16 copy of x), and
//         idx_slow[pos] = t.
// CTA 0 also writes the counts and empties the GEMM's tile queue.
template <int K>
__global__ void __launch_bounds__(256) partition_gather_kernel(
    const __nv_bfloat16* x, const float* G,
    const uint8_t* gate, int T, int d, int max_T, int32_t* idx_fast,
    int32_t* idx_slow, int32_t* count, __nv_bfloat16* Gf,
    __nv_bfloat16* Xs) {
  __shared__ int s_red[2][8];
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // this token's x row and g row are loaded together with the gate bytes
  // (one round trip to memory instead of two); the branch uses one of them
  constexpr int kXR = 8;  // 16-byte chunks of x per thread held in registers
  const int nch = d / 8;
  const bool x_in_regs = nch <= kXR * int(blockDim.x);
  uint4 xr[kXR];
  const uint4* src = reinterpret_cast<const uint4*>(x + size_t(t) * d);
  if (x_in_regs) {
#pragma unroll
    for (int u = 0; u < kXR; ++u) {
      const int i = tid + u * int(blockDim.x);
      xr[u] = i < nch ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  float gr[(K + 255) / 256];
#pragma unroll
  for (int u = 0; u < (K + 255) / 256; ++u) {
    const int a = tid + u * 256;
    gr[u] = a < K ? G[size_t(t) * K + a] : 0.f;
  }
  int before = 0, total = 0;
  for (int i = tid; i < T; i += blockDim.x) {
    const int f = gate[i] != 0;
    total += f;
    if (i < t) before += f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xFFFFFFFFu, before, o);
    total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
  }
  if (lane == 0) {
    s_red[0][warp] = before;
    s_red[1][warp] = total;
  }
  __syncthreads();
  before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    before += s_red[0][w];
    total += s_red[1][w];
  }
  if (t == 0 && tid == 0) {
    count[0] = T - total;  // n_fast
    count[1] = total;      // n_slow
    count[2] = 0;          // the GEMM's tile queue starts empty
  }
  if (gate[t] == 0) {
    const int pos = t - before;
    if (tid == 0) idx_fast[pos] = t;
#pragma unroll
    for (int u = 0; u < (K + 255) / 256; ++u) {
      const int a = tid + u * 256;
      if (a < K) {
        const float g = gr[u];
        const __nv_bfloat16 hi = __float2bfloat16_rn(g);
        const __nv_bfloat16 lo = __float2bfloat16_rn(g - __bfloat162float(hi));
        Gf[size_t(pos) * K + a] = hi;
        Gf[(size_t(max_T) + pos) * K + a] = lo;
      }
    }
  } else {
    const int pos = before;
    if (tid == 0) idx_slow[pos] = t;
    uint4* dst = reinterpret_cast<uint4*>(Xs + size_t(pos) * d);
    if (x_in_regs) {
#pragma unroll
      for (int u = 0; u < kXR; ++u) {
        const int i = tid + u * int(blockDim.x);
        if (i < nch) dst[i] = xr[u];
      }
    } else {
      for (int i = tid; i < nch; i += blockDim.x) dst[i] = src[i];
    }
  }
}

template <int K>
gsi_status_t launch_front(gsi_handle* h, const void* x, int T, uint8_t* gate, float* rho,
                          cudaStream_t s) {
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  // projection: tensor cores (k = 128, 256) into partials, else CUDA cores
  // accumulating into G
  int S = 0;
  if (tc_proj_supported(h) && h->bP) {
    int kb_per = 0;
    S = tc_proj_splits(h, T, &kb_per);
    const gsi_status_t st = tc_proj_launch(h, x, T, S, kb_per, s);
    if (st != GSI_OK) return st;
  } else {
    if (cudaMemsetAsync(h->bG, 0, size_t(T) * K * sizeof(float), s) != cudaSuccess) return GSI_ERR_CUDA;
    if (cudaMemsetAsync(h->bsx, 0, size_t(T) * sizeof(float), s) != cudaSuccess) return GSI_ERR_CUDA;
    dim3 pg(unsigned((h->d + kProjRows - 1) / kProjRows), unsigned((T + kProjTok - 1) / kProjTok));
    proj_kernel<K><<<pg, 256, 0, s>>>(xb, h->V, T, int(h->d), h->bG, h->bsx);
  }
  if constexpr (K >= 64 && K <= 256) {
    if (h->cr_F) {
      if (launch_pdl(gate_mma_kernel<K>, dim3((T + kGateMmaTok - 1) / kGateMmaTok),
                     dim3(kGateMmaThreads), gate_mma_smem<K>(), s, h->bG, h->bP, S,
                     size_t(h->max_T) * K, xb, h->cr_F, T, int(h->d), h->eps, h->bgate, gate,
                     rho, h->status, S > 0 ? static_cast<const float*>(h->bsxp) : nullptr,
                     size_t(h->max_T)) != cudaSuccess)
        return GSI_ERR_CUDA;
    } else {
      gate_kernel<K><<<(T + kGateTok - 1) / kGateTok, 256, 0, s>>>(h->bG, h->bsx, h->gram, T,
                                                                   h->eps, h->bgate, gate, rho);
    }
  } else {
    gate_kernel<K><<<(T + kGateTok - 1) / kGateTok, 256, 0, s>>>(h->bG, h->bsx, h->gram, T, h->eps,
                                                                 h->bgate, gate, rho);
  }
  if (launch_pdl(partition_gather_kernel<K>, dim3(T), dim3(256), 0, s, xb, h->bG, h->bgate, T,
                 int(h->d), int(h->max_T), h->bidx_fast, h->bidx_slow, h->bcount, h->bGf,
                 h->bXs) != cudaSuccess)
    return GSI_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

size_t batched_workspace_bytes(int64_t max_T, int64_t d, int64_t k) {
  size_t b = 0;
  b += align256(size_t(max_T) * k * 4);      // bG
  b += align256(size_t(max_T) * 4);          // bsx
  b += align256(size_t(max_T));              // bgate
  b += align256(size_t(max_T) * 4) * 2;      // idx lists
  b += align256(16);                         // counts
  b += align256(size_t(max_T) * 2 * k * 2);  // bGf
  b += align256(size_t(max_T) * d * 2);      // bXs
  if (k == 128 || k == 256) {
    b += align256(size_t(k) * d * 2);                          // bVT
    b += align256(size_t(kProjMaxSplits) * max_T * k * 4);     // bP
    b += align256(size_t(kProjMaxSplits) * max_T * 4);         // bsxp
  }
  return b;
}

// The MMA gate kernel's shared memory exceeds the default 48 KB for k = 256:
// raise its limit once per function (a property of the function, not of a
// handle).
template <int K>
bool gate_mma_prepare() {
  static bool done = false;
  if (!done)
    done = cudaFuncSetAttribute(gate_mma_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(gate_mma_smem<K>())) == cudaSuccess;
  return done;
}

void batched_bind_workspace(gsi_handle* h, void* base, int64_t max_T) {
  gate_mma_prepare<64>();
  gate_mma_prepare<128>();
  gate_mma_prepare<256>();
  char* p = static_cast<char*>(base);
  auto take = [&](size_t bytes) { char* r = p; p += align256(bytes); return r; };
  h->bG = reinterpret_cast<float*>(take(size_t(max_T) * h->k * 4));
  h->bsx = reinterpret_cast<float*>(take(size_t(max_T) * 4));
  h->bgate = reinterpret_cast<uint8_t*>(take(size_t(max_T)));
  h->bidx_fast = reinterpret_cast<int32_t*>(take(size_t(max_T) * 4));
  h->bidx_slow = reinterpret_cast<int32_t*>(take(size_t(max_T) * 4));
  h->bcount = reinterpret_cast<int32_t*>(take(16));
  h->bGf = reinterpret_cast<__nv_bfloat16*>(take(size_t(max_T) * 2 * h->k * 2));
  h->bXs = reinterpret_cast<__nv_bfloat16*>(take(size_t(max_T) * h->d * 2));
  h->bVT = nullptr;
  h->bP = nullptr;
  h->bsxp = nullptr;
  if (h->k == 128 || h->k == 256) {
    h->bVT = reinterpret_cast<__nv_bfloat16*>(take(size_t(h->k) * h->d * 2));
    h->bP = reinterpret_cast<float*>(take(size_t(kProjMaxSplits) * max_T * h->k * 4));
    h->bsxp = reinterpret_cast<float*>(take(size_t(kProjMaxSplits) * max_T * 4));
  }
  h->max_T = max_T;
}

int batched_launch_count(const gsi_handle* h, int64_t T) {
  (void)h;
  return T > 1 ? 3 + tc_gemm_launch_count() : 0;
}

gsi_status_t batched_prepare(gsi_handle* h) {
  if (h->bVT) {
    dim3 grid(unsigned((h->k + 31) / 32), unsigned((h->d + 31) / 32));
    transpose_kernel<<<grid, 256>>>(h->V, int(h->d), int(h->k), h->bVT);
    if (cudaGetLastError() != cudaSuccess) return GSI_ERR_CUDA;
  }
  return tc_proj_prepare(h);
}

gsi_status_t batched_launch(gsi_handle* h, const void* x, int64_t T, float* y, uint8_t* gate,
                            float* rho, cudaStream_t s) {
  gsi_status_t st;
  switch (h->k) {
    case 16: st = launch_front<16>(h, x, int(T), gate, rho, s); break;
    case 32: st = launch_front<32>(h, x, int(T), gate, rho, s); break;
    case 64: st = launch_front<64>(h, x, int(T), gate, rho, s); break;
    case 128: st = launch_front<128>(h, x, int(T), gate, rho, s); break;
    case 256: st = launch_front<256>(h, x, int(T), gate, rho, s); break;
    case 512: st = launch_front<512>(h, x, int(T), gate, rho, s); break;
    default: return GSI_ERR_UNSUPPORTED_SHAPE;
  }
  if (st != GSI_OK) return st;
  TcGemmArgs g;
  g.W = h->W;
  g.M = h->M;
  g.Gf = h->bGf;
  g.Xs = h->bXs;
  g.idx_fast = h->bidx_fast;
  g.idx_slow = h->bidx_slow;
  g.count = h->bcount;
  g.tile_counter = h->bcount + 2;
  g.y = y;
  g.T = int(T);
  g.d_out = int(h->d_out);
  g.d = int(h->d);
  g.k = int(h->k);
  g.status = h->status;
  return tc_gemm_launch(h, g, s);
}

}  // namespace gsi
