// gsi_prep.cu -- one-off operand preparation for the GSI gated linear map.
//
//   gram:         Gm = V_k^T V_k (k x k), accumulated in fp64 and stored fp32,
//                 and the upper 16 x 16 tiles of E = Gm - I (off-diagonal
//                 tiles doubled) stored bf16 in MMA operand order: the
//                 one-barrier decode kernel's correction term g^T E g.
//                 Used by the batched path to form ||r||^2 without a second
//                 pass over V_k: ||x - V_k g||^2 = ||x||^2 - 2 g.g + g^T Gm g,
//                 an identity for any V_k (eq. 1 of section 2.1 of the page
//                 "Technical summary: Gated Subspace Inference for
//                 transformer acceleration", with g = V_k^T x).
//   precompute_M: the cached image of section 2.1, eq. 2: M = bf16(W V_k),
//                 fp32 accumulation, one round-to-nearest-even per entry.
// Neither is on the per-token path; both run once per operand set.
#include "gsi_device.cuh"
#include "gsi_internal.h"

namespace gsi {
namespace {

constexpr int kGramTile = 16;
constexpr int kGramRows = 64;

// One CTA per 16 x 16 tile of Gm; V_k rows staged 64 at a time.
__global__ void __launch_bounds__(256) gram_kernel(const __nv_bfloat16* __restrict__ V, int d, int k,
                                                   float* __restrict__ gram,
                                                   __nv_bfloat16* __restrict__ F) {
  __shared__ float sa[kGramRows][kGramTile];
  __shared__ float sb[kGramRows][kGramTile];
  const int a0 = blockIdx.y * kGramTile, b0 = blockIdx.x * kGramTile;
  const int ta = threadIdx.x / kGramTile, tb = threadIdx.x % kGramTile;
  double acc = 0.0;
  for (int i0 = 0; i0 < d; i0 += kGramRows) {
    for (int t = threadIdx.x; t < kGramRows * kGramTile; t += blockDim.x) {
      const int r = t / kGramTile, c = t % kGramTile;
      const int i = i0 + r;
      sa[r][c] = i < d ? __bfloat162float(V[size_t(i) * k + a0 + c]) : 0.f;
      sb[r][c] = i < d ? __bfloat162float(V[size_t(i) * k + b0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int r = 0; r < kGramRows; ++r) acc += double(sa[r][ta]) * double(sb[r][tb]);
    __syncthreads();
  }
  const int a = a0 + ta, b = b0 + tb;
  gram[size_t(a) * k + b] = float(acc);
  // F from the fp64 sum, so the small entries of E = Gm - I keep their precision
  if (F && blockIdx.y <= blockIdx.x) {
    const double e = acc - (a == b ? 1.0 : 0.0);
    const double f = blockIdx.y < blockIdx.x ? 2.0 * e : e;
    const int tile = corr_tile_index(blockIdx.y, blockIdx.x, k / kGramTile);
    F[size_t(tile) * 256 + corr_tile_pos(ta, tb)] = __double2bfloat16(f);
  }
}

constexpr int kMTileO = 64;  // rows of W / M per CTA
constexpr int kMTileA = 64;  // columns of V / M per CTA
constexpr int kMTileI = 32;  // reduction step

// M tile (64 x 64) per CTA, 256 threads, 4 x 4 outputs per thread.
__global__ void __launch_bounds__(256) precompute_M_kernel(const __nv_bfloat16* __restrict__ W,
                                                           const __nv_bfloat16* __restrict__ V,
                                                           __nv_bfloat16* __restrict__ M,
                                                           int d_out, int d, int k) {
  __shared__ float sw[kMTileI][kMTileO + 1];
  __shared__ float sv[kMTileI][kMTileA];
  const int o0 = blockIdx.y * kMTileO, a0 = blockIdx.x * kMTileA;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int i0 = 0; i0 < d; i0 += kMTileI) {
    for (int t = threadIdx.x; t < kMTileO * kMTileI; t += blockDim.x) {
      const int o = t / kMTileI, i = t % kMTileI;
      const int go = o0 + o, gi = i0 + i;
      sw[i][o] = (go < d_out && gi < d) ? __bfloat162float(W[size_t(go) * d + gi]) : 0.f;
    }
    for (int t = threadIdx.x; t < kMTileI * kMTileA; t += blockDim.x) {
      const int i = t / kMTileA, a = t % kMTileA;
      const int gi = i0 + i, ga = a0 + a;
      sv[i][a] = (gi < d && ga < k) ? __bfloat162float(V[size_t(gi) * k + ga]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < kMTileI; ++i) {
      float wv[4], vv[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) wv[p] = sw[i][ty * 4 + p];
#pragma unroll
      for (int q = 0; q < 4; ++q) vv[q] = sv[i][tx * 4 + q];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(wv[p], vv[q], acc[p][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int o = o0 + ty * 4 + p;
    if (o >= d_out) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = a0 + tx * 4 + q;
      if (a < k) M[size_t(o) * k + a] = __float2bfloat16_rn(acc[p][q]);
    }
  }
}

}  // namespace

gsi_status_t gram_launch(const __nv_bfloat16* V, int64_t d, int64_t k, float* gram,
                         __nv_bfloat16* F, cudaStream_t s) {
  dim3 grid(unsigned(k / kGramTile), unsigned(k / kGramTile));
  gram_kernel<<<grid, 256, 0, s>>>(V, int(d), int(k), gram, F);
  return cudaGetLastError() == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

gsi_status_t precompute_M_launch(const __nv_bfloat16* W, const __nv_bfloat16* V, __nv_bfloat16* M,
                                 int64_t d_out, int64_t d, int64_t k, cudaStream_t s) {
  dim3 grid(unsigned((k + kMTileA - 1) / kMTileA), unsigned((d_out + kMTileO - 1) / kMTileO));
  precompute_M_kernel<<<grid, 256, 0, s>>>(W, V, M, int(d_out), int(d), int(k));
  return cudaGetLastError() == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

}  // namespace gsi
