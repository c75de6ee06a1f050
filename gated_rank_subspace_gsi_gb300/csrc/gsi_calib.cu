// gsi_calib.cu -- calibration of the rank-k basis V_k on the GPU.
//
// Page: "Technical summary: Gated Subspace Inference for transformer
// acceleration" [GSI], section 2.3: the basis is computed once from one
// forward pass over a representative calibration sequence; the page names no
// algorithm.  Here V_k spans the top-k eigenvectors of the uncentred second
// moment C = X^T X of the n calibration tokens X (n x d) -- the rank-k
// subspace with the least summed squared residual r of section 2.1 (eq. 1)
// -- approached by block power iteration from a caller-supplied start block.
// One iteration, with every block stored transposed (k rows) so that both
// operands of each GEMM are K-major rows for the tensor maps:
//
//   Z^T = Q^T X^T          tcgen05 split-K GEMM: A = X (n x d), B = Q^T, K = d
//   Y^T = Z^T X            tcgen05 split-K GEMM: A = X^T (d x n), B = Z^T, K = n
//   Q^T = orth(Y^T)        CholeskyQR in fp32 on the k x d block:
//                            G = Y^T Y;  D = diag(G)^(-1/2);
//                            D G D + s I = L L^T;  Q^T = L^-1 D Y^T
//
// The orthonormalisation runs twice (CholeskyQR2).  The first pass adds a
// small shift s to the unit-diagonal Gram matrix, so that it cannot break
// down on an ill-conditioned block; its triangular transform still preserves
// the span exactly.  The second, unshifted pass restores orthonormality.  In
// the middle of the iteration only the span matters, so the second pass runs
// only when the first one's smallest pivot says its block is far from
// orthonormal (a device flag; the kernels of a skipped pass return at once).
// The last iteration always runs both passes and writes V_k (d x k, bf16).
//
// Kernels: a bf16 transpose, the tcgen05 GEMM of gsi_tc_gemm.cu, a fixed-order
// sum of split-K partials, the Gram matrix (fp32 CUDA cores, split over d,
// deterministic last-CTA reduction), a one-CTA blocked Cholesky with the
// inverses of its 32 x 32 diagonal blocks (k <= 256: the lower triangle fits
// in shared memory), and a blocked forward substitution that applies L^-1 D
// to 32-column slices of the block.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gsi.h"
#include "gsi_device.cuh"
#include "gsi_internal.h"
#include "gsi_tc_gemm.h"

namespace gsi {
namespace {

constexpr uint32_t kStatusRank = 4u;      // a vanished column or a pivot below the floor
constexpr int kCB = 32;                   // Cholesky block edge
constexpr int kCalMaxK = 256;             // lower triangle of k x k fp32 in shared memory
constexpr int kCalMaxNb = kCalMaxK / kCB;
constexpr int kBlk = kCB * (kCB + 1);     // one 32 x 33 block (padded rows)
constexpr int kPtStride = 36;             // row stride of transposed panel blocks (16-byte rows)
constexpr int kPtBlk = kCB * kPtStride;
constexpr float kShift1 = 1.0f / 8192.0f;        // first-pass shift on the unit diagonal
constexpr float kPivotSkip2 = 1.0f / 4096.0f;    // first-pass pivots all above this: skip pass 2
constexpr float kPivotFloor = 1.0f / 1048576.0f; // a pivot below this: breakdown (status)

__host__ __device__ constexpr int tri(int n) { return n * (n + 1) / 2; }

// index (I, J), I >= J, of lower block number p in row-major packed order
__device__ __forceinline__ void unpack_tri(int p, int& I, int& J) {
  I = 0;
  while (tri(I + 1) <= p) ++I;
  J = p - tri(I);
}

// Control words at the start of the workspace (one 256-byte line each group).
struct CalCtl {
  uint32_t status;        // kStatus* bits
  int32_t need2;          // set by a first pass whose block needs the second pass
  uint32_t pad[62];
  uint32_t counters[64];  // Gram last-CTA tickets, one per 32 x 32 tile
};
static_assert(sizeof(CalCtl) == 512, "control block layout");

// ---- bf16 transpose: out (cols x rows) = in (rows x cols)^T -----------------
template <typename OutT>
__device__ __forceinline__ void store_val(OutT* p, float v);
template <>
__device__ __forceinline__ void store_val<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_val<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename OutT>
__global__ void __launch_bounds__(256) cal_transpose_kernel(const __nv_bfloat16* in,
                                                            int rows, int cols,
                                                            OutT* out) {
  __shared__ float tile[32][33];
  pdl_launch_dependents();
  pdl_wait();
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int q = threadIdx.x; q < 1024; q += 256) {
    const int r = q >> 5, c = q & 31;
    tile[r][c] = (r0 + r < rows && c0 + c < cols)
                     ? __bfloat162float(in[size_t(r0 + r) * cols + c0 + c])
                     : 0.f;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < 1024; q += 256) {
    const int r = q >> 5, c = q & 31;  // out row c0 + r, column r0 + c
    if (c0 + r < cols && r0 + c < rows) store_val(&out[size_t(c0 + r) * rows + r0 + c], tile[c][r]);
  }
}

// ---- sum of S split-K partials, fixed order (count % 4 == 0) ---------------
template <typename OutT>
__global__ void __launch_bounds__(256) cal_sum_kernel(const float* P, int S,
                                                      size_t stride, size_t count,
                                                      OutT* out) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t n4 = count / 4;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += size_t(gridDim.x) * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(P)[i];
    for (int s = 1; s < S; ++s) {
      const float4 v = reinterpret_cast<const float4*>(P + size_t(s) * stride)[i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    store_val(&out[4 * i + 0], acc.x);
    store_val(&out[4 * i + 1], acc.y);
    store_val(&out[4 * i + 2], acc.z);
    store_val(&out[4 * i + 3], acc.w);
  }
}

// ---- Gram matrix G = Q Q^T of a k x d fp32 block (lower 32 x 32 tiles) -----
// Grid (tri(nb) tiles, S slices of d).  Each CTA sums one tile over one slice
// (four groups of 64 threads over interleaved columns, each thread a 4 x 4
// patch), writes its partial, and the last CTA of the tile to arrive adds the
// S partials in slice order and stores the tile of G (kp x kp).
constexpr int kGThreads = 256;
constexpr int kGChunk = 64;

__global__ void __launch_bounds__(kGThreads) cal_gram_kernel(const float* Q, int k,
                                                             int d, int cs, float* Gp,
                                                             float* G, int kp,
                                                             CalCtl* ctl,
                                                             uint32_t* counters,
                                                             int only_if_need2) {
  __shared__ __align__(16) float As[kGChunk][kPtStride];
  __shared__ __align__(16) float Bs[kGChunk][kPtStride];
  __shared__ float red[3][kCB][kCB + 1];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();
  if (only_if_need2 && *reinterpret_cast<volatile int32_t*>(&ctl->need2) == 0) return;
  const int p = blockIdx.x, sl = blockIdx.y, S = gridDim.y;
  int I, J;
  unpack_tri(p, I, J);
  const int tid = threadIdx.x, g = tid >> 6, u = tid & 63, ty = u >> 3, tx = u & 7;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int c_begin = sl * cs, c_end = min(d, c_begin + cs);
  // the next chunk is loaded into registers while the current one is used
  constexpr int kPer = kCB * kGChunk / kGThreads;  // 8 elements per operand
  float na[kPer], nbv[kPer];
  auto fetch = [&](int c0) {
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int q = tid + u * kGThreads, r = q / kGChunk, col = c0 + q % kGChunk;
      const int ra = I * kCB + r, rb = J * kCB + r;
      const bool okc = col < c_end;
      na[u] = (okc && ra < k) ? Q[size_t(ra) * d + col] : 0.f;
      nbv[u] = (okc && rb < k) ? Q[size_t(rb) * d + col] : 0.f;
    }
  };
  if (c_begin < c_end) fetch(c_begin);
  for (int c0 = c_begin; c0 < c_end; c0 += kGChunk) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int q = tid + u * kGThreads, r = q / kGChunk, m = q % kGChunk;
      As[m][r] = na[u];
      Bs[m][r] = nbv[u];
    }
    __syncthreads();
    if (c0 + kGChunk < c_end) fetch(c0 + kGChunk);
#pragma unroll 4
    for (int m = g; m < kGChunk; m += 4) {
      const float4 a = *reinterpret_cast<const float4*>(&As[m][4 * ty]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[m][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  if (g > 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) red[g - 1][4 * ty + i][4 * tx + j] = acc[i][j];
  }
  __syncthreads();
  float* part = Gp + (size_t(p) * S + sl) * (kCB * kCB);
  if (g == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 4 * ty + i, c = 4 * tx + j;
        part[r * kCB + c] = ((acc[i][j] + red[0][r][c]) + red[1][r][c]) + red[2][r][c];
      }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&counters[p], 1u) == unsigned(S - 1)) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int e = tid; e < kCB * kCB; e += kGThreads) {
    float v = 0.f;
    for (int s2 = 0; s2 < S; ++s2) v += __ldcg(&Gp[(size_t(p) * S + s2) * (kCB * kCB) + e]);
    G[size_t(I * kCB + (e >> 5)) * kp + J * kCB + (e & 31)] = v;
  }
  if (tid == 0) counters[p] = 0;
}

// ---- one-CTA blocked Cholesky of D G D + shift I -----------------------------
// Right-looking over 32-wide block columns.  Shared memory holds the lower
// blocks (32 x 33 rows), the current panel transposed (for the register-tiled
// trailing update) and the inverse of the current diagonal block.  Outputs:
// L (kp x kp, lower blocks; rows/cols >= k padded with the identity), the
// inverses of its diagonal blocks (nb x 32 x 32), D (kp; 0 past k).  Pivots
// below kPivotFloor (or NaN) are replaced by 1 and raise kStatusRank; a first
// pass whose pivots are all >= kPivotSkip2 leaves need2 = 0.
constexpr int kCThreads = 512;

size_t chol_smem_bytes(int nb) {
  return size_t(tri(nb)) * kBlk * 4 + size_t(std::max(1, nb - 1)) * kPtBlk * 4 + 2 * size_t(kPtBlk) * 4 +
         size_t(nb) * kCB * 4 + size_t(kCB) * 4;
}

// Factor the diagonal block AJJ in place (lower triangle, zeros above); one
// warp.  Also writes 1 / L_ii to Dinv (32, shared) and the columns of L_JJ to
// LR (below) for the panel's forward substitution, and flags pivots below
// the floor (replaced by 1) and below the skip threshold.
//
// Lane i keeps row i in registers; the 32 steps are unrolled, so step c
// updates only the columns m > c that are still live.  Column c of L is
// published through row c of LR (32 x kPtStride, shared scratch) and read
// back as 16-byte broadcasts.  The next pivot is lane c + 1's diagonal entry
// after step c, which needs only that lane's own new entry of L: its
// broadcast and square root start before the column broadcast and overlap
// it.  The arithmetic (each entry's updates, in step order) is that of plain
// right-looking elimination.
__device__ __forceinline__ void chol_diag_factor(float* AJJ, float* Dinv, float* LR, int lane,
                                                 int* s_bad, int* s_small) {
  constexpr unsigned kAll = 0xffffffffu;
  // Start converged: a warp that arrives here split (after lane-divergent
  // code) would run every shuffle below as a rendezvous of its splits, which
  // costs about 25x the converged loop.
  __syncwarp();
  float a[kCB];
#pragma unroll
  for (int m = 0; m < kCB; ++m) a[m] = AJJ[lane * (kCB + 1) + m];
  bool bad = false, small = false;
  float piv = __shfl_sync(kAll, a[0], 0);
#pragma unroll
  for (int c = 0; c < kCB; ++c) {
    // piv: A[c][c] after the updates of steps 0 .. c - 1
    if (!(piv >= kPivotFloor)) {
      bad = true;
      piv = 1.f;
    }
    if (piv < kPivotSkip2) small = true;
    // rsqrtf's error (a few ulp) scales column c of L by 1 + O(1e-7): the
    // span of the transformed block does not change and its orthonormality
    // moves by that much, far below the fp32 Gram matrix's own rounding
    const float inv = rsqrtf(piv);
    const float l = (lane == c) ? piv * inv : ((lane > c) ? a[c] * inv : 0.f);
    if (lane == c) Dinv[c] = inv;
    AJJ[lane * (kCB + 1) + c] = l;
    if (c + 1 < kCB) {
      // lane c + 1: its entry c + 1 after this step (the same fma as below)
      const float pn = fmaf(-l, l, a[c + 1]);
      const float piv_next = __shfl_sync(kAll, pn, c + 1);
      float* row = LR + c * kPtStride;  // row c: L[m][c] at m
      row[lane] = l;
      __syncwarp();
#pragma unroll
      for (int m4 = ((c + 1) / 4) * 4; m4 < kCB; m4 += 4) {
        const float4 q = *reinterpret_cast<const float4*>(row + m4);
        if (m4 + 0 > c) a[m4 + 0] = fmaf(-l, q.x, a[m4 + 0]);
        if (m4 + 1 > c) a[m4 + 1] = fmaf(-l, q.y, a[m4 + 1]);
        if (m4 + 2 > c) a[m4 + 2] = fmaf(-l, q.z, a[m4 + 2]);
        if (m4 + 3 > c) a[m4 + 3] = fmaf(-l, q.w, a[m4 + 3]);
      }
      piv = piv_next;
    }
  }
  if (lane == 0) {
    if (bad) *s_bad = 1;
    if (small) *s_small = 1;
  }
  __syncwarp();
}

// Inverse of a factored 32 x 32 diagonal block (AJJ, rows of 33) by forward
// substitution on the unit vectors, written to LIg (row-major 32 x 32); one
// warp, lane j owning column j as a sliding window (x[m] holds entry i + m at
// step i).  The block's columns are first copied to R (32 x kPtStride,
// shared scratch) rotated as in chol_diag_factor, so that each step reads
// them as 16-byte broadcasts.  Off the factorisation's critical path: only
// the forward substitution kernel that follows reads these.
__device__ __forceinline__ void chol_diag_inverse(const float* AJJ, float* R, float* LIg, int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  __syncwarp();
  for (int c = 0; c < kCB; ++c) R[c * kPtStride + ((lane - c - 1) & (kCB - 1))] = AJJ[lane * (kCB + 1) + c];
  const float my_inv = 1.0f / AJJ[lane * (kCB + 1) + lane];
  __syncwarp();
  float x[kCB];
#pragma unroll
  for (int m = 0; m < kCB; ++m) x[m] = (m == lane) ? 1.f : 0.f;
#pragma unroll 1
  for (int i = 0; i < kCB; ++i) {
    const float xi = x[0] * __shfl_sync(kAll, my_inv, i);
    LIg[i * kCB + lane] = xi;
    const float* row = R + i * kPtStride;
#pragma unroll
    for (int m4 = 0; m4 < kCB; m4 += 4) {
      const float4 q = *reinterpret_cast<const float4*>(row + m4);
      x[m4 + 1] = fmaf(-q.x, xi, x[m4 + 1]);
      if (m4 + 2 < kCB) x[m4 + 2] = fmaf(-q.y, xi, x[m4 + 2]);
      if (m4 + 3 < kCB) x[m4 + 3] = fmaf(-q.z, xi, x[m4 + 3]);
      if (m4 + 4 < kCB) x[m4 + 4] = fmaf(-q.w, xi, x[m4 + 4]);
    }
#pragma unroll
    for (int m = 0; m + 1 < kCB; ++m) x[m] = x[m + 1];
  }
}

__global__ void __launch_bounds__(kCThreads, 1)
    cal_chol_kernel(const float* G, int k, int kp, float shift, int first_pass,
                    float* Lg, float* LIg, float* Dg,
                    CalCtl* ctl, int only_if_need2) {
  extern __shared__ __align__(16) float csm[];
  __shared__ int s_bad;
  __shared__ int s_small;
  pdl_launch_dependents();
  pdl_wait();
  if (only_if_need2 && *reinterpret_cast<volatile int32_t*>(&ctl->need2) == 0) return;
  const int nb = kp / kCB, np = tri(nb);
  float* A = csm;
  float* PT = A + size_t(np) * kBlk;
  float* LN = PT + size_t(max(1, nb - 1)) * kPtBlk;  // scratch for the diagonal-block inverses
  float* LTd = LN + kPtBlk;                            // current diagonal block of L: row c = column c
  float* Ds = LTd + kPtBlk;                            // D (kp), then 1 / L_ii of the block (32)
  float* Dinv = Ds + kp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kWarps = kCThreads / 32;
  if (tid == 0) {
    s_bad = 0;
    s_small = 0;
  }
  __syncthreads();
  for (int i = tid; i < kp; i += kCThreads) {
    float dv = 0.f;
    if (i < k) {
      const float gii = G[size_t(i) * kp + i];
      if (gii > 0.f && gii <= 3.0e38f)
        dv = 1.0f / sqrtf(gii);
      else
        s_bad = 1;
    }
    Ds[i] = dv;
    Dg[i] = dv;
  }
  __syncthreads();
  // row i of the lower blocks (columns 0 .. 32 (I + 1) - 1, the diagonal
  // block in full) is contiguous in G: one warp per row, all loads first
  for (int i0 = warp; i0 < kp; i0 += 2 * kWarps) {
    float v[2][kCalMaxNb];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = i0 + h * kWarps, ncol = ((i >> 5) + 1) * kCB;
#pragma unroll
      for (int u = 0; u < kCalMaxNb; ++u) {
        const int j = u * kCB + lane;
        v[h][u] = (i < kp && j < ncol && i < k && j < k) ? G[size_t(i) * kp + j] : 0.f;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = i0 + h * kWarps;
      if (i >= kp) break;
      const int I = i >> 5, r = i & 31, ncol = (I + 1) * kCB;
      const float di = Ds[i];
#pragma unroll
      for (int u = 0; u < kCalMaxNb; ++u) {
        const int j = u * kCB + lane;
        if (j >= ncol) break;
        float a = v[h][u] * di * Ds[j];
        if (i == j) a = (i < k && di > 0.f) ? a + shift : 1.f;
        A[size_t(tri(I) + u) * kBlk + r * (kCB + 1) + lane] = a;
      }
    }
  }
  __syncthreads();

  // step J: the panel below diagonal block J, the trailing update, and (warp
  // 0, overlapped with the update) the factorisation of diagonal block J + 1;
  // step -1 only factors block 0
  for (int J = -1; J < nb; ++J) {
    if (J >= 0) {
      // panel: L_IJ solves L_IJ L_JJ^T = A_IJ for the block rows below, by
      // forward substitution: one warp per block row, lane r holding row r
      // (a, then the solution x) in registers.  Right-looking and unrolled:
      // x[c] is final once columns 0 .. c - 1 are eliminated, and then updates
      // the live columns m > c with column c of L_JJ (row c of LTd, 16-byte
      // broadcasts), so each step is a few independent FMAs rather than a
      // dot product over all earlier columns.  The result goes to L (global)
      // and, transposed, to PT for the trailing update; A_IJ itself is not
      // needed again.
      for (int I = J + 1 + warp; I < nb; I += kWarps) {
        const float* AIJ = A + size_t(tri(I) + J) * kBlk;
        float x[kCB];
#pragma unroll
        for (int m = 0; m < kCB; ++m) x[m] = AIJ[lane * (kCB + 1) + m];
#pragma unroll
        for (int c = 0; c < kCB; ++c) {
          x[c] *= Dinv[c];
          if (c + 1 < kCB) {
            const float* col = LTd + c * kPtStride;  // L_JJ[m][c] at m
#pragma unroll
            for (int m4 = ((c + 1) / 4) * 4; m4 < kCB; m4 += 4) {
              const float4 q = *reinterpret_cast<const float4*>(col + m4);
              if (m4 + 0 > c) x[m4 + 0] = fmaf(-x[c], q.x, x[m4 + 0]);
              if (m4 + 1 > c) x[m4 + 1] = fmaf(-x[c], q.y, x[m4 + 1]);
              if (m4 + 2 > c) x[m4 + 2] = fmaf(-x[c], q.z, x[m4 + 2]);
              if (m4 + 3 > c) x[m4 + 3] = fmaf(-x[c], q.w, x[m4 + 3]);
            }
          }
        }
        float* pt = PT + size_t(I - J - 1) * kPtBlk;
#pragma unroll
        for (int c = 0; c < kCB; ++c) pt[c * kPtStride + lane] = x[c];
        __syncwarp();
        // the block to L in global memory, one coalesced row per step
        for (int r = 0; r < kCB; ++r)
          Lg[size_t(I * kCB + r) * kp + J * kCB + lane] = pt[lane * kPtStride + r];
      }
      __syncthreads();
      // trailing update A_IL -= L_IJ L_LJ^T, J < L <= I; one warp per block pair,
      // each lane a 4 x 8 patch
      const int n1 = nb - 1 - J;
      const int lr = lane >> 2, lc = lane & 3;
      // warp 0 updates block (J+1, J+1) first and factors it while the other
      // warps update the rest (pairs 1.. over warps 1..)
      for (int pp = (warp == 0) ? 0 : warp; pp < tri(n1); pp += (warp == 0) ? tri(n1) : kWarps - 1) {
        int Ip, Lp;
        unpack_tri(pp, Ip, Lp);
        const float* PI = PT + size_t(Ip) * kPtBlk;
        const float* PL = PT + size_t(Lp) * kPtBlk;
        float acc[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 4
        for (int m = 0; m < kCB; ++m) {
          const float4 av = *reinterpret_cast<const float4*>(PI + m * kPtStride + 4 * lr);
          const float4 b0 = *reinterpret_cast<const float4*>(PL + m * kPtStride + 8 * lc);
          const float4 b1 = *reinterpret_cast<const float4*>(PL + m * kPtStride + 8 * lc + 4);
          const float a4[4] = {av.x, av.y, av.z, av.w};
          const float b8[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a4[i], b8[j], acc[i][j]);
        }
        float* AIL = A + size_t(tri(J + 1 + Ip) + J + 1 + Lp) * kBlk;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) AIL[(4 * lr + i) * (kCB + 1) + 8 * lc + j] -= acc[i][j];
      }
    }
    if (warp == 0 && J + 1 < nb)
      chol_diag_factor(A + size_t(tri(J + 1) + J + 1) * kBlk, Dinv, LTd, lane, &s_bad,
                       &s_small);
    __syncthreads();
  }
  // the inverses of the diagonal blocks, one warp each, for the forward
  // substitution kernel
  // (scratch: the panel buffer PT, then LN and LTd, contiguous: nb + 1 blocks)
  for (int J = warp; J < nb; J += kWarps)
    chol_diag_inverse(A + size_t(tri(J) + J) * kBlk, PT + size_t(J) * kPtBlk,
                      LIg + size_t(J) * kCB * kCB, lane);
  // the diagonal blocks of L (the panels went to Lg as they were formed)
  for (int q = tid; q < nb * kCB * kCB; q += kCThreads) {
    const int J = q >> 10, e = q & 1023, r = e >> 5, c = e & 31;
    Lg[size_t(J * kCB + r) * kp + J * kCB + c] = A[size_t(tri(J) + J) * kBlk + r * (kCB + 1) + c];
  }
  if (tid == 0) {
    if (s_bad) atomicOr(&ctl->status, kStatusRank);
    if (first_pass) ctl->need2 = s_small ? 1 : 0;
  }
}

// ---- apply: Q^T[:, slice] = L^-1 D Y^T[:, slice] (blocked forward substitution)
// One CTA per 32 columns of d.  The CTA first stages all of L it needs in
// shared memory -- the panels left of each diagonal block, transposed, and
// the inverses of the diagonal blocks, transposed -- with every load in
// flight at once, then runs the substitution from shared memory only: block
// row I of the D-scaled slice is updated by the blocks to its left and
// multiplied by the inverse of L_II.  Outputs (any may be null): outF fp32
// k x d, outB bf16 k x d, outV bf16 d x k (the basis layout).
constexpr int kAThreads = 256;
constexpr int kACols = 32;

size_t apply_smem_bytes(int nb) {
  return size_t(nb) * kCB * (kACols + 1) * 4        // slice
         + size_t(tri(nb - 1)) * kPtBlk * 4         // panels left of the diagonal, transposed
         + size_t(nb) * kPtBlk * 4                  // inverses of the diagonal blocks, transposed
         + size_t(kCB) * (kACols + 1) * 4;          // block row before its inverse
}

__global__ void __launch_bounds__(kAThreads)
    cal_apply_kernel(const float* Y, int k, int d, int kp, const float* Dg,
                     const float* Lg, const float* LIg,
                     float* outF, __nv_bfloat16* outB,
                     __nv_bfloat16* outV, const CalCtl* ctl,
                     int only_if_need2) {
  extern __shared__ __align__(16) float asm_[];
  pdl_launch_dependents();
  pdl_wait();
  if (only_if_need2 && *reinterpret_cast<const volatile int32_t*>(&ctl->need2) == 0) return;
  const int nb = kp / kCB;
  float* Xs = asm_;                                     // kp x 33
  float* LT = Xs + size_t(kp) * (kACols + 1);           // panel I at kPtBlk * tri(I - 1): [32 I][36]
  float* LIt = LT + size_t(tri(nb - 1)) * kPtBlk;       // nb x [32][36]
  float* Ts = LIt + size_t(nb) * kPtBlk;                // 32 x 33
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = blockIdx.x * kACols;
  const bool col_ok = c0 + lane < d;
  for (int r = warp; r < kp; r += kAThreads / 32)
    Xs[r * (kACols + 1) + lane] = (r < k && col_ok) ? Dg[r] * Y[size_t(r) * d + c0 + lane] : 0.f;
  // L panels: row r of block row I, columns 0 .. 32 I - 1, as float4
  for (int I = 1; I < nb; ++I) {
    float* dst = LT + size_t(tri(I - 1)) * kPtBlk;
    const int w4 = I * kCB / 4;
#pragma unroll 4
    for (int q = tid; q < kCB * w4; q += kAThreads) {
      const int r = q / w4, m = 4 * (q % w4);
      const float4 l4 = *reinterpret_cast<const float4*>(&Lg[size_t(I * kCB + r) * kp + m]);
      dst[(m + 0) * kPtStride + r] = l4.x;
      dst[(m + 1) * kPtStride + r] = l4.y;
      dst[(m + 2) * kPtStride + r] = l4.z;
      dst[(m + 3) * kPtStride + r] = l4.w;
    }
  }
#pragma unroll 4
  for (int q = tid; q < nb * kCB * kCB / 4; q += kAThreads) {
    const int I = q >> 8, e = 4 * (q & 255), r = e >> 5, m = e & 31;
    const float4 l4 = *reinterpret_cast<const float4*>(&LIg[size_t(I) * kCB * kCB + e]);
    float* dst = LIt + size_t(I) * kPtBlk;
    dst[(m + 0) * kPtStride + r] = l4.x;
    dst[(m + 1) * kPtStride + r] = l4.y;
    dst[(m + 2) * kPtStride + r] = l4.z;
    dst[(m + 3) * kPtStride + r] = l4.w;
  }
  __syncthreads();
  for (int I = 0; I < nb; ++I) {
    const int w = kCB * I;  // columns of L left of the diagonal block
    const float* Lp = LT + size_t(tri(I - 1)) * kPtBlk;
    float acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = Xs[(I * kCB + 4 * warp + q) * (kACols + 1) + lane];
#pragma unroll 8
    for (int m = 0; m < w; ++m) {
      const float4 l4 = *reinterpret_cast<const float4*>(Lp + m * kPtStride + 4 * warp);
      const float x = Xs[m * (kACols + 1) + lane];
      acc[0] = fmaf(-l4.x, x, acc[0]);
      acc[1] = fmaf(-l4.y, x, acc[1]);
      acc[2] = fmaf(-l4.z, x, acc[2]);
      acc[3] = fmaf(-l4.w, x, acc[3]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) Ts[(4 * warp + q) * (kACols + 1) + lane] = acc[q];
    __syncthreads();
    const float* Li = LIt + size_t(I) * kPtBlk;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int m = 0; m < kCB; ++m) {
      const float4 l4 = *reinterpret_cast<const float4*>(Li + m * kPtStride + 4 * warp);
      const float t = Ts[m * (kACols + 1) + lane];
      o[0] = fmaf(l4.x, t, o[0]);
      o[1] = fmaf(l4.y, t, o[1]);
      o[2] = fmaf(l4.z, t, o[2]);
      o[3] = fmaf(l4.w, t, o[3]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) Xs[(I * kCB + 4 * warp + q) * (kACols + 1) + lane] = o[q];
    __syncthreads();
  }
  if (outF || outB) {
    for (int r = warp; r < k; r += kAThreads / 32) {
      if (!col_ok) continue;
      const float v = Xs[r * (kACols + 1) + lane];
      if (outF) outF[size_t(r) * d + c0 + lane] = v;
      if (outB) outB[size_t(r) * d + c0 + lane] = __float2bfloat16_rn(v);
    }
  }
  if (outV) {
    // row c0 + c of V holds column c of the slice; lanes cover pairs of rows r
    for (int c = warp; c < kACols; c += kAThreads / 32) {
      if (c0 + c >= d) continue;
      for (int r = 2 * lane; r < k; r += 64) {
        __nv_bfloat162 v2;
        v2.x = __float2bfloat16_rn(Xs[r * (kACols + 1) + c]);
        v2.y = __float2bfloat16_rn(Xs[(r + 1) * (kACols + 1) + c]);
        *reinterpret_cast<__nv_bfloat162*>(&outV[size_t(c0 + c) * k + r]) = v2;
      }
    }
  }
}

#include "gsi_rank1.cuh"

// ---- host side ----------------------------------------------------------------

struct CalLayout {
  size_t ctl, XT, QT, ZT, P1, Y, P2, Q1, Gp, G, L, LI, D, total;
};

constexpr int kMaxGramSlices = 32;

CalLayout cal_layout(int64_t n, int64_t d, int64_t k) {
  const int64_t kp = (k + kCB - 1) / kCB * kCB, nb = kp / kCB;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  CalLayout o{};
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t here = at;
    at += up(bytes);
    return here;
  };
  o.ctl = take(sizeof(CalCtl));
  o.XT = take(size_t(d) * n * 2);
  o.QT = take(size_t(k) * d * 2);
  o.ZT = take(size_t(k) * n * 2);
  o.P1 = take(size_t(kProjMaxSplits) * k * n * 4);
  o.Y = take(size_t(k) * d * 4);
  o.P2 = take(size_t(kProjMaxSplits) * k * d * 4);
  o.Q1 = take(size_t(k) * d * 4);
  o.Gp = take(size_t(kMaxGramSlices) * tri(int(nb)) * kCB * kCB * 4);
  o.G = take(size_t(kp) * kp * 4);
  o.L = take(size_t(kp) * kp * 4);
  o.LI = take(size_t(nb) * kCB * kCB * 4);
  o.D = take(size_t(kp) * 4);
  o.total = at;
  return o;
}

bool cal_shape_ok(int64_t n, int64_t d, int64_t k) {
  const bool k_ok = k == 16 || k == 32 || k == 64 || k == 128 || k == 256;
  return k_ok && d >= k && n >= k && d % 8 == 0 && n % 8 == 0 && d <= (int64_t(1) << 30) &&
         n <= (int64_t(1) << 30) && size_t(d) * size_t(n) <= (size_t(1) << 40);
}

// Optional per-launch timing (gsi_calibrate_timed): an event pair around
// every kernel launch, on the launching stream.
enum CalKind { kKindTranspose = 0, kKindGemm, kKindSum, kKindGram, kKindChol, kKindApply };
struct CalTimer {
  std::vector<cudaEvent_t> ev;  // start, stop per launch
  std::vector<int> kind;
  bool failed = false;
  void begin(int kd, cudaStream_t s) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
      failed = true;
      return;
    }
    ev.push_back(a);
    ev.push_back(b);
    kind.push_back(kd);
    if (cudaEventRecord(a, s) != cudaSuccess) failed = true;
  }
  void end(cudaStream_t s) {
    if (!ev.empty() && cudaEventRecord(ev.back(), s) != cudaSuccess) failed = true;
  }
  ~CalTimer() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
  }
};

struct CalRun {
  CalTimer* tm = nullptr;
  int64_t n, d, k, kp, nb;
  CalLayout lay;
  unsigned char* ws;
  CalCtl* ctl;
  int sms;
  cudaStream_t s;
  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
  void tb(int kd) const {
    if (tm) tm->begin(kd, s);
  }
  void te() const {
    if (tm) tm->end(s);
  }
};

gsi_status_t orth_pass(const CalRun& r, const float* Yin, bool first, int only_if_need2,
                       float* outF, __nv_bfloat16* outB, __nv_bfloat16* outV) {
  const int np = tri(int(r.nb));
  const int d = int(r.d);
  int S = std::max(1, std::min(kMaxGramSlices, (2 * r.sms + np - 1) / np));
  S = std::min(S, std::max(1, d / 256));
  int cs = (d + S - 1) / S;
  cs = (cs + kGChunk - 1) / kGChunk * kGChunk;
  S = (d + cs - 1) / cs;
  float* Gp = r.at<float>(r.lay.Gp);
  float* G = r.at<float>(r.lay.G);
  float* L = r.at<float>(r.lay.L);
  float* LI = r.at<float>(r.lay.LI);
  float* D = r.at<float>(r.lay.D);
  r.tb(kKindGram);
  cudaError_t e = launch_pdl(cal_gram_kernel, dim3(unsigned(np), unsigned(S)), dim3(kGThreads), 0,
                             r.s, Yin, int(r.k), d, cs, Gp, G, int(r.kp), r.ctl,
                             r.ctl->counters, only_if_need2);
  r.te();
  if (e != cudaSuccess) return GSI_ERR_CUDA;
  r.tb(kKindChol);
  e = launch_pdl(cal_chol_kernel, dim3(1), dim3(kCThreads), chol_smem_bytes(int(r.nb)), r.s,
                 (const float*)G, int(r.k), int(r.kp), first ? kShift1 : 0.f, first ? 1 : 0, L, LI, D,
                 r.ctl, only_if_need2);
  r.te();
  if (e != cudaSuccess) return GSI_ERR_CUDA;
  const unsigned ncta = unsigned((r.d + kACols - 1) / kACols);
  r.tb(kKindApply);
  e = launch_pdl(cal_apply_kernel, dim3(ncta), dim3(kAThreads), apply_smem_bytes(int(r.nb)), r.s,
                 Yin, int(r.k), d, int(r.kp), (const float*)D, (const float*)L, (const float*)LI, outF,
                 outB, outV, (const CalCtl*)r.ctl, only_if_need2);
  r.te();
  return e == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

gsi_status_t cal_prepare() {
  static bool done = false;
  if (done) return GSI_OK;
  if (cudaFuncSetAttribute(cal_chol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(chol_smem_bytes(kCalMaxNb))) != cudaSuccess ||
      cudaFuncSetAttribute(cal_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(apply_smem_bytes(kCalMaxNb))) != cudaSuccess ||
      cudaFuncSetAttribute(r1_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (kRMaxK * (kRW + 1) + kRMaxVec) * 4) != cudaSuccess)
    return GSI_ERR_CUDA;
  const gsi_status_t st = tc_nt_prepare();
  if (st != GSI_OK) return st;
  done = true;
  return GSI_OK;
}

// Launches per call, for the accounting entry point.
int cal_launches(int64_t n, int64_t d, int64_t k, int iters, int sms) {
  const int per_pass = 3;
  if (iters == 0) return 1 + 2 * per_pass;
  int kb1, kb2;
  const int S2 = tc_nt_splits(d, k, n, sms, &kb2);
  (void)tc_nt_splits(n, k, d, sms, &kb1);
  const int per_iter = 3 + (S2 > 1 ? 1 : 0) + 2 * per_pass;
  return 2 + iters * per_iter;
}

}  // namespace
}  // namespace gsi

using namespace gsi;

extern "C" {

gsi_status_t gsi_calibrate_workspace_size(int64_t n, int64_t d, int64_t k, size_t* bytes) {
  if (!bytes) return GSI_ERR_INVALID_ARG;
  *bytes = 0;
  if (!cal_shape_ok(n, d, k)) return GSI_ERR_UNSUPPORTED_SHAPE;
  *bytes = cal_layout(n, d, k).total;
  return GSI_OK;
}

int gsi_calibrate_launch_count(int64_t n, int64_t d, int64_t k, int iters) {
  if (!cal_shape_ok(n, d, k) || iters < 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return cal_launches(n, d, k, iters, sms);
}

}  // extern "C"

namespace gsi {
namespace {

gsi_status_t calibrate_impl(const void* X, int64_t n, int64_t d, int64_t k, const void* Q0,
                            int iters, void* V_k, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream, CalTimer* tm, bool clear_status = true) {
  if (!X || !Q0 || !V_k || !workspace || iters < 0 || iters > 10000) return GSI_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q0) || !aligned16(V_k) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return GSI_ERR_INVALID_ARG;
  if (!cal_shape_ok(n, d, k)) return GSI_ERR_UNSUPPORTED_SHAPE;
  CalRun r;
  r.tm = tm;
  r.n = n;
  r.d = d;
  r.k = k;
  r.kp = (k + kCB - 1) / kCB * kCB;
  r.nb = r.kp / kCB;
  r.lay = cal_layout(n, d, k);
  if (workspace_bytes < r.lay.total) return GSI_ERR_WORKSPACE;
  r.ws = static_cast<unsigned char*>(workspace);
  r.ctl = r.at<CalCtl>(r.lay.ctl);
  r.s = stream;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&r.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GSI_ERR_CUDA;
  gsi_status_t st = cal_prepare();
  if (st != GSI_OK) return st;
  // the Gram tickets return to zero after every use; the status word is
  // cleared at the start of a call (of a cascade)
  if (clear_status && cudaMemsetAsync(r.ctl, 0, sizeof(CalCtl), stream) != cudaSuccess)
    return GSI_ERR_CUDA;

  const auto* Xb = static_cast<const __nv_bfloat16*>(X);
  const auto* Q0b = static_cast<const __nv_bfloat16*>(Q0);
  auto* XT = r.at<__nv_bfloat16>(r.lay.XT);
  auto* QT = r.at<__nv_bfloat16>(r.lay.QT);
  auto* ZT = r.at<__nv_bfloat16>(r.lay.ZT);
  float* P1 = r.at<float>(r.lay.P1);
  float* Y = r.at<float>(r.lay.Y);
  float* P2 = r.at<float>(r.lay.P2);
  float* Q1 = r.at<float>(r.lay.Q1);
  auto* V = static_cast<__nv_bfloat16*>(V_k);
  uint32_t* status = &r.ctl->status;
  const dim3 tb(256);

  if (iters == 0) {
    // V_k = orth(Q0): the block itself, in fp32, through both passes
    const dim3 g(unsigned((k + 31) / 32), unsigned((d + 31) / 32));
    r.tb(kKindTranspose);
    const cudaError_t e = launch_pdl(cal_transpose_kernel<float>, g, tb, 0, stream, Q0b, int(d),
                                     int(k), Y);
    r.te();
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    if ((st = orth_pass(r, Y, true, 0, Q1, nullptr, nullptr)) != GSI_OK) return st;
    return orth_pass(r, Q1, false, 0, nullptr, nullptr, V);
  }

  {
    const dim3 gx(unsigned((d + 31) / 32), unsigned((n + 31) / 32));
    r.tb(kKindTranspose);
    cudaError_t e = launch_pdl(cal_transpose_kernel<__nv_bfloat16>, gx, tb, 0, stream, Xb, int(n),
                               int(d), XT);
    r.te();
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    const dim3 gq(unsigned((k + 31) / 32), unsigned((d + 31) / 32));
    r.tb(kKindTranspose);
    e = launch_pdl(cal_transpose_kernel<__nv_bfloat16>, gq, tb, 0, stream, Q0b, int(d), int(k), QT);
    r.te();
    if (e != cudaSuccess) return GSI_ERR_CUDA;
  }
  int kb1, kb2;
  const int S1 = tc_nt_splits(n, k, d, r.sms, &kb1);
  const int S2 = tc_nt_splits(d, k, n, r.sms, &kb2);
  const size_t kn = size_t(k) * n, kd = size_t(k) * d;
  const unsigned sum_grid1 = unsigned(std::min<size_t>(4 * size_t(r.sms), (kn / 4 + 255) / 256));
  const unsigned sum_grid2 = unsigned(std::min<size_t>(4 * size_t(r.sms), (kd / 4 + 255) / 256));
  for (int it = 0; it < iters; ++it) {
    const bool last = it + 1 == iters;
    // Z^T = Q^T X^T: P1[s][j][t]
    r.tb(kKindGemm);
    st = tc_nt_gemm(Xb, n, QT, k, d, P1, kn, S1, kb1, status, stream);
    r.te();
    if (st != GSI_OK) return st;
    r.tb(kKindSum);
    cudaError_t e = launch_pdl(cal_sum_kernel<__nv_bfloat16>, dim3(std::max(1u, sum_grid1)), tb, 0,
                               stream, (const float*)P1, S1, kn, kn, ZT);
    r.te();
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    // Y^T = Z^T X: P2[s][j][i]
    float* Ydst = (S2 > 1) ? P2 : Y;
    r.tb(kKindGemm);
    st = tc_nt_gemm(XT, d, ZT, k, n, Ydst, kd, S2, kb2, status, stream);
    r.te();
    if (st != GSI_OK) return st;
    if (S2 > 1) {
      r.tb(kKindSum);
      e = launch_pdl(cal_sum_kernel<float>, dim3(std::max(1u, sum_grid2)), tb, 0, stream,
                     (const float*)P2, S2, kd, kd, Y);
      r.te();
      if (e != cudaSuccess) return GSI_ERR_CUDA;
    }
    // CholeskyQR2 (the second pass only where needed, except at the end)
    if ((st = orth_pass(r, Y, true, 0, Q1, last ? nullptr : QT, nullptr)) != GSI_OK) return st;
    if ((st = orth_pass(r, Q1, false, last ? 0 : 1, nullptr, last ? nullptr : QT,
                        last ? V : nullptr)) != GSI_OK)
      return st;
  }
  return GSI_OK;
}

}  // namespace
}  // namespace gsi

extern "C" {

gsi_status_t gsi_calibrate(const void* X, int64_t n, int64_t d, int64_t k, const void* Q0,
                           int iters, void* V_k, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  return calibrate_impl(X, n, d, k, Q0, iters, V_k, workspace, workspace_bytes, stream, nullptr);
}

gsi_status_t gsi_calibrate_cascade(const void* const* X, int layers, int64_t n, int64_t d,
                                   int64_t k, const void* Q0, int iters_first, int iters_next,
                                   void* const* V, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  if (!X || !V || layers < 1 || iters_next < 0) return GSI_ERR_INVALID_ARG;
  for (int l = 0; l < layers; ++l) {
    if (!X[l] || !V[l]) return GSI_ERR_INVALID_ARG;
    for (int m = 0; m < l; ++m)
      if (V[m] == V[l]) return GSI_ERR_INVALID_ARG;  // each layer keeps its own basis
  }
  for (int l = 0; l < layers; ++l) {
    const gsi_status_t st =
        calibrate_impl(X[l], n, d, k, l == 0 ? Q0 : V[l - 1], l == 0 ? iters_first : iters_next,
                       V[l], workspace, workspace_bytes, stream, nullptr, l == 0);
    if (st != GSI_OK) return st;
  }
  return GSI_OK;
}

gsi_status_t gsi_calibrate_timed(const void* X, int64_t n, int64_t d, int64_t k, const void* Q0,
                                 int iters, void* V_k, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream, float* launch_ms, int* launch_kind,
                                 int max_launches, int* n_launches) {
  if (!launch_ms || !launch_kind || !n_launches || max_launches < 0) return GSI_ERR_INVALID_ARG;
  *n_launches = 0;
  CalTimer tm;
  const gsi_status_t st =
      calibrate_impl(X, n, d, k, Q0, iters, V_k, workspace, workspace_bytes, stream, &tm);
  if (st != GSI_OK) return st;
  if (tm.failed || cudaStreamSynchronize(stream) != cudaSuccess) return GSI_ERR_CUDA;
  const int cnt = int(tm.kind.size());
  for (int i = 0; i < cnt && i < max_launches; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, tm.ev[2 * i], tm.ev[2 * i + 1]) != cudaSuccess) return GSI_ERR_CUDA;
    launch_ms[i] = ms;
    launch_kind[i] = tm.kind[i];
  }
  *n_launches = std::min(cnt, max_launches);
  return GSI_OK;
}

gsi_status_t gsi_calibrate_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return GSI_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GSI_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GSI_ERR_CUDA;
  if (word & kStatusBadLaunch) return GSI_ERR_LAUNCH;
  if (word & kStatusTimeout) return GSI_ERR_TIMEOUT;
  return (word & kStatusRank) ? GSI_ERR_RANK : GSI_OK;
}

}  // extern "C"

// ---- rank-1 refinement of a start basis (the depth cascade's corrections) --

namespace gsi {
namespace {

struct R1Layout {
  CalLayout cal;
  size_t VP, G2, Gp2, cnt2, ctl, H, pn, cs2, h, r, q, c, w, part, tot, tick, total;
  int kp2, nb2, G, pstride;
};

R1Layout r1_layout(int64_t n, int64_t d, int64_t k) {
  R1Layout o{};
  o.cal = cal_layout(n, d, k);
  size_t at = o.cal.total;
  auto take = [&](size_t bytes) {
    const size_t here = at;
    at += (bytes + 255) & ~size_t(255);
    return here;
  };
  o.kp2 = int((2 * k + kCB - 1) / kCB * kCB);
  o.nb2 = o.kp2 / kCB;
  o.G = int((d + kRW - 1) / kRW);
  o.pstride = int((2 * k + 3 + 3) / 4 * 4);
  o.VP = take(size_t(2) * k * d * 4);
  o.G2 = take(size_t(o.kp2) * o.kp2 * 4);
  o.Gp2 = take(size_t(kMaxGramSlices) * tri(o.nb2) * kCB * kCB * 4);
  o.cnt2 = take(size_t(tri(o.nb2)) * 4);
  o.ctl = take(sizeof(R1Ctl));
  o.H = take(size_t(k) * k * 4);
  o.pn = take(size_t(k) * 8);
  o.cs2 = take(size_t(k) * 8);
  o.h = take(size_t(k) * 4);
  o.r = take(size_t(d) * 4);
  o.q = take(size_t(d) * 4);
  o.c = take(size_t(d) * 4);
  o.w = take(size_t(n) * 4);
  o.part = take(size_t(o.G) * o.pstride * 4);
  o.tot = take(size_t(o.pstride) * 4);
  o.tick = take(2 * 4);  // [0] the init kernel's ticket, [1] the grid barrier's counter
  o.total = at;
  return o;
}

int r1_launches(int64_t n, int64_t d, int64_t k, int corrections, int sms) {
  const int start = 1 + 2 * 3;  // transpose of V_in, CholeskyQR2
  if (corrections == 0) return start + 1;
  int kb1, kb2;
  const int S2 = tc_nt_splits(d, k, n, sms, &kb2);
  (void)tc_nt_splits(n, k, d, sms, &kb1);
  // X^T, the two products and the first sum, the second sum, Gram of [V; P], init
  const int prep = 1 + 3 + (S2 > 1 ? 1 : 0) + 1 + 1;
  return start + prep + 1;  // + the persistent launch (all corrections, then V_out)
}

gsi_status_t refine_impl(const void* X, int64_t n, int64_t d, int64_t k, const void* V_in,
                         int corrections, void* V_out, int32_t* order, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream, bool clear_status) {
  if (!X || !V_in || !V_out || !workspace || corrections < 0 || corrections > (1 << 20))
    return GSI_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(V_in) || !aligned16(V_out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      (reinterpret_cast<uintptr_t>(order) & 3u) != 0)
    return GSI_ERR_INVALID_ARG;
  if (!cal_shape_ok(n, d, k)) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (corrections > 0 && std::max(n, d) > kRMaxVec) return GSI_ERR_UNSUPPORTED_SHAPE;
  const R1Layout lay = r1_layout(n, d, k);
  if (workspace_bytes < lay.total) return GSI_ERR_WORKSPACE;
  CalRun r;
  r.n = n;
  r.d = d;
  r.k = k;
  r.kp = (k + kCB - 1) / kCB * kCB;
  r.nb = r.kp / kCB;
  r.lay = lay.cal;
  r.ws = static_cast<unsigned char*>(workspace);
  r.ctl = r.at<CalCtl>(r.lay.ctl);
  r.s = stream;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&r.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GSI_ERR_CUDA;
  gsi_status_t st = cal_prepare();
  if (st != GSI_OK) return st;
  if (clear_status && cudaMemsetAsync(r.ctl, 0, sizeof(CalCtl), stream) != cudaSuccess)
    return GSI_ERR_CUDA;
  uint32_t* cnt2 = r.at<uint32_t>(lay.cnt2);
  if (cudaMemsetAsync(cnt2, 0, size_t(tri(lay.nb2)) * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(r.at<uint32_t>(lay.tick), 0, 2 * 4, stream) !=
          cudaSuccess)
    return GSI_ERR_CUDA;

  const auto* Xb = static_cast<const __nv_bfloat16*>(X);
  auto* XT = r.at<__nv_bfloat16>(r.lay.XT);
  auto* QT = r.at<__nv_bfloat16>(r.lay.QT);
  auto* ZT = r.at<__nv_bfloat16>(r.lay.ZT);
  float* P1 = r.at<float>(r.lay.P1);
  float* Y = r.at<float>(r.lay.Y);
  float* P2 = r.at<float>(r.lay.P2);
  float* Q1 = r.at<float>(r.lay.Q1);
  float* V = r.at<float>(lay.VP);
  float* P = V + size_t(k) * d;
  uint32_t* status = &r.ctl->status;
  const dim3 tb(256);

  R1Args a{};
  a.V = V;
  a.P = P;
  a.H = r.at<float>(lay.H);
  a.pn = r.at<double>(lay.pn);
  a.cs2 = r.at<double>(lay.cs2);
  a.h = r.at<float>(lay.h);
  a.r = r.at<float>(lay.r);
  a.q = r.at<float>(lay.q);
  a.c = r.at<float>(lay.c);
  a.w = r.at<float>(lay.w);
  a.part = r.at<float>(lay.part);
  a.tot = r.at<float>(lay.tot);
  a.X = Xb;
  a.XT = XT;
  a.ctl = r.at<R1Ctl>(lay.ctl);
  a.status = status;
  a.order = order;
  a.n = int(n);
  a.d = int(d);
  a.k = int(k);
  a.G = lay.G;
  a.pstride = lay.pstride;

  // the start basis: the positive-diagonal QR factor of V_in (CholeskyQR2)
  {
    const dim3 g(unsigned((k + 31) / 32), unsigned((d + 31) / 32));
    const cudaError_t e = launch_pdl(cal_transpose_kernel<float>, g, tb, 0, stream,
                                     static_cast<const __nv_bfloat16*>(V_in), int(d), int(k), Y);
    if (e != cudaSuccess) return GSI_ERR_CUDA;
  }
  if ((st = orth_pass(r, Y, true, 0, Q1, nullptr, nullptr)) != GSI_OK) return st;
  if ((st = orth_pass(r, Q1, false, 0, V, corrections > 0 ? QT : nullptr, nullptr)) != GSI_OK)
    return st;

  const unsigned G = unsigned(lay.G);
  if (corrections > 0) {
    // P = C V = X^T (X V) on the tensor cores (V and X V rounded to bf16)
    const dim3 gx(unsigned((d + 31) / 32), unsigned((n + 31) / 32));
    cudaError_t e = launch_pdl(cal_transpose_kernel<__nv_bfloat16>, gx, tb, 0, stream, Xb, int(n),
                               int(d), XT);
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    int kb1, kb2;
    const int S1 = tc_nt_splits(n, k, d, r.sms, &kb1);
    const int S2 = tc_nt_splits(d, k, n, r.sms, &kb2);
    const size_t kn = size_t(k) * n, kd = size_t(k) * d;
    const unsigned sum_grid1 = unsigned(std::min<size_t>(4 * size_t(r.sms), (kn / 4 + 255) / 256));
    const unsigned sum_grid2 = unsigned(std::min<size_t>(4 * size_t(r.sms), (kd / 4 + 255) / 256));
    if ((st = tc_nt_gemm(Xb, n, QT, k, d, P1, kn, S1, kb1, status, stream)) != GSI_OK) return st;
    e = launch_pdl(cal_sum_kernel<__nv_bfloat16>, dim3(std::max(1u, sum_grid1)), tb, 0, stream,
                   (const float*)P1, S1, kn, kn, ZT);
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    if ((st = tc_nt_gemm(XT, d, ZT, k, n, S2 > 1 ? P2 : P, kd, S2, kb2, status, stream)) != GSI_OK)
      return st;
    if (S2 > 1) {
      e = launch_pdl(cal_sum_kernel<float>, dim3(std::max(1u, sum_grid2)), tb, 0, stream,
                     (const float*)P2, S2, kd, kd, P);
      if (e != cudaSuccess) return GSI_ERR_CUDA;
    }
    // Gram matrix of the stacked block [V; P]: H = V P^T, ||p_i||^2
    const int np2 = tri(lay.nb2);
    int S = std::max(1, std::min(kMaxGramSlices, (2 * r.sms + np2 - 1) / np2));
    S = std::min(S, std::max(1, int(d) / 256));
    int cs = int((d + S - 1) / S);
    cs = (cs + kGChunk - 1) / kGChunk * kGChunk;
    S = int((d + cs - 1) / cs);
    float* G2 = r.at<float>(lay.G2);
    e = launch_pdl(cal_gram_kernel, dim3(unsigned(np2), unsigned(S)), dim3(kGThreads), 0, stream,
                   (const float*)V, int(2 * k), int(d), cs, r.at<float>(lay.Gp2), G2, lay.kp2, r.ctl,
                   cnt2, 0);
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    e = launch_pdl(r1_init_kernel, dim3(unsigned((k + kRThreads / 32 - 1) / (kRThreads / 32))),
                   dim3(kRThreads), 0, stream, a, (const float*)G2, lay.kp2,
                   r.at<uint32_t>(lay.tick));
    if (e != cudaSuccess) return GSI_ERR_CUDA;
    // every correction in one launch whose CTAs wait on one another at grid
    // barriers: all of them must be resident at once
    const size_t dyn = (size_t(k) * (kRW + 1) + size_t(std::max(n, d))) * 4;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, r1_persistent_kernel, kRThreads,
                                                      dyn) != cudaSuccess)
      return GSI_ERR_CUDA;
    if (per_sm < 1) return GSI_ERR_UNSUPPORTED_SHAPE;
    const unsigned grid = unsigned(std::min<int64_t>(lay.G, int64_t(per_sm) * r.sms));
    e = launch_pdl(r1_persistent_kernel, dim3(grid), dim3(kRThreads), dyn, stream, a, corrections,
                   r.at<uint32_t>(lay.tick) + 1, static_cast<__nv_bfloat16*>(V_out));
    return e == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
  }
  const cudaError_t e = launch_pdl(r1_finish_kernel, dim3(G), dim3(kRThreads), 0, stream, a, 0,
                                   static_cast<__nv_bfloat16*>(V_out));
  return e == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

}  // namespace
}  // namespace gsi

extern "C" {

gsi_status_t gsi_refine_rank1_workspace_size(int64_t n, int64_t d, int64_t k, size_t* bytes) {
  if (!bytes) return GSI_ERR_INVALID_ARG;
  *bytes = 0;
  if (!cal_shape_ok(n, d, k)) return GSI_ERR_UNSUPPORTED_SHAPE;
  *bytes = r1_layout(n, d, k).total;
  return GSI_OK;
}

gsi_status_t gsi_refine_rank1(const void* X, int64_t n, int64_t d, int64_t k, const void* V_in,
                              int corrections, void* V_out, int32_t* order, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  return refine_impl(X, n, d, k, V_in, corrections, V_out, order, workspace, workspace_bytes,
                     stream, true);
}

gsi_status_t gsi_calibrate_cascade_rank1(const void* const* X, int layers, int64_t n, int64_t d,
                                         int64_t k, const void* Q0, int iters_first,
                                         int corrections, void* const* V, int32_t* order,
                                         void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
  if (!X || !V || layers < 1 || corrections < 0) return GSI_ERR_INVALID_ARG;
  for (int l = 0; l < layers; ++l) {
    if (!X[l] || !V[l]) return GSI_ERR_INVALID_ARG;
    for (int m = 0; m < l; ++m)
      if (V[m] == V[l]) return GSI_ERR_INVALID_ARG;
  }
  if (!cal_shape_ok(n, d, k)) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (workspace_bytes < r1_layout(n, d, k).total) return GSI_ERR_WORKSPACE;
  gsi_status_t st = calibrate_impl(X[0], n, d, k, Q0, iters_first, V[0], workspace,
                                   workspace_bytes, stream, nullptr, true);
  if (st != GSI_OK) return st;
  for (int l = 1; l < layers; ++l) {
    int32_t* od = order ? order + size_t(l - 1) * corrections : nullptr;
    st = refine_impl(X[l], n, d, k, V[l - 1], corrections, V[l], od, workspace, workspace_bytes,
                     stream, false);
    if (st != GSI_OK) return st;
  }
  return GSI_OK;
}

int gsi_refine_rank1_launch_count(int64_t n, int64_t d, int64_t k, int corrections) {
  if (!cal_shape_ok(n, d, k) || corrections < 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return r1_launches(n, d, k, corrections, sms);
}

}  // extern "C"
