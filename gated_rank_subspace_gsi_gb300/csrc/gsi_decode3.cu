// gsi_decode3.cu -- the T = 1 (decode) path of the GSI gated linear map as one
// persistent kernel per call with ONE grid-wide exchange (k in {64, 128, 256}).
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
// (gsi_internal.h).
//
// Work split.  G co-resident CTAs (at most one per SM); CTA c owns d / G rows
// of V_k and d_out / G output rows.  Before it waits on the previous kernel
// (programmatic dependent launch) each CTA loads, with 2-D TMA tensor copies
// in the 128-byte swizzled layout, its V_k rows and its M rows (64-column
// blocks, rows rounded up to 16), plus the correction tiles with a 1-D bulk
// copy: none depends on x, so these reads overlap the previous kernel's tail.
// All three contractions run on warp-level bf16 MMAs (m16n8k16, fp32
// accumulation), their A operands read from the swizzled tiles without bank
// conflicts:
//   phase 1   partial g_c = V_c^T x_c: A = V_c^T (ldmatrix.trans), B = x_c
//             (exact in bf16); warp w owns 16 entries of g over all of the
//             CTA's rows, and adds them with vector red.add into one of
//             kCopies accumulator copies (copy c % 8, which spreads the atomic
//             traffic); ||x_c||^2 in fp32; then the grid barrier (release add,
//             acquire poll)
//   phase 2   every CTA sums the copies in a fixed order (the same g, bit for
//             bit, in every CTA, hence the same gate) and writes g's bf16
//             high part and remainder as the B operand of the MMAs below
//             (g = hi + lo to ~2^-17); then g^T E g over the correction
//             tiles, and the speculative fast-path rows M_c g (A = M_c rows
//             by ldmatrix), spread over all warps
//   phase 3   thread 0 forms rho and the gate in fp32; the CTA stores M_c g,
//             or, on the rare slow token, streams its rows of W from HBM for
//             W_c x.
// With a prefetch link (gsi_set_prefetch) the last warp also issues, right
// after the barrier, L2 prefetches of its 1 / G share of the next call's
// V_k, M and correction tiles, so the next call stages them from L2.
// The accumulators are double-buffered by a launch epoch kept on the device:
// CTA 0 zeroes the buffer the next launch uses, so no memset is needed and
// the kernel replays in a CUDA graph.
#include <cuda.h>

#include <algorithm>
#include <cfloat>
#include <cstring>

#include "gsi_device.cuh"
#include "gsi_internal.h"
#include "gsi_tc_gemm.h"

namespace gsi {
namespace {

constexpr int kThreads = 512;               // compute threads (16 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads + 32;       // + one warp that issues the L2 prefetches
constexpr int kCopies = 8;        // accumulator copies of (g, ||x||^2)
constexpr int kMaxBoxRows = 256;  // TMA box limit
constexpr int kMaxPf = 12;        // prefetch ranges (3 per handle, up to 4 handles)

struct Decode3Args {
  const __nv_bfloat16* W;
  const __nv_bfloat16* F;
  const __nv_bfloat16* x;
  float* y;
  uint8_t* gate;
  float* rho;
  int d_out, d;
  float eps;
  int rows_M, rows_V;  // rows owned per CTA
  int box_M, box_V;    // TMA box rows (multiples of 16, <= 256)
  int nbox_M, nbox_V;  // row boxes per CTA (rows staged = nbox x box)
  float* acc;          // [2][kCopies][acc_stride]
  int acc_stride;      // >= k + 1, multiple of 4
  uint32_t* bar;       // [0] arrival counter, [1] launch epoch, [2] counter base
  uint32_t* status;
  // operands of the next call to prefetch into L2 (bytes 0: none); CTA
  // pf_part0 + c of pf_parts prefetches its share of each range
  const char* pf[kMaxPf];
  uint32_t pf_bytes[kMaxPf];
  int pf_part0, pf_parts;
};

// Up to kMaxGroup one-token calls in one launch (gsi_group_forward): member m
// owns CTAs [cta0[m], cta0[m + 1]).
struct GroupMaps {
  CUtensorMap m[2 * kMaxGroup];  // V_k and M maps of each member
};
struct GroupArgs {
  Decode3Args a[kMaxGroup];
  int cta0[kMaxGroup + 1];
  int n;
};

__device__ __forceinline__ void red_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Prefetch [p, p + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// Barriers of the 16 compute warps only (named barrier 1), so that the
// prefetch warp, whose bulk-prefetch instructions can stall it for a
// microsecond or more, never holds them up.
__device__ __forceinline__ void sync_compute() {
  asm volatile("bar.sync 1, %0;" :: "n"(kThreads) : "memory");
}
__device__ __forceinline__ bool sync_compute_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r) : "r"(uint32_t(v)), "n"(kThreads) : "memory");
  return r != 0;
}
// Named barrier 2 (all kBlock threads): the compute warps arrive without
// waiting once the grid exchange is done; the prefetch warp waits for that.
__device__ __forceinline__ void signal_prefetch_warp() {
  asm volatile("bar.arrive 2, %0;" :: "n"(kBlock) : "memory");
}
__device__ __forceinline__ void wait_for_compute_warps() {
  asm volatile("bar.sync 2, %0;" :: "n"(kBlock) : "memory");
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t v;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
  return v;
}

// D += A B for one 16 x 16 (A, row-major) by 16 x 8 (B, column-major) bf16
// product with fp32 accumulation (registers in the PTX fragment layout).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// Four 8 x 8 bf16 matrices from shared memory (lane l gives the address of row
// l % 8 of matrix l / 8); register j holds matrix j, optionally transposed.
__device__ __forceinline__ uint4 ldsm_x4(uint32_t addr) {
  uint4 r;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}
__device__ __forceinline__ uint4 ldsm_x4_trans(uint32_t addr) {
  uint4 r;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

// Shared address of 16-byte chunk `chunk` (0..7) of row `row` in a block of
// 128-byte rows written by TMA's 128-byte swizzle (block base 1024-aligned).
__device__ __forceinline__ uint32_t swz(uint32_t block, int row, int chunk) {
  return block + uint32_t(row) * 128u + (uint32_t(chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ float warp_sum_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Dynamic shared-memory layout (byte offsets from a 1024-aligned base),
// identical on host and device.  sM / sV: K / 64 column blocks of
// rows x 128 bytes each (TMA swizzled).
struct Smem3 {
  size_t sM, sV, sF, xb, g, ys, yp, bfrag, total;
};
__host__ __device__ inline size_t al3(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline Smem3 smem3_layout(int K, int rowsM, int rowsV) {
  Smem3 s;
  size_t o = 0;
  s.sM = o;    o = al3(o + size_t(K / 64) * rowsM * 128, 1024);
  s.sV = o;    o = al3(o + size_t(K / 64) * rowsV * 128, 1024);
  s.sF = o;    o = al3(o + corr_tiles_elems(K) * 2, 128);
  s.xb = o;    o = al3(o + size_t(rowsV) * 2, 16);
  s.g = o;     o = al3(o + size_t(K) * 4, 16);
  s.ys = o;    o = al3(o + size_t(rowsM) * 4, 16);
  s.yp = o;    o = al3(o + size_t(kWarps) * 16 * 4, 16);
  s.bfrag = o; o = al3(o + size_t(K / 16) * 32 * 8, 128);
  s.total = o;
  return s;
}
constexpr size_t kSmemSlack = 1024;  // to align the dynamic base to 1024 bytes

// One one-token call on CTAs 0..G-1 of its own (cta = this CTA's index).
template <int K>
__device__ __forceinline__ void decode3_body(const CUtensorMap* tmV, const CUtensorMap* tmM,
                                             const Decode3Args& a, const int cta, const int G) {
  static_assert(K == 64 || K == 128 || K == 256, "k in {64, 128, 256}");
  static_assert(K < kThreads, "one compute thread is free to read ||x||^2 beside the g loads");
  constexpr int T16 = K / 16;  // 16-wide blocks of g
  constexpr int KC = K / 64;   // 64-column (128-byte) blocks of a row
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t s_bar[2];  // [0] V_k slice, [1] correction tiles and M slice
  __shared__ uint32_t s_epoch, s_base;
  __shared__ int s_ok;
  __shared__ float s_sx;
  __shared__ float s_qw[kWarps], s_ggw[kWarps];
  __shared__ float s_rho;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int rowsM = a.nbox_M * a.box_M, rowsV = a.nbox_V * a.box_V;
  const Smem3 lay = smem3_layout(K, rowsM, rowsV);
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  // Launch self-check (uniform over the grid, before any wait): a launch that
  // does not cover d and d_out or got less shared memory than its layout
  // does nothing and reports it.
  if (blockDim.x != kBlock || int64_t(G) * a.rows_M < a.d_out || int64_t(G) * a.rows_V < a.d ||
      rowsM < a.rows_M || rowsV < a.rows_V || dynamic_smem_bytes() < lay.total + pad) {
    if (cta == 0 && tid == 0) atomicOr(a.status, kStatusBadLaunch);
    return;
  }
  unsigned char* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const int m0 = cta * a.rows_M;
  const int nM = max(0, min(a.d_out, m0 + a.rows_M) - m0);
  const int v0 = cta * a.rows_V;
  const int nV = max(0, min(a.d, v0 + a.rows_V) - v0);

  __nv_bfloat16* sF = reinterpret_cast<__nv_bfloat16*>(smem + lay.sF);
  __nv_bfloat16* s_xb = reinterpret_cast<__nv_bfloat16*>(smem + lay.xb);  // [rowsV]
  float* s_g = reinterpret_cast<float*>(smem + lay.g);                    // [K]
  float* s_ys = reinterpret_cast<float*>(smem + lay.ys);                  // [rowsM]
  float* s_yp = reinterpret_cast<float*>(smem + lay.yp);                  // [kWarps][16]
  uint2* s_bfrag = reinterpret_cast<uint2*>(smem + lay.bfrag);            // [T16][32]

  // ---- prologue: stage this CTA's weights (independent of x) ------------
  const uint32_t box_bytes_M = uint32_t(a.box_M) * 128, box_bytes_V = uint32_t(a.box_V) * 128;
  const uint32_t bytes_F = uint32_t(corr_tiles_elems(K)) * 2;
  if (tid == 32) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmV)) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmM)) : "memory");
  }
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kWarps) {
    // The prefetch warp: once the compute warps are past the grid exchange
    // (the rest of the call works from shared memory), this CTA's share of the
    // next call's operands, into L2; then it exits.  Weights only: it reads
    // nothing the previous kernel writes.
    pdl_launch_dependents();
    wait_for_compute_warps();
    const uint32_t part = uint32_t(a.pf_part0 + cta), parts = uint32_t(a.pf_parts);
#pragma unroll 1
    for (int o = 0; o < kMaxPf; ++o) {
      const uint32_t bytes = a.pf_bytes[o];
      if (bytes == 0) continue;
      const uint32_t share = (bytes / 16 + parts - 1) / parts * 16;
      const uint32_t lo = min(bytes, part * share), hi = min(bytes, lo + share);
      constexpr uint32_t kPiece = 16384;
      for (uint32_t off = lo + uint32_t(lane) * kPiece; off < hi; off += 32u * kPiece)
        prefetch_l2(a.pf[o] + off, min(kPiece, hi - off));
    }
    return;
  }
  // staging issued by warp 1: fetching a tensor map's descriptor stalls the
  // issuing thread, and thread 0 must reach the dependent-launch wait first
  // Two completion groups: phase 1 needs only the V_k slice, so it does not
  // wait for the correction tiles or the (larger) M slice.
  if (tid == 32) {
    mbar_arrive_expect_tx(&s_bar[0], KC * a.nbox_V * box_bytes_V);
    for (int kc = 0; kc < KC; ++kc)
      for (int b = 0; b < a.nbox_V; ++b)
        tma_load_2d(smem + lay.sV + size_t(kc) * rowsV * 128 + size_t(b) * box_bytes_V, tmV,
                    kc * 64, v0 + b * a.box_V, &s_bar[0]);
    mbar_arrive_expect_tx(&s_bar[1], KC * a.nbox_M * box_bytes_M + bytes_F);
    constexpr uint32_t kChunk = 32768;
    const char* gF = reinterpret_cast<const char*>(a.F);
    for (uint32_t off = 0; off < bytes_F; off += kChunk)
      bulk_g2s(reinterpret_cast<char*>(sF) + off, gF + off, min(kChunk, bytes_F - off), &s_bar[1]);
    for (int kc = 0; kc < KC; ++kc)
      for (int b = 0; b < a.nbox_M; ++b)
        tma_load_2d(smem + lay.sM + size_t(kc) * rowsM * 128 + size_t(b) * box_bytes_M, tmM,
                    kc * 64, m0 + b * a.box_M, &s_bar[1]);
  }
  // work that needs neither x nor the previous kernel: the zero part of the
  // B operands (columns 2..7)
  for (int t = tid; t < T16 * 24; t += kThreads) s_bfrag[(t / 24) * 32 + 8 + t % 24] = make_uint2(0u, 0u);
  pdl_launch_dependents();
  pdl_wait();  // x and this handle's workspace are now safe to touch

  // ---- phase 1: x slice, partial g and ||x_c||^2 ---------------------------
  if (tid == 0) {
    s_epoch = ld_cg_u32(a.bar + 1);
    s_base = ld_cg_u32(a.bar + 2);
  }
  for (int i = tid; i < rowsV; i += kThreads)
    s_xb[i] = i < nV ? a.x[v0 + i] : __float2bfloat16_rn(0.f);
  bool ok = mbar_wait_bounded(&s_bar[0], 0, a.status);
  ok = sync_compute_and(ok);
  const uint32_t e = s_epoch;
  float* acc = a.acc + size_t(e & 1u) * kCopies * a.acc_stride;
  if (cta == 0) {  // clear the buffers the next launch accumulates into
    float* nxt = a.acc + size_t((e + 1u) & 1u) * kCopies * a.acc_stride;
    for (int i = tid; i < kCopies * a.acc_stride; i += kThreads) nxt[i] = 0.f;
  }
  const int nVw = ok ? nV : 0;
  float* my_copy = acc + size_t(cta % kCopies) * a.acc_stride;
  if (nVw > 0) {
    // warp w: entries [16 mb, 16 mb + 16) of g over row blocks kb = w / T16,
    // w / T16 + 16 / T16, ...; rows past nV hold x = 0
    const int mb = warp % T16, kb0 = warp / T16;
    constexpr int kStep = kWarps / T16;
    const int nkb = (nVw + 15) / 16;
    const int j = lane >> 3, rr = lane & 7;
    const int col = mb * 16 + (j & 1) * 8;  // A rows m = entries of g
    const uint32_t blk = sbase + uint32_t(lay.sV) + uint32_t(col / 64) * uint32_t(rowsV) * 128u;
    const int chunk = (col % 64) / 8;
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(s_xb);
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    int kb = kb0;
    for (; kb + kStep < nkb; kb += 2 * kStep) {
      const uint4 A0 = ldsm_x4_trans(swz(blk, kb * 16 + rr + (j >> 1) * 8, chunk));
      const uint4 A1 = ldsm_x4_trans(swz(blk, (kb + kStep) * 16 + rr + (j >> 1) * 8, chunk));
      const uint32_t b00 = grp == 0 ? xw[kb * 8 + tig] : 0u;
      const uint32_t b01 = grp == 0 ? xw[kb * 8 + 4 + tig] : 0u;
      const uint32_t b10 = grp == 0 ? xw[(kb + kStep) * 8 + tig] : 0u;
      const uint32_t b11 = grp == 0 ? xw[(kb + kStep) * 8 + 4 + tig] : 0u;
      mma_16816(d0, A0, b00, b01);
      mma_16816(d1, A1, b10, b11);
    }
    if (kb < nkb) {
      const uint4 A0 = ldsm_x4_trans(swz(blk, kb * 16 + rr + (j >> 1) * 8, chunk));
      mma_16816(d0, A0, grp == 0 ? xw[kb * 8 + tig] : 0u, grp == 0 ? xw[kb * 8 + 4 + tig] : 0u);
    }
    // column 0 of D: lanes with tig == 0 hold entries grp and grp + 8
    const float v0g = d0[0] + d1[0], v8g = d0[2] + d1[2];
    const int src = lane & 16;
    float u[4], w4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      u[q] = __shfl_sync(0xFFFFFFFFu, v0g, src + 4 * q);
      w4[q] = __shfl_sync(0xFFFFFFFFu, v8g, src + 4 * q);
    }
    if (kb0 < nkb && (lane & 15) == 0) {
      const int a0 = mb * 16 + (lane >> 4) * 4;
      red_add_v4_f32(my_copy + a0, u[0], u[1], u[2], u[3]);
      red_add_v4_f32(my_copy + a0 + 8, w4[0], w4[1], w4[2], w4[3]);
    }
    if (warp == kWarps - 1) {  // ||x_c||^2 (x_i^2 is exact in fp32 for bf16 x_i)
      float sx = 0.f;
      for (int i = lane; i < nVw; i += 32) {
        const float xv = __bfloat162float(s_xb[i]);
        sx = fmaf(xv, xv, sx);
      }
      sx = warp_sum_all(sx);
      if (lane == 0) red_add_f32(my_copy + K, sx);
    }
  }

  // ---- the grid barrier ---------------------------------------------------
  // Thread 0 arrives once every warp's atomics are issued; while the arrival
  // propagates, all threads load their correction tiles into registers, then
  // thread 0 polls.
  sync_compute();
  // the counter stood at s_base when this launch started (launches of one
  // handle may use different CTA counts)
  const uint32_t target = s_base + uint32_t(G);
  if (tid == 0) red_release_u32(a.bar, 1u);

  // Tiles (I, J), I <= J, are taken by column: columns J and T16 - 1 - J pair
  // up (T16 + 1 tiles), the kWpp warps of a pair split its tiles into
  // segments of at most kSeg.  Step s of a pair: column J1 = p for s <= p
  // (row I = s), else column J2 = T16 - 1 - p (row I = s - p - 1).
  constexpr int kPairs = T16 / 2, kWpp = kWarps / kPairs;
  constexpr int kSeg = (T16 + 1 + kWpp - 1) / kWpp;
  const int qp = warp / kWpp, qh = warp % kWpp;
  const int J1 = qp, J2 = T16 - 1 - qp;
  uint4 fa[kSeg];
  const bool staged = mbar_wait_bounded(&s_bar[1], 0, a.status);
  {
    const uint4* tiles = reinterpret_cast<const uint4*>(sF);
#pragma unroll
    for (int st = 0; st < kSeg; ++st) {
      const int s = qh * kSeg + st;
      const bool first = s <= J1;
      const int I = first ? s : s - J1 - 1, J = first ? J1 : J2;
      fa[st] = s <= T16 ? tiles[corr_tile_index(I, J, T16) * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (tid == 0) {
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
  ok = sync_compute_and(staged) && ok && s_ok;
  const int nMw = ok ? nM : 0;
  signal_prefetch_warp();

  // ---- phase 2: g (same order in every CTA), g^T E g, g.g, speculative M g --
  float g2 = 0.f;
  for (int t = tid; t < K; t += kThreads) {
    float gsum = 0.f;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) gsum += ld_cg_f32(acc + size_t(c) * a.acc_stride + t);
    s_g[t] = gsum;
    g2 = fmaf(gsum, gsum, g2);
    // B operands: g_t is row kk = t % 16 of column block t / 16: register
    // kk / 8, lane pair (kk % 8) / 2, half kk % 2 of lanes pair (high part)
    // and 4 + pair (remainder)
    const __nv_bfloat16 hi = __float2bfloat16_rn(gsum);
    const __nv_bfloat16 lo = __float2bfloat16_rn(gsum - __bfloat162float(hi));
    const int kk = t & 15, pos = (kk >> 3) * 2 + (kk & 1), pr = (kk & 7) >> 1;
    __nv_bfloat16* bf = reinterpret_cast<__nv_bfloat16*>(s_bfrag + (t >> 4) * 32);
    bf[pr * 4 + pos] = hi;
    bf[(4 + pr) * 4 + pos] = lo;
  }
  if (warp < K / 32) {
    g2 = warp_sum_all(g2);
    if (lane == 0) s_ggw[warp] = g2;
  }
  if (tid == kThreads - 1) {  // idle in the loop above (K < kThreads): the loads overlap
    float sx = 0.f;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) sx += ld_cg_f32(acc + size_t(c) * a.acc_stride + K);
    s_sx = sx;
  }
  sync_compute();
  {
    // g^T E g = sum over tiles I <= J of g_I . (F_IJ g_J), one independent
    // MMA per tile from the registers loaded before the barrier; B = g_J is
    // loaded once per column
    const uint2 bJ1 = s_bfrag[J1 * 32 + lane], bJ2 = s_bfrag[J2 * 32 + lane];
    float qsum = 0.f;
#pragma unroll
    for (int st = 0; st < kSeg; ++st) {
      const int s = qh * kSeg + st;
      if (s <= T16) {
        const bool first = s <= J1;
        const int I = first ? s : s - J1 - 1;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(d, fa[st], first ? bJ1.x : bJ2.x, first ? bJ1.y : bJ2.y);
        // columns 0 (high) and 1 (low) of rows grp and grp + 8 (lanes with
        // tig == 0; the other lanes hold the zero columns)
        qsum = fmaf(s_g[I * 16 + grp], d[0] + d[1], qsum);
        qsum = fmaf(s_g[I * 16 + grp + 8], d[2] + d[3], qsum);
      }
    }
    if (tig != 0) qsum = 0.f;
    qsum = warp_sum_all(qsum);
    if (lane == 0) s_qw[warp] = qsum;
  }
  {
    // speculative fast path: rows of M_c g, A = 16 rows of M_c, B = g (hi,
    // lo); with fewer than 16 row blocks a row block's K / 16 steps are split
    // over wpr warps, whose partial sums meet in s_yp[warp]
    const int RB = (nMw + 15) / 16;
    if (RB > 0) {
      const int wpr = RB >= kWarps ? 1 : kWarps / RB;
      const int j = lane >> 3, rr = lane & 7;
      const uint32_t blkM = sbase + uint32_t(lay.sM);
      for (int rb = warp / wpr; rb < RB; rb += kWarps / wpr) {
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        const int row = rb * 16 + rr + (j & 1) * 8;
        int kb = warp % wpr;
        for (; kb + wpr < T16; kb += 2 * wpr) {
          const int c0 = kb * 16 + (j >> 1) * 8, c1 = c0 + wpr * 16;
          const uint4 A0 = ldsm_x4(swz(blkM + uint32_t(c0 / 64) * uint32_t(rowsM) * 128u, row, (c0 % 64) / 8));
          const uint4 A1 = ldsm_x4(swz(blkM + uint32_t(c1 / 64) * uint32_t(rowsM) * 128u, row, (c1 % 64) / 8));
          const uint2 b0 = s_bfrag[kb * 32 + lane], b1 = s_bfrag[(kb + wpr) * 32 + lane];
          mma_16816(d0, A0, b0.x, b0.y);
          mma_16816(d1, A1, b1.x, b1.y);
        }
        if (kb < T16) {
          const int c0 = kb * 16 + (j >> 1) * 8;
          const uint4 A0 = ldsm_x4(swz(blkM + uint32_t(c0 / 64) * uint32_t(rowsM) * 128u, row, (c0 % 64) / 8));
          const uint2 b0 = s_bfrag[kb * 32 + lane];
          mma_16816(d0, A0, b0.x, b0.y);
        }
        if (tig == 0) {
          const float y0 = (d0[0] + d0[1]) + (d1[0] + d1[1]);
          const float y8 = (d0[2] + d0[3]) + (d1[2] + d1[3]);
          float* dst = wpr == 1 ? s_ys + rb * 16 : s_yp + warp * 16;
          dst[grp] = y0;
          dst[grp + 8] = y8;
        }
      }
    }
  }
  sync_compute();

  // ---- gate ------------------------------------------------------------------
  if (tid == 0) {
    // fp32 throughout: the sums' relative error (~1e-7 of ||x||^2) moves rho by
    // ~1e-6 near any practical eps, and fp64 is slow on this part
    float quad = 0.f, gg = 0.f;
    for (int w = 0; w < kWarps; ++w) quad += s_qw[w];
    for (int w = 0; w < K / 32; ++w) gg += s_ggw[w];
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
  sync_compute();
  const bool slow = !(s_rho < a.eps);

  // ---- phase 3: the branch the gate picked ---------------------------------
  if (ok) {
    if (!slow) {
      // the split the M g phase used: one warp per row block (rows in s_ys)
      // or wpr warps per row block (partials in s_yp)
      const int RB = (nMw + 15) / 16;
      const int wpr = RB >= kWarps ? 1 : kWarps / max(RB, 1);
      if (wpr == 1) {
        for (int r = tid; r < nMw; r += kThreads) a.y[m0 + r] = s_ys[r];
      } else {
        for (int r = tid; r < nMw; r += kThreads) {
          const float* src = s_yp + (r / 16) * wpr * 16 + (r % 16);
          float v = 0.f;
          for (int q = 0; q < wpr; ++q) v += src[q * 16];
          a.y[m0 + r] = v;
        }
      }
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
        int jj = lane;
        for (; jj + 32 < nch; jj += 64) {
          uint4 w0[4], w1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            w0[q] = ld_stream_v4(wr[q] + jj);
            w1[q] = ld_stream_v4(wr[q] + jj + 32);
          }
          float xa[8], xb[8];
          bf16x8_to_f32(x4[jj], xa);
          bf16x8_to_f32(x4[jj + 32], xb);
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
        for (; jj < nch; jj += 32) {
          float xa[8];
          bf16x8_to_f32(x4[jj], xa);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float f[8];
            bf16x8_to_f32(ld_stream_v4(wr[q] + jj), f);
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
    a.bar[2] = s_base + uint32_t(G);
    a.bar[1] = e + 1u;  // every CTA read the epoch and base before the barrier
  }
}

template <int K>
__global__ void __launch_bounds__(kBlock, 1)
    gsi_decode3_kernel(const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmM, const __grid_constant__ Decode3Args a) {
  decode3_body<K>(&tmV, &tmM, a, int(blockIdx.x), int(gridDim.x));
}

template <int K>
__global__ void __launch_bounds__(kBlock, 1)
    gsi_decode3_group_kernel(const __grid_constant__ GroupMaps maps,
                             const __grid_constant__ GroupArgs g) {
  int m = 0;
  while (m + 1 < g.n && int(blockIdx.x) >= g.cta0[m + 1]) ++m;
  decode3_body<K>(&maps.m[2 * m], &maps.m[2 * m + 1], g.a[m], int(blockIdx.x) - g.cta0[m],
                  g.cta0[m + 1] - g.cta0[m]);
}

const void* decode3_kernel_for(int64_t k, bool group) {
  switch (k) {
    case 64: return group ? reinterpret_cast<const void*>(&gsi_decode3_group_kernel<64>)
                          : reinterpret_cast<const void*>(&gsi_decode3_kernel<64>);
    case 128: return group ? reinterpret_cast<const void*>(&gsi_decode3_group_kernel<128>)
                           : reinterpret_cast<const void*>(&gsi_decode3_kernel<128>);
    case 256: return group ? reinterpret_cast<const void*>(&gsi_decode3_group_kernel<256>)
                           : reinterpret_cast<const void*>(&gsi_decode3_kernel<256>);
    default: return nullptr;
  }
}

int acc3_stride(int64_t k) { return int((k + 1 + 3) / 4 * 4); }

// Row boxes for `rows` owned rows: box rows a multiple of 16 and <= 256.
void row_boxes(int rows, int* box, int* nbox) {
  const int padded = (rows + 15) / 16 * 16;
  *nbox = (padded + kMaxBoxRows - 1) / kMaxBoxRows;
  *box = ((padded + *nbox - 1) / *nbox + 15) / 16 * 16;
}

// Largest dynamic shared memory a kernel of this k may use on this device
// (raised to that limit once: the limit belongs to the function).
gsi_status_t smem_limit(const void* fn, int device, int* limit) {
  int max_optin = 0;
  if (cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
    return GSI_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return GSI_ERR_CUDA;
  *limit = max_optin - int(fa.sharedSizeBytes);
  if (fa.maxDynamicSharedSizeBytes < *limit &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, *limit) != cudaSuccess)
    return GSI_ERR_CUDA;
  return GSI_OK;
}

// Rows, TMA boxes, shared memory and tensor maps of handle h run on G CTAs.
gsi_status_t plan_member(const gsi_handle* h, int G, int limit, Dec3Plan* p, void* tmV, void* tmM) {
  p->G = G;
  p->rows_M = int((h->d_out + G - 1) / G);
  p->rows_V = int((h->d + G - 1) / G);
  row_boxes(p->rows_M, &p->box_M, &p->nbox_M);
  row_boxes(p->rows_V, &p->box_V, &p->nbox_V);
  p->smem = smem3_layout(int(h->k), p->nbox_M * p->box_M, p->nbox_V * p->box_V).total + kSmemSlack;
  if (p->smem > size_t(limit)) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (!tma_encode_bf16_2d(tmV, h->V, uint64_t(h->d), uint64_t(h->k), uint32_t(p->box_V), 64) ||
      !tma_encode_bf16_2d(tmM, h->M, uint64_t(h->d_out), uint64_t(h->k), uint32_t(p->box_M), 64))
    return GSI_ERR_CUDA;
  return GSI_OK;
}

// Prefetch ranges of a target handle or group (operands above 64 MiB are
// not prefetched: a large share of L2).  Returns the number of ranges.
int prefetch_ranges(const gsi_handle* nh, const gsi_group* ng, const char** p, uint32_t* b) {
  const gsi_handle* list[kMaxGroup];
  int nl = 0;
  if (nh) list[nl++] = nh;
  if (ng)
    for (int m = 0; m < ng->n && nl < kMaxGroup; ++m) list[nl++] = ng->h[m];
  const int64_t kMaxPrefetch = int64_t(64) << 20;
  int n = 0;
  for (int i = 0; i < nl; ++i) {
    const gsi_handle* t = list[i];
    const int64_t bytes[3] = {t->d * t->k * 2, t->d_out * t->k * 2,
                              t->dec3_F ? int64_t(corr_tiles_elems(int(t->k))) * 2 : 0};
    const void* ptr[3] = {t->V, t->M, t->dec3_F};
    for (int o = 0; o < 3; ++o)
      if (bytes[o] > 0 && bytes[o] <= kMaxPrefetch && n < kMaxPf) {
        p[n] = static_cast<const char*>(ptr[o]);
        b[n] = uint32_t(bytes[o]);
        ++n;
      }
  }
  for (int i = n; i < kMaxPf; ++i) {
    p[i] = nullptr;
    b[i] = 0u;
  }
  return n;
}

void fill_args(Decode3Args* a, const gsi_handle* h, const Dec3Plan& p, const void* x, float* y,
               uint8_t* gate, float* rho) {
  a->W = h->W;
  a->F = h->dec3_F;
  a->x = static_cast<const __nv_bfloat16*>(x);
  a->y = y;
  a->gate = gate;
  a->rho = rho;
  a->d_out = int(h->d_out);
  a->d = int(h->d);
  a->eps = h->eps;
  a->rows_M = p.rows_M;
  a->rows_V = p.rows_V;
  a->box_M = p.box_M;
  a->box_V = p.box_V;
  a->nbox_M = p.nbox_M;
  a->nbox_V = p.nbox_V;
  a->acc = h->dec3_acc;
  a->acc_stride = acc3_stride(h->k);
  a->bar = h->dec3_bar;
  a->status = h->status;
}

cudaLaunchConfig_t launch_config(dim3 grid, size_t smem, cudaStream_t s, bool pdl,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.numAttrs = 0;
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
  }
  cfg.attrs = attr;
  return cfg;
}

}  // namespace

size_t decode3_acc_floats(int64_t k) { return size_t(2) * kCopies * acc3_stride(k); }

gsi_status_t decode3_configure(gsi_handle* h) {
  const void* fn = decode3_kernel_for(h->k, false);
  const void* fng = decode3_kernel_for(h->k, true);
  if (!fn || !fng) return GSI_ERR_UNSUPPORTED_SHAPE;
  int limit = 0;
  gsi_status_t st = smem_limit(fn, h->device, &limit);
  if (st == GSI_OK) {
    int limit_g = 0;
    st = smem_limit(fng, h->device, &limit_g);
  }
  if (st != GSI_OK) return st;
  const int64_t rows_hint = (std::max(h->d_out, h->d) + 7) / 8;
  const int G = int(std::max<int64_t>(1, std::min<int64_t>(h->num_sms, rows_hint)));
  Dec3Plan p;
  st = plan_member(h, G, limit, &p, h->dec3_tmaps[0], h->dec3_tmaps[1]);
  if (st != GSI_OK) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBlock, p.smem) != cudaSuccess)
    return GSI_ERR_CUDA;
  // The CTAs wait on one another: all of them must fit at once.
  if (per_sm < 1 || int64_t(per_sm) * h->num_sms < G) return GSI_ERR_UNSUPPORTED_SHAPE;
  h->dec3_plan = p;
  return GSI_OK;
}

gsi_status_t decode3_launch(gsi_handle* h, const void* x, float* y, uint8_t* gate, float* rho,
                            cudaStream_t s) {
  Decode3Args a;
  fill_args(&a, h, h->dec3_plan, x, y, gate, rho);
  prefetch_ranges(h->pf_next, h->pf_group, a.pf, a.pf_bytes);
  a.pf_part0 = 0;
  a.pf_parts = h->dec3_plan.G;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(dim3(h->dec3_plan.G), h->dec3_plan.smem, s, h->use_pdl, attr);
  const CUtensorMap* maps = reinterpret_cast<const CUtensorMap*>(h->dec3_tmaps);
  cudaError_t err;
  switch (h->k) {
    case 64: err = cudaLaunchKernelEx(&cfg, gsi_decode3_kernel<64>, maps[0], maps[1], a); break;
    case 128: err = cudaLaunchKernelEx(&cfg, gsi_decode3_kernel<128>, maps[0], maps[1], a); break;
    case 256: err = cudaLaunchKernelEx(&cfg, gsi_decode3_kernel<256>, maps[0], maps[1], a); break;
    default: return GSI_ERR_UNSUPPORTED_SHAPE;
  }
  return err == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

gsi_status_t group_configure(gsi_group* g) {
  const gsi_handle* h0 = g->h[0];
  const void* fn = decode3_kernel_for(h0->k, true);
  if (!fn) return GSI_ERR_UNSUPPORTED_SHAPE;
  int limit = 0;
  gsi_status_t st = smem_limit(fn, h0->device, &limit);
  if (st != GSI_OK) return st;
  // CTAs in proportion to each member's operand bytes (V_k + M), at least one
  // each, all co-resident (one per SM)
  const int S = h0->num_sms;
  if (g->n > S) return GSI_ERR_UNSUPPORTED_SHAPE;
  double w[kMaxGroup], wsum = 0.0;
  for (int m = 0; m < g->n; ++m) {
    w[m] = double(g->h[m]->d + g->h[m]->d_out) * double(g->h[m]->k);
    wsum += w[m];
  }
  int Gm[kMaxGroup], used = 0;
  for (int m = 0; m < g->n; ++m) {
    const int64_t rows_hint = (std::max(g->h[m]->d_out, g->h[m]->d) + 7) / 8;
    Gm[m] = int(std::max<int64_t>(1, std::min<int64_t>(rows_hint, int64_t(S * w[m] / wsum))));
    used += Gm[m];
  }
  for (int m = 0; used > S; m = (m + 1) % g->n)  // rounding never overshoots by much
    if (Gm[m] > 1) {
      --Gm[m];
      --used;
    }
  size_t smem = 0;
  g->cta0[0] = 0;
  for (int m = 0; m < g->n; ++m) {
    st = plan_member(g->h[m], Gm[m], limit, &g->plan[m], g->tmaps[2 * m], g->tmaps[2 * m + 1]);
    if (st != GSI_OK) return st;
    smem = std::max(smem, g->plan[m].smem);
    g->cta0[m + 1] = g->cta0[m] + Gm[m];
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBlock, smem) != cudaSuccess)
    return GSI_ERR_CUDA;
  if (per_sm < 1 || int64_t(per_sm) * S < g->cta0[g->n]) return GSI_ERR_UNSUPPORTED_SHAPE;
  g->smem = smem;
  return GSI_OK;
}

gsi_status_t group_launch(gsi_group* g, const void* const* x, float* const* y,
                          uint8_t* const* gate, float* const* rho, cudaStream_t s) {
  GroupMaps maps;
  GroupArgs ga;
  std::memset(&maps, 0, sizeof maps);
  std::memset(&ga, 0, sizeof ga);
  std::memcpy(maps.m, g->tmaps, size_t(2) * g->n * sizeof(CUtensorMap));
  ga.n = g->n;
  const char* pfp[kMaxPf];
  uint32_t pfb[kMaxPf];
  prefetch_ranges(g->pf_next, nullptr, pfp, pfb);
  for (int m = 0; m < g->n; ++m) {
    fill_args(&ga.a[m], g->h[m], g->plan[m], x[m], y[m], gate ? gate[m] : nullptr,
              rho ? rho[m] : nullptr);
    std::memcpy(ga.a[m].pf, pfp, sizeof pfp);
    std::memcpy(ga.a[m].pf_bytes, pfb, sizeof pfb);
    ga.a[m].pf_part0 = g->cta0[m];
    ga.a[m].pf_parts = g->cta0[g->n];
  }
  for (int m = 0; m <= g->n; ++m) ga.cta0[m] = g->cta0[m];
  for (int m = g->n + 1; m <= kMaxGroup; ++m) ga.cta0[m] = g->cta0[g->n];
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(dim3(g->cta0[g->n]), g->smem, s, true, attr);
  cudaError_t err;
  switch (g->k) {
    case 64: err = cudaLaunchKernelEx(&cfg, gsi_decode3_group_kernel<64>, maps, ga); break;
    case 128: err = cudaLaunchKernelEx(&cfg, gsi_decode3_group_kernel<128>, maps, ga); break;
    case 256: err = cudaLaunchKernelEx(&cfg, gsi_decode3_group_kernel<256>, maps, ga); break;
    default: return GSI_ERR_UNSUPPORTED_SHAPE;
  }
  return err == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

}  // namespace gsi
