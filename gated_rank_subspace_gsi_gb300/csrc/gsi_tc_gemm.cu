// gsi_tc_gemm.cu -- the two dense contractions of the batched GSI path on
// the sm_103a tcgen05 tensor cores, written with inline PTX (TMA, mbarrier,
// tcgen05.mma / commit / ld, TMEM alloc).
//
// Page: "Technical summary: Gated Subspace Inference for transformer
// acceleration" [GSI], section 2.2: fast tokens take y = M g, slow tokens
// take y = W x.  After compaction (gsi_batched.cu) both are GEMMs:
//   Y_slow^T (d_out x n_slow) = W (d_out x d)  . X_slow^T
//   Y_fast^T (d_out x n_fast) = M (d_out x k)  . (G_hi + G_lo)^T
// Weights sit in the MMA's M dimension ("swap AB"), so each weight tile is
// read from HBM by exactly one CTA and the token count sets N (16..256, a
// runtime value in the instruction descriptor).  G_fast is carried as two
// bf16 planes hi = bf16(g), lo = bf16(g - hi); both accumulate into the same
// TMEM tile, which keeps g to ~2^-16 relative although the operands are bf16.
//
// Persistent CTAs (192 threads, one per SM) take 128-row x 256-token slow
// tiles and 128-row x 128-token fast tiles from a device-side queue, slow
// tiles first: warp 0 issues TMA loads (one elected lane), warp 1 allocates
// TMEM and issues tcgen05.mma (one elected lane) into one of two 256-column
// accumulators, warps 2-5 drain the other (tcgen05.ld 32x32b) and scatter
// each token column to its row of y.  Operands stream through mbarrier rings
// of 128-byte-swizzled bf16 boxes that run on across a CTA's tiles: the slow
// ring (a 128x64 box of W and the X_slow boxes of the token tile per stage)
// and the fast ring (a 128x64 box of M and 128 rows of both g planes).
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "gsi_device.cuh"
#include "gsi_internal.h"
#include "gsi_tc_gemm.h"

namespace gsi {
namespace {

constexpr int kBM = 128;           // weight rows per tile (MMA M)
constexpr int kBN = 256;           // slow token rows per tile (max MMA N)
constexpr int kBNF = 128;          // fast token rows per tile (both g planes in one stage)
constexpr int kBK = 64;            // K elements per stage (128 bytes of bf16)
constexpr int kStages = 4;          // stages of the fast ring
constexpr int kMaxSlowStages = 8;   // at most, on the slow ring
constexpr int kABytes = kBM * kBK * 2;   // 16 KiB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kRingBytes = 216 * 1024;  // both rings share this memory
constexpr int kTcThreads = 192;
constexpr int kTmemCols = 512;  // two 256-column accumulators
constexpr size_t kTcSmem = size_t(kRingBytes) + 1024;  // + alignment slack
// The GEMM kernel has two TMA rings over the same shared memory.  The slow
// ring's stage is one A box of W and the one or two boxes of X_slow that
// cover the first slow token tile (128 + 32 rows for 154 tokens: 36 KB, six
// stages); the fast ring has 4 stages of 48 KB (A 128 x 64 and both g planes
// of 128 tokens).  A shorter token tile loads B as boxes of 32, 64, 128 or 256
// rows that just cover it.  A CTA takes its slow tiles before its fast ones,
// so it switches rings at most once, after every slow stage is released.
constexpr int kBoxRows[4] = {256, 128, 64, 32};  // host: the maps' box heights
__host__ __device__ constexpr int box_rows(int i) { return 256 >> i; }  // = kBoxRows[i]
struct TcMaps {
  CUtensorMap W, M;
  CUtensorMap Xs[4], Ghi[4], Glo[4];  // B operands, box heights kBoxRows[]
};

// ---- tcgen05 wrappers ------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_addr(dst_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      :: "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile whose rows are 128 bytes
// (64 bf16) and swizzled in 8-row / 1024-byte atoms by TMA's 128-byte mode:
// start address >> 4 in bits 0-13, leading-byte offset 16 B (unused by this
// layout), stride-byte offset 1024 B between 8-row groups, descriptor
// version 1 (bits 46-47), layout type 2 = 128-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= uint64_t((saddr >> 4) & 0x3FFFu);
  desc |= uint64_t(1u) << 16;
  desc |= uint64_t(1024u >> 4) << 32;
  desc |= uint64_t(1u) << 46;
  desc |= uint64_t(2u) << 61;
  return desc;
}
// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* status,
                                             int* s_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(s_abort)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      *reinterpret_cast<volatile int*>(s_abort) = 1;
      return false;
    }
  }
  return true;
}

// index into kBoxRows of the smallest box of at least r rows (r <= 128), and
// the two boxes that cover a tile of N rows: a 256-row box for N > 192, else
// a 128-row box followed by the smallest box that covers the rest
__device__ __forceinline__ int box_index(int r) { return r <= 32 ? 3 : (r <= 64 ? 2 : 1); }

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

// One tile of the two GEMMs: 128 output rows (o0) x up to 256 slow tokens or
// up to 128 fast tokens (j0).  Slow tiles come first in the numbering (the
// long ones start first), then fast tiles; within a kind, consecutive tiles
// share a token tile and walk the output rows, so their B operand stays in
// L2.  A fast tile's stage holds one A box of M and the same rows of both g
// planes (hi, lo) beside it, so M is read once per tile.
struct Tile {
  bool slow;
  int o0, j0, nvalid, N, num_kb, bx1, bx2, b_bytes;
};

__device__ __forceinline__ Tile decode_tile(int t, int n_slow_tiles, int n_mt, int n_fast,
                                            int n_slow, const TcGemmArgs& a) {
  Tile u;
  u.slow = t < n_slow_tiles;
  const int tt = u.slow ? t : t - n_slow_tiles;
  const int mt = tt % n_mt, jt = tt / n_mt;
  const int bn = u.slow ? kBN : kBNF;
  u.o0 = mt * kBM;
  u.j0 = jt * bn;
  u.nvalid = min(bn, (u.slow ? n_slow : n_fast) - u.j0);
  u.N = (u.nvalid + 15) & ~15;
  u.num_kb = u.slow ? (a.d + kBK - 1) / kBK : (a.k + kBK - 1) / kBK;
  u.bx1 = u.N > 192 ? 0 : box_index(u.N);
  u.bx2 = (u.slow && u.N > 128 && u.N <= 192) ? box_index(u.N - 128) : -1;
  // slow: one or two boxes of X_slow; fast: one box of each g plane
  u.b_bytes = (u.slow ? box_rows(u.bx1) + (u.bx2 >= 0 ? box_rows(u.bx2) : 0)
                      : 2 * box_rows(u.bx1)) * kBK * 2;
  return u;
}

// Persistent: one CTA per SM takes tiles from a device-wide counter (zeroed
// by the partition-and-gather kernel) until none are left.  Warp 0 (one lane)
// takes each tile, publishes it to the other roles through a two-slot queue
// in shared memory, and streams its operands through the slow or the fast TMA
// ring; warp 1 (one lane) issues the tile's MMAs into one of two TMEM
// accumulators; warps 2-5 drain the other accumulator of the previous tile
// meanwhile and scatter it to y.  Every wait is bounded.
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, TcGemmArgs a) {
  constexpr int kQ = 2;  // tiles in flight: queue slots and TMEM accumulators
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full_bar[kStages];   // fast ring
  __shared__ uint64_t empty_bar[kStages];
  __shared__ uint64_t sfull_bar[kMaxSlowStages];   // slow ring
  __shared__ uint64_t sempty_bar[kMaxSlowStages];
  __shared__ uint64_t tq_full[kQ], tq_empty[kQ], acc_full[kQ], acc_empty[kQ];
  __shared__ int s_tile[kQ];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued, s_issued_slow;

  pdl_launch_dependents();
  pdl_wait();  // token counts, index lists, gathered operands and the tile counter are visible
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_fast = a.count[0], n_slow = a.count[1];
  const int n_mt = (a.d_out + kBM - 1) / kBM;
  const int n_slow_tiles = n_mt * ((n_slow + kBN - 1) / kBN);
  const int total = n_slow_tiles + n_mt * ((n_fast + kBNF - 1) / kBNF);
  // the slow ring: stage = A + the first (largest) slow token tile's B boxes
  const int slow_stage =
      n_slow_tiles > 0 ? kABytes + decode_tile(0, n_slow_tiles, n_mt, n_fast, n_slow, a).b_bytes
                       : kStageBytes;
  const int S = min(kMaxSlowStages, kRingBytes / slow_stage);

  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* tiles = smem_raw + (base - smem_addr(smem_raw));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kMaxSlowStages; ++s) {
      mbar_init(&sfull_bar[s], 1);
      mbar_init(&sempty_bar[s], 1);
    }
    for (int q = 0; q < kQ; ++q) {
      mbar_init(&tq_full[q], 1);
      mbar_init(&tq_empty[q], 5);   // the MMA lane and the 4 epilogue warps
      mbar_init(&acc_full[q], 1);
      mbar_init(&acc_empty[q], 4);  // the 4 epilogue warps
    }
    s_abort = 0;
    s_issued = 0;
    s_issued_slow = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      int g = 0;   // K steps issued on the fast ring: stage g % kStages
      int gs = 0;  // K steps issued on the slow ring: stage gs % S
      bool drained = false;
      for (int i = 0;; ++i) {
        const int q = i % kQ;
        if (i >= kQ && !wait_bounded(&tq_empty[q], ((i / kQ) & 1) ^ 1, a.status, &s_abort)) break;
        int t = atomicAdd(a.tile_counter, 1);
        if (t >= total) t = -1;
        s_tile[q] = t;
        mbar_arrive_cta(&tq_full[q]);
        if (t < 0) break;
        const Tile u = decode_tile(t, n_slow_tiles, n_mt, n_fast, n_slow, a);
        bool ok = true;
        if (!u.slow && !drained) {
          // the fast ring reuses the slow ring's memory: every slow stage
          // issued must have been released by its MMAs first
          for (int h = max(0, gs - S); h < gs && ok; ++h)
            ok = wait_bounded(&sempty_bar[h % S], (h / S) & 1, a.status, &s_abort);
          drained = true;
        }
        for (int kb = 0; ok && kb < u.num_kb; ++kb) {
          const int kc = kb * kBK;
          if (u.slow) {
            const int s = gs % S;
            if (gs >= S && !wait_bounded(&sempty_bar[s], ((gs / S) & 1) ^ 1, a.status, &s_abort)) {
              ok = false;
              break;
            }
            unsigned char* sa = tiles + size_t(s) * slow_stage;
            unsigned char* sb = sa + kABytes;
            mbar_arrive_expect_tx(&sfull_bar[s], uint32_t(kABytes + u.b_bytes));
            tma_load_2d(sa, &maps.W, kc, u.o0, &sfull_bar[s]);
            tma_load_2d(sb, &maps.Xs[u.bx1], kc, u.j0, &sfull_bar[s]);
            if (u.bx2 >= 0)
              tma_load_2d(sb + box_rows(u.bx1) * kBK * 2, &maps.Xs[u.bx2], kc,
                          u.j0 + box_rows(u.bx1), &sfull_bar[s]);
            ++gs;
          } else {
            const int s = g % kStages;
            if (g >= kStages &&
                !wait_bounded(&empty_bar[s], ((g / kStages) & 1) ^ 1, a.status, &s_abort)) {
              ok = false;
              break;
            }
            unsigned char* sa = tiles + size_t(s) * kStageBytes;
            unsigned char* sb = sa + kABytes;
            mbar_arrive_expect_tx(&full_bar[s], uint32_t(kABytes + u.b_bytes));
            tma_load_2d(sa, &maps.M, kc, u.o0, &full_bar[s]);
            tma_load_2d(sb, &maps.Ghi[u.bx1], kc, u.j0, &full_bar[s]);
            tma_load_2d(sb + box_rows(u.bx1) * kBK * 2, &maps.Glo[u.bx1], kc, u.j0, &full_bar[s]);
            ++g;
          }
        }
        if (!ok) break;
      }
      s_issued = g;
      s_issued_slow = gs;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int g = 0, gs = 0;  // K steps consumed on the fast and the slow ring
      for (int i = 0;; ++i) {
        const int q = i % kQ;
        if (!wait_bounded(&tq_full[q], (i / kQ) & 1, a.status, &s_abort)) break;
        const int t = s_tile[q];
        mbar_arrive_cta(&tq_empty[q]);
        if (t < 0) break;
        const Tile u = decode_tile(t, n_slow_tiles, n_mt, n_fast, n_slow, a);
        if (i >= kQ && !wait_bounded(&acc_empty[q], ((i / kQ) & 1) ^ 1, a.status, &s_abort)) break;
        tc_fence_after();
        const uint32_t acc = tmem + uint32_t(q * kBN);
        const uint32_t idesc = idesc_bf16_f32(kBM, u.N);
        bool ok = true;
        for (int kb = 0; kb < u.num_kb; ++kb) {
          const int s = u.slow ? gs % S : g % kStages;
          uint64_t* fb = u.slow ? &sfull_bar[s] : &full_bar[s];
          uint64_t* eb = u.slow ? &sempty_bar[s] : &empty_bar[s];
          const uint32_t par = u.slow ? (gs / S) & 1 : (g / kStages) & 1;
          if (!wait_bounded(fb, par, a.status, &s_abort)) {
            ok = false;
            break;
          }
          if (u.slow) ++gs; else ++g;
          tc_fence_after();
          const uint32_t sa = base + uint32_t(s) * uint32_t(u.slow ? slow_stage : kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_bf16(acc, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb + kk * 32), idesc,
                        (kb | kk) != 0 ? 1u : 0u);
          if (!u.slow) {
            // the lo plane of the same tokens, against the same A box
            const uint32_t sb2 = sb + uint32_t(box_rows(u.bx1) * kBK * 2);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc_mma_bf16(acc, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb2 + kk * 32),
                          idesc, 1u);
          }
          tc_commit(eb);
        }
        if (!ok) break;
        tc_commit(&acc_full[q]);
      }
    }
  } else {
    // epilogue: warps 2..5 own TMEM lane quarters (warp % 4)
    const int qw = warp & 3;
    for (int i = 0;; ++i) {
      const int q = i % kQ;
      if (!wait_bounded(&tq_full[q], (i / kQ) & 1, a.status, &s_abort)) break;
      const int t = s_tile[q];
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&tq_empty[q]);
      if (t < 0) break;
      const Tile u = decode_tile(t, n_slow_tiles, n_mt, n_fast, n_slow, a);
      const bool ok = wait_bounded(&acc_full[q], (i / kQ) & 1, a.status, &s_abort);
      tc_fence_after();
      const int o = u.o0 + qw * 32 + lane;
      const int32_t* idx = u.slow ? a.idx_slow : a.idx_fast;
      if (ok) {
        for (int c0 = 0; c0 < u.N; c0 += 32) {
          // lane l holds the token of column c0 + l; each column's is broadcast
          const int my_tok = c0 + lane < u.nvalid ? *(idx + u.j0 + c0 + lane) : 0;
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + (uint32_t(qw * 32) << 16) + uint32_t(q * kBN + c0), r);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int tok = __shfl_sync(0xFFFFFFFFu, my_tok, jj);
            if (c0 + jj < u.nvalid && o < a.d_out)
              a.y[size_t(tok) * a.d_out + o] = __uint_as_float(r[jj]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acc_empty[q]);
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) {
    // make sure no bulk copy is still writing into this CTA's shared memory
    const int issued = s_issued, issued_slow = s_issued_slow;
    for (int g = max(0, issued - kStages); g < issued; ++g) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&full_bar[g % kStages], (g / kStages) & 1) &&
             globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    for (int g = max(0, issued_slow - S); g < issued_slow; ++g) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&sfull_bar[g % S], (g / S) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- projection G = X V_k as a GEMM (T > 1) ------------------------------
// D (128 entries of g x 64 tokens) = V^T rows (A, K-major: the handle's
// transposed copy of V_k) . X rows (B, K-major), over one of S slices of the
// reduction dimension d; each CTA writes its fp32 partial to P[s] (16-byte
// stores staged through the drained ring), and the gate kernel sums the S
// partials in a fixed order.  Same warp roles as tc_gemm_kernel.  For the
// batched path (a_fixed) the V^T boxes of the first stages load before the
// dependent-launch wait, and the CTAs of entries 0..127 also sum the squares
// of each staged x tile on their epilogue warps (||x||^2 over the slice).
constexpr int kPN = 64;  // tokens per tile (MMA N)
constexpr int kPStages = 4;       // ring depth when the grid is more than one wave
constexpr int kPMaxStages = 8;    // when every CTA is resident at once: a whole slice in flight
constexpr int kPABytes = kBM * kBK * 2;  // 16 KiB
constexpr int kPBBytes = kPN * kBK * 2;  // 8 KiB
constexpr int kPStageBytes = kPABytes + kPBBytes;
constexpr int kPTmemCols = 64;
constexpr size_t kPMaxSmem = size_t(kPMaxStages) * kPStageBytes + 1024;

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_proj_kernel(const __grid_constant__ CUtensorMap tmVT, const __grid_constant__ CUtensorMap tmX,
                   TcProjArgs a) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full_bar[kPMaxStages];
  __shared__ uint64_t empty_bar[kPMaxStages];
  __shared__ uint64_t accum_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued;

  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM, t0 = blockIdx.y * kPN, sl = blockIdx.z;
  const int nkb_all = (a.d + kBK - 1) / kBK;
  const int kb0 = min(nkb_all, sl * a.kb_per), kb1 = min(nkb_all, kb0 + a.kb_per);
  const int num_kb = kb1 - kb0;
  const int nvalid = min(kPN, a.T - t0);
  const int stages = min(max(a.stages, 1), kPMaxStages);
  // stages whose A box is loaded before the wait (A fixed for the launch)
  const int pre = a.a_fixed ? min(num_kb, stages) : 0;
  // the CTAs of entries 0..127 also sum the squares of their staged x tiles:
  // a stage is released by the MMAs' commit and by the 4 epilogue warps
  const bool do_sx = a.sxp != nullptr && blockIdx.x == 0;

  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* tiles = smem_raw + (base - smem_addr(smem_raw));
  if (threadIdx.x == 0) {
    for (int st = 0; st < stages; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], do_sx ? 5 : 1);
    }
    mbar_init(&accum_bar, 1);
    s_abort = 0;
    s_issued = 0;
    fence_mbar_init();
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full_bar[i], kPStageBytes);
      tma_load_2d(tiles + size_t(i) * kPStageBytes, &tmVT, (kb0 + i) * kBK, m0, &full_bar[i]);
    }
  }
  pdl_wait();  // x may come from the previous kernel
  if (warp == 1) tmem_alloc(&s_tmem, kPTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      for (; i < num_kb; ++i) {
        const int st = i % stages;
        if (i >= stages &&
            !wait_bounded(&empty_bar[st], ((i / stages) & 1) ^ 1, a.status, &s_abort))
          break;
        unsigned char* sa = tiles + size_t(st) * kPStageBytes;
        if (i >= pre) {
          mbar_arrive_expect_tx(&full_bar[st], kPStageBytes);
          tma_load_2d(sa, &tmVT, (kb0 + i) * kBK, m0, &full_bar[st]);
        }
        tma_load_2d(sa + kPABytes, &tmX, (kb0 + i) * kBK, t0, &full_bar[st]);
      }
      s_issued = i;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kPN);
      for (int i = 0; i < num_kb; ++i) {
        const int st = i % stages;
        if (!wait_bounded(&full_bar[st], (i / stages) & 1, a.status, &s_abort)) break;
        tc_fence_after();
        const uint32_t sa = base + uint32_t(st) * kPStageBytes;
        const uint32_t sb = sa + kPABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma_bf16(tmem, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb + kk * 32), idesc,
                      (i | kk) != 0 ? 1u : 0u);
        tc_commit(&empty_bar[st]);
      }
      tc_commit(&accum_bar);
    }
  } else {
    // epilogue: warps 2..5 own TMEM lane quarters (warp % 4); entry m0 + row
    const int q = warp & 3;
    if (do_sx) {
      // ||x||^2 over this slice: warp q takes tokens 16 q .. 16 q + 15 of the
      // tile, lane l token 16 q + l / 2 and half l % 2 of its 128-byte row
      // (the row's chunks are swizzled, which a sum of squares ignores);
      // rows past T are the tensor map's zero fill
      float sxl = 0.f;
      const int r = 16 * q + (lane >> 1);
      for (int i = 0; i < num_kb; ++i) {
        const int st = i % stages;
        if (!wait_bounded(&full_bar[st], (i / stages) & 1, a.status, &s_abort)) break;
        const uint4* xrow = reinterpret_cast<const uint4*>(tiles + size_t(st) * kPStageBytes +
                                                           kPABytes + size_t(r) * 128) +
                            (lane & 1) * 4;
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float f[8];
          bf16x8_to_f32(xrow[c], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) part = fmaf(f[e], f[e], part);
        }
        sxl += part;
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(&empty_bar[st]);
      }
      sxl += __shfl_xor_sync(0xFFFFFFFFu, sxl, 1);
      if ((lane & 1) == 0 && r < nvalid)
        a.sxp[size_t(sl) * a.sxp_stride + size_t(t0 + r)] = num_kb > 0 ? sxl : 0.f;
    }
    const bool ok = wait_bounded(&accum_bar, 0, a.status, &s_abort);
    tc_fence_after();
    const int row = m0 + q * 32 + lane;
    float* P = a.P + size_t(sl) * a.split_stride;
    if (ok && num_kb > 0 && a.k % 4 == 0 && (reinterpret_cast<uintptr_t>(P) & 15) == 0) {
      // Each 32 x 32 chunk goes through shared memory (the ring, drained
      // once the accumulator is complete) so that the warp writes 16-byte
      // vectors: lane (token j = lane / 8 + 4 p, rows 4 (lane % 8) .. + 3).
      float* stg = reinterpret_cast<float*>(tiles) + q * (32 * 33);
      const int jq = lane >> 3, o4 = (lane & 7) * 4;
      const int rq = m0 + q * 32 + o4;
      for (int c0 = 0; c0 < kPN; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(c0), r);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) stg[jj * 33 + lane] = __uint_as_float(r[jj]);
        __syncwarp();
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int jj = 4 * p + jq, j = c0 + jj;
          const float* src = stg + jj * 33 + o4;
          if (j < nvalid && rq < a.k)
            *reinterpret_cast<float4*>(P + size_t(t0 + j) * a.k + rq) =
                make_float4(src[0], src[1], src[2], src[3]);
        }
        __syncwarp();
      }
    } else {
      for (int c0 = 0; c0 < kPN; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(c0), r);
        if (row < a.k) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = c0 + jj;
            // a slice with no reduction steps contributes zero
            if (j < nvalid)
              P[size_t(t0 + j) * a.k + row] = (ok && num_kb > 0) ? __uint_as_float(r[jj]) : 0.f;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) {
    const int issued = s_issued;
    for (int i = max(0, issued - stages); i < issued; ++i) {
      const int st = i % stages;
      const uint64_t tw = globaltimer_ns();
      while (!mbar_try_wait(&full_bar[st], (i / stages) & 1) &&
             globaltimer_ns() - tw < kWaitLimitNs) {
      }
    }
  }
  if (warp == 1) {
    if (lane == 0) {
      const uint64_t tw = globaltimer_ns();
      while (!mbar_try_wait(&accum_bar, 0) && globaltimer_ns() - tw < kWaitLimitNs) {
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

// ---- host side: tensor maps ---------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return tma_encode_bf16_2d(map, base, rows, cols, box_rows, kBK);
}

}  // namespace

// 2-D bf16 row-major tensor (rows x cols), box of box_rows x box_cols, 128-byte
// swizzle (box_cols * 2 must be 128), zero fill outside the tensor.
bool tma_encode_bf16_2d(void* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int tc_gemm_launch_count() { return 1; }

// Ring depth of a projection launch: a whole slice in flight (up to 8 stages,
// about 193 KB of shared memory, one CTA per SM) when every CTA of the grid is
// resident at once; else 4 stages, so that two CTAs share an SM.
int proj_stages(int64_t ctas, int kb_per, int num_sms) {
  return ctas <= num_sms ? std::max(1, std::min(kPMaxStages, kb_per)) : kPStages;
}
size_t proj_smem(int stages) { return size_t(stages) * kPStageBytes + 1024; }

bool tc_proj_supported(const gsi_handle* h) { return h->k == 128 || h->k == 256; }

gsi_status_t tc_proj_prepare(gsi_handle* h) {
  if (!tc_proj_supported(h)) return GSI_OK;
  if (!tma_encode_bf16_2d(h->tmaps_proj, h->bVT, uint64_t(h->k), uint64_t(h->d), uint32_t(kBM), kBK))
    return GSI_ERR_CUDA;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(tc_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPMaxSmem)) != cudaSuccess)
      return GSI_ERR_CUDA;
    attr = true;
  }
  return GSI_OK;
}

int tc_proj_splits(const gsi_handle* h, int64_t T, int* kb_per) {
  const int nkb = int((h->d + kBK - 1) / kBK);
  const int tiles = int(h->k / kBM) * int((T + kPN - 1) / kPN);
  int S = std::max(1, std::min({kProjMaxSplits, nkb, (h->num_sms + tiles - 1) / tiles}));
  *kb_per = (nkb + S - 1) / S;
  S = (nkb + *kb_per - 1) / *kb_per;  // no empty slices
  return S;
}

gsi_status_t tc_nt_prepare() {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(tc_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPMaxSmem)) != cudaSuccess)
      return GSI_ERR_CUDA;
    attr = true;
  }
  return GSI_OK;
}

int tc_nt_splits(int64_t rows_a, int64_t rows_b, int64_t K, int num_sms, int* kb_per) {
  const int nkb = int((K + kBK - 1) / kBK);
  const int tiles = int((rows_a + kBM - 1) / kBM) * int((rows_b + kPN - 1) / kPN);
  int S = std::max(1, std::min({kProjMaxSplits, nkb, (num_sms + tiles - 1) / tiles}));
  *kb_per = (nkb + S - 1) / S;
  return (nkb + *kb_per - 1) / *kb_per;  // no empty slices
}

gsi_status_t tc_nt_gemm(const void* A, int64_t rows_a, const void* B, int64_t rows_b, int64_t K,
                        float* P, size_t split_stride, int S, int kb_per, uint32_t* status,
                        cudaStream_t s) {
  if (rows_a <= 0 || rows_b <= 0 || K <= 0 || K % 8 != 0 || !aligned16(A) || !aligned16(B))
    return GSI_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap tmA, tmB;
  if (!tma_encode_bf16_2d(&tmA, A, uint64_t(rows_a), uint64_t(K), uint32_t(kBM), kBK) ||
      !tma_encode_bf16_2d(&tmB, B, uint64_t(rows_b), uint64_t(K), uint32_t(kPN), kBK))
    return GSI_ERR_CUDA;
  TcProjArgs a;
  a.P = P;
  a.T = int(rows_b);
  a.d = int(K);
  a.k = int(rows_a);
  a.kb_per = kb_per;
  a.split_stride = split_stride;
  a.status = status;
  dim3 grid(unsigned((rows_a + kBM - 1) / kBM), unsigned((rows_b + kPN - 1) / kPN), unsigned(S));
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GSI_ERR_CUDA;
  }
  a.stages = proj_stages(int64_t(grid.x) * grid.y * grid.z, kb_per, sms);
  a.a_fixed = 0;  // A may be written by an earlier kernel of the stream
  a.sxp = nullptr;
  a.sxp_stride = 0;
  return launch_pdl(tc_proj_kernel, grid, dim3(kTcThreads), proj_smem(a.stages), s, tmA, tmB, a) ==
                 cudaSuccess
             ? GSI_OK
             : GSI_ERR_CUDA;
}

gsi_status_t tc_proj_launch(gsi_handle* h, const void* x, int64_t T, int S, int kb_per, cudaStream_t s) {
  CUtensorMap tmX;
  if (!tma_encode_bf16_2d(&tmX, x, uint64_t(T), uint64_t(h->d), uint32_t(kPN), kBK)) return GSI_ERR_CUDA;
  TcProjArgs a;
  a.P = h->bP;
  a.T = int(T);
  a.d = int(h->d);
  a.k = int(h->k);
  a.kb_per = kb_per;
  a.split_stride = size_t(h->max_T) * h->k;
  a.status = h->status;
  dim3 grid(unsigned(h->k / kBM), unsigned((T + kPN - 1) / kPN), unsigned(S));
  a.stages = proj_stages(int64_t(grid.x) * grid.y * grid.z, kb_per, h->num_sms);
  a.a_fixed = 1;  // the handle's V_k^T, written once when the workspace was bound
  a.sxp = h->bsxp;
  a.sxp_stride = size_t(h->max_T);
  const CUtensorMap* vt = reinterpret_cast<const CUtensorMap*>(h->tmaps_proj);
  return launch_pdl(tc_proj_kernel, grid, dim3(kTcThreads), proj_smem(a.stages), s, *vt, tmX, a) ==
                 cudaSuccess
             ? GSI_OK
             : GSI_ERR_CUDA;
}

gsi_status_t tc_gemm_prepare(gsi_handle* h) {
  static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
  static_assert(sizeof(TcMaps) <= sizeof(h->tmaps), "tensor map storage");
  TcMaps* maps = reinterpret_cast<TcMaps*>(h->tmaps);
  const uint64_t mt = uint64_t(h->max_T);
  bool ok = encode_2d(&maps->W, h->W, uint64_t(h->d_out), uint64_t(h->d), kBM) &&
            encode_2d(&maps->M, h->M, uint64_t(h->d_out), uint64_t(h->k), kBM);
  for (int b = 0; b < 4 && ok; ++b) {
    const uint32_t rows = uint32_t(kBoxRows[b]);
    ok = encode_2d(&maps->Xs[b], h->bXs, mt, uint64_t(h->d), rows) &&
         encode_2d(&maps->Ghi[b], h->bGf, mt, uint64_t(h->k), rows) &&
         encode_2d(&maps->Glo[b], h->bGf + size_t(mt) * h->k, mt, uint64_t(h->k), rows);
  }
  if (!ok) return GSI_ERR_CUDA;
  if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kTcSmem)) != cudaSuccess)
    return GSI_ERR_CUDA;
  return GSI_OK;
}

gsi_status_t tc_gemm_launch(gsi_handle* h, const TcGemmArgs& a, cudaStream_t s) {
  const TcMaps* maps = reinterpret_cast<const TcMaps*>(h->tmaps);
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GSI_ERR_CUDA;
  }
  // at most one CTA per SM (the ring takes most of shared memory), and no more
  // CTAs than tiles could exist (slow tiles of 256 tokens, fast of 128)
  const int n_tiles = (a.T + kBNF - 1) / kBNF;
  const int max_tiles = ((a.d_out + kBM - 1) / kBM) * (n_tiles + 1);
  dim3 grid(unsigned(std::max(1, std::min(sms, max_tiles))));
  return launch_pdl(tc_gemm_kernel, grid, dim3(kTcThreads), kTcSmem, s, *maps, a) == cudaSuccess
             ? GSI_OK
             : GSI_ERR_CUDA;
}

}  // namespace gsi
