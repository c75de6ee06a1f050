// gsi_decode_cr.cu -- the T = 1 (decode) path of the GSI gated linear map:
// one kernel per call with ONE exchange between CTAs, sized so that two CTAs
// fit on an SM (k in {64, 128, 256}).
//
// Page: "Technical summary: Gated Subspace Inference for transformer
// acceleration" [GSI].  Per token x (section 2.1 eq. 1-2, section 2.2):
//   g = V_k^T x,  rho = ||x - V_k g|| / ||x||,
//   y = M g if rho < eps (fast path), y = W x otherwise (slow path).
//
// Why two CTAs per SM.  Decode tokens are sequential, so one call's kernel
// cannot read its x before the previous kernel has finished; what it can do
// is stage the weights it will need (its slices of V_k and M), which do not
// depend on x.  With at most ~113 KB of shared memory and 288 threads per
// CTA, the next call's CTAs become resident beside this call's (programmatic
// dependent launch) and stage their slices from HBM while this call runs its
// exchange, so a call starts with its operands already on chip.
//
// Roles.  A call runs on G co-resident CTAs.  CTA 0 is the gate CTA: it
// stages the correction tiles of E = V_k^T V_k - I (bf16, MMA operand order)
// and computes the exact residual ratio
//   rho^2 = (||x||^2 - g.g + g^T E g) / ||x||^2
// (the Gram identity for any V_k, since g = V_k^T x), writes gate and rho, and
// publishes the gate.  CTAs 1..G-1 each own d / (G-1) rows of V_k and
// d_out / (G-1) output rows; they stage those rows of V_k and M (2-D TMA,
// 128-byte swizzle) before the dependent-launch wait.  They decide the gate
// themselves from
//   |g^T E g| <= ||E||_2 g.g
// (||E||_2 bounded above once per handle), with directed rounding so that a
// decision they take is the one the gate CTA takes; only for a token whose
// rho is within that bound of eps (about 5% of eps at k = 256) do they wait
// for the gate CTA's published gate.  The correction is therefore off the
// critical path of every other CTA.
//
// Exchange.  Every CTA reads all of x: ||x||^2 (a fixed-order fp32 sum), the
// non-finite test and the exponent of max|x_i| are then the same, bit for
// bit, in every CTA without an exchange.  The partial projections
// V_c^T x_c (warp-level bf16 MMAs, fp32 accumulation) are turned into fixed
// point at a scale set by max|x| and split into two 19-bit integer digits,
// each an exact fp32 integer; the digits are added with vector red.add into
// one of 8 accumulator copies (at most 19 contributors each, so every sum is
// an exact integer below 2^24).  Integer addition is associative, so g does
// not depend on the order in which the CTAs' atomics arrive: g, rho and the
// gate are reproducible bit for bit, and calls on handles that hold
// different rows of the same W (one per GPU) take identical gates.
//
// Phases (CTAs 1..G-1):
//   0  x (all of it): ||x||^2, max|x|, this CTA's slice of x
//   1  partial g over its V_k rows, digits, red.add; grid barrier
//   2  g from the 16 digit sums of each entry; g.g; gate decision
//   3  fast: M_c g (units of 64 columns of M, partials added in a fixed
//      order); slow: W_c x, W streamed from HBM.
// The accumulators are double-buffered by a launch epoch kept on the device
// (the gate CTA clears the buffer the next launch uses), so the kernel
// replays in a CUDA graph without a memset.  Every wait is bounded.
#include <cuda.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstring>

#include "gsi_device.cuh"
#include "gsi_internal.h"
#include "gsi_tc_gemm.h"

namespace gsi {
namespace {

constexpr int kThreads = 256;               // compute threads (8 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads + 32;       // + one warp that issues the L2 prefetches
constexpr int kCopies = 8;                  // accumulator copies (every CTA reads all of them)
constexpr int kPerCopy = 63;                // contributors per copy (the count field)
constexpr int kMaxGrid = kCopies * kPerCopy + 1;
constexpr int kDigitBits = 19;
constexpr int kFixBits = 38;                // |partial| < 2^38 units of the fixed point
constexpr int kCountShift = 58;             // arrivals above the summed fixed point
constexpr int kMaxBoxRows = 256;            // TMA box limit
constexpr int kMaxPf = 12;                  // prefetch ranges (3 per handle, up to 4 handles)
constexpr size_t kCoresidentSmem = 115712;  // 2 x (this + 1 KB reserved) <= 228 KB per SM
constexpr int kSlowAhead = 2;               // slow path: units of W prefetched ahead per warp
constexpr int kMaxXChunks = 8;              // 16-byte chunks of x per thread: d <= 16384
constexpr int kMaxD = kMaxXChunks * kThreads * 8;

struct CrArgs {
  const __nv_bfloat16* W;
  const __nv_bfloat16* F;
  const __nv_bfloat16* x;
  float* y;
  uint8_t* gate;
  float* rho;
  int d_out, d;
  float eps;
  float normE;          // upper bound of ||E||_2 (E as its bf16 tiles represent it)
  int vbits;            // 2^vbits >= sqrt(rows_V) x max column norm of V_k (partial bound)
  int rows_M, rows_V;   // rows owned per CTA 1..G-1
  int box_M, box_V;     // TMA box rows (multiples of 16, <= 256)
  int nbox_M, nbox_V;   // row boxes per CTA
  uint64_t* acc;        // [2][kCopies][K] counted fixed-point words
  uint32_t* bar;        // [1] launch epoch, [4..5] published gate word
  uint32_t* status;
  const char* pf[kMaxPf];
  uint32_t pf_bytes[kMaxPf];
  int pf_part0, pf_parts;
};

struct CrGroupMaps {
  CUtensorMap m[2 * kMaxGroup];  // V_k and M maps of each member
};
struct CrGroupArgs {
  CrArgs a[kMaxGroup];
  int cta0[kMaxGroup + 1];
  int n;
};

// Small per-CTA state at the end of the dynamic shared memory (the kernel has
// no static shared memory, so the dynamic base is the CTA's first byte).
struct CrCtl {
  uint64_t mbar[2];          // [0] V_k slice, [1] M slice (or correction tiles)
  float sxw[kWarps];         // per-warp ||x||^2 partials
  uint32_t mxw[kWarps];      // per-warp max |x| (fp32 bits; >= 0x7F800000: NaN or Inf)
  float ggw[kWarps];         // per-warp g.g partials
  float qw[kWarps];          // per-warp correction partials (gate CTA)
  uint32_t epoch;
  int ok, dec;
  float rho;
};

// Dynamic shared-memory layout (byte offsets from the 1024-aligned base),
// identical on host and device.
//   A   [0, B): the M slice (K / 64 column blocks of rowsM x 128 bytes, TMA
//       swizzled); x on the slow path, then (d a multiple of 1024) its
//       per-segment row sums where they fit (else at the head of B)
//   B   [B, B + b): the V_k slice (same layout)
//   aux g, the B fragments of g and the M g partials: the tail of B (dead
//       once the projection is done) when they fit, else after it
// The gate CTA, which stages neither slice, keeps the correction tiles at
// [0, F), which ends before aux.  x slice and control words follow.
struct CrLay {
  size_t B, part, g, bfrag, yp, xs, ctl, total;
};
__host__ __device__ inline size_t cr_al(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline CrLay cr_layout(int K, int d, int rowsM, int rowsV) {
  CrLay s;
  const size_t a_M = size_t(K / 64) * rowsM * 128;
  const size_t a_x = size_t(d) * 2;
  const size_t a_F = corr_tiles_elems(K) * 2;
  s.B = cr_al(a_M > a_x ? a_M : a_x, 1024);
  const size_t b = size_t(K / 64) * rowsV * 128;
  const size_t n_g = cr_al(size_t(K) * 4, 16), n_bf = cr_al(size_t(K / 16) * 64, 16);
  const size_t n_yp = cr_al(size_t(rowsM) * (K / 64) * 4, 16);
  const size_t aux = n_g + n_bf + n_yp;
  // The slow path's per-segment row sums (d a multiple of 1024): after x in
  // A, else at the head of the V_k slice (dead by then) ahead of aux, else
  // in A grown to hold them.
  const size_t n_part = d % 1024 == 0 ? size_t(rowsM) * (d / 1024) * 4 : 0;
  if (a_x + n_part <= s.B) {
    s.part = a_x;
  } else if (aux <= b && n_part <= b - aux) {
    s.part = s.B;
  } else {
    s.part = a_x;
    s.B = cr_al(a_x + n_part, 1024);
  }
  size_t ax = aux <= b ? s.B + b - aux : s.B + b;
  ax = ax > cr_al(a_F, 16) ? ax : cr_al(a_F, 16);
  s.g = ax;
  s.bfrag = ax + n_g;
  s.yp = s.bfrag + n_bf;
  const size_t end = s.B + b > ax + aux ? s.B + b : ax + aux;
  s.xs = cr_al(end, 16);
  s.ctl = cr_al(s.xs + size_t(rowsV) * 2, 16);
  s.total = s.ctl + cr_al(sizeof(CrCtl), 16);
  return s;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}
// x is written by the kernel before this one: read it at L2 (coherent), not
// through the non-coherent or L1 paths.
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

// Named barrier 1: the 8 compute warps only (the prefetch warp's bulk
// prefetches can stall it for a microsecond or more).
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
// Named barrier 2 (all kBlock threads): the compute warps arrive once the grid
// exchange is done; the prefetch warp waits for that.
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

// D += A B, one 16 x 16 (A, row-major) by 16 x 8 (B, column-major) bf16
// product with fp32 accumulation (PTX fragment layout).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
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

// v 2^n for a power-of-two factor, exact while the result is a normal
// number: two factors 2^(n/2) and 2^(n - n/2), each inside the fp32 exponent
// range for |n| <= 252.
__device__ __forceinline__ float scale_pow2(float v, int n) {
  const int n1 = n / 2, n2 = n - n1;
  return (v * __int_as_float((127 + n1) << 23)) * __int_as_float((127 + n2) << 23);
}

// The nearest integer q to v 2^-lsb (|v| < 2^(lsb + kFixBits), so
// |q| <= 2^38), in fp32 arithmetic only (64-bit conversions are slow on this
// part): r = rint(v 2^-lsb) is exact in fp32, r = h 2^19 + l with
// h = floor(r 2^-19) and 0 <= l < 2^19 both exact, then q from the integers.
__device__ __forceinline__ long long to_fixed(float v, int lsb) {
  const float r = rintf(scale_pow2(v, -lsb));
  const float h = floorf(r * (1.f / float(1 << kDigitBits)));
  const float l = fmaf(-h, float(1 << kDigitBits), r);
  return (long long)__float2int_rz(h) * (1ll << kDigitBits) + __float2int_rz(l);
}
__device__ __forceinline__ void red_add_u64(uint64_t* p, uint64_t v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

// One one-token call on CTAs 0..G-1 of its own (cta = this CTA's index).
template <int K>
__device__ __forceinline__ void cr_body(const CUtensorMap* tmV, const CUtensorMap* tmM,
                                        const CrArgs& a, const int cta, const int G) {
  static_assert(K == 64 || K == 128 || K == 256, "k in {64, 128, 256}");
  constexpr int T16 = K / 16;  // 16-wide blocks of g
  constexpr int KC = K / 64;   // 64-column (128-byte) blocks of a row
  constexpr int S = K / 64;    // M g units per row block (4 blocks of 16 columns each)
  static_assert(kWarps % S == 0, "each warp keeps one column range of M");
  extern __shared__ __align__(1024) unsigned char smem[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int rowsM = a.nbox_M * a.box_M, rowsV = a.nbox_V * a.box_V;
  const CrLay lay = cr_layout(K, a.d, rowsM, rowsV);
  const uint32_t sbase = smem_addr(smem);
  // Launch self-check (uniform over the grid, before any wait): a launch that
  // does not cover d and d_out, got less shared memory than its layout, or
  // whose shared memory is not 1024-aligned (the swizzle) does nothing.
  if (blockDim.x != kBlock || G < 2 || G > kMaxGrid || (sbase & 1023u) != 0u ||
      int64_t(G - 1) * a.rows_M < a.d_out || int64_t(G - 1) * a.rows_V < a.d ||
      rowsM < a.rows_M || rowsV < a.rows_V || dynamic_smem_bytes() < lay.total) {
    if (cta == 0 && tid == 0) atomicOr(a.status, kStatusBadLaunch);
    return;
  }
  const bool gate_cta = cta == 0;
  const int m0 = gate_cta ? 0 : (cta - 1) * a.rows_M;
  const int nM = gate_cta ? 0 : max(0, min(a.d_out, m0 + a.rows_M) - m0);
  const int v0 = gate_cta ? 0 : (cta - 1) * a.rows_V;
  const int nV = gate_cta ? 0 : max(0, min(a.d, v0 + a.rows_V) - v0);

  CrCtl& ctl = *reinterpret_cast<CrCtl*>(smem + lay.ctl);
  __nv_bfloat16* s_xs = reinterpret_cast<__nv_bfloat16*>(smem + lay.xs);  // [rowsV]
  float* s_g = reinterpret_cast<float*>(smem + lay.g);                    // [K]
  __nv_bfloat16* s_bf = reinterpret_cast<__nv_bfloat16*>(smem + lay.bfrag);  // [T16][8 lanes][4]
  float* s_yp = reinterpret_cast<float*>(smem + lay.yp);                  // [row blocks][S][16]

  // ---- prologue: stage this CTA's weights (independent of x) ------------
  if (tid == 0) {
    mbar_init(&ctl.mbar[0], 1);
    mbar_init(&ctl.mbar[1], 1);
    fence_mbar_init();
  }
  for (int i = tid; i < rowsV / 2; i += kBlock) reinterpret_cast<uint32_t*>(s_xs)[i] = 0u;
  __syncthreads();
  if (warp == kWarps) {
    // The staging and prefetch warp.  Staging: this CTA's rows of V_k and M
    // (or the correction tiles), which do not depend on x, issued as soon as
    // the CTA is resident (while the previous call runs, when it became
    // resident beside it).
    pdl_launch_dependents();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmV)) : "memory");
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmM)) : "memory");
      if (!gate_cta) {
        const uint32_t bytes_V = uint32_t(a.box_V) * 128, bytes_M = uint32_t(a.box_M) * 128;
        mbar_arrive_expect_tx(&ctl.mbar[0], KC * a.nbox_V * bytes_V);
        for (int kc = 0; kc < KC; ++kc)
          for (int b = 0; b < a.nbox_V; ++b)
            tma_load_2d(smem + lay.B + size_t(kc) * rowsV * 128 + size_t(b) * bytes_V, tmV, kc * 64,
                        v0 + b * a.box_V, &ctl.mbar[0]);
        mbar_arrive_expect_tx(&ctl.mbar[1], KC * a.nbox_M * bytes_M);
        for (int kc = 0; kc < KC; ++kc)
          for (int b = 0; b < a.nbox_M; ++b)
            tma_load_2d(smem + size_t(kc) * rowsM * 128 + size_t(b) * bytes_M, tmM, kc * 64,
                        m0 + b * a.box_M, &ctl.mbar[1]);
      } else {
        const uint32_t bytes_F = uint32_t(corr_tiles_elems(K)) * 2;
        mbar_arrive_expect_tx(&ctl.mbar[1], bytes_F);
        constexpr uint32_t kChunk = 32768;
        const char* gF = reinterpret_cast<const char*>(a.F);
        for (uint32_t off = 0; off < bytes_F; off += kChunk)
          bulk_g2s(smem + off, gF + off, min(kChunk, bytes_F - off), &ctl.mbar[1]);
      }
      // This CTA's share of x (whole 128-byte lines) into L2 before the
      // dependent-launch wait.  A prefetch reads nothing into the program,
      // so it is safe while the previous kernel may still be writing x:
      // those writes land in L2, which every later read of x goes through.
      const uint32_t xbytes = uint32_t(a.d) * 2u;
      const uint32_t xshare = max(128u, (xbytes / uint32_t(G) + 127u) & ~127u);
      const uint32_t xlo = uint32_t(cta) * xshare;
      if (xlo < xbytes)
        prefetch_l2(reinterpret_cast<const char*>(a.x) + xlo, min(xshare, xbytes - xlo));
    }
    __syncwarp();
    // Prefetch: once the compute warps are past the exchange, this CTA's
    // share of the linked call's operands, into L2; then the warp exits.
    // Weights only: it reads nothing the previous kernel writes.
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
  pdl_launch_dependents();
  pdl_wait();  // x and this handle's workspace are now safe to touch

  // ---- phase 0: all of x: ||x||^2, max|x|, this CTA's slice ---------------
  if (tid == 0) {
    ctl.epoch = ld_cg_u32(a.bar + 1);
    ctl.ok = 1;
  }
  {
    float sxp = 0.f;
    uint32_t mx = 0u;
    const uint4* x4 = reinterpret_cast<const uint4*>(a.x);
    const int nch = a.d / 8;
    // all of this thread's chunks are requested before any is used: one
    // round trip to memory, not one per chunk
    uint4 xv[kMaxXChunks];
#pragma unroll
    for (int j = 0; j < kMaxXChunks; ++j)
      if (tid + j * kThreads < nch) xv[j] = ld_cg_v4(x4 + tid + j * kThreads);
#pragma unroll
    for (int j = 0; j < kMaxXChunks; ++j) {
      const int i = tid + j * kThreads;
      if (i >= nch) break;
      const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t lo = w[q] << 16, hi = w[q] & 0xFFFF0000u;
        const float fl = __uint_as_float(lo), fh = __uint_as_float(hi);
        sxp = fmaf(fl, fl, sxp);
        sxp = fmaf(fh, fh, sxp);
        mx = max(mx, max(lo & 0x7FFFFFFFu, hi & 0x7FFFFFFFu));
      }
      const int e0 = 8 * i;
      if (e0 + 8 > v0 && e0 < v0 + nV) {
        const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&xv[j]);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (e0 + q >= v0 && e0 + q < v0 + nV) s_xs[e0 + q - v0] = xb[q];
      }
    }
    sxp = warp_sum_all(sxp);
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) {
      ctl.sxw[warp] = sxp;
      ctl.mxw[warp] = mx;
    }
  }
  bool ok = gate_cta ? true : mbar_wait_bounded(&ctl.mbar[0], 0, a.status);
  ok = sync_compute_and(ok);
  float sx = 0.f;
  uint32_t mxall = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {  // same order in every thread and CTA
    sx += ctl.sxw[w];
    mxall = max(mxall, ctl.mxw[w]);
  }
  const bool nonfinite = mxall >= 0x7F800000u;
  // max|x| < 2^ex; the partials of g are below 2^(ex + vbits)
  const int ex = mxall == 0u ? 0 : int((mxall >> 23) & 0xFFu) - 126;
  const int lsb = ex + a.vbits - kFixBits;
  const uint32_t e = ctl.epoch;
  uint64_t* acc = a.acc + size_t(e & 1u) * kCopies * K;
  if (gate_cta) {  // clear the words the next launch accumulates into
    uint64_t* nxt = a.acc + size_t((e + 1u) & 1u) * kCopies * K;
    for (int i = tid; i < kCopies * K; i += kThreads) nxt[i] = 0u;
  }

  // ---- phase 1: partial g over this CTA's rows of V_k, added as counted words --
  // CTAs 1..P (those that own rows of V_k) each add every entry of their
  // partial projection once, into copy (cta - 1) % kCopies.  A word is
  //   (arrivals << 58) + sum over arrivals of (q + 2^38),
  // q the partial in fixed point (|q| <= 2^38): one 64-bit atomic adds a
  // partial and its arrival together, so a reader that sees the full count
  // has every partial, with no fence and no separate barrier.
  const int P = min(G - 1, (a.d + a.rows_V - 1) / a.rows_V);
  if (nV > 0 && !nonfinite && warp < T16) {
    constexpr int kGB = T16 >= kWarps ? T16 / kWarps : 1;  // g blocks per warp (1 or 2)
    const int nkb = (nV + 15) / 16;
    const int j8 = lane >> 3, rr = lane & 7;
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(s_xs);
    float v0g[kGB], v8g[kGB];
#pragma unroll
    for (int gb = 0; gb < kGB; ++gb) {
      const int mb = warp + gb * kWarps;
      const int col = mb * 16 + (j8 & 1) * 8;  // A rows = entries of g
      const uint32_t blk = sbase + uint32_t(lay.B) + uint32_t(col / 64) * uint32_t(rowsV) * 128u;
      const int chunk = (col % 64) / 8;
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      int kb = 0;
      for (; kb + 1 < nkb; kb += 2) {
        const uint4 A0 = ldsm_x4_trans(swz(blk, kb * 16 + rr + (j8 >> 1) * 8, chunk));
        const uint4 A1 = ldsm_x4_trans(swz(blk, (kb + 1) * 16 + rr + (j8 >> 1) * 8, chunk));
        const uint32_t b00 = grp == 0 ? xw[kb * 8 + tig] : 0u;
        const uint32_t b01 = grp == 0 ? xw[kb * 8 + 4 + tig] : 0u;
        const uint32_t b10 = grp == 0 ? xw[(kb + 1) * 8 + tig] : 0u;
        const uint32_t b11 = grp == 0 ? xw[(kb + 1) * 8 + 4 + tig] : 0u;
        mma_16816(d0, A0, b00, b01);
        mma_16816(d1, A1, b10, b11);
      }
      if (kb < nkb) {
        const uint4 A0 = ldsm_x4_trans(swz(blk, kb * 16 + rr + (j8 >> 1) * 8, chunk));
        mma_16816(d0, A0, grp == 0 ? xw[kb * 8 + tig] : 0u, grp == 0 ? xw[kb * 8 + 4 + tig] : 0u);
      }
      // column 0 of D: lanes with tig == 0 hold entries grp (d[0]) and grp + 8 (d[2])
      v0g[gb] = d0[0] + d1[0];
      v8g[gb] = d0[2] + d1[2];
    }
    // lane l takes entry l % 16 of g block l / 16
    const int src = 4 * (lane & 7);
    float val = 0.f;
#pragma unroll
    for (int gb = 0; gb < kGB; ++gb) {
      const float a0 = __shfl_sync(0xFFFFFFFFu, v0g[gb], src);
      const float a8 = __shfl_sync(0xFFFFFFFFu, v8g[gb], src);
      if ((lane >> 4) == gb) val = (lane & 8) ? a8 : a0;
    }
    if ((lane >> 4) < kGB) {
      // a CTA whose staging timed out still counts its arrival (with zero),
      // so that the others do not wait for it; the status word reports it
      const long long q = to_fixed(ok ? val : 0.f, lsb);
      const uint64_t add = (uint64_t(1) << kCountShift) + uint64_t(q + (1ll << kFixBits));
      const int entry = (warp + (lane >> 4) * kWarps) * 16 + (lane & 15);
      red_add_u64(acc + size_t((cta - 1) % kCopies) * K + entry, add);
    }
  }

  // ---- phase 2: g from the counted words (the same bits in every CTA) -------
  // thread t reads entry t of every copy until each copy's count is complete
  float g2 = 0.f;
  int good = 1;
  if (tid < K && !nonfinite) {
    uint64_t w[kCopies];
#pragma unroll
    for (int c = 0; c < kCopies; ++c) w[c] = ld_relaxed_u64(acc + size_t(c) * K + tid);
    auto complete = [&]() {
      bool all = true;
#pragma unroll
      for (int c = 0; c < kCopies; ++c)
        all = all && int(w[c] >> kCountShift) == P / kCopies + (c < P % kCopies ? 1 : 0);
      return all;
    };
    if (!complete()) {
      const uint64_t t0 = globaltimer_ns();
      while (true) {
#pragma unroll
        for (int c = 0; c < kCopies; ++c)
          if (int(w[c] >> kCountShift) != P / kCopies + (c < P % kCopies ? 1 : 0))
            w[c] = ld_relaxed_u64(acc + size_t(c) * K + tid);
        if (complete()) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(a.status, kStatusTimeout);
          good = 0;
          break;
        }
      }
    }
    long long qs = 0;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) {
      const long long n = (long long)(w[c] >> kCountShift);
      qs += (long long)(w[c] & ((uint64_t(1) << kCountShift) - 1)) - (n << kFixBits);
    }
    // qs 2^lsb in fp32: a fixed function of the exact integer sum
    const float q = fmaf(float(int(qs >> kDigitBits)), float(1 << kDigitBits),
                         float(int(qs & ((1ll << kDigitBits) - 1))));
    const float gt = scale_pow2(q, lsb);
    s_g[tid] = gt;
    g2 = gt * gt;
    // B operand of the MMAs below: g_t is row kk = t % 16 of column block
    // t / 16; lanes 0..3 hold the high part (column 0), lanes 4..7 the
    // remainder (column 1), register kk / 8, half kk % 2, lane pair (kk % 8) / 2
    const __nv_bfloat16 h = __float2bfloat16_rn(gt);
    const __nv_bfloat16 l = __float2bfloat16_rn(gt - __bfloat162float(h));
    const int kk = tid & 15, reg = kk >> 3, half = kk & 1, pr = (kk & 7) >> 1;
    __nv_bfloat16* bf = s_bf + (tid >> 4) * 32;
    bf[(pr * 2 + reg) * 2 + half] = h;
    bf[((4 + pr) * 2 + reg) * 2 + half] = l;
  }
  ok = sync_compute_and(good != 0) && ok;
  signal_prefetch_warp();
  g2 = warp_sum_all(g2);
  if (lane == 0) ctl.ggw[warp] = g2;
  sync_compute();
  float gg = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) gg += ctl.ggw[w];
  const float d0 = sx - gg;

  // ---- the gate ---------------------------------------------------------------
  if (gate_cta) {
    // exact correction g^T E g over the tiles (I, J), I <= J
    const bool staged = mbar_wait_bounded(&ctl.mbar[1], 0, a.status);
    ok = sync_compute_and(staged) && ok;
    float qsum = 0.f;
    if (ok) {
      // Tiles (I, J), I <= J, by column: columns J1 = p and J2 = T16 - 1 - p
      // hold T16 + 1 tiles together; the kWpp warps of pair p split them into
      // segments of kSeg.  Step s of a pair: column J1 for s <= J1 (row
      // I = s), else column J2 (row I = s - J1 - 1).  Tiles are loaded in
      // batches, their MMAs are independent.
      constexpr int kPairs = T16 / 2, kWpp = kWarps / kPairs;
      constexpr int kSeg = (T16 + 1 + kWpp - 1) / kWpp;
      constexpr int kBatch = kSeg < 6 ? kSeg : 6;
      const int p = warp / kWpp, qh = warp % kWpp;
      const int J1 = p, J2 = T16 - 1 - p;
      const uint4* tiles = reinterpret_cast<const uint4*>(smem);
      const uint2* bfr = reinterpret_cast<const uint2*>(s_bf);
      const uint2 bJ1 = lane < 8 ? bfr[J1 * 8 + lane] : make_uint2(0u, 0u);
      const uint2 bJ2 = lane < 8 ? bfr[J2 * 8 + lane] : make_uint2(0u, 0u);
#pragma unroll
      for (int b0 = 0; b0 < kSeg; b0 += kBatch) {
        uint4 fa[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int st = qh * kSeg + b0 + q;
          const bool first = st <= J1;
          const int I = first ? st : st - J1 - 1, J = first ? J1 : J2;
          fa[q] = (b0 + q < kSeg && st <= T16) ? tiles[corr_tile_index(I, J, T16) * 32 + lane]
                                                : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int st = qh * kSeg + b0 + q;
          if (b0 + q < kSeg && st <= T16) {
            const bool first = st <= J1;
            const int I = first ? st : st - J1 - 1;
            float dd[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(dd, fa[q], first ? bJ1.x : bJ2.x, first ? bJ1.y : bJ2.y);
            // columns 0 (high) and 1 (remainder) of rows grp and grp + 8
            qsum = fmaf(s_g[I * 16 + grp], dd[0] + dd[1], qsum);
            qsum = fmaf(s_g[I * 16 + grp + 8], dd[2] + dd[3], qsum);
          }
        }
      }
    }
    if (tig != 0) qsum = 0.f;
    qsum = warp_sum_all(qsum);
    if (lane == 0) ctl.qw[warp] = qsum;
    sync_compute();
    if (tid == 0) {
      float quad = 0.f;
      for (int w = 0; w < kWarps; ++w) quad += ctl.qw[w];
      float rho;
      if (!(fabsf(sx) <= FLT_MAX)) {
        rho = __int_as_float(0x7FC00000);  // non-finite x: NaN, slow path
      } else if (sx == 0.f) {
        rho = 0.f;
      } else {
        float sr = d0 + quad;
        if (!(sr >= 0.f)) sr = (sr == sr) ? 0.f : sr;
        rho = sqrtf(sr / sx);
      }
      if (!ok) rho = __int_as_float(0x7FC00000);  // a wait ran out: say so in the outputs
      const uint32_t gt = (rho < a.eps) ? 0u : 1u;
      if (a.gate) a.gate[0] = uint8_t(gt);
      if (a.rho) a.rho[0] = rho;
      // the gate word carries its own launch tag: no other data is published
      // with it, so it needs no fence; the epoch and base are read by the
      // next launch only after this kernel has completed
      st_relaxed_u64(reinterpret_cast<uint64_t*>(a.bar + 4), (uint64_t(e + 1u) << 32) | gt);
      a.bar[1] = e + 1u;  // every CTA read the epoch before its first exchange word
    }
    return;
  }

  // CTAs 1..G-1: the gate from the bound |g^T E g| <= ||E||_2 g.g, with
  // rounding directed so that a decision taken here is the gate CTA's.
  if (tid == 0) {
    int dec;  // 0 fast, 1 slow, 2 ask the gate CTA
    if (!(fabsf(sx) <= FLT_MAX)) {
      dec = 1;
    } else if (sx == 0.f) {
      dec = (0.f < a.eps) ? 0 : 1;
    } else if (!(a.eps > 0.f)) {
      dec = 1;  // rho >= 0 >= eps
    } else {
      // The gate CTA takes rho = sqrt(sr / sx) with sr = d0 + q, |q| <= Q.
      // Compare d0 +- Q with eps^2 sx instead, each side moved by a relative
      // 1e-5, which covers the roundings of these few operations and of the
      // gate CTA's division and square root (a few 2^-24 each).
      const float Q = a.normE * gg * 1.02f;
      const float t = a.eps * a.eps * sx;
      if (!(Q <= FLT_MAX) || d0 != d0) {
        dec = 2;
      } else if ((d0 + Q) * 1.00001f < t * 0.99999f) {
        dec = 0;
      } else if ((d0 - Q) * 0.99999f > t * 1.00001f) {
        dec = 1;
      } else {
        dec = 2;
      }
    }
    if (dec == 2 && ok) {
      const uint64_t want = uint64_t(e + 1u);
      const uint64_t* word = reinterpret_cast<const uint64_t*>(a.bar + 4);
      uint64_t w = ld_relaxed_u64(word);
      if ((w >> 32) != want) {
        const uint64_t t0 = globaltimer_ns();
        while (((w = ld_relaxed_u64(word)) >> 32) != want) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.status, kStatusTimeout);
            ctl.ok = 0;
            break;
          }
        }
      }
      dec = int(w & 1u);
    }
    ctl.dec = dec;
  }
  const bool staged = mbar_wait_bounded(&ctl.mbar[1], 0, a.status);
  ok = sync_compute_and(staged) && ok && ctl.ok;
  const bool slow = ctl.dec != 0;

  // ---- phase 3: the branch the gate picked --------------------------------------
  if (!ok) {
    for (int r = tid; r < nM; r += kThreads) a.y[m0 + r] = __int_as_float(0x7FC00000);
  } else if (!slow) {
    // M_c g in units of (16 rows) x (64 columns); warp w always takes the
    // column range w % S, so its B operands are loaded once
    const int RB = (nM + 15) / 16;
    const int s = warp % S;
    uint2 b[4];
    const uint2* bfr = reinterpret_cast<const uint2*>(s_bf);
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = lane < 8 ? bfr[(s * 4 + q) * 8 + lane] : make_uint2(0u, 0u);
    const int j8 = lane >> 3, rr = lane & 7;
    const uint32_t blkM = sbase + uint32_t(s) * uint32_t(rowsM) * 128u;
    // two units at a time (units u and u + kWarps: the same column range),
    // four independent MMA chains
    for (int u = warp; u < RB * S; u += 2 * kWarps) {
      const int u2 = u + kWarps;
      const bool two = u2 < RB * S;
      const int row = (u / S) * 16 + rr + (j8 & 1) * 8;
      const int row2 = (two ? u2 / S : u / S) * 16 + rr + (j8 & 1) * 8;
      float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
      float f0[4] = {0.f, 0.f, 0.f, 0.f}, f1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 4; q += 2) {
        const uint4 A0 = ldsm_x4(swz(blkM, row, q * 2 + (j8 >> 1)));
        const uint4 A1 = ldsm_x4(swz(blkM, row, (q + 1) * 2 + (j8 >> 1)));
        const uint4 B0 = ldsm_x4(swz(blkM, row2, q * 2 + (j8 >> 1)));
        const uint4 B1 = ldsm_x4(swz(blkM, row2, (q + 1) * 2 + (j8 >> 1)));
        mma_16816(e0, A0, b[q].x, b[q].y);
        mma_16816(e1, A1, b[q + 1].x, b[q + 1].y);
        mma_16816(f0, B0, b[q].x, b[q].y);
        mma_16816(f1, B1, b[q + 1].x, b[q + 1].y);
      }
      if (tig == 0) {
        float* dst = s_yp + size_t(u) * 16;
        dst[grp] = (e0[0] + e0[1]) + (e1[0] + e1[1]);
        dst[grp + 8] = (e0[2] + e0[3]) + (e1[2] + e1[3]);
        if (two) {
          float* dst2 = s_yp + size_t(u2) * 16;
          dst2[grp] = (f0[0] + f0[1]) + (f1[0] + f1[1]);
          dst2[grp + 8] = (f0[2] + f0[3]) + (f1[2] + f1[3]);
        }
      }
    }
    sync_compute();
    for (int r = tid; r < nM; r += kThreads) {
      const float* src = s_yp + size_t(r / 16) * S * 16 + (r % 16);
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < S; ++q) v += src[q * 16];
      a.y[m0 + r] = v;
    }
  } else {
    // W_c x, W streamed from HBM: 4 rows per warp at a time, 4 16-byte
    // pieces per row and lane in flight, refilled half at a time (the next
    // step's pieces 0-1 load while pieces 2-3 are summed), so that the loads in
    // flight never drain to zero; the order of each row's sum does not depend
    // on which CTA or warp owns the row
    const int nch = a.d / 8;
    const uint64_t pol = l2_evict_first_policy();  // W is read once per call
    uint4* x4 = reinterpret_cast<uint4*>(smem);  // the M slice is not needed here
    {
      uint4 xv[kMaxXChunks];
      const uint4* gx = reinterpret_cast<const uint4*>(a.x);
#pragma unroll
      for (int j = 0; j < kMaxXChunks; ++j)
        if (tid + j * kThreads < nch) xv[j] = ld_cg_v4(gx + tid + j * kThreads);
#pragma unroll
      for (int j = 0; j < kMaxXChunks; ++j)
        if (tid + j * kThreads < nch) x4[tid + j * kThreads] = xv[j];
    }
    sync_compute();
    if (nch % 128 == 0) {
      // d a multiple of 1024: the work is cut into units of 4 rows x one
      // 1024-element segment, dealt to the warps in turn so that every warp
      // streams the same number of bytes; the next unit's pieces load while
      // this unit's are summed.  A row's sum is the sum, in segment order, of
      // its segments' warp sums (each a lane chain of 4 pieces, then the xor
      // tree), staged in shared memory: its order depends on d alone.
      const int P = nch / 128;
      const int nU = (nM + 3) / 4 * P;
      float* s_part = reinterpret_cast<float*>(smem + lay.part);  // [row][P]
      int u = warp;
      const uint4* wr[4];
      auto unit_ptrs = [&](int uu) {
        const int r0 = uu / P * 4, c0 = (uu - uu / P * P) * 128 + lane;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          wr[q] = reinterpret_cast<const uint4*>(a.W + size_t(m0 + min(r0 + q, nM - 1)) * a.d) + c0;
      };
      // Lanes 0-3 prefetch into L2 the 2 KB row segments of this warp's unit
      // kSlowAhead turns ahead, so that more of W is in flight than the
      // registers hold and the register loads find it in L2.
      auto unit_prefetch = [&](int uu) {
        if (lane < 4 && uu < nU) {
          const int r = min(uu / P * 4 + lane, nM - 1), c = (uu - uu / P * P) * 1024;
          prefetch_l2(a.W + size_t(m0 + r) * a.d + c, 2048u);
        }
      };
      if (u < nU) {
#pragma unroll 1
        for (int i = 1; i <= kSlowAhead; ++i) unit_prefetch(u + i * kWarps);
        unit_ptrs(u);
        uint4 wa[4][2], wb[4][2];  // pieces 0-1 and 2-3 of the unit
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            wa[q][p] = ld_stream_v4(wr[q] + 32 * p, pol);
            wb[q][p] = ld_stream_v4(wr[q] + 32 * (p + 2), pol);
          }
        while (true) {
          const int un = u + kWarps;
          const bool next = un < nU;
          const int gi = u / P, seg = u - gi * P;
          const uint4* xs4 = x4 + seg * 128 + lane;
          if (next) unit_ptrs(un);  // all of this unit's pieces are loaded
          unit_prefetch(u + (kSlowAhead + 1) * kWarps);
          float acc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float xf[8];
            bf16x8_to_f32(xs4[32 * p], xf);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
              bf16x8_to_f32(wa[q][p], f);
#pragma unroll
              for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xf[t], acc4[q]);
            }
          }
          if (next) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int p = 0; p < 2; ++p) wa[q][p] = ld_stream_v4(wr[q] + 32 * p, pol);
          }
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float xf[8];
            bf16x8_to_f32(xs4[32 * (p + 2)], xf);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
              bf16x8_to_f32(wb[q][p], f);
#pragma unroll
              for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xf[t], acc4[q]);
            }
          }
          if (next) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int p = 0; p < 2; ++p) wb[q][p] = ld_stream_v4(wr[q] + 32 * (p + 2), pol);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float v = warp_sum_xor<32>(acc4[q]);
            if (lane == q && gi * 4 + q < nM) s_part[(gi * 4 + q) * P + seg] = v;
          }
          u = un;
          if (!next) break;
        }
      }
      sync_compute();
      for (int r = tid; r < nM; r += kThreads) {
        float v = 0.f;
        for (int q = 0; q < P; ++q) v += s_part[r * P + q];
        a.y[m0 + r] = v;
      }
    } else
    for (int rb = warp * 4; rb < nM; rb += kWarps * 4) {
      float acc4[4] = {0.f, 0.f, 0.f, 0.f};
      const uint4* wr[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = min(rb + q, nM - 1);
        wr[q] = reinterpret_cast<const uint4*>(a.W + size_t(m0 + r) * a.d);
      }
      int jj = lane;
      if (jj + 96 < nch) {
        uint4 wa[4][2], wb[4][2];  // pieces 0-1 and 2-3 of the step at jj
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            wa[q][p] = ld_stream_v4(wr[q] + jj + 32 * p, pol);
            wb[q][p] = ld_stream_v4(wr[q] + jj + 32 * (p + 2), pol);
          }
        while (true) {
          const int jn = jj + 128;
          const bool next = jn + 96 < nch;
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float xf[8];
            bf16x8_to_f32(x4[jj + 32 * p], xf);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
              bf16x8_to_f32(wa[q][p], f);
#pragma unroll
              for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xf[t], acc4[q]);
            }
          }
          if (next) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int p = 0; p < 2; ++p) wa[q][p] = ld_stream_v4(wr[q] + jn + 32 * p, pol);
          }
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float xf[8];
            bf16x8_to_f32(x4[jj + 32 * (p + 2)], xf);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
              bf16x8_to_f32(wb[q][p], f);
#pragma unroll
              for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xf[t], acc4[q]);
            }
          }
          jj = jn;
          if (!next) break;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int p = 0; p < 2; ++p) wb[q][p] = ld_stream_v4(wr[q] + jj + 32 * (p + 2), pol);
        }
      }
      for (; jj < nch; jj += 32) {
        float xf[8];
        bf16x8_to_f32(x4[jj], xf);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
          bf16x8_to_f32(ld_stream_v4(wr[q] + jj, pol), f);
#pragma unroll
          for (int t = 0; t < 8; ++t) acc4[q] = fmaf(f[t], xf[t], acc4[q]);
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

// The one kernel of every one-token call with this K: a single handle's call
// is a group of one.  (Two kernels alternating in the decode step, one for
// single calls and one for groups, cost 0.24 us per gated linear more: the
// SMs ran each phase of code that the other kernel had just displaced.)
template <int K>
__global__ void __launch_bounds__(kBlock, 2)
    gsi_decode_cr_group_kernel(const __grid_constant__ CrGroupMaps maps,
                               const __grid_constant__ CrGroupArgs g) {
  int m = 0;
  while (m + 1 < g.n && int(blockIdx.x) >= g.cta0[m + 1]) ++m;
  cr_body<K>(&maps.m[2 * m], &maps.m[2 * m + 1], g.a[m], int(blockIdx.x) - g.cta0[m],
             g.cta0[m + 1] - g.cta0[m]);
}

const void* cr_kernel_for(int64_t k) {
  switch (k) {
    case 64: return reinterpret_cast<const void*>(&gsi_decode_cr_group_kernel<64>);
    case 128: return reinterpret_cast<const void*>(&gsi_decode_cr_group_kernel<128>);
    case 256: return reinterpret_cast<const void*>(&gsi_decode_cr_group_kernel<256>);
    default: return nullptr;
  }
}


// Row boxes for `rows` owned rows: box rows a multiple of 16 and <= 256.
void row_boxes(int rows, int* box, int* nbox) {
  const int padded = (rows + 15) / 16 * 16;
  *nbox = (padded + kMaxBoxRows - 1) / kMaxBoxRows;
  *box = ((padded + *nbox - 1) / *nbox + 15) / 16 * 16;
}

// Largest dynamic shared memory a kernel may use on this device (raised to
// that limit once: the limit belongs to the function), with the whole
// shared/L1 carveout as shared memory, so that kernels of different handles
// and groups can share an SM.
gsi_status_t smem_limit(const void* fn, int device, int* limit) {
  int max_optin = 0;
  if (cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
    return GSI_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return GSI_ERR_CUDA;
  *limit = max_optin - int(fa.sharedSizeBytes);
  if (fa.maxDynamicSharedSizeBytes < *limit) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, *limit) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return GSI_ERR_CUDA;
  }
  return GSI_OK;
}

// Operand bytes one of CTAs 1..G-1 of handle h reads (its V_k and M rows).
double member_load(const gsi_handle* h, int G) {
  return double(h->d + h->d_out) * double(h->k) * 2.0 / double(G - 1);
}

// Rows, TMA boxes, shared memory and tensor maps of handle h run on G CTAs.
gsi_status_t plan_member(const gsi_handle* h, int G, int limit, CrPlan* p, void* tmV, void* tmM) {
  p->G = G;
  p->rows_M = int((h->d_out + G - 2) / (G - 1));
  p->rows_V = int((h->d + G - 2) / (G - 1));
  row_boxes(p->rows_M, &p->box_M, &p->nbox_M);
  row_boxes(p->rows_V, &p->box_V, &p->nbox_V);
  p->smem = cr_layout(int(h->k), int(h->d), p->nbox_M * p->box_M, p->nbox_V * p->box_V).total;
  if (p->smem > size_t(limit)) return GSI_ERR_UNSUPPORTED_SHAPE;
  // 2^vbits >= sqrt(rows_V) x the largest column norm of V_k (with margin):
  // no partial projection of a CTA exceeds max|x| 2^vbits
  const double bound = std::sqrt(double(p->rows_V)) * double(h->cr_vmax) * 1.01 + 1e-30;
  p->vbits = std::max(0, int(std::ceil(std::log2(bound))));
  if (p->vbits > 60) return GSI_ERR_UNSUPPORTED_SHAPE;
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
                              t->cr_F ? int64_t(corr_tiles_elems(int(t->k))) * 2 : 0};
    const void* ptr[3] = {t->V, t->M, t->cr_F};
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

void fill_args(CrArgs* a, const gsi_handle* h, const CrPlan& p, const void* x, float* y,
               uint8_t* gate, float* rho) {
  a->W = h->W;
  a->F = h->cr_F;
  a->x = static_cast<const __nv_bfloat16*>(x);
  a->y = y;
  a->gate = gate;
  a->rho = rho;
  a->d_out = int(h->d_out);
  a->d = int(h->d);
  a->eps = h->eps;
  a->normE = h->cr_normE;
  a->vbits = p.vbits;
  a->rows_M = p.rows_M;
  a->rows_V = p.rows_V;
  a->box_M = p.box_M;
  a->box_V = p.box_V;
  a->nbox_M = p.nbox_M;
  a->nbox_V = p.nbox_V;
  a->acc = reinterpret_cast<uint64_t*>(h->cr_acc);
  a->bar = h->cr_bar;
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

// Launch the one-token kernel on `grid` CTAs for a filled argument block.
gsi_status_t cr_launch(int64_t k, const CrGroupMaps& maps, const CrGroupArgs& ga, int grid,
                       size_t smem, bool pdl, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(dim3(grid), smem, s, pdl, attr);
  cudaError_t err;
  switch (k) {
    case 64: err = cudaLaunchKernelEx(&cfg, gsi_decode_cr_group_kernel<64>, maps, ga); break;
    case 128: err = cudaLaunchKernelEx(&cfg, gsi_decode_cr_group_kernel<128>, maps, ga); break;
    case 256: err = cudaLaunchKernelEx(&cfg, gsi_decode_cr_group_kernel<256>, maps, ga); break;
    default: return GSI_ERR_UNSUPPORTED_SHAPE;
  }
  return err == cudaSuccess ? GSI_OK : GSI_ERR_CUDA;
}

}  // namespace

size_t decode_cr_acc_floats(int64_t k) { return size_t(2) * kCopies * 2 * size_t(k); }

gsi_status_t decode_cr_configure(gsi_handle* h) {
  const void* fn = cr_kernel_for(h->k);
  if (!fn) return GSI_ERR_UNSUPPORTED_SHAPE;
  if (h->d > kMaxD) return GSI_ERR_UNSUPPORTED_SHAPE;  // every CTA reads all of x
  int limit = 0;
  gsi_status_t st = smem_limit(fn, h->device, &limit);
  if (st != GSI_OK) return st;
  const int64_t rows_hint = (std::max(h->d_out, h->d) + 7) / 8 + 1;
  const int G = int(std::max<int64_t>(2, std::min<int64_t>({int64_t(h->num_sms), rows_hint,
                                                            int64_t(kMaxGrid)})));
  CrPlan p;
  st = plan_member(h, G, limit, &p, h->cr_tmaps[0], h->cr_tmaps[1]);
  if (st != GSI_OK) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBlock, p.smem) != cudaSuccess)
    return GSI_ERR_CUDA;
  // The CTAs wait on one another: all of them must fit at once.
  if (per_sm < 1 || int64_t(per_sm) * h->num_sms < G) return GSI_ERR_UNSUPPORTED_SHAPE;
  p.coresident = per_sm >= 2 && p.smem <= kCoresidentSmem;
  h->cr_plan = p;
  return GSI_OK;
}

gsi_status_t decode_cr_launch(gsi_handle* h, const void* x, float* y, uint8_t* gate, float* rho,
                              cudaStream_t s) {
  CrGroupMaps maps;
  CrGroupArgs ga;
  std::memset(&maps, 0, sizeof maps);
  std::memset(&ga, 0, sizeof ga);
  std::memcpy(maps.m, h->cr_tmaps, 2 * sizeof(CUtensorMap));
  ga.n = 1;
  CrArgs& a = ga.a[0];
  fill_args(&a, h, h->cr_plan, x, y, gate, rho);
  prefetch_ranges(h->pf_next, h->pf_group, a.pf, a.pf_bytes);
  a.pf_part0 = 0;
  a.pf_parts = h->cr_plan.G;
  ga.cta0[0] = 0;
  for (int m = 1; m <= kMaxGroup; ++m) ga.cta0[m] = h->cr_plan.G;
  return cr_launch(h->k, maps, ga, h->cr_plan.G, h->cr_plan.smem, h->use_pdl, s);
}

gsi_status_t group_configure(gsi_group* g) {
  const gsi_handle* h0 = g->h[0];
  const void* fn = cr_kernel_for(h0->k);
  if (!fn) return GSI_ERR_UNSUPPORTED_SHAPE;
  int limit = 0;
  gsi_status_t st = smem_limit(fn, h0->device, &limit);
  if (st != GSI_OK) return st;
  // CTAs per member: start from two each (a gate CTA and one more), then give
  // each further CTA to the member whose per-CTA operand bytes are largest
  // (the split that minimises the slowest member's share)
  const int S = std::min(h0->num_sms, g->n * kMaxGrid);
  if (2 * g->n > S) return GSI_ERR_UNSUPPORTED_SHAPE;
  int Gm[kMaxGroup];
  for (int m = 0; m < g->n; ++m) Gm[m] = 2;
  for (int used = 2 * g->n; used < S; ++used) {
    int best = -1;
    double worst = -1.0;
    for (int m = 0; m < g->n; ++m) {
      const int64_t rows_hint = (std::max(g->h[m]->d_out, g->h[m]->d) + 7) / 8 + 1;
      if (Gm[m] >= kMaxGrid || Gm[m] >= rows_hint) continue;
      const double l = member_load(g->h[m], Gm[m]);
      if (l > worst) {
        worst = l;
        best = m;
      }
    }
    if (best < 0) break;
    ++Gm[best];
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
  if (per_sm < 1 || int64_t(per_sm) * h0->num_sms < g->cta0[g->n]) return GSI_ERR_UNSUPPORTED_SHAPE;
  g->smem = smem;
  return GSI_OK;
}

gsi_status_t group_launch(gsi_group* g, const void* const* x, float* const* y,
                          uint8_t* const* gate, float* const* rho, cudaStream_t s) {
  CrGroupMaps maps;
  CrGroupArgs ga;
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
  return cr_launch(g->k, maps, ga, g->cta0[g->n], g->smem, true, s);
}

}  // namespace gsi
