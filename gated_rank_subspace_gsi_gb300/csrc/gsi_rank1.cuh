// gsi_rank1.cuh -- kernels of the rank-1 refinement of a start basis: the
// depth cascade of section 2.3 of "Technical summary: Gated Subspace
// Inference for transformer acceleration" [GSI], where layer l + 1's basis
// starts from layer l's and is refined by a few rank-1 corrections whose new
// directions are re-orthogonalised by DGKS (classical Gram-Schmidt, repeated
// once when the first projection kept less than 1/sqrt(2) of the norm).
// Included by gsi_calib.cu, inside its namespace; the host side is there.
//
// One correction of the basis V (d x k, orthonormal) for C = X^T X:
//   j   = the column whose residual (I - V V^T) C v_j is largest
//   r   = C v_j - V (V^T C v_j)
//   q   = r re-orthogonalised against V (DGKS), normalised
//   v_j <- cos(t) v_j + sin(t) q, the unit vector of span(v_j, q) with the
//          largest Rayleigh quotient: t = atan2(2 s, a - b) / 2 with
//          a = v_j^T C v_j, b = q^T C q, s = v_j^T C q
// The state lives in the calibration workspace, every d-long vector stored as
// a row (the blocks are k x d, "transposed"):
//   V, P   k x d fp32, P = C V (one 2k x d block)
//   H      k x k fp32, H[m][i] = v_m . p_i, so column i of the residual has
//          squared norm pn[i] - cs2[i]
//   pn     k fp64, ||p_i||^2;  cs2  k fp64, sum over m of H[m][i]^2
// All corrections run in one persistent launch (r1_persistent_kernel) whose
// CTAs are all resident at once; grid-wide phases are separated by the
// bounded grid barrier of gsi_device.cuh.  Per correction:
//   A   (32-column slices of d) the previous correction's rotation applied
//       to row j' of V and P; r = p_j - sum over m of H[m][j] v_m; partial
//       rows of V^T r and ||r||^2
//   A'  (entries over warps) h = V^T r and ||r||^2, each entry summed over
//       the slices in slice order
//   B   (slices) q = r - V h; partial ||q||^2; every CTA then takes the DGKS
//       test on the same sums (A, A', B again on q when it asks)
//   C   (tokens) w = X q / ||q||
//   D   (slices) c = X^T w = C q; partial rows of V^T c, P^T q, q.c, p_j.c,
//       ||c||^2
//   D'  (entries over warps) their totals
//   E   (every CTA, the same arithmetic) the 2 x 2 problem, row and column j
//       of H (each CTA writes its share), pn and cs2 (a copy per CTA), and the
//       next column
// Every sum runs in a fixed order, so a call is reproducible bit for bit.

constexpr int kRW = 32;          // columns of the d axis per CTA
constexpr int kRThreads = 512;
constexpr int kRWarps = kRThreads / 32;
constexpr int kRMaxK = 256;
constexpr int kRBatch = 8;       // loads a thread keeps in flight
constexpr int kRMaxVec = 32768;  // largest d and n of a refinement (their vector is staged)

// Control block of a refinement (256 bytes).
struct R1Ctl {
  uint32_t pad1[4];
  int32_t j;           // the column the current correction works on
  int32_t jp;          // the column of the rotation not yet applied to V and P (-1: none)
  int32_t dgks2;       // the second Gram-Schmidt pass runs in this correction
  int32_t step;        // corrections done
  float cs, sn;        // that rotation
  float rr;            // ||r||^2
  float qq;            // ||q||^2 after the last pass
  float qinv;          // 1 / ||q|| (0: q vanished, no rotation)
  float pad0[3];
  uint32_t pad[48];
};
static_assert(sizeof(R1Ctl) == 256, "control block layout");

struct R1Args {
  float* V;                  // k x d
  float* P;                  // k x d
  float* H;                  // k x k
  double* pn;                // k
  double* cs2;               // k
  float* h;                  // k: V^T of the vector being projected
  float* r;                  // d
  float* q;                  // d (not normalised)
  float* c;                  // d: C q / ||q||
  float* w;                  // n: X q / ||q||
  float* part;               // G x pstride partials, one row per slice
  float* tot;                // pstride totals of the partial rows
  const __nv_bfloat16* X;    // n x d
  const __nv_bfloat16* XT;   // d x n
  R1Ctl* ctl;
  uint32_t* status;
  int32_t* order;            // corrections entries, or null
  int n, d, k, G, pstride;   // G: 32-column slices of d
};

// V's slice of 32 columns into shared memory (rows of 33, zero past d),
// 2 x kRBatch rows per warp in flight.
__device__ __forceinline__ void r1_load_slice(const float* V, int k, int d, int x0,
                                              float* Vs) {
  constexpr int kW = kRThreads / 32, kB = 2 * kRBatch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int x = x0 + lane;
  const bool ok = x < d;
  for (int m0 = warp; m0 < k; m0 += kW * kB) {
    float v[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int m = m0 + u * kW;
      v[u] = (ok && m < k) ? V[size_t(m) * d + x] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int m = m0 + u * kW;
      if (m < k) Vs[m * (kRW + 1) + lane] = v[u];
    }
  }
}

// y[lane] = sum over m of Vs[m][lane] * coef[m], in a fixed order: eight
// partial sums over m = warp (mod 8), then added in warp order by warp 0.
// Returns the value in warp 0's lanes (others: 0).
__device__ __forceinline__ float r1_combine(const float* Vs, const float* coef, int k,
                                            float (*red)[kRW]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int m = warp; m < k; m += kRThreads / 32) acc = fmaf(Vs[m * (kRW + 1) + lane], coef[m], acc);
  red[warp][lane] = acc;
  __syncthreads();
  float s = 0.f;
  if (warp == 0) {
#pragma unroll
    for (int u = 0; u < kRThreads / 32; ++u) s += red[u][lane];
  }
  return s;
}

// A column index read from the control block, kept inside [0, k) (-1 stays
// -1 where allowed): no launch can address past V, P or H.
__device__ __forceinline__ int r1_col(int j, int k, bool allow_none) {
  if (allow_none && j < 0) return -1;
  return (j >= 0 && j < k) ? j : 0;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// acc + the 8 products of one 16-byte chunk of bf16 with 8 fp32 values.
__device__ __forceinline__ float r1_dot8(const uint4& xv, const float4& va, const float4& vb,
                                         float acc) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&xv);
  const float2 f0 = __bfloat1622float2(b[0]), f1 = __bfloat1622float2(b[1]);
  const float2 f2 = __bfloat1622float2(b[2]), f3 = __bfloat1622float2(b[3]);
  acc = fmaf(f0.x, va.x, acc);
  acc = fmaf(f0.y, va.y, acc);
  acc = fmaf(f1.x, va.z, acc);
  acc = fmaf(f1.y, va.w, acc);
  acc = fmaf(f2.x, vb.x, acc);
  acc = fmaf(f2.y, vb.y, acc);
  acc = fmaf(f3.x, vb.z, acc);
  return fmaf(f3.y, vb.w, acc);
}

// ---- the persistent form ---------------------------------------------------

// A value held as an unevaluated sum hi + lo of two fp32 numbers (about 48
// bits), for the running column norms: FP64 is slow on this GPU, and these
// sums stay in the update's dependent chain.  Error-free sum (Knuth) and
// product (one FMA).
struct R1F2 {
  float hi, lo;
};
__device__ __forceinline__ R1F2 r1_two_sum(float a, float b) {
  const float s = a + b, bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ R1F2 r1_add(R1F2 x, R1F2 y) {
  const R1F2 s = r1_two_sum(x.hi, y.hi);
  const float lo = s.lo + (x.lo + y.lo);
  const float h = s.hi + lo;
  return {h, lo - (h - s.hi)};
}
__device__ __forceinline__ R1F2 r1_sq(float x) {
  const float p = x * x;
  return {p, fmaf(x, x, -p)};
}
__device__ __forceinline__ R1F2 r1_neg(R1F2 x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ float r1_f(R1F2 x) { return x.hi + x.lo; }

// The dot product of a bf16 row (len8 16-byte chunks) with an fp32 vector in
// shared memory (staged once per CTA), lanes over chunks with kRBatch chunks
// of the row in flight; the total in every lane of the warp (fixed order:
// each lane's chunks, then a butterfly).
__device__ __forceinline__ float r1_row_dot_s(const __nv_bfloat16* row,
                                              const float* vs, int len8) {
  const int lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(row);
  const float4* vr = reinterpret_cast<const float4*>(vs);
  float acc = 0.f;
  int i0 = lane;
  for (; i0 + 32 * (kRBatch - 1) < len8; i0 += 32 * kRBatch) {
    uint4 xv[kRBatch];
#pragma unroll
    for (int u = 0; u < kRBatch; ++u) xv[u] = *(xr + i0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kRBatch; ++u)
      acc = r1_dot8(xv[u], vr[2 * (i0 + 32 * u)], vr[2 * (i0 + 32 * u) + 1], acc);
  }
  for (; i0 < len8; i0 += 32) acc = r1_dot8(*(xr + i0), vr[2 * i0], vr[2 * i0 + 1], acc);
  return warp_sum(acc);
}

// r1_row_dot_s for two rows at once (both rows' chunks in flight together).
__device__ __forceinline__ float2 r1_row_dot2_s(const __nv_bfloat16* r0,
                                                const __nv_bfloat16* r1,
                                                const float* vs, int len8) {
  const int lane = threadIdx.x & 31;
  const uint4* x0 = reinterpret_cast<const uint4*>(r0);
  const uint4* x1 = reinterpret_cast<const uint4*>(r1);
  const float4* vr = reinterpret_cast<const float4*>(vs);
  float a0 = 0.f, a1 = 0.f;
  int i0 = lane;
  for (; i0 + 32 * (kRBatch - 1) < len8; i0 += 32 * kRBatch) {
    uint4 xa[kRBatch], xb[kRBatch];
#pragma unroll
    for (int u = 0; u < kRBatch; ++u) {
      xa[u] = *(x0 + i0 + 32 * u);
      xb[u] = *(x1 + i0 + 32 * u);
    }
#pragma unroll
    for (int u = 0; u < kRBatch; ++u) {
      const float4 va = vr[2 * (i0 + 32 * u)], vb = vr[2 * (i0 + 32 * u) + 1];
      a0 = r1_dot8(xa[u], va, vb, a0);
      a1 = r1_dot8(xb[u], va, vb, a1);
    }
  }
  for (; i0 < len8; i0 += 32) {
    const float4 va = vr[2 * i0], vb = vr[2 * i0 + 1];
    a0 = r1_dot8(*(x0 + i0), va, vb, a0);
    a1 = r1_dot8(*(x1 + i0), va, vb, a1);
  }
  return make_float2(warp_sum(a0), warp_sum(a1));
}

// Copy `count` floats (count % 4 == 0) written by other CTAs of this launch
// into shared memory, through L2.
__device__ __forceinline__ void r1_stage(float* dst, const float* src, int count) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
  float4* d4 = reinterpret_cast<float4*>(dst);
  for (int i = threadIdx.x; i < count / 4; i += kRThreads) d4[i] = __ldcg(s4 + i);
}

// Sum over the G slices of entry e of the partial rows, by one warp: each lane
// adds slices lane, lane + 32, ... in order, then a butterfly (a fixed order).
__device__ __forceinline__ float r1_slice_sum(const R1Args& a, int e) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int q0 = lane; q0 < a.G; q0 += 32 * 4) {  // four loads in flight, added in order
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + 32 * u;
      v[u] = q < a.G ? __ldcg(&a.part[size_t(q) * a.pstride + e]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (q0 + 32 * u < a.G) s += v[u];
  }
  return warp_sum(s);
}

// Phases A' and D': the totals of entries [0, ne) into a.tot, one entry per
// warp of the grid at a time.
__device__ __forceinline__ void r1_totals(const R1Args& a, int ne) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = int(blockIdx.x) * kRWarps + warp; e < ne; e += int(gridDim.x) * kRWarps) {
    const float v = r1_slice_sum(a, e);
    if (lane == 0) a.tot[e] = v;
  }
}

// ||q||^2 from the slices' partials (entry k + 1, which no phase between B
// and D writes), the same sum in every CTA.
__device__ __forceinline__ float r1_sum_qq(const R1Args& a, float* s_qq) {
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) {
    const float v = r1_slice_sum(a, a.k + 1);
    if ((threadIdx.x & 31) == 0) *s_qq = v;
  }
  __syncthreads();
  return *s_qq;
}

// Phase A on slice sl: mode 0 applies the pending rotation (row jp of V and
// P) and forms r = p_j - sum over m of coef[m] v_m; mode 1 (the second DGKS
// pass) takes q.  Writes the slice's partial row of V^T(vector), and ||r||^2 in
// mode 0.  Vs holds the slice on return (loaded unless `load` is false).
// Every vector entry of the slice is written by this CTA only (the slice's
// owner), so plain loads see it.
__device__ void r1_project_slice(const R1Args& a, int sl, int mode, int j, int jp, float cs,
                                 float sn, float qinv_prev, const float* coef, float* Vs,
                                 float (*red)[kRW], float* vec, bool load) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, d = a.d, x0 = sl * kRW, x = x0 + lane;
  const bool ok = x < d;
  __syncthreads();
  if (load) r1_load_slice(a.V, k, d, x0, Vs);
  __syncthreads();
  if (mode == 0) {
    if (warp == 0) {
      if (jp >= 0 && ok) {
        const float v = fmaf(cs, Vs[jp * (kRW + 1) + lane], sn * (qinv_prev * a.q[x]));
        Vs[jp * (kRW + 1) + lane] = v;
        a.V[size_t(jp) * d + x] = v;
        const size_t pi = size_t(jp) * d + x;
        a.P[pi] = fmaf(cs, a.P[pi], sn * a.c[x]);
      }
      vec[lane] = ok ? a.P[size_t(j) * d + x] : 0.f;
    }
    __syncthreads();
    const float s = r1_combine(Vs, coef, k, red);
    if (warp == 0) {
      const float rv = ok ? vec[lane] - s : 0.f;
      vec[lane] = rv;
      if (ok) a.r[x] = rv;
    }
  } else {
    if (warp == 0) vec[lane] = ok ? a.q[x] : 0.f;
  }
  __syncthreads();
  float* part = a.part + size_t(sl) * a.pstride;
  for (int m = tid; m < k; m += kRThreads) {
    float acc = 0.f;
#pragma unroll 8
    for (int l = 0; l < kRW; ++l) acc = fmaf(Vs[m * (kRW + 1) + l], vec[l], acc);
    part[m] = acc;
  }
  if (mode == 0 && warp == 0) {
    const float rr = warp_sum(vec[lane] * vec[lane]);
    if (lane == 0) part[k] = rr;
  }
}

// Phase B on slice sl: q = (mode 0: r, mode 1: q) - sum over m of coef[m] v_m;
// the slice's ||q||^2 into entry k + 1 of its partial row.
__device__ void r1_subtract_slice(const R1Args& a, int sl, int mode, const float* coef, float* Vs,
                                  float (*red)[kRW], bool load) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = a.k, d = a.d, x0 = sl * kRW, x = x0 + lane;
  const bool ok = x < d;
  __syncthreads();
  if (load) r1_load_slice(a.V, k, d, x0, Vs);
  __syncthreads();
  const float s = r1_combine(Vs, coef, k, red);
  if (warp == 0) {
    const float src = ok ? (mode == 0 ? a.r[x] : a.q[x]) : 0.f;
    const float qv = ok ? src - s : 0.f;
    if (ok) a.q[x] = qv;
    const float qq = warp_sum(qv * qv);
    if (lane == 0) a.part[size_t(sl) * a.pstride + k + 1] = qq;
  }
}

// Phase D on slice sl: c = X^T w on its 32 columns (four per warp, rows of
// X^T; w staged in shared memory as ws), then its partial row of V^T c,
// P^T q^, q^.c, p_j.c and ||c||^2 (q^ = q / ||q||).
__device__ void r1_apply_c_slice(const R1Args& a, int sl, int j, float qinv, float* cvec,
                                 float* qvec, const float* ws) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, d = a.d, x0 = sl * kRW;
  __syncthreads();
  static_assert(kRW == 2 * kRWarps, "two columns of the slice per warp");
  {
    const int xl = 2 * warp, x = x0 + xl;
    float2 acc = make_float2(0.f, 0.f);
    if (x + 1 < d) {
      acc = r1_row_dot2_s(a.XT + size_t(x) * a.n, a.XT + size_t(x + 1) * a.n, ws, a.n / 8);
    } else if (x < d) {
      acc.x = r1_row_dot_s(a.XT + size_t(x) * a.n, ws, a.n / 8);
    }
    if (lane == 0) {
      if (x < d) a.c[x] = acc.x;
      if (x + 1 < d) a.c[x + 1] = acc.y;
      cvec[xl] = acc.x;
      cvec[xl + 1] = acc.y;
    }
  }
  if (warp == 0) qvec[lane] = (x0 + lane < d) ? qinv * a.q[x0 + lane] : 0.f;
  __syncthreads();
  float* part = a.part + size_t(sl) * a.pstride;
  const bool full = x0 + kRW <= d;
  for (int m = tid; m < k; m += kRThreads) {
    const float* vr = a.V + size_t(m) * d + x0;
    const float* pr = a.P + size_t(m) * d + x0;
    float vc = 0.f, pq = 0.f, pc = 0.f;
    if (full) {
#pragma unroll
      for (int l4 = 0; l4 < kRW / 4; ++l4) {
        const float4 v = reinterpret_cast<const float4*>(vr)[l4];
        const float4 p = reinterpret_cast<const float4*>(pr)[l4];
        const int l = 4 * l4;
        vc = fmaf(v.x, cvec[l], vc);
        vc = fmaf(v.y, cvec[l + 1], vc);
        vc = fmaf(v.z, cvec[l + 2], vc);
        vc = fmaf(v.w, cvec[l + 3], vc);
        pq = fmaf(p.x, qvec[l], pq);
        pq = fmaf(p.y, qvec[l + 1], pq);
        pq = fmaf(p.z, qvec[l + 2], pq);
        pq = fmaf(p.w, qvec[l + 3], pq);
        pc = fmaf(p.x, cvec[l], pc);
        pc = fmaf(p.y, cvec[l + 1], pc);
        pc = fmaf(p.z, cvec[l + 2], pc);
        pc = fmaf(p.w, cvec[l + 3], pc);
      }
    } else {
      for (int l = 0; l < kRW && x0 + l < d; ++l) {
        vc = fmaf(vr[l], cvec[l], vc);
        pq = fmaf(pr[l], qvec[l], pq);
        pc = fmaf(pr[l], cvec[l], pc);
      }
    }
    part[m] = vc;
    part[k + m] = pq;
    if (m == j) part[2 * k + 1] = pc;
  }
  if (warp == 0) {
    const float qc = warp_sum(qvec[lane] * cvec[lane]);
    const float cc = warp_sum(cvec[lane] * cvec[lane]);
    if (lane == 0) {
      part[2 * k] = qc;
      part[2 * k + 2] = cc;
    }
  }
}

// All corrections in one launch; every CTA of the grid is resident at once
// (the host checks occupancy), slices sl = CTA, CTA + grid, ... belong to one
// CTA for the whole launch.  Dynamic shared memory: the V slice, k rows of 33
// floats, then max(d, n) floats for the vector that phases C and D read whole
// (q, then w).  A barrier that runs out (1 s) sets the timeout bit and ends the
// launch in every CTA; V_out is then not written.
__global__ void __launch_bounds__(kRThreads) r1_persistent_kernel(R1Args a, int corrections,
                                                                  uint32_t* bar,
                                                                  __nv_bfloat16* Vout) {
  extern __shared__ __align__(16) float r1_dyn[];
  float* Vs = r1_dyn;
  float* vsh = r1_dyn + a.k * (kRW + 1);  // 16-byte aligned: k is a multiple of 16
  __shared__ float coef[kRMaxK];
  __shared__ float red[kRWarps][kRW];
  __shared__ float vec[kRW], cvec[kRW], qvec[kRW];
  __shared__ float orow[kRMaxK], ocol[kRMaxK];  // H's row and column j before this update
  __shared__ float nrow[kRMaxK], ncol[kRMaxK];  // ... after it (the next correction's jp)
  __shared__ float s_vc[kRMaxK], s_pq[kRMaxK], s_sc[4];
  __shared__ R1F2 s_pn[kRMaxK], s_cs2[kRMaxK];  // this CTA's copy, updated like every other
  __shared__ R1F2 s_dd[kRWarps];
  __shared__ float s_kv[kRWarps];
  __shared__ int s_ii[kRThreads];
  __shared__ float s_qq;
  __shared__ int s_ok;
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, grid = int(gridDim.x), cta = int(blockIdx.x);
  const bool reload = a.G > grid;  // more than one slice per CTA: Vs must be reloaded
  uint32_t nb = 0;
#define R1_BARRIER()                                                              \
  do {                                                                            \
    ++nb;                                                                         \
    if (!grid_barrier(bar, nb * uint32_t(grid), a.status, &s_ok)) return;         \
  } while (0)

  for (int i = tid; i < k; i += kRThreads) {
    const double p = __ldcg(&a.pn[i]), c = __ldcg(&a.cs2[i]);
    s_pn[i] = {float(p), float(p - double(float(p)))};
    s_cs2[i] = {float(c), float(c - double(float(c)))};
  }
  int j = r1_col(__ldcg(&a.ctl->j), k, false);
  int jp = -1;
  float cs = 1.f, sn = 0.f, qinv_prev = 0.f;
  __syncthreads();

  for (int step = 0; step < corrections; ++step) {
    // H[:, j] after every earlier update: from memory, except row and column
    // jp, whose owners may still be writing them
    for (int m = tid; m < k; m += kRThreads)
      coef[m] = (jp >= 0 && j == jp)   ? ncol[m]
                : (jp >= 0 && m == jp) ? nrow[j]
                                       : __ldcg(&a.H[size_t(m) * k + j]);
    // A, A': h = V^T r, ||r||^2
    for (int sl = cta; sl < a.G; sl += grid)
      r1_project_slice(a, sl, 0, j, jp, cs, sn, qinv_prev, coef, Vs, red, vec, true);
    R1_BARRIER();
    r1_totals(a, k + 1);
    R1_BARRIER();
    __syncthreads();
    for (int m = tid; m < k; m += kRThreads) coef[m] = __ldcg(&a.tot[m]);
    const float rr = __ldcg(&a.tot[k]);
    // B: q = r - V h; the DGKS test on the same sums in every CTA
    for (int sl = cta; sl < a.G; sl += grid) r1_subtract_slice(a, sl, 0, coef, Vs, red, reload);
    R1_BARRIER();
    float qq = r1_sum_qq(a, &s_qq);
    if (qq < 0.5f * rr) {
      for (int sl = cta; sl < a.G; sl += grid)
        r1_project_slice(a, sl, 1, j, -1, 1.f, 0.f, 0.f, coef, Vs, red, vec, reload);
      R1_BARRIER();
      r1_totals(a, k);
      R1_BARRIER();
      __syncthreads();
      for (int m = tid; m < k; m += kRThreads) coef[m] = __ldcg(&a.tot[m]);
      for (int sl = cta; sl < a.G; sl += grid) r1_subtract_slice(a, sl, 1, coef, Vs, red, reload);
      R1_BARRIER();
      qq = r1_sum_qq(a, &s_qq);
    }
    float qinv = 0.f;
    if (!isfinite(qq)) {
      if (cta == 0 && tid == 0) atomicOr(a.status, kStatusRank);
    } else if (qq > 1e-30f * s_pn[j].hi && qq > 0.f) {
      qinv = 1.0f / sqrtf(qq);
    }
    // C: w = X q / ||q||, one token per warp of the grid
    __syncthreads();
    r1_stage(vsh, a.q, a.d);
    __syncthreads();
    for (int t = cta * kRWarps + warp; t < a.n; t += grid * kRWarps) {
      const float acc = r1_row_dot_s(a.X + size_t(t) * a.d, vsh, a.d / 8);
      if (lane == 0) a.w[t] = acc * qinv;
    }
    R1_BARRIER();
    // D, D': H's row and column j as they stand, c = C q^ and the totals
    for (int i = tid; i < k; i += kRThreads) {
      orow[i] = __ldcg(&a.H[size_t(j) * k + i]);
      ocol[i] = __ldcg(&a.H[size_t(i) * k + j]);
    }
    __syncthreads();
    r1_stage(vsh, a.w, a.n);
    for (int sl = cta; sl < a.G; sl += grid) r1_apply_c_slice(a, sl, j, qinv, cvec, qvec, vsh);
    R1_BARRIER();
    r1_totals(a, 2 * k + 3);
    R1_BARRIER();
    // E: the same update in every CTA
    for (int e = tid; e < 2 * k + 3; e += kRThreads) {
      const float v = __ldcg(&a.tot[e]);
      if (e < k) s_vc[e] = v;
      else if (e < 2 * k) s_pq[e - k] = v;
      else s_sc[e - 2 * k] = v;  // q^.c, p_j.c, ||c||^2
    }
    __syncthreads();
    const float av = ocol[j], bv = s_sc[0], sv = s_vc[j];
    float ncs = 1.f, nsn = 0.f;
    const bool rotate = qinv > 0.f;  // q vanished: nothing changes
    if (rotate) {
      const float t = 0.5f * atan2f(2.f * sv, av - bv);
      sincosf(t, &nsn, &ncs);
    }
    const int i0 = int(int64_t(k) * cta / grid), i1 = int(int64_t(k) * (cta + 1) / grid);
    R1F2 colv2 = {0.f, 0.f};
    const int i = tid;
    if (i < k) {
      float nr = orow[i], nc = ocol[i];
      if (rotate) {
        if (i != j) {
          nr = fmaf(ncs, orow[i], nsn * s_pq[i]);
          nc = fmaf(ncs, ocol[i], nsn * s_vc[i]);
          s_cs2[i] = r1_add(s_cs2[i], r1_add(r1_sq(nr), r1_neg(r1_sq(orow[i]))));
        } else {
          nr = ncs * ncs * av + ncs * nsn * (sv + s_pq[j]) + nsn * nsn * bv;
          nc = nr;
        }
        if (i >= i0 && i < i1) {  // this CTA's share of the writes
          a.H[size_t(j) * k + i] = nr;
          a.H[size_t(i) * k + j] = nc;
        }
      }
      nrow[i] = nr;
      ncol[i] = nc;
      colv2 = r1_sq(nc);
    }
    // sum of the new column's squares: a butterfly in each warp, then the
    // warps' sums in warp order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const R1F2 other = {__shfl_xor_sync(0xffffffffu, colv2.hi, o),
                          __shfl_xor_sync(0xffffffffu, colv2.lo, o)};
      colv2 = (lane & o) ? r1_add(other, colv2) : r1_add(colv2, other);
    }
    if (lane == 0) s_dd[warp] = colv2;
    __syncthreads();
    if (tid == 0 && rotate) {
      R1F2 c2sum = {0.f, 0.f};
      for (int w = 0; w < kRWarps; ++w) c2sum = r1_add(c2sum, s_dd[w]);
      s_cs2[j] = c2sum;
      // ||cs p_j + sn c||^2 = cs^2 ||p_j||^2 + 2 cs sn p_j.c + sn^2 ||c||^2
      const R1F2 pj = s_pn[j];
      const float c2 = ncs * ncs, sc2 = 2.f * ncs * nsn, s2 = nsn * nsn;
      const R1F2 t0 = {c2 * pj.hi, c2 * pj.lo};
      s_pn[j] = r1_add(t0, r1_two_sum(sc2 * s_sc[1], s2 * s_sc[2]));
    }
    __syncthreads();
    // the next column: the largest pn - cs2, the first of equals (a butterfly
    // in each warp, then over the warps' winners)
    {
      float v = -INFINITY;
      if (tid < k) v = r1_f(r1_add(s_pn[tid], r1_neg(s_cs2[tid])));
      int ix = tid;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, ix, o);
        if (v2 > v || (v2 == v && i2 < ix)) {
          v = v2;
          ix = i2;
        }
      }
      if (lane == 0) {
        s_kv[warp] = v;
        s_ii[warp] = ix;
      }
      __syncthreads();
      if (warp == 0) {
        v = lane < kRWarps ? s_kv[lane] : -INFINITY;
        ix = lane < kRWarps ? s_ii[lane] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, ix, o);
          if (v2 > v || (v2 == v && i2 < ix)) {
            v = v2;
            ix = i2;
          }
        }
        if (lane == 0) s_ii[kRWarps] = ix;
      }
      __syncthreads();
    }
    if (cta == 0 && tid == 0 && a.order) a.order[step] = j;
    const int jn = r1_col(s_ii[kRWarps], k, false);
    __syncthreads();
    jp = rotate ? j : -1;
    cs = ncs;
    sn = nsn;
    qinv_prev = qinv;
    j = jn;
  }
#undef R1_BARRIER
  // the last rotation, then V as the d x k bf16 basis
  for (int sl = cta; sl < a.G; sl += grid) {
    const int x0 = sl * kRW, x = x0 + lane;
    __syncthreads();
    r1_load_slice(a.V, k, a.d, x0, Vs);
    __syncthreads();
    if (warp == 0 && jp >= 0 && x < a.d)
      Vs[jp * (kRW + 1) + lane] = fmaf(cs, Vs[jp * (kRW + 1) + lane], sn * (qinv_prev * a.q[x]));
    __syncthreads();
    for (int xl = 0; xl < kRW && x0 + xl < a.d; ++xl)
      for (int m = tid; m < k; m += kRThreads)
        Vout[size_t(x0 + xl) * k + m] = __float2bfloat16_rn(Vs[m * (kRW + 1) + xl]);
  }
}


// init: H, pn and cs2 from the Gram matrix of the stacked block [V; P] (G2,
// kp2 x kp2, lower tiles: G2[k + i][m] = p_i . v_m), one row i per warp with
// the lanes over m, k / 8 CTAs; the CTA that finishes last (a ticket, no
// wait) picks the first column and clears the control block.
__global__ void __launch_bounds__(kRThreads) r1_init_kernel(R1Args a, const float* G2,
                                                            int kp2, uint32_t* tick) {
  constexpr int kW = kRThreads / 32;
  __shared__ double s_dd[kRThreads];
  __shared__ int s_ii[kRThreads];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, k = a.k;
  const int i = blockIdx.x * kW + warp;
  if (i < k) {
    const float* row = G2 + size_t(k + i) * kp2;
    float hv[kRMaxK / 32];
#pragma unroll
    for (int u = 0; u < kRMaxK / 32; ++u) {
      const int m = lane + 32 * u;
      hv[u] = (m < k) ? row[m] : 0.f;
    }
    double acc = 0.0;
#pragma unroll
    for (int u = 0; u < kRMaxK / 32; ++u) {
      const int m = lane + 32 * u;
      if (m < k) {
        a.H[size_t(m) * k + i] = hv[u];
        acc += double(hv[u]) * hv[u];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      a.pn[i] = double(row[k + i]);
      a.cs2[i] = acc;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = (atomicAdd(tick, 1u) == gridDim.x - 1) ? 1 : 0;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  s_dd[tid] = (tid < k) ? __ldcg(&a.pn[tid]) - __ldcg(&a.cs2[tid]) : -INFINITY;
  s_ii[tid] = tid;
  __syncthreads();
  for (int o = kRThreads / 2; o > 0; o >>= 1) {
    if (tid < o) {
      const double v2 = s_dd[tid + o];
      if (v2 > s_dd[tid] || (v2 == s_dd[tid] && s_ii[tid + o] < s_ii[tid])) {
        s_dd[tid] = v2;
        s_ii[tid] = s_ii[tid + o];
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    R1Ctl* ctl = a.ctl;
    ctl->j = s_ii[0];
    ctl->jp = -1;
    ctl->dgks2 = 0;
    ctl->step = 0;
    ctl->cs = 1.f;
    ctl->sn = 0.f;
    ctl->rr = 0.f;
    ctl->qq = 0.f;
    ctl->qinv = 0.f;
    *tick = 0;
  }
}

// finish: the pending rotation applied to this slice of V, and V written as
// the d x k bf16 basis.  With no correction (jp = -1) V is the start basis.
__global__ void __launch_bounds__(kRThreads) r1_finish_kernel(R1Args a, int any,
                                                              __nv_bfloat16* Vout) {
  __shared__ float Vs[kRMaxK * (kRW + 1)];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, d = a.d, x0 = blockIdx.x * kRW, x = x0 + lane;
  r1_load_slice(a.V, k, d, x0, Vs);
  __syncthreads();
  const int jp = any ? r1_col(a.ctl->jp, k, true) : -1;
  if (warp == 0 && jp >= 0 && x < d) {
    const float cs = a.ctl->cs, sn = a.ctl->sn, qinv = a.ctl->qinv;
    Vs[jp * (kRW + 1) + lane] = fmaf(cs, Vs[jp * (kRW + 1) + lane], sn * (qinv * a.q[x]));
  }
  __syncthreads();
  for (int xl = 0; xl < kRW && x0 + xl < d; ++xl)
    for (int m = tid; m < k; m += kRThreads)
      Vout[size_t(x0 + xl) * k + m] = __float2bfloat16_rn(Vs[m * (kRW + 1) + xl]);
}
