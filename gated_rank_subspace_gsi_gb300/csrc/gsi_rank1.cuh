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
// The kernels of one correction, each a grid over 32-column slices of d (or
// over tokens) whose last CTA to finish reduces the partials in CTA order:
//   project   the previous correction's rotation applied to row j' of V and
//             P; r = p_j - sum over m of H[m][j] v_m; partials of V^T r, ||r||^2
//   subtract  q = r - V h; partial ||q||^2; the last CTA takes the DGKS test
//   project / subtract again on q when the test asked for it (the launches
//             return at once otherwise)
//   xq        w = X q / ||q||                               (token slices)
//   xtw       c = X^T w = C q; partial V^T c, P^T q, q.c, p_j.c, ||c||^2; the
//             last CTA solves the 2 x 2 problem and updates H, pn, cs2 and
//             the choice of the next column
// The rotation itself is applied to V and P by the next project (or finish)
// launch, slice by slice.  No CTA waits on another: the reductions take
// tickets (the last CTA of each group of 16 sums the group's partials, the
// last group's finisher sums the groups), so no wait can hang, and the sums
// run in a fixed order whichever CTA does them.

constexpr int kRW = 32;          // columns of the d axis per CTA
constexpr int kRThreads = 256;
constexpr int kRWideThreads = 512;  // the X^T w kernel: two columns per warp
constexpr int kRTok = kRThreads / 32;  // tokens per CTA of the X q product (one per warp)
constexpr int kRMaxK = 256;
constexpr int kRGrp = 16;        // CTAs per first-level group of a reduction
constexpr int kRBatch = 8;       // loads a thread keeps in flight

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
  float* part;               // G x pstride partials, one row per CTA
  float* gpart;              // ngrp x pstride group sums
  uint32_t* tick;            // 3 x (1 + ngrp) tickets (project, subtract, xtw), zero between launches
  const __nv_bfloat16* X;    // n x d
  const __nv_bfloat16* XT;   // d x n
  R1Ctl* ctl;
  uint32_t* status;
  int32_t* order;            // corrections entries, or null
  int n, d, k, G, ngrp, pstride;
};

// Sum over the G CTAs of the partial rows part[g][0..ne), called by every
// thread of every CTA once its row is written.  The last CTA of each group of
// kRGrp sums the group's rows (in row order) into a group row; the last group
// to finish sums the group rows (in group order).  True in that one CTA, with
// the totals in tot[0..ne) (shared memory).  tick: 1 + ngrp counters, zero on
// entry and again when the call returns.
__device__ bool r1_reduce(const R1Args& a, uint32_t* tick, int ne, float* tot, int* s_flag) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int grp = blockIdx.x / kRGrp, g0 = grp * kRGrp, gn = min(a.G, g0 + kRGrp) - g0;
  // the CTA's writes are ordered before thread 0's fence by the barrier, and
  // the fence (cumulative) orders them before the ticket
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    *s_flag = (atomicAdd(&tick[1 + grp], 1u) == unsigned(gn - 1)) ? 1 : 0;
    if (*s_flag) __threadfence();
  }
  __syncthreads();
  if (*s_flag == 0) return false;
  for (int e = tid; e < ne; e += nt) {
    float v[kRGrp];
#pragma unroll
    for (int u = 0; u < kRGrp; ++u)
      v[u] = (u < gn) ? __ldcg(&a.part[size_t(g0 + u) * a.pstride + e]) : 0.f;
    float sum = v[0];
#pragma unroll
    for (int u = 1; u < kRGrp; ++u)
      if (u < gn) sum += v[u];
    a.gpart[size_t(grp) * a.pstride + e] = sum;
  }
  __syncthreads();
  if (tid == 0) {
    tick[1 + grp] = 0;
    __threadfence();
    *s_flag = (atomicAdd(&tick[0], 1u) == unsigned(a.ngrp - 1)) ? 1 : 0;
    if (*s_flag) __threadfence();
  }
  __syncthreads();
  if (*s_flag == 0) return false;
  for (int e = tid; e < ne; e += nt) {
    float sum = 0.f;
    int q = 0;
    for (; q + kRBatch <= a.ngrp; q += kRBatch) {
      float v[kRBatch];
#pragma unroll
      for (int u = 0; u < kRBatch; ++u) v[u] = __ldcg(&a.gpart[size_t(q + u) * a.pstride + e]);
#pragma unroll
      for (int u = 0; u < kRBatch; ++u) sum += v[u];
    }
    for (; q < a.ngrp; ++q) sum += __ldcg(&a.gpart[size_t(q) * a.pstride + e]);
    tot[e] = sum;
  }
  if (tid == 0) tick[0] = 0;
  __syncthreads();
  return true;
}

// V's slice of 32 columns into shared memory (rows of 33, zero past d),
// 2 x kRBatch rows per warp in flight.
__device__ __forceinline__ void r1_load_slice(const float* __restrict__ V, int k, int d, int x0,
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

// project: mode 0 applies the pending rotation and forms r = p_j - V H[:, j];
// mode 1 (the second DGKS pass, only when asked) takes the vector q.  Both
// write partials of V^T(vector) and, in mode 0, ||r||^2; the last CTA sums
// them into h (and rr).
__global__ void __launch_bounds__(kRThreads) r1_project_kernel(R1Args a, int mode) {
  __shared__ float Vs[kRMaxK * (kRW + 1)];
  __shared__ float coef[kRMaxK];
  __shared__ float red[kRThreads / 32][kRW];
  __shared__ float vec[kRW];
  __shared__ float tot[kRMaxK + 4];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();
  R1Ctl* ctl = a.ctl;
  if (mode == 1 && *reinterpret_cast<volatile int32_t*>(&ctl->dgks2) == 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, d = a.d, x0 = blockIdx.x * kRW, x = x0 + lane;
  const bool ok = x < d;
  const int j = r1_col(ctl->j, k, false);
  r1_load_slice(a.V, k, d, x0, Vs);
  if (mode == 0) {
    for (int m = tid; m < k; m += kRThreads) coef[m] = a.H[size_t(m) * k + j];
  }
  __syncthreads();
  if (mode == 0) {
    const int jp = r1_col(ctl->jp, k, true);
    if (warp == 0) {
      if (jp >= 0 && ok) {
        const float cs = ctl->cs, sn = ctl->sn, qinv = ctl->qinv;
        const float v = fmaf(cs, Vs[jp * (kRW + 1) + lane], sn * (qinv * a.q[x]));
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
  float* part = a.part + size_t(blockIdx.x) * a.pstride;
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
  if (!r1_reduce(a, a.tick, mode == 0 ? k + 1 : k, tot, &s_last)) return;
  for (int m = tid; m < k; m += kRThreads) a.h[m] = tot[m];
  if (mode == 0 && tid == 0) ctl->rr = tot[k];
}

// subtract: q = (mode 0: r, mode 1: q) - V h; partial ||q||^2.  The last CTA
// takes the DGKS test in mode 0 (a second pass when ||q||^2 < ||r||^2 / 2)
// and sets 1 / ||q||, or 0 when q vanished (non-finite: status bit).
__global__ void __launch_bounds__(kRThreads) r1_subtract_kernel(R1Args a, int mode) {
  __shared__ float Vs[kRMaxK * (kRW + 1)];
  __shared__ float coef[kRMaxK];
  __shared__ float red[kRThreads / 32][kRW];
  __shared__ float tot[4];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();
  R1Ctl* ctl = a.ctl;
  if (mode == 1 && *reinterpret_cast<volatile int32_t*>(&ctl->dgks2) == 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, d = a.d, x0 = blockIdx.x * kRW, x = x0 + lane;
  const bool ok = x < d;
  r1_load_slice(a.V, k, d, x0, Vs);
  for (int m = tid; m < k; m += kRThreads) coef[m] = a.h[m];
  __syncthreads();
  const float s = r1_combine(Vs, coef, k, red);
  float* part = a.part + size_t(blockIdx.x) * a.pstride;
  if (warp == 0) {
    const float src = ok ? (mode == 0 ? a.r[x] : a.q[x]) : 0.f;
    const float qv = ok ? src - s : 0.f;
    if (ok) a.q[x] = qv;
    const float qq = warp_sum(qv * qv);
    if (lane == 0) part[0] = qq;
  }
  if (!r1_reduce(a, a.tick + (1 + a.ngrp), 1, tot, &s_last)) return;
  if (tid == 0) {
    const float qq = tot[0];
    ctl->qq = qq;
    if (mode == 0) ctl->dgks2 = (qq < 0.5f * ctl->rr) ? 1 : 0;
    const float pj = float(a.pn[r1_col(ctl->j, a.k, false)]);
    float qinv = 0.f;
    if (!isfinite(qq)) {
      atomicOr(a.status, kStatusRank);
    } else if (qq > 1e-30f * pj && qq > 0.f) {
      qinv = 1.0f / sqrtf(qq);
    }
    ctl->qinv = qinv;
  }
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

// The dot product of a bf16 row (len8 16-byte chunks) with an fp32 vector,
// lanes over chunks with kRBatch chunks of both in flight; the total in
// every lane of the warp (fixed order: each lane's chunks, then a butterfly).
__device__ __forceinline__ float r1_row_dot(const __nv_bfloat16* __restrict__ row,
                                            const float* __restrict__ v, int len8) {
  const int lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(row);
  const float4* vr = reinterpret_cast<const float4*>(v);
  float acc = 0.f;
  int i0 = lane;
  // whole batches: every load of the batch issued before the first product
  for (; i0 + 32 * (kRBatch - 1) < len8; i0 += 32 * kRBatch) {
    uint4 xv[kRBatch];
    float4 va[kRBatch], vb[kRBatch];
#pragma unroll
    for (int u = 0; u < kRBatch; ++u) xv[u] = __ldg(xr + i0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kRBatch; ++u) {
      va[u] = __ldg(vr + 2 * (i0 + 32 * u));
      vb[u] = __ldg(vr + 2 * (i0 + 32 * u) + 1);
    }
#pragma unroll
    for (int u = 0; u < kRBatch; ++u) acc = r1_dot8(xv[u], va[u], vb[u], acc);
  }
  for (; i0 < len8; i0 += 32) acc = r1_dot8(__ldg(xr + i0), __ldg(vr + 2 * i0), __ldg(vr + 2 * i0 + 1), acc);
  return warp_sum(acc);
}

// xq: w[t] = (x_t . q) / ||q||, one token per warp.
__global__ void __launch_bounds__(kRThreads) r1_xq_kernel(R1Args a) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRTok + warp;
  if (t >= a.n) return;
  const float qinv = a.ctl->qinv;
  const float acc = r1_row_dot(a.X + size_t(t) * a.d, a.q, a.d / 8);
  if (lane == 0) a.w[t] = acc * qinv;
}

// xtw: c = X^T w on this CTA's 32 columns (two per warp, rows of X^T), then
// partials of V^T c, P^T q^, q^.c, p_j.c and ||c||^2 (q^ = q / ||q||).  The
// CTA that finishes the reduction finishes the correction: the angle, H's
// row and column j, pn[j], cs2, and the next column (the largest residual,
// the first of equals).
__global__ void __launch_bounds__(kRWideThreads) r1_xtw_kernel(R1Args a) {
  constexpr int kWarps = kRWideThreads / 32;
  __shared__ float cvec[kRW], qvec[kRW];
  __shared__ float tot[2 * kRMaxK + 4];
  __shared__ double s_dd[kRWideThreads];
  __shared__ int s_ii[kRWideThreads];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();
  R1Ctl* ctl = a.ctl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, d = a.d, x0 = blockIdx.x * kRW;
  const int j = r1_col(ctl->j, k, false);
  const float qinv = ctl->qinv;
  for (int u = 0; u < kRW / kWarps; ++u) {
    const int xl = warp * (kRW / kWarps) + u, x = x0 + xl;
    float acc = 0.f;
    if (x < d) {
      acc = r1_row_dot(a.XT + size_t(x) * a.n, a.w, a.n / 8);
      if (lane == 0) a.c[x] = acc;
    }
    if (lane == 0) cvec[xl] = acc;
  }
  if (warp == 0) qvec[lane] = (x0 + lane < d) ? qinv * a.q[x0 + lane] : 0.f;
  __syncthreads();
  float* part = a.part + size_t(blockIdx.x) * a.pstride;
  const bool full = x0 + kRW <= d;
  for (int m = tid; m < k; m += kRWideThreads) {
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
  if (!r1_reduce(a, a.tick + 2 * (1 + a.ngrp), 2 * k + 3, tot, &s_last)) return;
  const float* s_vc = tot;          // V^T c
  const float* s_pq = tot + k;      // P^T q^
  const float* s_sc = tot + 2 * k;  // q^.c, p_j.c, ||c||^2

  // q vanished (qinv = 0): nothing changes, and no rotation is pending
  float* H = a.H;
  const float av = H[size_t(j) * k + j], bv = s_sc[0], sv = s_vc[j];
  float cs = 1.f, sn = 0.f;
  const bool rotate = qinv > 0.f;
  if (rotate) {
    const float t = 0.5f * atan2f(2.f * sv, av - bv);
    sincosf(t, &sn, &cs);
  }
  const int i = tid;
  double colv2 = 0.0;
  if (rotate && i < k) {
    float colv;
    if (i != j) {
      const float old_r = H[size_t(j) * k + i];
      const float new_r = fmaf(cs, old_r, sn * s_pq[i]);
      H[size_t(j) * k + i] = new_r;
      a.cs2[i] += double(new_r) * new_r - double(old_r) * old_r;
      const float old_c = H[size_t(i) * k + j];
      colv = fmaf(cs, old_c, sn * s_vc[i]);
      H[size_t(i) * k + j] = colv;
    } else {
      colv = cs * cs * av + cs * sn * (sv + s_pq[j]) + sn * sn * bv;
      H[size_t(j) * k + j] = colv;
    }
    colv2 = double(colv) * colv;
  }
  s_dd[tid] = colv2;
  __syncthreads();
  for (int o = kRWideThreads / 2; o > 0; o >>= 1) {
    if (tid < o) s_dd[tid] += s_dd[tid + o];
    __syncthreads();
  }
  if (tid == 0 && rotate) {
    a.cs2[j] = s_dd[0];
    const double c2 = double(cs) * cs, sc = double(cs) * sn, s2 = double(sn) * sn;
    a.pn[j] = c2 * a.pn[j] + 2.0 * sc * double(s_sc[1]) + s2 * double(s_sc[2]);
  }
  __syncthreads();
  // the next column: largest pn - cs2, the first of equals
  s_dd[tid] = (i < k) ? a.pn[i] - a.cs2[i] : -INFINITY;
  s_ii[tid] = i;
  __syncthreads();
  for (int o = kRWideThreads / 2; o > 0; o >>= 1) {
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
    const int step = ctl->step;
    if (a.order) a.order[step] = j;
    ctl->jp = rotate ? j : -1;
    ctl->cs = cs;
    ctl->sn = sn;
    ctl->j = s_ii[0];
    ctl->step = step + 1;
  }
}

// init (one CTA): H, pn and cs2 from the Gram matrix of the stacked block
// [V; P] (G2, kp2 x kp2, lower tiles: G2[k + i][m] = p_i . v_m), one row per
// warp at a time with the lanes over m; then the first column and a clean
// control block.
__global__ void __launch_bounds__(kRThreads) r1_init_kernel(R1Args a, const float* __restrict__ G2,
                                                            int kp2) {
  constexpr int kW = kRThreads / 32;
  __shared__ double s_dd[kRThreads];
  __shared__ int s_ii[kRThreads];
  __shared__ double s_rho[kRMaxK];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, k = a.k;
  for (int i = warp; i < k; i += kW) {
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
      const double p2 = double(row[k + i]);
      a.pn[i] = p2;
      a.cs2[i] = acc;
      s_rho[i] = p2 - acc;
    }
  }
  __syncthreads();
  s_dd[tid] = (tid < k) ? s_rho[tid] : -INFINITY;
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
  }
}

// finish: the pending rotation applied to this slice of V, and V written as
// the d x k bf16 basis.  With no correction (jp = -1) V is the start basis.
__global__ void __launch_bounds__(kRThreads) r1_finish_kernel(R1Args a, int any,
                                                              __nv_bfloat16* __restrict__ Vout) {
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
