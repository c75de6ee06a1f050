// gsi_internal.h -- host-side handle layout and the launchers that the C ABI
// (gsi_api.cu) calls.  Not part of the public interface (include/gsi.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gsi.h"

struct gsi_group;

namespace gsi {
constexpr int kMaxGroup = 4;  // one-token calls per gsi_group_forward launch
// Launch plan of the one-exchange decode kernel for one handle on G CTAs
// (CTA 0 decides the gate; CTAs 1..G-1 own rows_V rows of V_k and rows_M
// output rows each).
struct CrPlan {
  int G = 0, rows_M = 0, rows_V = 0;
  int box_M = 0, nbox_M = 0, box_V = 0, nbox_V = 0;  // TMA row boxes
  int vbits = 0;            // bound of a CTA's partial projection, in powers of two of max|x|
  size_t smem = 0;
  bool coresident = false;  // two CTAs (of consecutive calls) fit on one SM
};
}  // namespace gsi

struct gsi_handle {
  // Borrowed operands (section 2.1 of the GSI summary): W (d_out x d),
  // V_k (d x k), M = W V_k (d_out x k), all bf16 row-major, device memory.
  const __nv_bfloat16* W = nullptr;
  const __nv_bfloat16* V = nullptr;
  const __nv_bfloat16* M = nullptr;
  int64_t d_out = 0, d = 0, k = 0;
  float eps = 0.f;
  int device = 0;
  int num_sms = 0;

  // ---- decode path (T = 1): one fused persistent kernel ------------------
  int dec_grid = 0;          // CTAs (all co-resident; one per SM at most)
  int dec_rows_M = 0;        // rows of M / W per CTA
  int dec_rows_V = 0;        // rows of V_k per CTA
  bool dec_stage_M = false;  // M slice staged in shared memory by bulk copy
  bool dec_stage_V = false;  // V slice staged in shared memory by bulk copy
  size_t dec_smem = 0;       // dynamic shared memory bytes
  bool use_pdl = true;       // programmatic dependent launch between kernels

  // ---- one-exchange decode kernel (k in {64, 128, 256}), used when it fits --
  bool cr_ok = false;
  gsi::CrPlan cr_plan;
  alignas(64) unsigned char cr_tmaps[2][128] = {};  // TMA maps of V_k and M (CUtensorMap)
  __nv_bfloat16* cr_F = nullptr;  // correction tiles (corr_tiles_elems(k))
  float* cr_acc = nullptr;        // decode_cr_acc_floats(k) fp32 digit accumulators
  uint32_t* cr_bar = nullptr;     // [0] arrival counter, [1] launch epoch, [2] counter base,
                                  // [4..5] published gate (64-bit)
  float cr_vmax = 0.f;            // largest column norm of V_k (from the Gram matrix)
  float cr_normE = 0.f;           // upper bound of ||E||_2 for the correction tiles

  // L2 prefetch link (gsi_set_prefetch, gsi_set_prefetch_group): each
  // one-token call on this handle prefetches the V_k, M and correction tiles
  // of pf_next, or of every member of pf_group, into L2.  pf_from and
  // pf_from_groups list the handles and groups whose link points here, so
  // destroying this handle unlinks them.
  gsi_handle* pf_next = nullptr;
  gsi_group* pf_group = nullptr;
  std::vector<gsi_handle*> pf_from;
  std::vector<gsi_group*> pf_from_groups;

  // ---- device workspace (one allocation) --------------------------------
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float* gram = nullptr;       // k x k fp32, V_k^T V_k (batched path)
  float* dec_acc = nullptr;    // 2 x acc_stride fp32: g (k), ||x||^2, ||r||^2
  int dec_acc_stride = 0;
  uint32_t* dec_bar = nullptr; // [0] arrival counter, [1] launch epoch
  uint32_t* status = nullptr;  // device status word (kStatus* bits)

  // batched path, sized for max_T tokens
  int64_t max_T = 0;
  void* bws = nullptr;         // separate allocation, regrown by gsi_reserve
  size_t bws_bytes = 0;
  float* bG = nullptr;         // max_T x k   projections g_t
  float* bsx = nullptr;        // max_T       ||x_t||^2
  uint8_t* bgate = nullptr;    // max_T       internal copy of the gates
  int32_t* bidx_fast = nullptr;// max_T       token indices of fast tokens
  int32_t* bidx_slow = nullptr;// max_T       token indices of slow tokens
  int32_t* bcount = nullptr;   // [0] n_fast, [1] n_slow
  __nv_bfloat16* bGf = nullptr;// [2][max_T][k] gathered g of fast tokens (hi, lo planes)
  __nv_bfloat16* bXs = nullptr;// max_T x d   gathered x of slow tokens
  __nv_bfloat16* bVT = nullptr;// k x d       V_k transposed (tensor-core projection)
  float* bP = nullptr;         // [8][max_T][k] projection partials (tensor-core projection)
  float* bsxp = nullptr;       // [8][max_T] ||x||^2 over each slice (tensor-core projection)
  alignas(64) unsigned char tmaps_proj[128] = {};  // TMA map of bVT
  // TMA tensor maps of the tcgen05 GEMMs (CUtensorMap, 128 bytes each):
  // W, M, G_fast hi plane, G_fast lo plane, X_slow
  alignas(64) unsigned char tmaps[14][128] = {};  // the batched GEMM's tensor maps

  // host staging for gsi_forward_host
  void* st_dev = nullptr;
  size_t st_bytes = 0;
  int64_t st_T = 0;
};

// Several one-token calls in one launch (gsi_group_create): members borrow
// their handles' operands and workspaces.
struct gsi_group {
  int n = 0, k = 0, device = 0;
  gsi_handle* h[gsi::kMaxGroup] = {};
  gsi::CrPlan plan[gsi::kMaxGroup];
  int cta0[gsi::kMaxGroup + 1] = {};  // member m owns CTAs [cta0[m], cta0[m + 1])
  size_t smem = 0;
  alignas(64) unsigned char tmaps[2 * gsi::kMaxGroup][128] = {};
  gsi_handle* pf_next = nullptr;        // prefetch target of the group's launches
  std::vector<gsi_handle*> pf_from;     // handles whose pf_group is this group
};

namespace gsi {

// Correction tiles of E = V_k^T V_k - I, for the identity
// g^T E g = sum_{I <= J} g_I^T F_IJ g_J over 16 x 16 blocks: F_II = E_II and
// F_IJ = 2 E_IJ for I < J (E is symmetric).  The k/16 (k/16 + 1) / 2 upper
// tiles are stored row by row (I, then J >= I), 256 bf16 each, in the order
// of the A operand of a 16 x 16 x 8 bf16 MMA: lane l (group l / 4, pair
// l % 4) owns 8 consecutive values, its registers a0..a3 = (rows group and
// group + 8) x (columns 2 pair, 2 pair + 1 and the same + 8), lower column in
// the lower half of each register.
__host__ __device__ inline int corr_tile_index(int I, int J, int t16) {
  return I * t16 - I * (I - 1) / 2 + (J - I);
}
__host__ __device__ inline size_t corr_tiles_elems(int k) {
  const size_t t = size_t(k) / 16;
  return t * (t + 1) / 2 * 256;
}
// Position of E block element (r, c) (0 <= r, c < 16) inside its tile.
__host__ __device__ inline int corr_tile_pos(int r, int c) {
  const int lane = (r & 7) * 4 + ((c & 7) >> 1);
  const int reg = (r >> 3) + 2 * (c >> 3);
  return lane * 8 + reg * 2 + (c & 1);
}

// Decode path (gsi_decode.cu)
gsi_status_t decode_configure(gsi_handle* h);
gsi_status_t decode_launch(gsi_handle* h, const void* x, float* y, uint8_t* gate,
                           float* rho, cudaStream_t s);

// One-exchange decode path (gsi_decode_cr.cu), k in {64, 128, 256}
size_t decode_cr_acc_floats(int64_t k);
gsi_status_t decode_cr_configure(gsi_handle* h);
gsi_status_t decode_cr_launch(gsi_handle* h, const void* x, float* y, uint8_t* gate,
                              float* rho, cudaStream_t s);
// Upper bound of the spectral norm of the symmetric matrix that the
// correction tiles (bf16, corr_tiles_elems(k) values) represent.
double corr_norm_bound(const uint16_t* tiles, int k);
gsi_status_t group_configure(gsi_group* g);
gsi_status_t group_launch(gsi_group* g, const void* const* x, float* const* y,
                          uint8_t* const* gate, float* const* rho, cudaStream_t s);

// Batched path (gsi_batched.cu)
gsi_status_t batched_launch(gsi_handle* h, const void* x, int64_t T, float* y,
                            uint8_t* gate, float* rho, cudaStream_t s);
int batched_launch_count(const gsi_handle* h, int64_t T);
size_t batched_workspace_bytes(int64_t max_T, int64_t d, int64_t k);
void batched_bind_workspace(gsi_handle* h, void* base, int64_t max_T);
gsi_status_t batched_prepare(gsi_handle* h);  // after binding: V_k^T, tensor maps

// One-off operand preparation (gsi_prep.cu)
gsi_status_t gram_launch(const __nv_bfloat16* V, int64_t d, int64_t k, float* gram,
                         __nv_bfloat16* F, cudaStream_t s);
gsi_status_t precompute_M_launch(const __nv_bfloat16* W, const __nv_bfloat16* V,
                                 __nv_bfloat16* M, int64_t d_out, int64_t d, int64_t k,
                                 cudaStream_t s);

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace gsi
