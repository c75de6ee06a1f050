// gsi_tc_gemm.h -- tcgen05 (5th-generation tensor core) GEMMs of the batched
// GSI path: Y_fast = G_fast M^T and Y_slow = X_slow W^T, scattered to y.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gsi.h"

struct gsi_handle;

namespace gsi {

struct TcGemmArgs {
  const __nv_bfloat16* W;   // d_out x d
  const __nv_bfloat16* M;   // d_out x k
  const __nv_bfloat16* Gf;  // [2][max_T][k]: hi and lo planes of fast tokens' g
  const __nv_bfloat16* Xs;  // max_T x d: slow tokens' x
  const int32_t* idx_fast;  // fast token indices (count[0] of them)
  const int32_t* idx_slow;  // slow token indices (count[1] of them)
  const int32_t* count;     // [0] n_fast, [1] n_slow (device)
  int32_t* tile_counter;    // device, zero at launch: the GEMM's tile queue
  float* y;                 // T x d_out
  int T, d_out, d, k;
  uint32_t* status;
};

// Encode a TMA map (CUtensorMap, 128 bytes at `map`) of a row-major bf16
// rows x cols tensor with a box_rows x box_cols box, 128-byte swizzle and zero
// fill outside the tensor.  False if the driver rejects it.
bool tma_encode_bf16_2d(void* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols);

// Projection G = X V_k on the tensor cores (T > 1, k in {128, 256}): S
// slices of the reduction dimension, fp32 partials in the handle's P buffer.
constexpr int kProjMaxSplits = 8;
__host__ __device__ constexpr int tc_proj_max_splits() { return kProjMaxSplits; }
struct TcProjArgs {
  float* P;             // [S][max_T][k] partials
  int T, d, k, kb_per;  // kb_per: 64-wide reduction steps per slice
  int stages;           // TMA ring depth (<= 8; the launch sizes shared memory to it)
  int a_fixed;          // 1: no kernel of the stream writes A (the handle's V_k^T), so
                        // the first stages' A boxes load before the dependent-launch wait
  size_t split_stride;  // floats between slices
  uint32_t* status;
  float* sxp;           // if set (the CTAs of the first 128 entries): ||x_t||^2 over the
                        // slice, sxp[s * sxp_stride + t]; the epilogue warps sum the
                        // staged x tiles while the MMAs run
  size_t sxp_stride;
};
bool tc_proj_supported(const gsi_handle* h);
gsi_status_t tc_proj_prepare(gsi_handle* h);
int tc_proj_splits(const gsi_handle* h, int64_t T, int* kb_per);
gsi_status_t tc_proj_launch(gsi_handle* h, const void* x, int64_t T, int S, int kb_per,
                            cudaStream_t s);

// The projection kernel as a general split-K product on the tensor cores:
// P[s][b][a] = sum over slice s of the K axis of A[a][:] . B[b][:], with A
// (rows_a x K) and B (rows_b x K) row-major bf16 (16-byte aligned,
// K % 8 == 0), fp32 partials with slice stride split_stride.  Ragged edges
// are read as zeros by the tensor maps.  S * kb_per * 64 must cover K.
gsi_status_t tc_nt_prepare();
int tc_nt_splits(int64_t rows_a, int64_t rows_b, int64_t K, int num_sms, int* kb_per);
gsi_status_t tc_nt_gemm(const void* A, int64_t rows_a, const void* B, int64_t rows_b, int64_t K,
                        float* P, size_t split_stride, int S, int kb_per, uint32_t* status,
                        cudaStream_t s);

// Build the TMA tensor maps of a handle (after its workspace is bound).
gsi_status_t tc_gemm_prepare(gsi_handle* h);
// One launch computing both GEMMs for T tokens.
gsi_status_t tc_gemm_launch(gsi_handle* h, const TcGemmArgs& a, cudaStream_t s);
int tc_gemm_launch_count();

}  // namespace gsi
