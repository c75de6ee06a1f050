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
  float* y;                 // T x d_out
  int T, d_out, d, k;
  uint32_t* status;
};

// Encode a TMA map (CUtensorMap, 128 bytes at `map`) of a row-major bf16
// rows x cols tensor with a box_rows x box_cols box, 128-byte swizzle and zero
// fill outside the tensor.  False if the driver rejects it.
bool tma_encode_bf16_2d(void* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols);

// Build the TMA tensor maps of a handle (after its workspace is bound).
gsi_status_t tc_gemm_prepare(gsi_handle* h);
// One launch computing both GEMMs for T tokens.
gsi_status_t tc_gemm_launch(gsi_handle* h, const TcGemmArgs& a, cudaStream_t s);
int tc_gemm_launch_count();

}  // namespace gsi
