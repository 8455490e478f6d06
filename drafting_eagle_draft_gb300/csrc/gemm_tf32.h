// The training step's plain products (see gemm_tf32.cu): tcgen05 TF32 GEMMs for bf16
// drafters, CUDA-core fp32 GEMMs for fp32 drafters.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace peagle {

struct TcGemmPlan;

struct TrainGemmCtx {
  TcGemmPlan* tc;          // tensor-map encoder (bf16 drafters); null: the fp32 kernel
  float* scratch_a;        // operands transposed (or re-strided) for the tensor cores
  float* scratch_b;
  size_t scratch_floats;   // capacity of each scratch buffer
  unsigned* err;           // device error word (timeouts of the bounded waits)
};

// out[c][r] = in[r][c] (in: rows x cols, row stride ld_in; out row stride ld_out), for
// `batch` matrices stride_in / stride_out floats apart.
void launch_transpose_f32(const float* in, int rows, int cols, int ld_in, float* out, int ld_out,
                          cudaStream_t s, int batch = 1, size_t stride_in = 0,
                          size_t stride_out = 0);

// Floats of a scratch buffer that holds a [rows][cols] operand with a padded row stride.
size_t tf32_scratch_floats(int rows, int cols);

// Row-major C [m x n] = alpha op(A) op(B) + beta C, op(A) [m x k] (A stored [m x k], or
// [k x m] when ta), op(B) [k x n] (B stored [k x n], or [n x k] when tb).  Asynchronous on
// s; PEAGLE_ERR_CAPACITY if a transposed operand does not fit the scratch buffers.
int train_gemm(const TrainGemmCtx& g, bool ta, bool tb, int m, int n, int k, float alpha,
               const float* A, int lda, const float* B, int ldb, float beta, float* C, int ldc,
               cudaStream_t s);

}  // namespace peagle
