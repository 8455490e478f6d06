// Tensor-core (tcgen05 + TMEM + TMA) GEMM of the bf16 draft pass: host interface.
#pragma once

#include <cuda_runtime.h>

#include "epilogue.cuh"

namespace peagle {

struct TcGemmPlan;

// Allocates the GEMM's workspace for up to rows_max activation rows and output /
// reduction dimensions up to max_dim.  *out stays NULL when the tensor-core path is
// not available in this build (the caller then uses the FFMA GEMM).
int tc_create(TcGemmPlan** out, int num_sms, int rows_max, int max_dim);
void tc_gemm(TcGemmPlan* p, const void* W, const void* X, int ldx, int Nout, int Kd, int R,
             const EpiArgs& epi, cudaStream_t s);
void tc_destroy(TcGemmPlan* p);

}  // namespace peagle
