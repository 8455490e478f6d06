// Tensor-core (tcgen05 + TMEM + TMA) GEMM of the bf16 draft pass: host interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"

namespace peagle {

struct TcGemmPlan;

// Allocates the GEMM's workspace (stream-K partial slots and tile counters) for up to
// rows_max activation rows and output dimensions up to max_dim; device-side timeouts are
// reported in *err.
int tc_create(TcGemmPlan** out, int num_sms, int rows_max, int max_dim, unsigned* err);
// Launches Y^T = W X^T with the fused epilogue `epi` on stream s (asynchronous).
//   W [Nout, Kd] bf16 row-major (device), X [rows, Kd] bf16 with row stride ldx elements;
//   rows = R, or 2R when epi.in_split (hi rows then lo rows).  Kd % 64 == 0.
// Returns PEAGLE_OK or a negative PEAGLE_ERR_* code (nothing launched on error).
int tc_gemm(TcGemmPlan* p, const void* W, const void* X, int ldx, int Nout, int Kd, int R,
            const EpiArgs& epi, cudaStream_t s);
void tc_destroy(TcGemmPlan* p);

// Pieces of the plan shared with the persistent pass kernel: a cached 2D bf16 tensor map
// (box 64 columns x box_rows rows, 128-byte swizzle), the partial slots
// [2 * num_sms][256][128] fp32 and the per-tile counters (zero between projections).
bool tc_tensor_map(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                   int ld, int box_rows);
// [rows][cols] bf16 (row stride ld, cols a multiple of 64) as ku-k-block boxes: one load
// brings ku consecutive 64-wide k-blocks of box_rows rows, each a 128-byte-swizzled tile
// (k-blocks past cols read as zero).
bool tc_tensor_map_ku(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                      int ld, int box_rows, int ku);
// [rows][cols] fp32 (row stride ld, a multiple of 4), boxes of 32 columns x box_rows rows
// (<= 256), 128-byte swizzle: the TF32 GEMM's K-major operands.
bool tc_tensor_map_f32(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                       int ld, int box_rows);
float* tc_partials(TcGemmPlan* p);
int tc_num_sms(TcGemmPlan* p);
unsigned* tc_tile_counters(TcGemmPlan* p);
int tc_max_tiles(TcGemmPlan* p);

}  // namespace peagle
