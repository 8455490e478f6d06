#include "gemm_tc.h"

namespace peagle {
struct TcGemmPlan {};
int tc_create(TcGemmPlan** out, int, int, int) { *out = nullptr; return 0; }
void tc_gemm(TcGemmPlan*, const void*, const void*, int, int, int, int, const EpiArgs&, cudaStream_t) {}
void tc_destroy(TcGemmPlan*) {}
}  // namespace peagle
