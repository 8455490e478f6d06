// Kernels of the training step (forward with saved activations, backward) on fp32 rows;
// see train_kernels.cu.  Row i of a call is (row_p[i], row_d[i]); rows outside the
// training contract are skipped (the rows-prepare kernels flag them).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace peagle {

// Attention geometry of one call: M rows, n positions, chain[i][t] = row of
// (p - t, d - t) for t = 0 .. d - 2, -1 elsewhere ([M][K - 1]).
struct TrainAttn {
  int M, n, K, nq, nkv, hd;
  float scale;
  const int* row_p;
  const int* row_d;
  const int* chain;
};

// tcgen05 forms of the fused prefix attention (train_attn_tc.cu): head_dim 64 and
// G = nq / nkv in {1, 2, 4, 8}.
struct TcGemmPlan;
struct TrainAttnTc {
  TcGemmPlan* tc;  // tensor-map encoder
  unsigned* err;   // device error word (bounded waits latch TIMEOUT)
  float* kvT;      // [nkv][64][ldn]: one layer's keys or values transposed
  int ldn;         // >= n, a multiple of 4
  float* qT;       // [nq][64][ldm]: queries transposed (backward)
  float* doT;      // [nq][64][ldm]: dO transposed (backward)
  int ldm;         // >= M, a multiple of 4
};

void launch_train_inputs(bool bf16, int M, int n, int K, int H, const int* row_p,
                         const int* row_d, const int* tokens, const void* hidden,
                         const void* embed, int Vt, const void* emb_mask, const void* h_shared,
                         float* E, float* Hin, unsigned* err, cudaStream_t s);
void launch_rms_fwd(int M, int D, const float* x, int ldx, const float* g, float eps, float* y,
                    int ldy, float* r, cudaStream_t s);
void launch_rms_bwd(int M, int D, const float* x, int ldx, const float* r, const float* g,
                    const float* dy, int ldy, float* dx, int lddx, bool acc, cudaStream_t s);
// out[h] += sum_i a[i][h] * (b ? b[i][h] : 1) * (rs ? rs[i] : 1), skipping depth-1 rows
// when skip_depth1_rows (row_d) is given
void launch_colsum(int M, int D, const float* a, int lda, const float* b, int ldb,
                   const float* rs, const int* skip_depth1_rows, float* out, cudaStream_t s);
void launch_swiglu_fwd(int M, int I, const float* gu, float* act, cudaStream_t s);
void launch_swiglu_bwd(int M, int I, const float* gu, const float* dact, float* dgu,
                       cudaStream_t s);
void launch_gu_split(int I, int H, const float* dw, float* dgate, float* dup, cudaStream_t s);
void launch_train_rope(int M, int n, int K, int nq, int nkv, int hd, const float* qkv,
                       const int* row_p, const int* row_d, const float2* tab, float* Qh,
                       float* Kr, float* Vr, float* K1, float* V1, bool tf32, cudaStream_t s);
void launch_train_rope_bwd(int M, int n, int K, int nq, int nkv, int hd, const float* dQh,
                           const float* dKr, const float* dVr, const int* row_p,
                           const int* row_d, const float2* tab, float* dqkv, cudaStream_t s);
void launch_chain(int M, int n, int K, int Kmax, const int* row_p, const int* row_d,
                  const int* row_index, int* chain, cudaStream_t s);
void launch_attn_fwd_softmax(const TrainAttn& a, int g, float* S1, const float* Qh,
                             const float* Kr, float* Pc, float* lse, cudaStream_t s);
void launch_attn_fwd_out(const TrainAttn& a, int g, const float* Oh, const float* Pc,
                         const float* Vr, float* O, cudaStream_t s);
void launch_attn_bwd_prep(const TrainAttn& a, const float* dO, const float* O, float* dOh,
                          float* Dv, bool tf32, cudaStream_t s);
void launch_attn_bwd_ds(const TrainAttn& a, int g, float* S1, float* dP1, const float* lse,
                        const float* Dv, const float* Qh, const float* Kr, const float* Vr,
                        const float* dOh, float* dQh, float* dKr, float* dVr, cudaStream_t s);
// The chain part of the backward (the prefix part on the fused kernels): dQh's chain part
// stored, the chain keys' dKr / dVr added; one launch for every kv head.  False (nothing
// launched) for K > 16 or head_dim other than 64 / 128.
bool launch_attn_bwd_chain(const TrainAttn& a, const float* lse, const float* Dv,
                           const float* Qh, const float* Kr, const float* Vr, const float* dOh,
                           float* dQh, float* dKr, float* dVr, cudaStream_t s);
void launch_kv1_scatter(int M, int n, int K, int nkv, int hd, const int* row_p, const int* row_d,
                        const float* dK1, const float* dV1, float* dKr, float* dVr,
                        cudaStream_t s);
// Fused prefix-attention backward on TF32 tensor cores (train_attn_mma.cu), for head_dim
// 64 and at most 8 q heads per kv head: dQh += dS K1 (dQh holds the chain part) and
// dK1 / dV1 (zero beforehand) += dS^T Q / P^T dO; row_index as from rows-prepare.  Qh, K1,
// V1 and dOh are stored rounded to TF32 by their producers (launch_train_rope and
// launch_attn_bwd_prep with tf32 set).
bool attn_bwd_fused_ok(const TrainAttn& a);
// The forward the same way (Q, K1, V1 stored rounded to TF32): the prefix's unnormalised
// output Op (per-head rows [nq][M][64]) with its row max / sum, then the chain keys joined
// per row: lse, Pc and O [M][nq hd].
// With tcx (and attn_tc_ok), the prefix part runs on the tcgen05 kernel.
int launch_attn_fwd_fused(const TrainAttn& a, float* Qh, const float* Kr, const float* Vr,
                          float* K1, float* V1, float* Op, float* mrow, float* lrow, float* Pc,
                          float* lse, float* O, const TrainAttnTc* tcx, cudaStream_t s);
// With tcx (and attn_tc_ok), the dQ part runs on the tcgen05 kernel.
int launch_attn_bwd_fused(const TrainAttn& a, const int* row_index, int Kmax, const float* Qh,
                          const float* dOh, const float* K1, const float* V1,
                          const float* lse, const float* Dv, float* dQh, float* dK1,
                          float* dV1, const TrainAttnTc* tcx, cudaStream_t s);
bool attn_tc_ok(const TrainAttn& a);
// The prefix part of the forward (Q, K1, V1 already rounded to TF32): Op, mrow, lrow as
// launch_attn_fwd_fused's prefix kernel writes them.  V1 is transposed into kvT first.
int launch_attn_fwd_prefix_tc(const TrainAttn& a, const TrainAttnTc& x, const float* Qh,
                              const float* K1, const float* V1, float* Op, float* mrow,
                              float* lrow, cudaStream_t s);
// dQh += dS K1 over the prefix (Q, dO, K1, V1 already rounded to TF32); K1 is
// transposed into kvT first.
int launch_attn_bwd_dq_tc(const TrainAttn& a, const TrainAttnTc& x, const float* Qh,
                          const float* dOh, const float* K1, const float* V1, const float* lse,
                          const float* Dv, float* dQh, cudaStream_t s);
// dK1 += dS^T Q, dV1 += P^T dO over the prefix (operands already rounded to TF32); Q and
// dO are transposed into qT / doT first.
int launch_attn_bwd_dkv_tc(const TrainAttn& a, const TrainAttnTc& x, const int* row_index,
                           int Kmax, const float* Qh, const float* dOh, const float* K1,
                           const float* V1, const float* lse, const float* Dv, float* dK1,
                           float* dV1, cudaStream_t s);
void launch_ce(int M, int V, float* logits, const int* labels, float* row_loss, float* loss,
               unsigned* err, cudaStream_t s);
void launch_embed_grad(int M, int n, int K, int H, int Vt, const int* row_p, const int* row_d,
                       const int* tokens, const float* dE, float* dembed, cudaStream_t s);
void launch_to_f32(size_t n, const void* src_bf16, float* dst, cudaStream_t s);
void launch_add(size_t n, const float* a, float* b, cudaStream_t s);

}  // namespace peagle
