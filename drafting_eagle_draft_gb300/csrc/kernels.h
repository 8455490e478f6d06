// Internal launchers of the P-EAGLE GB300 library (host side, C++).  Not part of the
// C ABI: peagle_api.cu composes them into the calls declared in include/peagle.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "epilogue.cuh"

namespace peagle {

struct AttnArgs {
  const void* q;          // [R, nq*hd] fp32 (post-RoPE)
  const void* kc;         // layer cache base [B][nkv][cap][hd]
  const void* vc;
  const int* seq_lens;    // [B]
  void* o;                // [R, nq*hd] (hi rows, then lo rows when split)
  int split;
  float* part;            // split-KV partials
  unsigned* counters;     // [B * nkv], zero between launches
  int B, K, nq, nkv, hd, cap, chunk, nchunk;
  int window;             // sliding window in positions (0: whole context); see attn_span
  float scale;
  unsigned* err;
};

struct MaskedAttnArgs {
  const void* q;          // [M, nq*hd] post-RoPE: fp32, or bf16 when q_bf16
  const void* k;          // [M, nkv, hd]   all rows
  const void* v;
  const void* k1;         // [n, nkv, hd]   depth-1 rows by position
  const void* v1;
  const int* row_p;       // [M]
  const int* row_d;       // [M]
  const int* row_index;   // [n * (Kmax + 1)] row of (p, d), -1 if absent
  void* o;                // [M, nq*hd] (hi rows, then lo rows when split)
  int split;
  int q_bf16;             // queries stored as bf16 (the tensor-core kernel only)
  int M, n, Kmax, nq, nkv, hd;
  float scale;
  unsigned* err;          // device error word (timeouts of the tensor-core kernel)
};

// fp32-accumulating FFMA GEMM: Y[r, m] = sum_k X[r, k] W[m, k]; then the fused epilogue.
void launch_gemm_simt(bool bf16, const void* W, const void* X, int ldx, float* Y, int ldy,
                      int Nout, int Kd, int R, const EpiArgs& epi, cudaStream_t s);

void launch_input_fusion(bool bf16, int mode, int R, int K, int n_src, int H, const void* embed,
                         int Vt,
                         const void* emb_mask, fx_t* F, const fx_t* f_shared,
                         const int* tokens, const int* row_p, const int* row_d,
                         const void* g_in, const void* g_hid, float eps, int split, void* X0,
                         fx_t* res, unsigned long long* keys, const int* seq_lens, int* row_pos,
                         unsigned* err, cudaStream_t s);

void launch_rmsnorm(bool bf16, int R, int H, const fx_t* res, const void* gamma, float eps,
                    int split, void* out, cudaStream_t s);

// bf16 draft pass: fixed-point q / k,v sums of one layer -> fp32 queries and the KV cache
// slots row_pos[r]; clears the sums
void launch_qkv_finalize(int R, int K, int nq, int nkv, int hd, int cap, fx_t* q_fx, fx_t* kv_fx,
                         float* Qf, void* kc, void* vc, const int* row_pos, unsigned* err,
                         cudaStream_t s);

void launch_attention_decode(bool bf16, const AttnArgs& a, cudaStream_t s);

void launch_masked_attention(bool bf16, const MaskedAttnArgs& a, cudaStream_t s);
// The same attention on tcgen05 tensor cores (bf16, head_dim 64, 128 % (nq / nkv) == 0);
// PEAGLE_ERR_UNSUPPORTED for other shapes (nothing launched).  `plan` encodes the TMA maps.
struct TcGemmPlan;
int masked_attn_tc_launch(TcGemmPlan* plan, const MaskedAttnArgs& a, cudaStream_t s);

// Efficient LM head: rank-r scores approx [R][Vd] of the fixed-point projection zfx [R][r]
// (r = 64, 128, 256 or 512) and their first-digit histogram, added into hist [R][2048];
// per-row top-k of approx -> cand [R][k] through the list gkey / gidx [R][4096] and the
// counters gcount / gdone [R] (the top-k launch clears hist, the counters and zfx); exact
// logits of the candidates -> argmax keys (+ logits, -inf elsewhere, when `logits` is
// given), decoded into out (token ids through d2t) by the last CTA, which also clears keys
// and the `done` counter.  H * 4 bytes of shared memory.
void launch_head_score(bool bf16, int R, int r, int Vd, const fx_t* zfx, const void* score,
                       float* approx, unsigned* hist, unsigned* err, int num_sms, cudaStream_t s);
void launch_topk(int R, int n, int k, const float* score, unsigned* hist, unsigned* gcount,
                 unsigned* gdone, unsigned* gkey, int* gidx, int* cand, fx_t* zfx, int zn,
                 int num_sms, cudaStream_t s);
void launch_cand_head(bool bf16, int R, int H, int k, const int* cand, const void* head,
                      const void* y, int split, unsigned long long* keys, float* logits, int Vd,
                      const int* d2t, int* out, unsigned* done, cudaStream_t s);
void launch_argmax_decode(int R, unsigned long long* keys, const int* d2t, int* out_tokens,
                          cudaStream_t s);

void launch_verify(int B, int K, const int* draft, const int* tgt, int* acc, int* bonus,
                   cudaStream_t s);

void launch_append_kv(bool bf16, int B, int N, int nkv, int hd, int cap, void* kc, void* vc,
                      int* seq_lens, const int* n_commit, int n_extra, const void* k_rows,
                      const void* v_rows, int n_max, int batch_slots, unsigned* err,
                      cudaStream_t s);

void launch_rows_prepare(int M, int n, int K, int Kmax, const int* row_p, const int* row_d,
                         int* row_index, unsigned* err, cudaStream_t s);

}  // namespace peagle
