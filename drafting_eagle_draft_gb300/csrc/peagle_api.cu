// C ABI of the P-EAGLE GB300 library (declared in include/peagle.h): argument
// validation, the drafter context (weights + workspaces, allocated once in
// peagle_create), and the kernel sequences of the draft pass, verification, KV commit
// and the training-style forward.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <memory>
#include <vector>


#include "gemm_tc.h"
#include "kernels.h"
#include "pass_kernel.h"
#include "tc_ptx.cuh"
#include "gemm_tf32.h"
#include "train_kernels.h"

using namespace peagle;

// pass-kernel calls whose phase times one timing read can report
constexpr int PASS_TRACE_SLOTS = 64;

// Training-step workspace, allocated by the first peagle_train_step for max_rows rows and
// max_seq positions: fp32 copies of the weights (bf16 contexts), the forward's saved
// activations per layer and the backward's buffers.
struct TrainWs {
  float *gscratch_a = nullptr, *gscratch_b = nullptr;  // transposed GEMM operands
  size_t gscratch_floats = 0;
  int Mmax = 0, nmax = 0;
  // fp32 weights (the context's own buffers on fp32 contexts); gate / up interleaved
  float *fc, *lm, *in_norm, *hid_norm, *fin_norm;
  std::vector<float*> qkv, o, gu, down, attn_norm, post_norm;
  // bf16 contexts: the projection weights transposed ([in][out]), the K-major B operand
  // of the backward's dX = dY W on the tensor cores (null on fp32 contexts)
  float *fcT = nullptr, *lmT = nullptr;
  std::vector<float*> qkvT, oT, guT, downT;
  // the tcgen05 prefix attention: one layer's keys or values transposed [nkv][64][ldn]
  float* kvT = nullptr;
  int ldn = 0;
  float *qT = nullptr, *doT = nullptr;  // [nq][64][ldm]: queries / dO transposed
  int ldm = 0;
  // forward (saved)
  int* chain;
  float *E, *Hin, *f, *r1, *r2, *x0, *y, *ry, *logits, *row_loss, *resL;
  std::vector<float*> res_in, a, ra, Qh, Kr, Vr, K1, V1, Pc, lse, O, res_mid, u, ru, GU, act;
  // scratch
  float *qkvb, *S1, *dP1, *Oh, *lrow;
  // backward
  float *bufA, *bufB, *dact, *dGU, *du, *dO, *dOh, *Dv, *dQh, *dKr, *dVr, *dK1, *dV1, *dqkv,
      *da, *dgu_w, *dE, *df, *dHin, *dy;
};

// The arguments a persistent-pass parameter block was built for: a call with the same
// ones reuses the block as it stands (no rebuild on the host before the launch).
struct PassKey {
  int B, K, all_ntp, capacity, batch;
  const void* k;
  const void* v;
  const void* seq_lens;
  const void* target_hidden;
  const void* new_token;
  const void* out_tokens;
  const void* out_logits;
};

struct peagle_ctx {
  peagle_dims d;
  bool bf;          // bf16 storage
  size_t es;        // element size
  int device;
  int num_sms;
  // weights (library-owned device memory)
  void *embed, *emb_mask, *h_shared, *fc, *input_norm, *hidden_norm, *final_norm, *lm_head;
  // efficient LM head (dims.lm_rank > 0): weights and per-pass buffers
  void *lm_proj, *lm_score;
  fx_t* lm_zfx;             // [rows][rank] fixed-point projection
  float* lm_approx;         // [rows][Vd] rank-r scores
  int* lm_cand;             // [rows][k] candidates
  unsigned* lm_hist;        // [rows][2048] first-digit histogram of the scores
  unsigned *lm_gcount, *lm_gdone;  // [rows] gathered keys / finished slices of the top-k
  unsigned* lm_gkey;        // [rows][4096] gathered keys and their indices
  int* lm_gidx;
  unsigned* lm_done;        // CTAs of the candidate head that have finished
  int* d2t;
  std::vector<void*> qkv, o, attn_norm, post_norm, gate_up, down;
  float2* rope;
  fx_t* f_shared;   // fc(h_shared) [H], fixed point
  // workspaces
  int rows_max;     // activation operand rows: 2 * max(max_batch * max_K, max_rows)
  fx_t* F;          // fc outputs [max(max_batch, max_seq), H], fixed point, zero between uses
  void* X0;         // [rows_max, 2H]
  fx_t* res;        // residual stream [rows_max, H], fixed point
  void* Xn;         // [rows_max, H]
  float* Qf;        // [max(max_batch*max_K, max_rows), nq*hd] fp32 post-RoPE queries
  void* O;          // [rows_max, nq*hd]
  void* act;        // [rows_max, I]
  float* Y;         // fp32 GEMM output (FFMA path) [rows_max, max_out]
  int ldY;
  unsigned long long* keys;  // [rows_max]
  int* row_pos;     // [max_batch * max_K] RoPE position / cache slot of each draft row
  float* att_part;
  unsigned* att_cnt;
  int att_chunks_max;
  // training-style forward
  void *Kr, *Vr, *K1, *V1;
  int* row_index;
  unsigned* err;
  unsigned last_err_bits;
  TcGemmPlan* tc;   // tensor-core GEMM state (bf16 only)
  // persistent pass kernel (bf16): phase counters + abort flag, host-side parameter block
  bool pass_on;     // available (bf16, cooperative launch, at most PASS_MAX_LAYERS layers)
  int pass_mode;    // peagle_set_pass_kernel: -1 up to 16 draft rows, 0 never, 1 always
  bool pp_valid;    // *pp holds a complete block built for pp_key (not in timing mode)
  PassKey pp_key;
  unsigned* pass_cnt;
  PassParams* pp;
  // timing of the pass kernel: per-call phase completion times (device slots) and the
  // stage of each phase (host)
  fx_t* pass_ss;    // [PASS_SS_SLOTS][PASS_MAX_ROWS] row sums of squares
  fx_t* pass_qfx;   // [PASS_MAX_ROWS, nq*hd] fixed-point queries
  fx_t* pass_kvfx;  // [PASS_MAX_ROWS][2][nkv*hd] fixed-point keys / values
  fx_t* mk_qfx;     // bf16 multi-kernel pass: [max_batch*max_K, nq*hd] fixed-point queries
  fx_t* mk_kvfx;    // and [max_batch*max_K][2][nkv*hd] keys / values (zero between layers)
  unsigned long long* pass_trace;
  std::vector<std::vector<int>> trace_stages;
  unsigned long long* pass_trace_cta;  // per-CTA signal times of the latest traced pass
  int trace_cta_phases;
  // bounded waits of the pass kernel (peagle_set_wait_limit)
  unsigned long long wait_ns;
  int stall_phase;
  size_t F_bytes;
  std::vector<void*> allocs;
  TrainWs* tw = nullptr;
  // optional per-stage timing: CUDA events recorded around each launch on its stream
  bool timing;
  std::vector<cudaEvent_t> ev;
  std::vector<int> ev_stage;
  size_t ev_used;
  int pending_stage;
};

// ---- per-stage timing ------------------------------------------------------------------
static void t_begin(peagle_ctx* c, int stage, cudaStream_t s) {
  if (!c->timing || c->ev_used + 2 > c->ev.size()) {
    c->pending_stage = -1;
    return;
  }
  cudaEventRecord(c->ev[c->ev_used], s);
  c->ev_stage[c->ev_used / 2] = stage;
  c->pending_stage = stage;
}
static void t_end(peagle_ctx* c, cudaStream_t s) {
  if (c->pending_stage < 0) return;
  cudaEventRecord(c->ev[c->ev_used + 1], s);
  c->ev_used += 2;
  c->pending_stage = -1;
}
#define TIMED(stage, call)      \
  do {                          \
    t_begin(c, (stage), s);     \
    call;                       \
    t_end(c, s);                \
  } while (0)

static int cuda_fail(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "peagle: %s: %s\n", what, cudaGetErrorString(e));
    return PEAGLE_ERR_CUDA;
  }
  return PEAGLE_OK;
}
#define CK(x)                                        \
  do {                                               \
    int _r = cuda_fail((x), #x);                     \
    if (_r != PEAGLE_OK) return _r;                  \
  } while (0)

static int dalloc(peagle_ctx* c, void** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  c->allocs.push_back(*p);
  return cudaMemset(*p, 0, bytes) == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

static int copy_in(peagle_ctx* c, void** dst, const void* src, size_t bytes) {
  if (!src) return PEAGLE_ERR_INVALID;
  int r = dalloc(c, dst, bytes);
  if (r) return r;
  CK(cudaMemcpy(*dst, src, bytes, cudaMemcpyDefault));
  return PEAGLE_OK;
}

static void free_ctx(peagle_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  for (void* p : c->allocs) cudaFree(p);
  if (c->tc) tc_destroy(c->tc);
  delete c->tw;
  delete c->pp;
  delete c;
}

static int validate_dims(const peagle_dims* d) {
  if (!d) return PEAGLE_ERR_INVALID;
  if (d->hidden <= 0 || d->n_layers <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 ||
      d->head_dim <= 0 || d->intermediate <= 0 || d->draft_vocab <= 0 || d->target_vocab <= 0 ||
      d->max_batch <= 0 || d->max_K <= 0 || d->max_positions <= 0 || d->max_rows < 0 ||
      d->max_seq < 0 || !(d->rms_eps >= 0.f) || !(d->rope_theta > 0.f))
    return PEAGLE_ERR_INVALID;
  if (d->dtype != PEAGLE_F32 && d->dtype != PEAGLE_BF16) return PEAGLE_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return PEAGLE_ERR_UNSUPPORTED;
  if (d->n_q_heads % d->n_kv_heads) return PEAGLE_ERR_UNSUPPORTED;
  if (d->hidden % 64 || d->intermediate % 64) return PEAGLE_ERR_UNSUPPORTED;
  if (d->hidden > 16384) return PEAGLE_ERR_UNSUPPORTED;
  if (((d->n_q_heads + 2 * d->n_kv_heads) * d->head_dim) % 128) return PEAGLE_ERR_UNSUPPORTED;
  if (d->max_K > 16 || d->max_batch * d->max_K > 256) return PEAGLE_ERR_CAPACITY;
  if (d->max_K * (d->n_q_heads / d->n_kv_heads) > 128) return PEAGLE_ERR_UNSUPPORTED;
  if (d->max_rows > 0 && d->max_seq <= 0) return PEAGLE_ERR_INVALID;
  if (d->attn_window < 0) return PEAGLE_ERR_INVALID;
  if (d->lm_rank < 0 || d->lm_topk < 0) return PEAGLE_ERR_INVALID;
  if (d->lm_rank > 0 &&
      ((d->lm_rank != 64 && d->lm_rank != 128 && d->lm_rank != 256 && d->lm_rank != 512) ||
       d->lm_topk < 1 || d->lm_topk > 1024 || d->hidden > 12288 ||
       d->draft_vocab > (1 << 24)))
    return PEAGLE_ERR_UNSUPPORTED;
  // the masked attention tile holds 64 (row, q head) pairs of one kv head
  if (d->max_rows > 0 && d->n_q_heads / d->n_kv_heads > 64) return PEAGLE_ERR_UNSUPPORTED;
  if (d->train != 0 && d->train != 1) return PEAGLE_ERR_INVALID;
  if (d->train && d->max_rows <= 0) return PEAGLE_ERR_INVALID;
  if (d->train && (d->attn_window > 0 || d->lm_rank > 0)) return PEAGLE_ERR_UNSUPPORTED;
  return PEAGLE_OK;
}

// ---- GEMM dispatch: tensor cores for bf16, FFMA for fp32 --------------------------------
static int gemm(peagle_ctx* c, const void* W, const void* X, int ldx, int Nout, int Kd, int R,
                const EpiArgs& epi, cudaStream_t s) {
  if (c->bf) return tc_gemm(c->tc, W, X, ldx, Nout, Kd, R, epi, s);
  launch_gemm_simt(false, W, X, ldx, c->Y, c->ldY, Nout, Kd, R, epi, s);
  return PEAGLE_OK;
}
#define GEMM(stage, ...)              \
  do {                                \
    t_begin(c, (stage), s);           \
    int _g = gemm(__VA_ARGS__);       \
    t_end(c, s);                      \
    if (_g != PEAGLE_OK) return _g;   \
  } while (0)

// The bf16 path carries every projection input as a bf16 hi + lo pair (2R operand rows):
// the weights are streamed once either way, and rounding then happens only where a value
// is stored in the bf16 KV cache.
static int use_split(const peagle_ctx* c) { return c->bf ? 1 : 0; }

static EpiArgs epi_base(peagle_ctx* c, int kind, int R, int Nout) {
  EpiArgs e;
  memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.R = R;
  e.Nout = Nout;
  e.err = c->err;
  e.nq = c->d.n_q_heads;
  e.nkv = c->d.n_kv_heads;
  e.hd = c->d.head_dim;
  e.rope = c->rope;
  e.max_pos = c->d.max_positions;
  e.I = c->d.intermediate;
  e.ld_res = c->d.hidden;
  return e;
}

static int train_ws(peagle_ctx* c);

extern "C" int peagle_create(const peagle_weights* w, const peagle_dims* dims, peagle_ctx** out) {
  if (!out) return PEAGLE_ERR_INVALID;
  *out = nullptr;
  int r = validate_dims(dims);
  if (r) return r;
  if (!w || !w->embed || !w->emb_mask || !w->h_shared || !w->fc || !w->input_norm ||
      !w->hidden_norm || !w->qkv || !w->o || !w->post_norm || !w->gate || !w->up || !w->down ||
      !w->final_norm || !w->lm_head || !w->d2t)
    return PEAGLE_ERR_INVALID;
  if (dims->lm_rank > 0 && (!w->lm_proj || !w->lm_score)) return PEAGLE_ERR_INVALID;
  const peagle_dims& d = *dims;
  for (int l = 0; l < d.n_layers; ++l)
    if (!w->qkv[l] || !w->o[l] || !w->post_norm[l] || !w->gate[l] || !w->up[l] || !w->down[l] ||
        (l > 0 && (!w->attn_norm || !w->attn_norm[l])))
      return PEAGLE_ERR_INVALID;

  peagle_ctx* c = new peagle_ctx();
  c->d = d;
  c->bf = d.dtype == PEAGLE_BF16;
  c->es = c->bf ? 2 : 4;
  c->tc = nullptr;
  c->last_err_bits = 0;
  c->timing = false;
  c->ev_used = 0;
  c->pending_stage = -1;
  c->wait_ns = PASS_DEFAULT_WAIT_NS;
  c->stall_phase = -1;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return PEAGLE_ERR_CUDA;
  }
  const size_t es = c->es;
  const int H = d.hidden, I = d.intermediate, nq = d.n_q_heads, nkv = d.n_kv_heads,
            hd = d.head_dim;
  const int qkv_out = (nq + 2 * nkv) * hd;
#define TRY(x)            \
  do {                    \
    int _r = (x);         \
    if (_r) {             \
      free_ctx(c);        \
      return _r;          \
    }                     \
  } while (0)
  TRY(copy_in(c, &c->embed, w->embed, (size_t)d.target_vocab * H * es));
  TRY(copy_in(c, &c->emb_mask, w->emb_mask, (size_t)H * es));
  TRY(copy_in(c, &c->h_shared, w->h_shared, (size_t)3 * H * es));
  TRY(copy_in(c, &c->fc, w->fc, (size_t)H * 3 * H * es));
  TRY(copy_in(c, &c->input_norm, w->input_norm, (size_t)H * es));
  TRY(copy_in(c, &c->hidden_norm, w->hidden_norm, (size_t)H * es));
  TRY(copy_in(c, &c->final_norm, w->final_norm, (size_t)H * es));
  TRY(copy_in(c, &c->lm_head, w->lm_head, (size_t)d.draft_vocab * H * es));
  TRY(copy_in(c, (void**)&c->d2t, w->d2t, (size_t)d.draft_vocab * 4));
  if (d.lm_rank > 0) {
    TRY(copy_in(c, &c->lm_proj, w->lm_proj, (size_t)d.lm_rank * H * es));
    TRY(copy_in(c, &c->lm_score, w->lm_score, (size_t)d.draft_vocab * d.lm_rank * es));
  }
  c->qkv.resize(d.n_layers);
  c->o.resize(d.n_layers);
  c->attn_norm.assign(d.n_layers, nullptr);
  c->post_norm.resize(d.n_layers);
  c->gate_up.resize(d.n_layers);
  c->down.resize(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) {
    const int din = l == 0 ? 2 * H : H;
    TRY(copy_in(c, &c->qkv[l], w->qkv[l], (size_t)qkv_out * din * es));
    TRY(copy_in(c, &c->o[l], w->o[l], (size_t)H * nq * hd * es));
    if (l > 0) TRY(copy_in(c, &c->attn_norm[l], w->attn_norm[l], (size_t)H * es));
    TRY(copy_in(c, &c->post_norm[l], w->post_norm[l], (size_t)H * es));
    TRY(copy_in(c, &c->down[l], w->down[l], (size_t)H * I * es));
    // gate/up interleaved in 64-row blocks: [gate 64 rows | up 64 rows] per block
    TRY(dalloc(c, &c->gate_up[l], (size_t)2 * I * H * es));
    const size_t blk = (size_t)64 * H * es;
    if (cudaMemcpy2D(c->gate_up[l], 2 * blk, w->gate[l], blk, blk, I / 64, cudaMemcpyDefault) ||
        cudaMemcpy2D((char*)c->gate_up[l] + blk, 2 * blk, w->up[l], blk, blk, I / 64,
                     cudaMemcpyDefault)) {
      free_ctx(c);
      return PEAGLE_ERR_CUDA;
    }
  }
  // RoPE table (cos, sin) for positions [0, max_positions), angles in double
  {
    const int half = hd / 2;
    std::vector<float2> tab((size_t)d.max_positions * half);
    for (int p = 0; p < d.max_positions; ++p)
      for (int i = 0; i < half; ++i) {
        double inv = pow((double)d.rope_theta, -2.0 * i / hd);
        double ang = (double)p * inv;
        tab[(size_t)p * half + i] = make_float2((float)cos(ang), (float)sin(ang));
      }
    TRY(copy_in(c, (void**)&c->rope, tab.data(), tab.size() * sizeof(float2)));
  }
  // workspaces
  const int logical_rows = d.max_batch * d.max_K > d.max_rows ? d.max_batch * d.max_K : d.max_rows;
  c->rows_max = 2 * logical_rows;
  const int R = c->rows_max;
  // fc outputs: one per request (draft pass), per row (catch-up) or per position (forward)
  const int fr = d.max_batch * d.max_K > d.max_seq ? d.max_batch * d.max_K : d.max_seq;
  c->F_bytes = (size_t)(fr > 1 ? fr : 1) * H * 8;
  TRY(dalloc(c, (void**)&c->F, c->F_bytes));
  TRY(dalloc(c, (void**)&c->f_shared, (size_t)H * 8));
  TRY(dalloc(c, &c->X0, (size_t)R * 2 * H * es));
  TRY(dalloc(c, (void**)&c->res, (size_t)R * H * 8));
  TRY(dalloc(c, &c->Xn, (size_t)R * H * es));
  TRY(dalloc(c, (void**)&c->Qf, (size_t)logical_rows * nq * hd * 4));
  TRY(dalloc(c, &c->O, (size_t)R * nq * hd * es));
  TRY(dalloc(c, &c->act, (size_t)R * I * es));
  TRY(dalloc(c, (void**)&c->keys, (size_t)R * 8));
  TRY(dalloc(c, (void**)&c->row_pos, (size_t)d.max_batch * d.max_K * 4));
  c->mk_qfx = nullptr;
  c->mk_kvfx = nullptr;
  if (c->bf) {
    TRY(dalloc(c, (void**)&c->mk_qfx, (size_t)d.max_batch * d.max_K * nq * hd * 8));
    TRY(dalloc(c, (void**)&c->mk_kvfx, (size_t)d.max_batch * d.max_K * 2 * nkv * hd * 8));
  }
  TRY(dalloc(c, (void**)&c->err, 64));
  int max_out = qkv_out;
  if (2 * I > max_out) max_out = 2 * I;
  if (H > max_out) max_out = H;
  if (d.draft_vocab > max_out) max_out = d.draft_vocab;
  c->ldY = (max_out + 127) / 128 * 128;
  if (!c->bf) TRY(dalloc(c, (void**)&c->Y, (size_t)R * c->ldY * 4));
  {
    const int G = nq / nkv;
    c->att_chunks_max = 64;
    TRY(dalloc(c, (void**)&c->att_part, (size_t)d.max_batch * nkv * c->att_chunks_max *
                                            (d.max_K * G) * (hd + 2) * 4));
    TRY(dalloc(c, (void**)&c->att_cnt, (size_t)d.max_batch * nkv * 4));
  }
  if (d.max_rows > 0) {
    TRY(dalloc(c, &c->Kr, (size_t)d.max_rows * nkv * hd * es));
    TRY(dalloc(c, &c->Vr, (size_t)d.max_rows * nkv * hd * es));
    TRY(dalloc(c, &c->K1, (size_t)d.max_seq * nkv * hd * es));
    TRY(dalloc(c, &c->V1, (size_t)d.max_seq * nkv * hd * es));
    TRY(dalloc(c, (void**)&c->row_index, (size_t)d.max_seq * 17 * 4));
  }
  if (d.lm_rank > 0) {
    const int dr = d.max_batch * d.max_K;  // draft rows
    const int k = d.lm_topk < d.draft_vocab ? d.lm_topk : d.draft_vocab;
    TRY(dalloc(c, (void**)&c->lm_zfx, (size_t)dr * d.lm_rank * 8));
    TRY(dalloc(c, (void**)&c->lm_approx, (size_t)dr * d.draft_vocab * 4));
    TRY(dalloc(c, (void**)&c->lm_cand, (size_t)dr * k * 4));
    TRY(dalloc(c, (void**)&c->lm_done, 4));
    TRY(dalloc(c, (void**)&c->lm_hist, (size_t)dr * 2048 * 4));
    TRY(dalloc(c, (void**)&c->lm_gcount, (size_t)dr * 4));
    TRY(dalloc(c, (void**)&c->lm_gdone, (size_t)dr * 4));
    TRY(dalloc(c, (void**)&c->lm_gkey, (size_t)dr * 4096 * 4));
    TRY(dalloc(c, (void**)&c->lm_gidx, (size_t)dr * 4096 * 4));
  }
  if (c->bf) TRY(tc_create(&c->tc, c->num_sms, R, max_out > 3 * H ? max_out : 3 * H, c->err));
  // fc(h_shared): constant for every MTP row, computed once with the pass's own GEMM
  {
    EpiArgs e = epi_base(c, EPI_STORE, 1, H);
    e.out_fx = c->f_shared;
    e.out_ld = H;
    int g = gemm(c, c->fc, c->h_shared, 3 * H, H, 3 * H, 1, e, 0);
    if (g != PEAGLE_OK || cudaDeviceSynchronize() != cudaSuccess) {
      free_ctx(c);
      return PEAGLE_ERR_CUDA;
    }
  }
  // the whole bf16 pass as one persistent kernel (peagle_set_pass_kernel chooses when)
  c->pass_on = false;
  c->pass_mode = -1;
  c->pp = nullptr;
  c->pp_valid = false;
  c->pass_cnt = nullptr;
  if (c->bf && d.n_layers <= PASS_MAX_LAYERS) {
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device);
    if (coop) {
      // phase counters, the abort flag, then the attention items' counts per layer,
      // request and kv head
      TRY(dalloc(c, (void**)&c->pass_cnt,
                 ((size_t)PASS_MAX_PHASE + 1 + (size_t)PASS_MAX_LAYERS * d.max_batch * nkv) * 4));
      TRY(dalloc(c, (void**)&c->pass_trace,
                 (size_t)PASS_TRACE_SLOTS * (PASS_MAX_PHASE + 1) * 8));
      TRY(dalloc(c, (void**)&c->pass_trace_cta, (size_t)PASS_MAX_PHASE * c->num_sms * 4 * 8));
      const size_t pr = (size_t)PASS_MAX_ROWS;
      TRY(dalloc(c, (void**)&c->pass_ss, (size_t)PASS_SS_SLOTS * pr * 8));
      TRY(dalloc(c, (void**)&c->pass_qfx, pr * nq * hd * 8));
      TRY(dalloc(c, (void**)&c->pass_kvfx, pr * 2 * nkv * hd * 8));
      c->pp = new PassParams();
      c->pass_on = true;
    }
  }
  // the training step's workspaces (fp32 weight copies, every layer's kept activations,
  // the GEMMs' scratch operands): made here, so that no other call allocates
  if (d.train) {
    const int tr = train_ws(c);
    if (tr != PEAGLE_OK) {
      free_ctx(c);
      return tr;
    }
  }
#undef TRY
  *out = c;
  return PEAGLE_OK;
}

// Keys a request's split-KV items cover: the whole cache, or with a sliding window of W
// positions at most W + K - 1 of them (row 0's window through the last draft row).
static int attention_span(peagle_ctx* c, int cap, int K) {
  const int w = c->d.attn_window;
  return (w > 0 && w + K < cap) ? w + K : cap;
}

static void attention_plan(peagle_ctx* c, int B, int cap, int* chunk, int* nchunk,
                           int waves = 2) {
  const int target = waves * c->num_sms;
  const int pairs = B * c->d.n_kv_heads;
  // one wave (the pass kernel: one item per CTA) must not spill a few items into a second
  int want = waves == 1 ? target / pairs : (target + pairs - 1) / pairs;
  if (want < 1) want = 1;
  if (want > c->att_chunks_max) want = c->att_chunks_max;
  int ch = (cap + want - 1) / want;
  ch = (ch + 63) / 64 * 64;
  if (ch < 64) ch = 64;
  *chunk = ch;
  *nchunk = (cap + ch - 1) / ch;
}

// ---- the draft pass as one persistent kernel (bf16) --------------------------------------
// Bytes of the pass kernel's counters a launch starts from zero: the phase counts, the abort
// flag and the attention items' counts per layer, request and kv head.
static size_t pass_cnt_bytes(const peagle_ctx* c, const PassParams& P) {
  return ((size_t)P.n_phase + 1 + (size_t)c->d.n_layers * P.B * c->d.n_kv_heads) * 4;
}

// Fills the kernel's parameter block with the same steps, epilogues and buffers as the
// multi-kernel path below.  Returns PEAGLE_ERR_UNSUPPORTED for shapes it does not cover
// (the caller then runs the multi-kernel path).
static int pass_draft(peagle_ctx* c, int B, const peagle_kv* kv, const int32_t* seq_lens,
                      const void* target_hidden, const int32_t* new_token, int K, bool all_ntp,
                      int32_t* out_tokens, float* out_logits, cudaStream_t s) {
  const peagle_dims& d = c->d;
  const int H = d.hidden, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim;
  const int R = B * K, G = nq / nkv;
  if (R > PASS_MAX_ROWS || K * G > 64 || d.n_layers > PASS_MAX_LAYERS)
    return PEAGLE_ERR_UNSUPPORTED;
  PassParams& P = *c->pp;
  const int grid = c->num_sms;
  PassKey key;
  memset(&key, 0, sizeof(key));
  key.B = B;
  key.K = K;
  key.all_ntp = all_ntp ? 1 : 0;
  key.capacity = kv->capacity;
  key.batch = kv->batch;
  key.k = kv->k;
  key.v = kv->v;
  key.seq_lens = seq_lens;
  key.target_hidden = target_hidden;
  key.new_token = new_token;
  key.out_tokens = out_tokens;
  key.out_logits = out_logits;
  P.wait_ns = c->wait_ns;
  P.stall_phase = c->stall_phase;
  if (!c->timing && c->pp_valid && memcmp(&key, &c->pp_key, sizeof(key)) == 0) {
    cudaError_t ce = cudaMemsetAsync(c->pass_cnt, 0, pass_cnt_bytes(c, P), s);
    if (ce != cudaSuccess) return cuda_fail(ce, "pass counters");
    return pass_launch(P, hd, grid, s);
  }
  c->pp_valid = false;
  P.n_gemm = 0;
  P.n_phase = 0;
  int bn_max = 16;
  bool fail = false;
  int cur_stage = PEAGLE_STAGE_FC;
  auto add_phase = [&](int kind, int layer, const void* gamma) {
    if (P.n_phase >= PASS_MAX_PHASE) {
      fail = true;
      return;
    }
    PassPhase& ph = P.ph[P.n_phase++];
    ph.kind = kind;
    ph.stage = kind == PP_GEMM ? cur_stage
               : kind == PP_ATTN ? PEAGLE_STAGE_ATTN
               : kind == PP_ARGMAX ? PEAGLE_STAGE_SMALL : PEAGLE_STAGE_NORM;
    ph.gemm = -1;
    ph.layer = layer;
    ph.slot = 0;
    ph.gamma = gamma;
  };
  // a projection Y = W X^T over the R draft rows (W [Nout, Kd] with row stride ldw);
  // `dep`: the phase its activation operand waits for (default: the phase before it)
  auto add_gemm = [&](const void* W, int ldw, const void* X, int ldx, int Nout, int Kd, int rows,
                      int split, const EpiArgs& e, int dep) {
    if (P.n_gemm >= PASS_MAX_GEMM || P.n_phase >= PASS_MAX_PHASE) {
      fail = true;
      return;
    }
    PassGemm& m = P.gemm[P.n_gemm];
    m.Nout = Nout;
    m.Kd = Kd;
    m.R = rows;
    m.split = split;
    m.additive =
        (e.kind == EPI_STORE || e.kind == EPI_RESID || e.kind == EPI_QKV_FX) ? 1 : 0;
    m.BN = ((split ? 2 * rows : rows) + 15) / 16 * 16;
    m.lo_col = split ? rows : 0;
    m.n_tiles = 1;
    m.KB = (Kd / 64 + PASS_KU - 1) / PASS_KU;  // k-units (the last may run past Kd: zeros)
    const long long tiles = (long long)((Nout + 127) / 128) * m.n_tiles;
    m.total = tiles * m.KB;
    m.Gm = (int)(m.total < grid ? m.total : grid);
    // A projection whose epilogue needs whole tiles (SwiGLU, LM head) pays a cross-CTA
    // fix-up at the end of every shared tile.  With between G/2 and G tiles, one whole tile
    // per CTA streams the same bytes from HBM (the idle CTAs' share is small) without it.
    if (!m.additive && tiles <= grid && 2 * tiles >= grid) m.Gm = (int)tiles;
    m.idesc = tc::idesc_bf16(128, m.BN);
    m.epi = e;
    if (tiles > tc_max_tiles(c->tc) || Kd % 64 || m.BN > 240) fail = true;
    if (!tc_tensor_map_ku(c->tc, &P.tm[2 * P.n_gemm], W, Nout, Kd, ldw, 128, PASS_KU) ||
        !tc_tensor_map_ku(c->tc, &P.tm[2 * P.n_gemm + 1], X, split ? 2 * rows : rows, Kd, ldx,
                          m.BN, PASS_KU))
      fail = true;
    if (m.BN > bn_max) bn_max = m.BN;
    m.phase = P.n_phase;
    m.dep = dep == -2 ? P.n_phase - 1 : dep;
    add_phase(PP_GEMM, -1, nullptr);
    P.ph[P.n_phase - 1].gemm = P.n_gemm++;
  };
  const int split = 1;
  const int qkv_out = (nq + 2 * nkv) * hd;
  const size_t es = c->es;
  const size_t layer_stride = (size_t)kv->batch * nkv * kv->capacity * hd * es;
  int slot = 2;  // sum-of-squares slots: 0 = e, 1 = f, then one per RMSNorm
  auto scaled = [&](EpiArgs& e, int sl) {
    e.row_ss = c->pass_ss + (size_t)sl * R;
    e.ss_inv_n = 1.f / (float)H;
    e.ss_eps = d.rms_eps;
  };
  {
    EpiArgs e = epi_base(c, EPI_STORE, B, H);
    e.out_fx = c->F;
    e.out_ld = H;
    cur_stage = PEAGLE_STAGE_FC;
    const int fc_rows = all_ntp ? R : B;  // catch-up: every row has its own hidden state
    e.R = fc_rows;
    add_gemm(c->fc, 3 * H, target_hidden, 3 * H, H, 3 * H, fc_rows, 0, e, -1);
  }
  add_phase(PP_INPUT, -1, nullptr);
  const int input_phase = P.n_phase - 1;
  for (int l = 0; l < d.n_layers; ++l) {
    EpiArgs e = epi_base(c, EPI_QKV_FX, R, qkv_out);
    e.in_split = split;
    e.q_fx = c->pass_qfx;
    e.kv_fx = c->pass_kvfx;
    e.row_pos = c->row_pos;
    cur_stage = PEAGLE_STAGE_QKV;
    if (l == 0) {
      // the first layer's 2H input [e * g_in || f * g_hid] has a norm scale per half:
      // two projections over the halves of W_qkv, each scaled by its own row sums
      scaled(e, 0);
      add_gemm(c->qkv[0], 2 * H, c->X0, 2 * H, qkv_out, H, R, split, e, input_phase);
      scaled(e, 1);
      add_gemm((const char*)c->qkv[0] + (size_t)H * es, 2 * H, (const char*)c->X0 + (size_t)H * es,
               2 * H, qkv_out, H, R, split, e, input_phase);
    } else {
      add_phase(PP_NORM, l, c->attn_norm[l]);
      P.ph[P.n_phase - 1].slot = slot;
      scaled(e, slot++);
      add_gemm(c->qkv[l], H, c->Xn, H, qkv_out, H, R, split, e, -2);
    }
    add_phase(PP_ATTN, l, nullptr);
    {
      EpiArgs eo = epi_base(c, EPI_RESID, R, H);
      eo.in_split = split;
      eo.resid = c->res;
      cur_stage = PEAGLE_STAGE_OPROJ;
      add_gemm(c->o[l], nq * hd, c->O, nq * hd, H, nq * hd, R, split, eo, -2);
    }
    add_phase(PP_NORM, l, c->post_norm[l]);
    P.ph[P.n_phase - 1].slot = slot;
    {
      EpiArgs eg = epi_base(c, EPI_SWIGLU, R, 2 * d.intermediate);
      eg.in_split = split;
      eg.out_split = split;
      eg.act_out = c->act;
      scaled(eg, slot++);
      cur_stage = PEAGLE_STAGE_GATEUP;
      add_gemm(c->gate_up[l], H, c->Xn, H, 2 * d.intermediate, H, R, split, eg, -2);
    }
    {
      EpiArgs ed = epi_base(c, EPI_RESID, R, H);
      ed.in_split = split;
      ed.resid = c->res;
      cur_stage = PEAGLE_STAGE_DOWN;
      add_gemm(c->down[l], d.intermediate, c->act, d.intermediate, H, d.intermediate, R, split,
               ed, -2);
    }
  }
  const bool lm = out_tokens || out_logits;  // the catch-up may skip the LM head
  if (lm) add_phase(PP_NORM, -1, c->final_norm);
  if (lm) P.ph[P.n_phase - 1].slot = slot;
  if (lm) {
    EpiArgs e = epi_base(c, EPI_LMHEAD, R, d.draft_vocab);
    e.in_split = split;
    e.logits = out_logits;
    e.keys = c->keys;
    scaled(e, slot++);
    cur_stage = PEAGLE_STAGE_LMHEAD;
    add_gemm(c->lm_head, H, c->Xn, H, d.draft_vocab, H, R, split, e, -2);
  }
  if (lm) add_phase(PP_ARGMAX, -1, nullptr);
  if (slot > PASS_SS_SLOTS) fail = true;
  if (fail) return PEAGLE_ERR_UNSUPPORTED;

  P.b_stage_bytes = bn_max * 128 * PASS_KU;
  P.acc_stride = bn_max + 16;
  uint32_t tc_cols = 32;
  while (tc_cols < (uint32_t)(2 * P.acc_stride)) tc_cols <<= 1;
  if (tc_cols > 512) return PEAGLE_ERR_UNSUPPORTED;
  P.tmem_cols = (int)tc_cols;
  const int att_bytes = pass_att_nbuf(hd) * 2 * 64 * hd * 2;
  P.uni_bytes = att_bytes > 32 * 128 * 4 ? att_bytes : 32 * 128 * 4;
  // dynamic shared memory: the 227 KB per-block limit minus the kernel's static part
  const size_t smem_cap = 223 * 1024;
  int stages = 2;
  while (stages < 16 && pass_smem_bytes(stages + 1, P.b_stage_bytes, P.uni_bytes) <= smem_cap)
    ++stages;
  if (pass_smem_bytes(stages, P.b_stage_bytes, P.uni_bytes) > smem_cap)
    return PEAGLE_ERR_UNSUPPORTED;
  P.stages = stages;
  P.B = B;
  P.K = K;
  P.R = R;
  P.H = H;
  P.split = split;
  P.Vt = d.target_vocab;
  P.eps = d.rms_eps;
  // one attention item per CTA: each CTA streams its chunk's tiles back to back
  int chunk, nchunk;
  attention_plan(c, B, attention_span(c, kv->capacity, K), &chunk, &nchunk, 1);
  P.chunk = chunk;
  P.nchunk = nchunk;
  AttnArgs& a = P.att;
  a.q = c->pass_qfx;
  a.split = split;
  a.kc = kv->k;
  a.vc = kv->v;
  a.seq_lens = seq_lens;
  a.o = c->O;
  a.part = c->att_part;
  a.counters = c->att_cnt;
  a.B = B;
  a.K = K;
  a.nq = nq;
  a.nkv = nkv;
  a.hd = hd;
  a.cap = kv->capacity;
  a.chunk = chunk;
  a.nchunk = nchunk;
  a.window = d.attn_window;
  a.scale = 1.f / sqrtf((float)hd);
  a.err = c->err;
  P.layer_stride = layer_stride;
  P.embed = c->embed;
  P.emb_mask = c->emb_mask;
  P.input_norm = c->input_norm;
  P.hidden_norm = c->hidden_norm;
  P.F = c->F;
  P.f_shared = c->f_shared;
  P.X0 = c->X0;
  P.Xn = c->Xn;
  P.res = c->res;
  P.ss = c->pass_ss;
  P.q_fx = c->pass_qfx;
  P.kv_fx = c->pass_kvfx;
  P.nq = nq;
  P.nkv = nkv;
  P.hd = hd;
  P.cap = kv->capacity;
  P.keys = c->keys;
  P.row_pos = c->row_pos;
  P.d2t = c->d2t;
  P.ws = tc_partials(c->tc);
  P.tile_cnt = tc_tile_counters(c->tc);
  P.phase_cnt = c->pass_cnt;
  P.err = c->err;
  P.seq_lens = seq_lens;
  P.new_token = new_token;
  P.all_ntp = all_ntp ? 1 : 0;
  P.out_tokens = out_tokens;
  P.trace = nullptr;
  P.trace_cta = nullptr;
  if (c->timing && c->trace_stages.size() < (size_t)PASS_TRACE_SLOTS) {
    P.trace_cta = c->pass_trace_cta;
    c->trace_cta_phases = P.n_phase;
    cudaError_t ze = cudaMemsetAsync(c->pass_trace_cta, 0, (size_t)P.n_phase * grid * 4 * 8, s);
    if (ze != cudaSuccess) return cuda_fail(ze, "pass trace");
    P.trace = c->pass_trace + c->trace_stages.size() * (PASS_MAX_PHASE + 1);
    std::vector<int> st(P.n_phase);
    for (int j = 0; j < P.n_phase; ++j) st[j] = P.ph[j].stage;
    c->trace_stages.push_back(st);
    cudaError_t te = cudaMemsetAsync(P.trace, 0, (size_t)(PASS_MAX_PHASE + 1) * 8, s);
    if (te != cudaSuccess) return cuda_fail(te, "pass trace");
  }
  cudaError_t ce = cudaMemsetAsync(c->pass_cnt, 0, pass_cnt_bytes(c, P), s);
  if (ce != cudaSuccess) return cuda_fail(ce, "pass counters");
  if (!c->timing) {
    c->pp_key = key;
    c->pp_valid = true;
  }
  return pass_launch(P, hd, grid, s);
}

// The draft pass (all_ntp = false: row 0 of each request NTP, rows 1.. MTP) and the
// catch-up pass (all_ntp: every row takes its own token and hidden state).
// Efficient LM head over the R draft rows whose final residual is in c->res: final norm,
// rank-r projection (fixed point), scores of the whole draft vocabulary, per-row top-k
// candidates, the full head on the candidates, argmax + d2t.
static int efficient_head(peagle_ctx* c, int R, int split, int32_t* out_tokens,
                          float* out_logits, cudaStream_t s) {
  const peagle_dims& d = c->d;
  const int H = d.hidden, r = d.lm_rank, Vd = d.draft_vocab;
  const int k = d.lm_topk < Vd ? d.lm_topk : Vd;
  TIMED(PEAGLE_STAGE_NORM,
        launch_rmsnorm(c->bf, R, H, c->res, c->final_norm, d.rms_eps, split, c->Xn, s));
  {
    EpiArgs e = epi_base(c, EPI_STORE, R, r);
    e.in_split = split;
    e.out_fx = c->lm_zfx;
    e.out_ld = r;
    GEMM(PEAGLE_STAGE_LMHEAD, c, c->lm_proj, c->Xn, H, r, H, R, e, s);
  }
  TIMED(PEAGLE_STAGE_LMHEAD, launch_head_score(c->bf, R, r, Vd, c->lm_zfx, c->lm_score,
                                               c->lm_approx, c->lm_hist, c->err, c->num_sms,
                                               s));
  TIMED(PEAGLE_STAGE_LMHEAD,
        launch_topk(R, Vd, k, c->lm_approx, c->lm_hist, c->lm_gcount, c->lm_gdone, c->lm_gkey,
                    c->lm_gidx, c->lm_cand, c->lm_zfx, r, c->num_sms, s));
  TIMED(PEAGLE_STAGE_LMHEAD, launch_cand_head(c->bf, R, H, k, c->lm_cand, c->lm_head, c->Xn,
                                              split, c->keys, out_logits, Vd, c->d2t,
                                              out_tokens, c->lm_done, s));
  cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "efficient LM head launch");
}

static int draft_impl(peagle_ctx* c, int32_t batch, const peagle_kv* kv,
                      const int32_t* seq_lens, const void* target_hidden,
                      const int32_t* new_token, int32_t K, bool all_ntp,
                      int32_t* out_draft_tokens, float* out_logits, cudaStream_t stream) {
  const peagle_dims& d = c->d;
  if (batch < 1 || K < 1) return PEAGLE_ERR_INVALID;
  if (batch > d.max_batch || K > d.max_K || batch > kv->batch) return PEAGLE_ERR_CAPACITY;
  if (kv->capacity < K || kv->capacity > d.max_positions) return PEAGLE_ERR_CAPACITY;
  cudaStream_t s = (cudaStream_t)stream;
  const int H = d.hidden, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim;
  const int qkv_out = (nq + 2 * nkv) * hd;
  const int R = batch * K;
  const int split = use_split(c);
  const size_t es = c->es;
  const size_t layer_stride = (size_t)kv->batch * nkv * kv->capacity * hd * es;
  // The persistent pass kernel wins when the pass is a chain of short steps (few draft
  // rows); with many rows its four worker warps per SM become the limit (attention over
  // long ragged contexts, the spread norm steps), and the multi-kernel path, whose
  // attention runs several CTAs per SM, is faster: decode_b1 (8 rows) 431 vs 448 us,
  // decode_b2 (16 rows) 613 vs 609 us, ragged_b16 (80 rows) 1927 vs 1465 us.
  const bool eff_head = d.lm_rank > 0 && (out_draft_tokens || out_logits);
  if (c->pass_on && c->pass_mode != 0 && (c->pass_mode == 1 || R <= 16)) {
    // with the efficient LM head the pass kernel stops at the last layer's residual
    const int r = pass_draft(c, batch, kv, seq_lens, target_hidden, new_token, K, all_ntp,
                             eff_head ? nullptr : out_draft_tokens,
                             eff_head ? nullptr : out_logits, s);
    if (r != PEAGLE_ERR_UNSUPPORTED)
      return (r == PEAGLE_OK && eff_head)
                 ? efficient_head(c, R, split, out_draft_tokens, out_logits, s)
                 : r;
  }

  // S1: fc over the NTP rows' target hidden states, then the fused input rows
  const int fc_rows = all_ntp ? R : batch;
  {
    EpiArgs e = epi_base(c, EPI_STORE, fc_rows, H);
    e.out_fx = c->F;
    e.out_ld = H;
    GEMM(PEAGLE_STAGE_FC, c, c->fc, target_hidden, 3 * H, H, 3 * H, fc_rows, e, s);
  }
  TIMED(PEAGLE_STAGE_NORM,
        launch_input_fusion(c->bf, all_ntp ? 2 : 0, R, K, fc_rows, H, c->embed, d.target_vocab,
                            c->emb_mask,
                            c->F, c->f_shared, new_token, nullptr, nullptr, c->input_norm,
                            c->hidden_norm, d.rms_eps, split, c->X0, c->res, c->keys, seq_lens,
                            c->row_pos, c->err, s));
  int chunk, nchunk;
  // about four items per SM: ragged contexts leave many items of a longer request than
  // average, and finer chunks spread them (ragged_b16: 449 us of attention with two items
  // per SM, 303 with four)
  attention_plan(c, batch, attention_span(c, kv->capacity, K), &chunk, &nchunk, 4);
  for (int l = 0; l < d.n_layers; ++l) {
    const void* a_in = c->X0;
    int din = 2 * H;
    if (l > 0) {
      TIMED(PEAGLE_STAGE_NORM,
            launch_rmsnorm(c->bf, R, H, c->res, c->attn_norm[l], d.rms_eps, split, c->Xn, s));
      a_in = c->Xn;
      din = H;
    }
    // S2: QKV projection + RoPE; k/v of row j go to cache slot seq_lens[b] + j.  bf16: the
    // additive fixed-point epilogue (every split-K contributor rotates and adds its own
    // partial, no cross-CTA reduction of partials), then one pass converts the sums
    if (c->bf) {
      EpiArgs e = epi_base(c, EPI_QKV_FX, R, qkv_out);
      e.in_split = split;
      e.q_fx = c->mk_qfx;
      e.kv_fx = c->mk_kvfx;
      e.row_pos = c->row_pos;
      GEMM(PEAGLE_STAGE_QKV, c, c->qkv[l], a_in, din, qkv_out, din, R, e, s);
      TIMED(PEAGLE_STAGE_QKV,
            launch_qkv_finalize(R, K, nq, nkv, hd, kv->capacity, c->mk_qfx, c->mk_kvfx, c->Qf,
                                (char*)kv->k + l * layer_stride, (char*)kv->v + l * layer_stride,
                                c->row_pos, c->err, s));
    } else {
      EpiArgs e = epi_base(c, EPI_QKV_ROPE, R, qkv_out);
      e.in_split = split;
      e.q_out = c->Qf;
      e.q_f32 = 1;
      e.k_dst = (char*)kv->k + l * layer_stride;
      e.v_dst = (char*)kv->v + l * layer_stride;
      e.row_pos = c->row_pos;
      e.decode = 1;
      e.K = K;
      e.cap = kv->capacity;
      GEMM(PEAGLE_STAGE_QKV, c, c->qkv[l], a_in, din, qkv_out, din, R, e, s);
    }
    // S3: split-KV attention over the cache + causal draft block
    {
      AttnArgs a;
      a.q = c->Qf;
      a.split = split;
      a.kc = (char*)kv->k + l * layer_stride;
      a.vc = (char*)kv->v + l * layer_stride;
      a.seq_lens = seq_lens;
      a.o = c->O;
      a.part = c->att_part;
      a.counters = c->att_cnt;
      a.B = batch;
      a.K = K;
      a.nq = nq;
      a.nkv = nkv;
      a.hd = hd;
      a.cap = kv->capacity;
      a.chunk = chunk;
      a.nchunk = nchunk;
      a.window = d.attn_window;
      a.scale = 1.f / sqrtf((float)hd);
      a.err = c->err;
      TIMED(PEAGLE_STAGE_ATTN, launch_attention_decode(c->bf, a, s));
    }
    // S4: o-proj + residual
    {
      EpiArgs e = epi_base(c, EPI_RESID, R, H);
      e.in_split = split;
      e.resid = c->res;
      GEMM(PEAGLE_STAGE_OPROJ, c, c->o[l], c->O, nq * hd, H, nq * hd, R, e, s);
    }
    // S5: SwiGLU MLP
    TIMED(PEAGLE_STAGE_NORM,
          launch_rmsnorm(c->bf, R, H, c->res, c->post_norm[l], d.rms_eps, split, c->Xn, s));
    {
      EpiArgs e = epi_base(c, EPI_SWIGLU, R, 2 * d.intermediate);
      e.in_split = split;
      e.out_split = split;
      e.act_out = c->act;
      GEMM(PEAGLE_STAGE_GATEUP, c, c->gate_up[l], c->Xn, H, 2 * d.intermediate, H, R, e, s);
    }
    {
      EpiArgs e = epi_base(c, EPI_RESID, R, H);
      e.in_split = split;
      e.resid = c->res;
      GEMM(PEAGLE_STAGE_DOWN, c, c->down[l], c->act, d.intermediate, H, d.intermediate, R, e, s);
    }
  }
  // S6: final norm, LM head with fused argmax, d2t remap (skipped by a catch-up pass that
  // asks for neither tokens nor logits)
  if (!out_draft_tokens && !out_logits) {
    cudaError_t ce = cudaGetLastError();
    return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "peagle_catch_up launch");
  }
  if (eff_head) return efficient_head(c, R, split, out_draft_tokens, out_logits, s);
  TIMED(PEAGLE_STAGE_NORM,
        launch_rmsnorm(c->bf, R, H, c->res, c->final_norm, d.rms_eps, split, c->Xn, s));
  {
    EpiArgs e = epi_base(c, EPI_LMHEAD, R, d.draft_vocab);
    e.in_split = split;
    e.logits = out_logits;
    e.keys = c->keys;
    GEMM(PEAGLE_STAGE_LMHEAD, c, c->lm_head, c->Xn, H, d.draft_vocab, H, R, e, s);
  }
  if (out_draft_tokens)
    TIMED(PEAGLE_STAGE_SMALL, launch_argmax_decode(R, c->keys, c->d2t, out_draft_tokens, s));
  else
    TIMED(PEAGLE_STAGE_SMALL, launch_argmax_decode(R, c->keys, c->d2t, nullptr, s));
  cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "peagle_draft launch");
}

extern "C" int peagle_draft(peagle_ctx* c, int32_t batch, const peagle_kv* kv,
                            const int32_t* seq_lens, const void* target_hidden,
                            const int32_t* new_token, int32_t K, int32_t* out_draft_tokens,
                            float* out_logits, void* stream) {
  if (!c || !kv || !kv->k || !kv->v || !seq_lens || !target_hidden || !new_token ||
      !out_draft_tokens)
    return PEAGLE_ERR_INVALID;
  return draft_impl(c, batch, kv, seq_lens, target_hidden, new_token, K, false,
                    out_draft_tokens, out_logits, (cudaStream_t)stream);
}

extern "C" int peagle_catch_up(peagle_ctx* c, int32_t batch, const peagle_kv* kv,
                               const int32_t* seq_lens, const void* hidden,
                               const int32_t* tokens, int32_t T, int32_t* out_tokens,
                               float* out_logits, void* stream) {
  if (!c || !kv || !kv->k || !kv->v || !seq_lens || !hidden || !tokens)
    return PEAGLE_ERR_INVALID;
  return draft_impl(c, batch, kv, seq_lens, hidden, tokens, T, true, out_tokens, out_logits,
                    (cudaStream_t)stream);
}

extern "C" int peagle_verify_greedy(int32_t batch, int32_t K, const int32_t* draft_tokens,
                                    const int32_t* target_argmax, int32_t* out_accept_len,
                                    int32_t* out_bonus, void* stream) {
  if (batch < 1 || K < 1 || K > 64 || !draft_tokens || !target_argmax || !out_accept_len ||
      !out_bonus)
    return PEAGLE_ERR_INVALID;
  launch_verify(batch, K, draft_tokens, target_argmax, out_accept_len, out_bonus,
                (cudaStream_t)stream);
  cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "peagle_verify_greedy launch");
}

extern "C" int peagle_append_kv(peagle_ctx* c, int32_t batch, const peagle_kv* kv,
                                int32_t* seq_lens, const int32_t* n_commit, int32_t n_extra,
                                const void* k_rows, const void* v_rows, int32_t n_max,
                                void* stream) {
  if (!c || !kv || !kv->k || !kv->v || !seq_lens || !n_commit) return PEAGLE_ERR_INVALID;
  if (batch < 1 || n_max < 0 || (k_rows == nullptr) != (v_rows == nullptr))
    return PEAGLE_ERR_INVALID;
  if (batch > kv->batch) return PEAGLE_ERR_CAPACITY;
  const peagle_dims& d = c->d;
  // in-place commits are bounded by the draft block (max_K rows); copies by n_max
  const int bound = k_rows ? n_max : d.max_K;
  cudaStream_t s = (cudaStream_t)stream;
  TIMED(PEAGLE_STAGE_SMALL,
        launch_append_kv(c->bf, batch, d.n_layers, d.n_kv_heads, d.head_dim, kv->capacity,
                         kv->k, kv->v, seq_lens, n_commit, n_extra, k_rows, v_rows, bound,
                         kv->batch, c->err, s));
  cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "peagle_append_kv launch");
}

extern "C" int peagle_forward_parallel(peagle_ctx* c, int32_t n, int32_t K, const int32_t* tokens,
                                       const void* hidden, const int32_t* row_p,
                                       const int32_t* row_d, int32_t M, int32_t* out_argmax,
                                       float* out_logits, void* stream) {
  if (!c || !tokens || !hidden || !row_p || !row_d || !out_argmax) return PEAGLE_ERR_INVALID;
  const peagle_dims& d = c->d;
  if (n < 1 || K < 1 || M < 1) return PEAGLE_ERR_INVALID;
  if (d.max_rows <= 0 || M > d.max_rows || n > d.max_seq || K > 16) return PEAGLE_ERR_CAPACITY;
  if (n > d.max_positions) return PEAGLE_ERR_CAPACITY;
  // the training mask has no window; the training forward scores the full head
  if (d.attn_window > 0 || d.lm_rank > 0) return PEAGLE_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  const int H = d.hidden, nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim;
  const int qkv_out = (nq + 2 * nkv) * hd;
  const int Kmax = 16;
  const int split = use_split(c);
  // bf16 drafters with head_dim 64 take the tensor-core masked attention, which reads the
  // queries as bf16 (its operand precision; the QKV epilogue rounds them once, RN, as the
  // kernel would); the mma.sync kernels read fp32 queries
  const bool tc_attn = c->bf && hd == 64 && 128 % (nq / nkv) == 0;
  TIMED(PEAGLE_STAGE_SMALL,
        launch_rows_prepare(M, n, K, Kmax, row_p, row_d, c->row_index, c->err, s));
  // the fc projection accumulates into F; clear every row of this sequence first (a row
  // list that skips a depth-1 position would otherwise leave it uncleared)
  if (cudaMemsetAsync(c->F, 0, (size_t)n * H * sizeof(fx_t), s) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  {
    EpiArgs e = epi_base(c, EPI_STORE, n, H);
    e.out_fx = c->F;
    e.out_ld = H;
    GEMM(PEAGLE_STAGE_FC, c, c->fc, hidden, 3 * H, H, 3 * H, n, e, s);
  }
  TIMED(PEAGLE_STAGE_NORM,
        launch_input_fusion(c->bf, 1, M, K, n, H, c->embed, d.target_vocab, c->emb_mask, c->F,
                            c->f_shared, tokens, row_p, row_d, c->input_norm, c->hidden_norm,
                            d.rms_eps, split, c->X0, c->res, c->keys, nullptr, nullptr, c->err,
                            s));
  for (int l = 0; l < d.n_layers; ++l) {
    const void* a_in = c->X0;
    int din = 2 * H;
    if (l > 0) {
      TIMED(PEAGLE_STAGE_NORM,
            launch_rmsnorm(c->bf, M, H, c->res, c->attn_norm[l], d.rms_eps, split, c->Xn, s));
      a_in = c->Xn;
      din = H;
    }
    {
      EpiArgs e = epi_base(c, EPI_QKV_ROPE, M, qkv_out);
      e.in_split = split;
      e.q_out = c->Qf;
      e.q_f32 = tc_attn ? 0 : 1;
      e.k_dst = c->Kr;
      e.v_dst = c->Vr;
      e.k1_dst = c->K1;
      e.v1_dst = c->V1;
      e.row_pos = row_p;
      e.row_depth = row_d;
      e.n_seq = n;
      e.decode = 0;
      GEMM(PEAGLE_STAGE_QKV, c, c->qkv[l], a_in, din, qkv_out, din, M, e, s);
    }
    {
      MaskedAttnArgs a;
      a.q = c->Qf;
      a.q_bf16 = tc_attn ? 1 : 0;
      a.split = split;
      a.k = c->Kr;
      a.v = c->Vr;
      a.k1 = c->K1;
      a.v1 = c->V1;
      a.row_p = row_p;
      a.row_d = row_d;
      a.row_index = c->row_index;
      a.o = c->O;
      a.M = M;
      a.n = n;
      a.Kmax = Kmax;
      a.nq = nq;
      a.nkv = nkv;
      a.hd = hd;
      a.scale = 1.f / sqrtf((float)hd);
      a.err = c->err;
      // tcgen05 kernel for bf16 and head_dim 64, else the mma.sync / fp32 kernels
      int ar = PEAGLE_OK;
      TIMED(PEAGLE_STAGE_ATTN, {
        if (tc_attn)
          ar = masked_attn_tc_launch(c->tc, a, s);
        else
          launch_masked_attention(c->bf, a, s);
      });
      if (ar != PEAGLE_OK) return ar;
    }
    {
      EpiArgs e = epi_base(c, EPI_RESID, M, H);
      e.in_split = split;
      e.resid = c->res;
      GEMM(PEAGLE_STAGE_OPROJ, c, c->o[l], c->O, nq * hd, H, nq * hd, M, e, s);
    }
    TIMED(PEAGLE_STAGE_NORM,
          launch_rmsnorm(c->bf, M, H, c->res, c->post_norm[l], d.rms_eps, split, c->Xn, s));
    {
      EpiArgs e = epi_base(c, EPI_SWIGLU, M, 2 * d.intermediate);
      e.in_split = split;
      e.out_split = split;
      e.act_out = c->act;
      GEMM(PEAGLE_STAGE_GATEUP, c, c->gate_up[l], c->Xn, H, 2 * d.intermediate, H, M, e, s);
    }
    {
      EpiArgs e = epi_base(c, EPI_RESID, M, H);
      e.in_split = split;
      e.resid = c->res;
      GEMM(PEAGLE_STAGE_DOWN, c, c->down[l], c->act, d.intermediate, H, d.intermediate, M, e, s);
    }
  }
  // Every projection input stays hi/lo here too: as plain bf16 the LM-head input alone
  // moved the training rows' logits to 1.1e-2 against the oracle (the attention output
  // as well: 1.5e-2), too close to the 2e-2 tolerance for 7% of the forward's time.
  const int split_y = split;
  TIMED(PEAGLE_STAGE_NORM,
        launch_rmsnorm(c->bf, M, H, c->res, c->final_norm, d.rms_eps, split_y, c->Xn, s));
  {
    EpiArgs e = epi_base(c, EPI_LMHEAD, M, d.draft_vocab);
    e.in_split = split_y;
    e.logits = out_logits;
    e.keys = c->keys;
    GEMM(PEAGLE_STAGE_LMHEAD, c, c->lm_head, c->Xn, H, d.draft_vocab, H, M, e, s);
  }
  TIMED(PEAGLE_STAGE_SMALL, launch_argmax_decode(M, c->keys, nullptr, out_argmax, s));
  cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "peagle_forward_parallel launch");
}

// ---- training step ("P-EAGLE: Parallel-Drafting EAGLE with Scalable Training", A2 section
// 2 and section 3): the training-style forward with its activations kept, the mean
// cross-entropy over the retained rows, and the gradient of every parameter.  fp32
// activations; the plain GEMMs (projections, the attention's depth-1 prefix products) run
// on this library's own kernels: TF32 tcgen05 MMAs for bf16 drafters, fp32 FMA tiles for
// fp32 drafters.  Every workspace is made by peagle_create.

#define TRY_RET(x)  \
  do {              \
    int _r = (x);   \
    if (_r) return _r; \
  } while (0)

static int train_ws(peagle_ctx* c) {
  if (c->tw) return PEAGLE_OK;
  const peagle_dims& d = c->d;
  const int M = d.max_rows, n = d.max_seq, H = d.hidden, I = d.intermediate;
  const int nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim;
  const int qkv_out = (nq + 2 * nkv) * hd, N = d.n_layers, Vd = d.draft_vocab;
  // built aside and attached only when complete (a failed call leaves no half workspace;
  // what it allocated stays on the context's list and is freed with it)
  std::unique_ptr<TrainWs> hold(new TrainWs());
  TrainWs* w = hold.get();
  w->Mmax = M;
  w->nmax = n;
  auto fl = [&](float** p, size_t count) { return dalloc(c, (void**)p, count * 4); };
  // fp32 weights
  auto wcopy = [&](float** dst, void* src, size_t count) -> int {
    if (!c->bf) {
      *dst = (float*)src;
      return PEAGLE_OK;
    }
    TRY_RET(fl(dst, count));
    launch_to_f32(count, src, *dst, 0);
    return PEAGLE_OK;
  };
  TRY_RET(wcopy(&w->fc, c->fc, (size_t)H * 3 * H));
  TRY_RET(wcopy(&w->lm, c->lm_head, (size_t)Vd * H));
  TRY_RET(wcopy(&w->in_norm, c->input_norm, H));
  TRY_RET(wcopy(&w->hid_norm, c->hidden_norm, H));
  TRY_RET(wcopy(&w->fin_norm, c->final_norm, H));
  w->qkv.resize(N);
  w->o.resize(N);
  w->gu.resize(N);
  w->down.resize(N);
  w->attn_norm.assign(N, nullptr);
  w->post_norm.resize(N);
  for (int l = 0; l < N; ++l) {
    const int din = l == 0 ? 2 * H : H;
    TRY_RET(wcopy(&w->qkv[l], c->qkv[l], (size_t)qkv_out * din));
    TRY_RET(wcopy(&w->o[l], c->o[l], (size_t)H * nq * hd));
    TRY_RET(wcopy(&w->gu[l], c->gate_up[l], (size_t)2 * I * H));
    TRY_RET(wcopy(&w->down[l], c->down[l], (size_t)H * I));
    if (l > 0) TRY_RET(wcopy(&w->attn_norm[l], c->attn_norm[l], H));
    TRY_RET(wcopy(&w->post_norm[l], c->post_norm[l], H));
  }
  w->qkvT.assign(N, nullptr);
  w->oT.assign(N, nullptr);
  w->guT.assign(N, nullptr);
  w->downT.assign(N, nullptr);
  if (c->bf) {
    // W [out][in] -> W^T [in][out] (every out dimension is a multiple of 4 floats)
    auto wT = [&](float** dst, const float* src, int out_dim, int in_dim) -> int {
      TRY_RET(fl(dst, (size_t)out_dim * in_dim));
      launch_transpose_f32(src, out_dim, in_dim, in_dim, *dst, out_dim, 0);
      return PEAGLE_OK;
    };
    TRY_RET(wT(&w->fcT, w->fc, H, 3 * H));
    TRY_RET(wT(&w->lmT, w->lm, Vd, H));
    for (int l = 0; l < N; ++l) {
      TRY_RET(wT(&w->qkvT[l], w->qkv[l], qkv_out, l == 0 ? 2 * H : H));
      TRY_RET(wT(&w->oT[l], w->o[l], H, nq * hd));
      TRY_RET(wT(&w->guT[l], w->gu[l], 2 * I, H));
      TRY_RET(wT(&w->downT[l], w->down[l], H, I));
    }
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return PEAGLE_ERR_CUDA;
  // forward, kept for the backward
  TRY_RET(dalloc(c, (void**)&w->chain, (size_t)M * 15 * 4));
  TRY_RET(fl(&w->E, (size_t)M * H));
  TRY_RET(fl(&w->Hin, (size_t)M * 3 * H));
  TRY_RET(fl(&w->f, (size_t)M * H));
  TRY_RET(fl(&w->r1, M));
  TRY_RET(fl(&w->r2, M));
  TRY_RET(fl(&w->x0, (size_t)M * 2 * H));
  TRY_RET(fl(&w->y, (size_t)M * H));
  TRY_RET(fl(&w->ry, M));
  TRY_RET(fl(&w->logits, (size_t)M * Vd));
  TRY_RET(fl(&w->row_loss, M));
  TRY_RET(fl(&w->resL, (size_t)M * H));
  for (auto* v : {&w->res_in, &w->a, &w->ra, &w->Qh, &w->Kr, &w->Vr, &w->K1, &w->V1, &w->Pc,
                  &w->lse, &w->O, &w->res_mid, &w->u, &w->ru, &w->GU, &w->act})
    v->assign(N, nullptr);
  for (int l = 0; l < N; ++l) {
    if (l > 0) {
      TRY_RET(fl(&w->res_in[l], (size_t)M * H));
      TRY_RET(fl(&w->a[l], (size_t)M * H));
      TRY_RET(fl(&w->ra[l], M));
    }
    TRY_RET(fl(&w->Qh[l], (size_t)nq * M * hd));
    TRY_RET(fl(&w->Kr[l], (size_t)M * nkv * hd));
    TRY_RET(fl(&w->Vr[l], (size_t)M * nkv * hd));
    TRY_RET(fl(&w->K1[l], (size_t)nkv * n * hd));
    TRY_RET(fl(&w->V1[l], (size_t)nkv * n * hd));
    TRY_RET(fl(&w->Pc[l], (size_t)nq * M * 15));
    TRY_RET(fl(&w->lse[l], (size_t)nq * M));
    TRY_RET(fl(&w->O[l], (size_t)M * nq * hd));
    TRY_RET(fl(&w->res_mid[l], (size_t)M * H));
    TRY_RET(fl(&w->u[l], (size_t)M * H));
    TRY_RET(fl(&w->ru[l], M));
    TRY_RET(fl(&w->GU[l], (size_t)M * 2 * I));
    TRY_RET(fl(&w->act[l], (size_t)M * I));
  }
  w->res_in[0] = w->f;
  w->a[0] = w->x0;
  TRY_RET(fl(&w->qkvb, (size_t)M * qkv_out));
  // the dense prefix score matrices [G M][n]: only where the fused attention does not apply
  TrainAttn probe;
  memset(&probe, 0, sizeof(probe));
  probe.nq = nq;
  probe.nkv = nkv;
  probe.hd = hd;
  const bool dense_attn = !(c->bf && attn_bwd_fused_ok(probe));
  w->S1 = w->dP1 = nullptr;
  if (dense_attn) {
    const size_t count = (size_t)(nq / nkv) * M * n;
    TRY_RET(dalloc(c, (void**)&w->S1, count * 4));
    TRY_RET(dalloc(c, (void**)&w->dP1, count * 4));
  }
  if (!dense_attn && attn_tc_ok(probe)) {
    w->ldn = (n + 3) / 4 * 4;
    TRY_RET(fl(&w->kvT, (size_t)nkv * 64 * w->ldn));
    w->ldm = (M + 3) / 4 * 4;
    TRY_RET(fl(&w->qT, (size_t)nq * 64 * w->ldm));
    TRY_RET(fl(&w->doT, (size_t)nq * 64 * w->ldm));
  }
  TRY_RET(fl(&w->Oh, (size_t)nq * M * hd));
  TRY_RET(fl(&w->lrow, (size_t)nq * M));
  // backward
  TRY_RET(fl(&w->bufA, (size_t)M * H));
  TRY_RET(fl(&w->bufB, (size_t)M * H));
  TRY_RET(fl(&w->dact, (size_t)M * I));
  TRY_RET(fl(&w->dGU, (size_t)M * 2 * I));
  TRY_RET(fl(&w->du, (size_t)M * H));
  TRY_RET(fl(&w->dO, (size_t)M * nq * hd));
  TRY_RET(fl(&w->dOh, (size_t)nq * M * hd));
  TRY_RET(fl(&w->Dv, (size_t)nq * M));
  TRY_RET(fl(&w->dQh, (size_t)nq * M * hd));
  TRY_RET(fl(&w->dKr, (size_t)M * nkv * hd));
  TRY_RET(fl(&w->dVr, (size_t)M * nkv * hd));
  TRY_RET(fl(&w->dK1, (size_t)nkv * n * hd));
  TRY_RET(fl(&w->dV1, (size_t)nkv * n * hd));
  TRY_RET(fl(&w->dqkv, (size_t)M * qkv_out));
  TRY_RET(fl(&w->da, (size_t)M * 2 * H));
  TRY_RET(fl(&w->dgu_w, (size_t)2 * I * H));
  TRY_RET(fl(&w->dE, (size_t)M * H));
  TRY_RET(fl(&w->df, (size_t)M * H));
  TRY_RET(fl(&w->dHin, (size_t)M * 3 * H));
  TRY_RET(fl(&w->dy, (size_t)M * H));
  // the tensor-core GEMMs' scratch operands (bf16 drafters): the largest operand that a
  // product reads transposed -- an activation [M][widest] or a weight [rows][cols]
  if (c->bf) {
    const int widest = std::max({3 * H, 2 * I, Vd, qkv_out, nq * hd, 2 * H});
    size_t cap = std::max(tf32_scratch_floats(M, widest), tf32_scratch_floats(widest, M));
    cap = std::max(cap, tf32_scratch_floats(widest, 3 * H));
    cap = std::max(cap, tf32_scratch_floats(widest, I));
    cap = std::max(cap, tf32_scratch_floats(widest, nq * hd));
    if (dense_attn) {
      // the dense prefix-attention path's operands: [G M][n] scores
      const int G = nq / nkv;
      cap = std::max(cap, tf32_scratch_floats(G * M, n));
      cap = std::max(cap, tf32_scratch_floats(n, G * M));
    }
    TRY_RET(fl(&w->gscratch_a, cap));
    TRY_RET(fl(&w->gscratch_b, cap));
    w->gscratch_floats = cap;
  }
  c->tw = hold.release();
  return PEAGLE_OK;
}

static int zero(float* p, size_t count, cudaStream_t s) {
  return cudaMemsetAsync(p, 0, count * 4, s) == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

extern "C" int peagle_train_step(peagle_ctx* c, int32_t n, int32_t K, const int32_t* tokens,
                                 const void* hidden, const int32_t* row_p, const int32_t* row_d,
                                 int32_t M, const int32_t* labels, float* out_loss,
                                 const peagle_grads* gr, void* stream) {
  if (!c || !tokens || !hidden || !row_p || !row_d || !labels || !out_loss || !gr)
    return PEAGLE_ERR_INVALID;
  if (!gr->emb_mask || !gr->h_shared || !gr->fc || !gr->input_norm || !gr->hidden_norm ||
      !gr->qkv || !gr->o || !gr->post_norm || !gr->gate || !gr->up || !gr->down ||
      !gr->final_norm || !gr->lm_head)
    return PEAGLE_ERR_INVALID;
  const peagle_dims& d = c->d;
  if (n < 1 || K < 1 || M < 1) return PEAGLE_ERR_INVALID;
  if (d.max_rows <= 0 || M > d.max_rows || n > d.max_seq || K > 16) return PEAGLE_ERR_CAPACITY;
  if (n > d.max_positions) return PEAGLE_ERR_CAPACITY;
  if (d.attn_window > 0 || d.lm_rank > 0) return PEAGLE_ERR_UNSUPPORTED;
  for (int l = 0; l < d.n_layers; ++l)
    if (!gr->qkv[l] || !gr->o[l] || !gr->post_norm[l] || !gr->gate[l] || !gr->up[l] ||
        !gr->down[l])
      return PEAGLE_ERR_INVALID;
  if (!c->tw) return PEAGLE_ERR_CAPACITY;  // workspaces are made by peagle_create
  TrainWs* w = c->tw;
  cudaStream_t s = (cudaStream_t)stream;
  TrainGemmCtx tg;
  tg.tc = c->bf ? c->tc : nullptr;
  tg.scratch_a = w->gscratch_a;
  tg.scratch_b = w->gscratch_b;
  tg.scratch_floats = w->gscratch_floats;
  tg.err = c->err;
  const int H = d.hidden, I = d.intermediate, Vd = d.draft_vocab, Vt = d.target_vocab;
  const int nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim, G = nq / nkv;
  const int qkv_out = (nq + 2 * nkv) * hd, N = d.n_layers, nqhd = nq * hd;
  const float eps = d.rms_eps, scale = 1.f / sqrtf((float)hd);
  const int Kmax = 16;
  int gerr = PEAGLE_OK;
  auto GM = [&](bool ta, bool tb, int m, int nn, int k, float alpha, const float* A, int lda,
                const float* B, int ldb, float beta, float* C, int ldc) {
    if (gerr == PEAGLE_OK)
      gerr = train_gemm(tg, ta, tb, m, nn, k, alpha, A, lda, B, ldb, beta, C, ldc, s);
  };
  // C [m x nn] = A W for a weight W stored [k][nn] (nn.Linear [out][in], k = out): from its
  // transposed copy WT [nn][k] where the context holds one
  auto GMW = [&](int m, int nn, int k, const float* A, int lda, const float* W,
                 const float* WT, float* C, int ldc) {
    if (WT)
      GM(false, true, m, nn, k, 1.f, A, lda, WT, k, 0.f, C, ldc);
    else
      GM(false, false, m, nn, k, 1.f, A, lda, W, nn, 0.f, C, ldc);
  };
  launch_rows_prepare(M, n, K, Kmax, row_p, row_d, c->row_index, c->err, s);
  launch_chain(M, n, K, Kmax, row_p, row_d, c->row_index, w->chain, s);
  TrainAttn ta;
  ta.M = M;
  ta.n = n;
  ta.K = K;
  ta.nq = nq;
  ta.nkv = nkv;
  ta.hd = hd;
  ta.scale = scale;
  ta.row_p = row_p;
  ta.row_d = row_d;
  ta.chain = w->chain;
  // bf16 drafters take the fused TF32 attention (fp32 drafters keep fp32 GEMMs over the
  // dense prefix score matrices, made by peagle_create)
  const bool fused_attn = c->bf && attn_bwd_fused_ok(ta);
  if (!fused_attn && !w->S1) return PEAGLE_ERR_UNSUPPORTED;
  TrainAttnTc atc;
  atc.tc = c->tc;
  atc.err = c->err;
  atc.kvT = w->kvT;
  atc.ldn = w->ldn;
  atc.qT = w->qT;
  atc.doT = w->doT;
  atc.ldm = w->ldm;

  // ---- forward
  launch_train_inputs(c->bf, M, n, K, H, row_p, row_d, tokens, hidden, c->embed, Vt, c->emb_mask,
                      c->h_shared, w->E, w->Hin, c->err, s);
  GM(false, true, M, H, 3 * H, 1.f, w->Hin, 3 * H, w->fc, 3 * H, 0.f, w->f, H);
  launch_rms_fwd(M, H, w->E, H, w->in_norm, eps, w->x0, 2 * H, w->r1, s);
  launch_rms_fwd(M, H, w->f, H, w->hid_norm, eps, w->x0 + H, 2 * H, w->r2, s);
  const float* res = w->f;
  for (int l = 0; l < N; ++l) {
    const int din = l == 0 ? 2 * H : H;
    if (l > 0) launch_rms_fwd(M, H, w->res_in[l], H, w->attn_norm[l], eps, w->a[l], H, w->ra[l], s);
    GM(false, true, M, qkv_out, din, 1.f, w->a[l], din, w->qkv[l], din, 0.f, w->qkvb, qkv_out);
    TRY_RET(zero(w->K1[l], (size_t)nkv * n * hd, s));
    TRY_RET(zero(w->V1[l], (size_t)nkv * n * hd, s));
    launch_train_rope(M, n, K, nq, nkv, hd, w->qkvb, row_p, row_d, c->rope, w->Qh[l], w->Kr[l],
                      w->Vr[l], w->K1[l], w->V1[l], fused_attn, s);
    if (fused_attn)  // online softmax over the prefix, then the chain keys per row
      TRY_RET(launch_attn_fwd_fused(ta, w->Qh[l], w->Kr[l], w->Vr[l], w->K1[l], w->V1[l], w->Oh,
                                    w->Dv, w->lrow, w->Pc[l], w->lse[l], w->O[l],
                                    w->kvT ? &atc : nullptr, s));
    for (int g = 0; g < nkv && !fused_attn; ++g) {
      const float* Qg = w->Qh[l] + (size_t)g * G * M * hd;
      const float* K1g = w->K1[l] + (size_t)g * n * hd;
      const float* V1g = w->V1[l] + (size_t)g * n * hd;
      GM(false, true, G * M, n, hd, scale, Qg, hd, K1g, hd, 0.f, w->S1, n);
      launch_attn_fwd_softmax(ta, g, w->S1, w->Qh[l], w->Kr[l], w->Pc[l], w->lse[l], s);
      GM(false, false, G * M, hd, n, 1.f, w->S1, n, V1g, hd, 0.f, w->Oh + (size_t)g * G * M * hd,
         hd);
      launch_attn_fwd_out(ta, g, w->Oh, w->Pc[l], w->Vr[l], w->O[l], s);
    }
    if (cudaMemcpyAsync(w->res_mid[l], res, (size_t)M * H * 4, cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return PEAGLE_ERR_CUDA;
    GM(false, true, M, H, nqhd, 1.f, w->O[l], nqhd, w->o[l], nqhd, 1.f, w->res_mid[l], H);
    launch_rms_fwd(M, H, w->res_mid[l], H, w->post_norm[l], eps, w->u[l], H, w->ru[l], s);
    GM(false, true, M, 2 * I, H, 1.f, w->u[l], H, w->gu[l], H, 0.f, w->GU[l], 2 * I);
    launch_swiglu_fwd(M, I, w->GU[l], w->act[l], s);
    float* res_out = l + 1 < N ? w->res_in[l + 1] : w->resL;
    if (cudaMemcpyAsync(res_out, w->res_mid[l], (size_t)M * H * 4, cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return PEAGLE_ERR_CUDA;
    GM(false, true, M, H, I, 1.f, w->act[l], I, w->down[l], I, 1.f, res_out, H);
    res = res_out;
  }
  launch_rms_fwd(M, H, w->resL, H, w->fin_norm, eps, w->y, H, w->ry, s);
  GM(false, true, M, Vd, H, 1.f, w->y, H, w->lm, H, 0.f, w->logits, Vd);
  launch_ce(M, Vd, w->logits, labels, w->row_loss, out_loss, c->err, s);  // logits -> dlogits

  // ---- backward
  GM(true, false, Vd, H, M, 1.f, w->logits, Vd, w->y, H, 0.f, gr->lm_head, H);
  GMW(M, H, Vd, w->logits, Vd, w->lm, w->lmT, w->dy, H);
  float* dres = w->bufA;
  float* dmid = w->bufB;
  launch_rms_bwd(M, H, w->resL, H, w->ry, w->fin_norm, w->dy, H, dres, H, false, s);
  TRY_RET(zero(gr->final_norm, H, s));
  launch_colsum(M, H, w->dy, H, w->resL, H, w->ry, nullptr, gr->final_norm, s);
  for (int l = N - 1; l >= 0; --l) {
    const int din = l == 0 ? 2 * H : H;
    // MLP
    GM(true, false, H, I, M, 1.f, dres, H, w->act[l], I, 0.f, gr->down[l], I);
    GMW(M, I, H, dres, H, w->down[l], w->downT[l], w->dact, I);
    launch_swiglu_bwd(M, I, w->GU[l], w->dact, w->dGU, s);
    GM(true, false, 2 * I, H, M, 1.f, w->dGU, 2 * I, w->u[l], H, 0.f, w->dgu_w, H);
    launch_gu_split(I, H, w->dgu_w, gr->gate[l], gr->up[l], s);
    GMW(M, H, 2 * I, w->dGU, 2 * I, w->gu[l], w->guT[l], w->du, H);
    if (cudaMemcpyAsync(dmid, dres, (size_t)M * H * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return PEAGLE_ERR_CUDA;
    launch_rms_bwd(M, H, w->res_mid[l], H, w->ru[l], w->post_norm[l], w->du, H, dmid, H, true, s);
    TRY_RET(zero(gr->post_norm[l], H, s));
    launch_colsum(M, H, w->du, H, w->res_mid[l], H, w->ru[l], nullptr, gr->post_norm[l], s);
    // attention
    GM(true, false, H, nqhd, M, 1.f, dmid, H, w->O[l], nqhd, 0.f, gr->o[l], nqhd);
    GMW(M, nqhd, H, dmid, H, w->o[l], w->oT[l], w->dO, nqhd);
    launch_attn_bwd_prep(ta, w->dO, w->O[l], w->dOh, w->Dv, fused_attn, s);
    TRY_RET(zero(w->dKr, (size_t)M * nkv * hd, s));
    TRY_RET(zero(w->dVr, (size_t)M * nkv * hd, s));
    if (fused_attn) {
      // chain part per row, then the prefix part on TF32 tensor cores without the dense
      // score matrices
      if (!launch_attn_bwd_chain(ta, w->lse[l], w->Dv, w->Qh[l], w->Kr[l], w->Vr[l], w->dOh,
                                 w->dQh, w->dKr, w->dVr, s))
        for (int g = 0; g < nkv; ++g)
          launch_attn_bwd_ds(ta, g, nullptr, nullptr, w->lse[l], w->Dv, w->Qh[l], w->Kr[l],
                             w->Vr[l], w->dOh, w->dQh, w->dKr, w->dVr, s);
      TRY_RET(zero(w->dK1, (size_t)nkv * n * hd, s));
      TRY_RET(zero(w->dV1, (size_t)nkv * n * hd, s));
      TRY_RET(launch_attn_bwd_fused(ta, c->row_index, Kmax, w->Qh[l], w->dOh, w->K1[l],
                                    w->V1[l], w->lse[l], w->Dv, w->dQh, w->dK1, w->dV1,
                                    w->kvT ? &atc : nullptr, s));
    }
    for (int g = 0; g < nkv && !fused_attn; ++g) {
      const float* Qg = w->Qh[l] + (size_t)g * G * M * hd;
      const float* K1g = w->K1[l] + (size_t)g * n * hd;
      const float* V1g = w->V1[l] + (size_t)g * n * hd;
      const float* dOg = w->dOh + (size_t)g * G * M * hd;
      float* dQg = w->dQh + (size_t)g * G * M * hd;
      GM(false, true, G * M, n, hd, scale, Qg, hd, K1g, hd, 0.f, w->S1, n);
      GM(false, true, G * M, n, hd, 1.f, dOg, hd, V1g, hd, 0.f, w->dP1, n);
      launch_attn_bwd_ds(ta, g, w->S1, w->dP1, w->lse[l], w->Dv, w->Qh[l], w->Kr[l], w->Vr[l],
                         w->dOh, w->dQh, w->dKr, w->dVr, s);
      GM(false, false, G * M, hd, n, 1.f, w->dP1, n, K1g, hd, 1.f, dQg, hd);
      GM(true, false, n, hd, G * M, 1.f, w->dP1, n, Qg, hd, 0.f, w->dK1 + (size_t)g * n * hd, hd);
      GM(true, false, n, hd, G * M, 1.f, w->S1, n, dOg, hd, 0.f, w->dV1 + (size_t)g * n * hd, hd);
    }
    launch_kv1_scatter(M, n, K, nkv, hd, row_p, row_d, w->dK1, w->dV1, w->dKr, w->dVr, s);
    launch_train_rope_bwd(M, n, K, nq, nkv, hd, w->dQh, w->dKr, w->dVr, row_p, row_d, c->rope,
                          w->dqkv, s);
    GM(true, false, qkv_out, din, M, 1.f, w->dqkv, qkv_out, w->a[l], din, 0.f, gr->qkv[l], din);
    GMW(M, din, qkv_out, w->dqkv, qkv_out, w->qkv[l], w->qkvT[l], w->da, din);
    if (l > 0) {
      launch_rms_bwd(M, H, w->res_in[l], H, w->ra[l], w->attn_norm[l], w->da, H, dmid, H, true, s);
      if (gr->attn_norm && gr->attn_norm[l]) {
        TRY_RET(zero(gr->attn_norm[l], H, s));
        launch_colsum(M, H, w->da, H, w->res_in[l], H, w->ra[l], nullptr, gr->attn_norm[l], s);
      }
    } else if (gr->attn_norm && gr->attn_norm[0]) {
      TRY_RET(zero(gr->attn_norm[0], H, s));  // layer 1 reads x0, not a norm of the residual
    }
    std::swap(dres, dmid);  // dres = the residual stream's gradient at the layer's input
  }
  // first-layer input x0 = [rms_in(E) || rms_hid(f)]; the residual stream starts at f
  launch_rms_bwd(M, H, w->E, H, w->r1, w->in_norm, w->da, 2 * H, w->dE, H, false, s);
  TRY_RET(zero(gr->input_norm, H, s));
  launch_colsum(M, H, w->da, 2 * H, w->E, H, w->r1, nullptr, gr->input_norm, s);
  launch_rms_bwd(M, H, w->f, H, w->r2, w->hid_norm, w->da + H, 2 * H, w->df, H, false, s);
  TRY_RET(zero(gr->hidden_norm, H, s));
  launch_colsum(M, H, w->da + H, 2 * H, w->f, H, w->r2, nullptr, gr->hidden_norm, s);
  launch_add((size_t)M * H, dres, w->df, s);
  GM(true, false, H, 3 * H, M, 1.f, w->df, H, w->Hin, 3 * H, 0.f, gr->fc, 3 * H);
  GMW(M, 3 * H, H, w->df, H, w->fc, w->fcT, w->dHin, 3 * H);
  TRY_RET(zero(gr->emb_mask, H, s));
  launch_colsum(M, H, w->dE, H, nullptr, 0, nullptr, row_d, gr->emb_mask, s);
  TRY_RET(zero(gr->h_shared, (size_t)3 * H, s));
  launch_colsum(M, 3 * H, w->dHin, 3 * H, nullptr, 0, nullptr, row_d, gr->h_shared, s);
  if (gr->embed) {
    TRY_RET(zero(gr->embed, (size_t)Vt * H, s));
    launch_embed_grad(M, n, K, H, Vt, row_p, row_d, tokens, w->dE, gr->embed, s);
  }
  if (gerr != PEAGLE_OK) return gerr;
  cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? PEAGLE_OK : cuda_fail(ce, "training step launch");
}

extern "C" int peagle_cod_rows(int32_t n, int32_t K, double ratio, const double* uniforms,
                               int32_t* out_p, int32_t* out_d, int32_t max_out) {
  if (n < 0 || K < 1 || K > 16 || !uniforms || !out_p || !out_d || max_out < 0)
    return PEAGLE_ERR_INVALID;
  // kept[d] for the previous position; depth 1 always kept
  std::vector<char> prev(K + 1, 0), cur(K + 1, 0);
  int count = 0;
  for (int p = 0; p < n; ++p) {
    for (int d = 1; d <= K; ++d) {
      bool keep;
      if (d == 1)
        keep = true;
      else if (p - d + 1 < 0)
        keep = false;
      else
        keep = prev[d - 1] && uniforms[(size_t)p * K + (d - 1)] < ratio;
      cur[d] = keep;
      if (keep) {
        if (count >= max_out) return PEAGLE_ERR_CAPACITY;
        out_p[count] = p;
        out_d[count] = d;
        ++count;
      }
    }
    prev.swap(cur);
  }
  return count;
}

extern "C" int peagle_sequence_partition(int32_t M, const int32_t* row_p, const int32_t* row_d,
                                         int32_t n_chunks, const int32_t* boundaries,
                                         int32_t* out_chunk) {
  if (M < 0 || n_chunks < 1 || !boundaries || (M > 0 && (!row_p || !row_d || !out_chunk)))
    return PEAGLE_ERR_INVALID;
  if (boundaries[0] != 0) return PEAGLE_ERR_INVALID;
  for (int s = 1; s < n_chunks; ++s)
    if (boundaries[s] <= boundaries[s - 1]) return PEAGLE_ERR_INVALID;
  constexpr int DMAX = 64;
  // chunk of (p, d) for the current and the previous position (rows are p-major)
  std::vector<int> prev(DMAX + 1, -1), cur(DMAX + 1, -1);
  int cur_p = -1, s = 0;
  for (int i = 0; i < M; ++i) {
    const int p = row_p[i], d = row_d[i];
    if (p < 0 || d < 1 || d > DMAX) return PEAGLE_ERR_INVALID;
    if (i > 0 && (p < row_p[i - 1] || (p == row_p[i - 1] && d <= row_d[i - 1])))
      return PEAGLE_ERR_INVALID;  // not p-major
    if (p != cur_p) {
      if (p == cur_p + 1) {
        prev.swap(cur);
      } else {
        std::fill(prev.begin(), prev.end(), -1);
      }
      std::fill(cur.begin(), cur.end(), -1);
      cur_p = p;
    }
    int ch;
    if (d <= 2) {
      while (s + 1 < n_chunks && boundaries[s + 1] <= p) ++s;  // p only grows
      ch = s;
    } else {
      ch = prev[d - 1];  // Chunk(p, d) = Chunk(p-1, d-1)
      if (ch < 0) return PEAGLE_ERR_INVALID;  // dependency not in the set
    }
    cur[d] = ch;
    out_chunk[i] = ch;
  }
  return PEAGLE_OK;
}

// After a pass that gave up on a bounded wait, the accumulators that the kernels clear as
// they consume them (fixed-point fc rows, q / k / v sums, GEMM tile counters, split-KV merge
// counters, the efficient head's counters) may hold a partial pass: zero them so the next
// call starts clean.
static int reset_after_timeout(peagle_ctx* c) {
  const peagle_dims& d = c->d;
  const size_t nq = d.n_q_heads, nkv = d.n_kv_heads, hd = d.head_dim;
  struct Z { void* p; size_t n; } z[] = {
      {c->F, c->F_bytes},
      {c->pass_qfx, (size_t)PASS_MAX_ROWS * nq * hd * 8},
      {c->pass_kvfx, (size_t)PASS_MAX_ROWS * 2 * nkv * hd * 8},
      {c->mk_qfx, (size_t)d.max_batch * d.max_K * nq * hd * 8},
      {c->mk_kvfx, (size_t)d.max_batch * d.max_K * 2 * nkv * hd * 8},
      {c->att_cnt, (size_t)d.max_batch * nkv * 4},
      {c->tc ? tc_tile_counters(c->tc) : nullptr, c->tc ? (size_t)tc_max_tiles(c->tc) * 4 : 0},
      {c->lm_done, 4},
      {c->lm_gcount, (size_t)d.max_batch * d.max_K * 4},
      {c->lm_gdone, (size_t)d.max_batch * d.max_K * 4},
      {c->lm_hist, (size_t)d.max_batch * d.max_K * 2048 * 4},
  };
  for (const Z& e : z)
    if (e.p && e.n && cudaMemset(e.p, 0, e.n) != cudaSuccess) return PEAGLE_ERR_CUDA;
  return cudaDeviceSynchronize() == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

extern "C" int peagle_status(peagle_ctx* c) {
  if (!c) return PEAGLE_ERR_INVALID;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "peagle_status");
  unsigned bits = 0;
  if (cudaMemcpy(&bits, c->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return PEAGLE_ERR_CUDA;
  c->last_err_bits = bits;
  if (bits) {
    cudaMemset(c->err, 0, 4);
    if ((bits & PEAGLE_DEV_TIMEOUT) && reset_after_timeout(c) != PEAGLE_OK) return PEAGLE_ERR_CUDA;
    return PEAGLE_ERR_DEVICE;
  }
  return PEAGLE_OK;
}

extern "C" int peagle_set_pass_kernel(peagle_ctx* c, int32_t mode) {
  if (!c || mode < -1 || mode > 1) return PEAGLE_ERR_INVALID;
  if (mode == 1 && !c->pass_on) return PEAGLE_ERR_UNSUPPORTED;
  c->pass_mode = mode;
  return PEAGLE_OK;
}

extern "C" int peagle_set_wait_limit(peagle_ctx* c, uint64_t limit_ns, int32_t unreachable_step) {
  if (!c || unreachable_step < -1 || unreachable_step >= PASS_MAX_PHASE) return PEAGLE_ERR_INVALID;
  c->wait_ns = limit_ns ? (unsigned long long)limit_ns : PASS_DEFAULT_WAIT_NS;
  c->stall_phase = unreachable_step;
  return PEAGLE_OK;
}

extern "C" int peagle_set_timing(peagle_ctx* c, int32_t enable) {
  if (!c) return PEAGLE_ERR_INVALID;
  if (enable && c->ev.empty()) {
    c->ev.resize(1024);
    c->ev_stage.assign(512, 0);
    for (auto& e : c->ev)
      if (cudaEventCreate(&e) != cudaSuccess) return PEAGLE_ERR_CUDA;
  }
  c->timing = enable != 0;
  c->ev_used = 0;
  c->trace_stages.clear();
  return PEAGLE_OK;
}

extern "C" int peagle_read_timing(peagle_ctx* c, float* stage_ms, int32_t* stage_launches) {
  if (!c || !stage_ms || !stage_launches) return PEAGLE_ERR_INVALID;
  for (int i = 0; i < PEAGLE_NUM_STAGES; ++i) {
    stage_ms[i] = 0.f;
    stage_launches[i] = 0;
  }
  for (size_t k = 0; k + 1 < c->ev_used; k += 2) {
    float ms = 0.f;
    if (cudaEventSynchronize(c->ev[k + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, c->ev[k], c->ev[k + 1]) != cudaSuccess)
      return PEAGLE_ERR_CUDA;
    const int st = c->ev_stage[k / 2];
    stage_ms[st] += ms;
    stage_launches[st] += 1;
  }
  c->ev_used = 0;
  // pass-kernel calls: the time from one phase's completion to the next is attributed to
  // the later phase's stage (one "launch" per phase)
  if (!c->trace_stages.empty()) {
    const size_t n = c->trace_stages.size();
    std::vector<unsigned long long> t(n * (PASS_MAX_PHASE + 1));
    if (cudaMemcpy(t.data(), c->pass_trace, t.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
      return PEAGLE_ERR_CUDA;
    for (size_t k = 0; k < n; ++k) {
      const unsigned long long* tk = t.data() + k * (PASS_MAX_PHASE + 1);
      const std::vector<int>& st = c->trace_stages[k];
      for (size_t j = 0; j < st.size(); ++j) {
        const double ms = tk[j + 1] > tk[j] ? (double)(tk[j + 1] - tk[j]) * 1e-6 : 0.0;
        stage_ms[st[j]] += (float)ms;
        stage_launches[st[j]] += 1;
      }
    }
    c->trace_stages.clear();
  }
  return PEAGLE_OK;
}

extern "C" int32_t peagle_read_pass_trace(peagle_ctx* c, uint64_t* out, int32_t max_entries,
                                          int32_t* out_phases, int32_t* out_ctas) {
  if (!c || !out || max_entries < 0 || !out_phases || !out_ctas) return PEAGLE_ERR_INVALID;
  *out_phases = 0;
  *out_ctas = 0;
  if (!c->pass_on || c->trace_cta_phases <= 0) return 0;
  const int n = c->trace_cta_phases * c->num_sms * 4;
  if (n > max_entries) return PEAGLE_ERR_CAPACITY;
  if (cudaMemcpy(out, c->pass_trace_cta, (size_t)n * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  *out_phases = c->trace_cta_phases;
  *out_ctas = c->num_sms;
  return n;
}

extern "C" int32_t peagle_device_error_bits(const peagle_ctx* c) {
  return c ? (int32_t)c->last_err_bits : 0;
}

extern "C" const char* peagle_strerror(int code) {
  switch (code) {
    case PEAGLE_OK: return "ok";
    case PEAGLE_ERR_INVALID: return "invalid argument";
    case PEAGLE_ERR_UNSUPPORTED: return "unsupported dimensions";
    case PEAGLE_ERR_CAPACITY: return "capacity exceeded";
    case PEAGLE_ERR_CUDA: return "CUDA error";
    case PEAGLE_ERR_DEVICE: return "device-side check failed";
    default: return "unknown error";
  }
}

extern "C" void peagle_destroy(peagle_ctx* c) { free_ctx(c); }
