// Persistent kernel of the bf16 draft pass: the whole pass (fc, input rows, N decoder
// layers, LM head, argmax) as one launch of one CTA per SM.  Host-side description.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "kernels.h"

namespace peagle {

constexpr int PASS_MAX_LAYERS = 8;
constexpr int PASS_MAX_GEMM = 3 + 4 * PASS_MAX_LAYERS;
constexpr int PASS_MAX_PHASE = 5 + 7 * PASS_MAX_LAYERS;
constexpr unsigned long long PASS_DEFAULT_WAIT_NS = 2000000000ull;  // bounded waits: 2 s
constexpr int PASS_MAX_ROWS = 120;                    // R = B*K (hi + lo rows <= 240)
// 64-wide k-blocks per ring stage: one tensor load brings PASS_KU k-blocks of a 128-row
// weight tile (32 KB).  A cold stream of 16 KB loads reached 3.9 TB/s over 152 SMs with 160
// KB in flight per SM; 32 KB loads with the same bytes in flight, 4.9 TB/s.
constexpr int PASS_KU = 2;
constexpr int PASS_SS_SLOTS = 2 + 2 * PASS_MAX_LAYERS;  // per-row sums of squares
// K/V tile buffers of an attention item (64 keys each).  Deeper pipelines (all four tiles
// of a 256-key chunk in flight) measured no faster: an item is bound by its compute and
// the step's latency chain, and the shared memory is worth more as weight-ring stages.
constexpr int pass_att_nbuf(int) { return 2; }

// RMSNorm is split in two: a step spread over all CTAs writes x * gamma (the projection's
// operand) and adds each row's sum of squares into a fixed-point slot; the consuming
// projection's epilogue scales its rows by rsqrt(mean + eps).
enum PassPhaseKind : int {
  PP_GEMM = 0,    // a projection on the tensor cores (its epilogue writes the next input)
  PP_INPUT = 1,   // NTP / MTP inputs: e * g_in, f * g_hid (+ sums of squares), residual = f
  PP_ATTN = 2,    // split-KV attention items (request, kv head, key chunk): the draft
                  // block's k / v into the cache, partials, then each item's share of the
                  // merge of its (request, kv head) -> O
  PP_NORM = 4,    // residual -> x * gamma (+ sums of squares)
  PP_ARGMAX = 5   // LM-head argmax keys -> draft tokens (d2t applied)
};

// One projection: stream-K over (128-feature tile, k-unit of PASS_KU 64-wide k-blocks)
// iterations, activation boxes of BN rows (hi rows [0,R), lo rows [R,2R) when split).
struct PassGemm {
  int Nout, Kd, R, split, additive, BN, lo_col, n_tiles, KB, Gm, phase;  // KB: k-units
  int dep;  // phase whose completion the activation operand waits for (-1: none)
  uint32_t idesc;
  long long total;
  EpiArgs epi;
};

struct PassPhase {
  int kind;
  int stage;           // PEAGLE_STAGE_* the step is reported under (timing)
  int gemm;            // PP_GEMM: index into PassParams::gemm
  int layer;           // PP_ATTN: decoder layer
  int slot;            // PP_NORM: sum-of-squares slot
  const void* gamma;   // PP_NORM: norm gain
};

// Scalars and pointers first: the kernel reads them often, the per-projection arrays at
// the end rarely (the block is ~22 KB of kernel parameters).
struct PassParams {
  int n_gemm, n_phase;
  int stages, b_stage_bytes, acc_stride, tmem_cols, uni_bytes;
  // shapes
  int B, K, R, H, split, Vt, chunk, nchunk;
  int nq, nkv, hd, cap;
  float eps;
  size_t layer_stride;
  // bounded waits: every wait of the kernel gives up after wait_ns nanoseconds (then the
  // device error word gets TIMEOUT and the CTAs leave); stall_phase >= 0 names a step whose
  // waits require one signal more than the grid gives, so that they run out (a test of
  // that path), -1 none
  unsigned long long wait_ns;
  int stall_phase;
  // library-owned buffers
  const void* embed;
  const void* emb_mask;
  const void* input_norm;
  const void* hidden_norm;
  fx_t* F;
  const fx_t* f_shared;
  void* X0;
  void* Xn;
  fx_t* res;
  fx_t* ss;              // [PASS_SS_SLOTS][R] row sums of squares (0: e, 1: f, 2..: norms)
  fx_t* q_fx;            // [R, nq*hd] fixed-point queries of the current layer
  fx_t* kv_fx;           // [R][2][nkv*hd] fixed-point keys / values of the current layer
  unsigned long long* keys;
  int* row_pos;
  const int* d2t;
  float* ws;             // stream-K partial slots
  unsigned* tile_cnt;    // per-tile contributor counters (zero between projections)
  unsigned* phase_cnt;   // [n_phase + 1]: phase completion counts, then the abort flag, then
                         // [layer][B][nkv] attention items that wrote their partials
  unsigned* err;
  unsigned long long* trace;  // timing: [0] start, [j+1] completion of phase j (ns), or null
  unsigned long long* trace_cta;  // timing: [phase][CTA][4] event times, or null
  // per call
  const int* seq_lens;
  const int* new_token;  // draft: [B] new tokens; catch-up: [B * K] tokens of the rows
  int all_ntp;           // catch-up: every row takes its own token and hidden state
  int* out_tokens;       // [R] or null
  AttnArgs att;        // per layer: kc / vc advanced by layer_stride bytes
  PassPhase ph[PASS_MAX_PHASE];
  PassGemm gemm[PASS_MAX_GEMM];
  CUtensorMap tm[2 * PASS_MAX_GEMM];  // per projection: weights, activations (PASS_KU-k-block
                                      // boxes, tc_tensor_map_ku)
};

// Bytes of dynamic shared memory the kernel needs for `stages` ring stages.
size_t pass_smem_bytes(int stages, int b_stage_bytes, int uni_bytes);
// Launches the pass on `grid` CTAs (one per SM, co-resident); PEAGLE_OK or an error code.
int pass_launch(const PassParams& P, int head_dim, int grid, cudaStream_t s);

}  // namespace peagle
