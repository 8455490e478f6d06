// Training step of the parallel-prediction forward ("P-EAGLE: Parallel-Drafting EAGLE with
// Scalable Training", A2 section 2 and section 3): the non-GEMM kernels of the forward
// with saved activations and of the backward, all on fp32 rows.  The projections and the
// prefix part of the attention are plain GEMMs (gemm_tf32.cu) issued by the host.
//
// Attention structure used throughout ("Speeding LLM inference with P-EAGLE in
// vLLM/Speculators", "Flex-attention mask"): row i = (p, d) sees the depth-1 rows at
// positions 0 .. p - d + 1 (its anchor) and the deeper members of its own chain,
// (p - t, d - t) for t = 0 .. d - 2.  The first set is a prefix of the depth-1 rows
// ordered by position, so its scores form a dense [rows x positions] matrix computed by
// GEMM and masked by the anchor; the chain holds at most K - 1 keys per row and is
// handled here per row.
#include <math.h>

#include "common.cuh"
#include "train_kernels.h"

namespace peagle {

namespace {

__device__ __forceinline__ bool row_ok(int p, int d, int n, int K) {
  return p >= 0 && p < n && d >= 1 && d <= K && p - d + 1 >= 0;
}

__device__ __forceinline__ float ld_any(const void* base, bool bf, size_t i) {
  return bf ? __bfloat162float(reinterpret_cast<const bf16*>(base)[i])
            : reinterpret_cast<const float*>(base)[i];
}

// ---- inputs -------------------------------------------------------------------------
__global__ void train_inputs_kernel(int M, int n, int K, int H, bool bf, const int* row_p,
                                    const int* row_d, const int* tokens, const void* hidden,
                                    const void* embed, int Vt, const void* emb_mask,
                                    const void* h_shared, float* E, float* Hin,
                                    unsigned* err) {
  const int i = blockIdx.x;
  const int p = row_p[i], d = row_d[i];
  const bool ok = row_ok(p, d, n, K);
  int tok = 0;
  if (ok && d == 1) {
    tok = tokens[p];
    if (tok < 0 || tok >= Vt) {
      if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_TOKEN);
      tok = -1;
    }
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float e = 0.f;
    if (ok) e = d == 1 ? (tok >= 0 ? ld_any(embed, bf, (size_t)tok * H + h) : 0.f)
                       : ld_any(emb_mask, bf, h);
    E[(size_t)i * H + h] = e;
  }
  for (int h = threadIdx.x; h < 3 * H; h += blockDim.x) {
    float x = 0.f;
    if (ok) x = d == 1 ? ld_any(hidden, bf, (size_t)p * 3 * H + h) : ld_any(h_shared, bf, h);
    Hin[(size_t)i * 3 * H + h] = x;
  }
}

// ---- RMSNorm ----------------------------------------------------------------------------
__global__ void rms_fwd_kernel(int D, const float* x, int ldx, const float* g, float eps,
                               float* y, int ldy, float* r) {
  __shared__ float red[32];
  const int i = blockIdx.x;
  const float* xr = x + (size_t)i * ldx;
  float ss = 0.f;
  for (int h = threadIdx.x; h < D; h += blockDim.x) ss += xr[h] * xr[h];
  ss = block_sum(ss, red);
  const float ri = rsqrtf(ss / D + eps);
  for (int h = threadIdx.x; h < D; h += blockDim.x) y[(size_t)i * ldy + h] = xr[h] * ri * g[h];
  if (threadIdx.x == 0 && r) r[i] = ri;
}

// dx = r z - r^3 x (z . x) / D with z = dy g (accumulated into dx when acc)
__global__ void rms_bwd_kernel(int D, const float* x, int ldx, const float* r, const float* g,
                               const float* dy, int ldy, float* dx, int lddx, int acc) {
  __shared__ float red[32];
  const int i = blockIdx.x;
  const float* xr = x + (size_t)i * ldx;
  const float* dyr = dy + (size_t)i * ldy;
  float zx = 0.f;
  for (int h = threadIdx.x; h < D; h += blockDim.x) zx += dyr[h] * g[h] * xr[h];
  zx = block_sum(zx, red);
  const float ri = r[i];
  const float c = ri * ri * ri * zx / D;
  for (int h = threadIdx.x; h < D; h += blockDim.x) {
    const float v = ri * dyr[h] * g[h] - c * xr[h];
    float* o = dx + (size_t)i * lddx + h;
    *o = acc ? *o + v : v;
  }
}

// out[h] (+)= sum over rows i of a[i][h] * (b ? b[i][h] : 1) * (rs ? rs[i] : 1), rows with
// sel (row_d) == 1 skipped when skip_depth1 is set.  Column blocks of 256, row chunks of
// 64, one atomic add per column and chunk.
__global__ void colsum_kernel(int M, int D, const float* a, int lda, const float* b, int ldb,
                              const float* rs, const int* row_d, float* out) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= D) return;
  const int i0 = blockIdx.y * 64, i1 = min(M, i0 + 64);
  float s = 0.f;
  for (int i = i0; i < i1; ++i) {
    if (row_d && row_d[i] == 1) continue;
    float v = a[(size_t)i * lda + h];
    if (b) v *= b[(size_t)i * ldb + h];
    if (rs) v *= rs[i];
    s += v;
  }
  atomicAdd(out + h, s);
}

// ---- SwiGLU (gate / up interleaved in 64-column blocks [gate 64 | up 64]) ------------
__device__ __forceinline__ int gu_col(int j, bool up) {
  return (j >> 6) * 128 + (up ? 64 : 0) + (j & 63);
}

__global__ void swiglu_fwd_kernel(int M, int I, const float* gu, float* act) {
  const size_t total = (size_t)M * I;
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total;
       t += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(t / I), j = (int)(t % I);
    const float g = gu[(size_t)i * 2 * I + gu_col(j, false)];
    const float u = gu[(size_t)i * 2 * I + gu_col(j, true)];
    act[t] = g / (1.f + expf(-g)) * u;
  }
}

// d gate = dact * up * silu'(gate), d up = dact * silu(gate); silu' = s (1 + x (1 - s))
__global__ void swiglu_bwd_kernel(int M, int I, const float* gu, const float* dact, float* dgu) {
  const size_t total = (size_t)M * I;
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total;
       t += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(t / I), j = (int)(t % I);
    const size_t cg = (size_t)i * 2 * I + gu_col(j, false), cu = (size_t)i * 2 * I + gu_col(j, true);
    const float g = gu[cg], u = gu[cu], da = dact[t];
    const float sg = 1.f / (1.f + expf(-g));
    dgu[cg] = da * u * sg * (1.f + g * (1.f - sg));
    dgu[cu] = da * g * sg;
  }
}

// [2I][H] interleaved gradient rows -> gate [I][H] and up [I][H]
__global__ void gu_split_kernel(int I, int H, const float* dw, float* dgate, float* dup) {
  const size_t total = (size_t)2 * I * H;
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total;
       t += (size_t)gridDim.x * blockDim.x) {
    const int rrow = (int)(t / H), h = (int)(t % H);
    const int blk = rrow >> 7, w = rrow & 127;
    const int j = blk * 64 + (w & 63);
    (w < 64 ? dgate : dup)[(size_t)j * H + h] = dw[t];
  }
}

// ---- RoPE (rotate-half pairs (c, c + hd/2), the table holds (cos, sin) per position) ----
// q rows -> head-major Qh [nq][M][hd]; k -> Kr [M][nkv][hd]; v -> Vr; the depth-1 rows'
// keys and values also to K1 / V1 [nkv][n][hd] by position.
// x rounded to TF32 (round to nearest, ties away), kept as fp32: the form the fused
// attention kernels' tensor-core products read their operands in
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// tf32: the queries and the depth-1 keys / values (K1, V1) are stored rounded to TF32
// (the operands of the fused attention); the all-row keys / values keep fp32
__global__ void train_rope_kernel(int M, int n, int K, int nq, int nkv, int hd, const float* qkv,
                                  const int* row_p, const int* row_d, const float2* tab,
                                  float* Qh, float* Kr, float* Vr, float* K1, float* V1,
                                  bool tf32) {
  const int i = blockIdx.x;
  const int p = row_p[i], d = row_d[i];
  const bool ok = row_ok(p, d, n, K);
  const int half = hd / 2, qkv_out = (nq + 2 * nkv) * hd;
  const float* src = qkv + (size_t)i * qkv_out;
  for (int t = threadIdx.x; t < (nq + nkv) * half; t += blockDim.x) {
    const int h = t / half, c = t % half;
    const float2 cs = ok ? tab[(size_t)p * half + c] : make_float2(1.f, 0.f);
    const float x1 = src[h * hd + c], x2 = src[h * hd + c + half];
    const float y1 = x1 * cs.x - x2 * cs.y, y2 = x2 * cs.x + x1 * cs.y;
    if (h < nq) {
      float* o = Qh + ((size_t)h * M + i) * hd;
      o[c] = tf32 ? round_tf32(y1) : y1;
      o[c + half] = tf32 ? round_tf32(y2) : y2;
    } else {
      const int g = h - nq;
      float* o = Kr + ((size_t)i * nkv + g) * hd;
      o[c] = y1;
      o[c + half] = y2;
      if (ok && d == 1) {
        float* o1 = K1 + ((size_t)g * n + p) * hd;
        o1[c] = tf32 ? round_tf32(y1) : y1;
        o1[c + half] = tf32 ? round_tf32(y2) : y2;
      }
    }
  }
  for (int t = threadIdx.x; t < nkv * hd; t += blockDim.x) {
    const float v = src[(nq + nkv) * hd + t];
    Vr[(size_t)i * nkv * hd + t] = v;
    if (ok && d == 1) V1[((size_t)(t / hd) * n + p) * hd + t % hd] = tf32 ? round_tf32(v) : v;
  }
}

// dq (head-major) and dk (rows) rotated back by the opposite angle into the fused
// gradient row dqkv [M][(nq + 2 nkv) hd]; dv copied
__global__ void train_rope_bwd_kernel(int M, int n, int K, int nq, int nkv, int hd,
                                      const float* dQh, const float* dKr, const float* dVr,
                                      const int* row_p, const int* row_d, const float2* tab,
                                      float* dqkv) {
  const int i = blockIdx.x;
  const int p = row_p[i], d = row_d[i];
  const bool ok = row_ok(p, d, n, K);
  const int half = hd / 2, qkv_out = (nq + 2 * nkv) * hd;
  float* dst = dqkv + (size_t)i * qkv_out;
  for (int t = threadIdx.x; t < (nq + nkv) * half; t += blockDim.x) {
    const int h = t / half, c = t % half;
    const float2 cs = ok ? tab[(size_t)p * half + c] : make_float2(1.f, 0.f);
    const float* s = h < nq ? dQh + ((size_t)h * M + i) * hd : dKr + ((size_t)i * nkv + h - nq) * hd;
    const float y1 = s[c], y2 = s[c + half];
    dst[h * hd + c] = y1 * cs.x + y2 * cs.y;
    dst[h * hd + c + half] = y2 * cs.x - y1 * cs.y;
  }
  for (int t = threadIdx.x; t < nkv * hd; t += blockDim.x)
    dst[(nq + nkv) * hd + t] = dVr[(size_t)i * nkv * hd + t];
}

// chain[i][t] = row of (p - t, d - t), t = 0 .. d - 2 (depths >= 2), -1 elsewhere
__global__ void chain_kernel(int M, int n, int K, int Kmax, const int* row_p, const int* row_d,
                             const int* row_index, int* chain) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M) return;
  const int p = row_p[i], d = row_d[i];
  const bool ok = row_ok(p, d, n, K);
  for (int t = 0; t < K - 1; ++t) {
    int r = -1;
    if (ok && t <= d - 2) r = row_index[(size_t)(p - t) * (Kmax + 1) + (d - t)];
    chain[(size_t)i * (K - 1) + t] = r;
  }
}

__device__ __forceinline__ int anchor_of(int p, int d, int n, int K) {
  return row_ok(p, d, n, K) ? p - d + 1 : -1;
}

// warp dot product of two hd-vectors (lane-strided)
__device__ __forceinline__ float wdot(const float* a, const float* b, int hd, int lane) {
  float s = 0.f;
  for (int c = lane; c < hd; c += 32) s += a[c] * b[c];
  return warp_sum(s);
}

// ---- attention forward: softmax over the masked prefix scores and the chain ----------
// One warp per (head of group g, row).  S1 [G][M][n] holds the scaled prefix scores; it
// becomes the probabilities (0 past the anchor).  Pc [nq][M][K-1], lse [nq][M].
__global__ void attn_fwd_softmax_kernel(TrainAttn a, int g, float* S1, const float* Qh,
                                        const float* Kr, float* Pc, float* lse) {
  const int G = a.nq / a.nkv, lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= G * a.M) return;
  const int hl = w / a.M, i = w % a.M, h = g * G + hl;
  const int K1n = a.K - 1;
  const int anc = anchor_of(a.row_p[i], a.row_d[i], a.n, a.K);
  float* srow = S1 + ((size_t)hl * a.M + i) * a.n;
  const float* q = Qh + ((size_t)h * a.M + i) * a.hd;
  float cs[16];
  float m = -INFINITY;
  for (int t = 0; t < K1n; ++t) {
    const int r = a.chain[(size_t)i * K1n + t];
    cs[t] = r >= 0 ? wdot(q, Kr + ((size_t)r * a.nkv + g) * a.hd, a.hd, lane) * a.scale : -INFINITY;
    m = fmaxf(m, cs[t]);
  }
  for (int j = lane; j <= anc; j += 32) m = fmaxf(m, srow[j]);
  m = warp_max(m);
  float l = 0.f;
  for (int j = lane; j <= anc; j += 32) l += expf(srow[j] - m);
  l = warp_sum(l);
  for (int t = 0; t < K1n; ++t) l += cs[t] > -INFINITY ? expf(cs[t] - m) : 0.f;
  const float L = (anc >= 0 || l > 0.f) ? m + logf(l) : 0.f;
  for (int j = lane; j < a.n; j += 32) srow[j] = j <= anc ? expf(srow[j] - L) : 0.f;
  if (lane < K1n)
    Pc[((size_t)h * a.M + i) * K1n + lane] = cs[lane] > -INFINITY ? expf(cs[lane] - L) : 0.f;
  if (lane == 0) lse[(size_t)h * a.M + i] = L;
}

// O rows [M][nq hd] of group g's heads: the prefix product Oh (head-major) plus the chain
__global__ void attn_fwd_out_kernel(TrainAttn a, int g, const float* Oh, const float* Pc,
                                    const float* Vr, float* O) {
  const int G = a.nq / a.nkv, K1n = a.K - 1;
  const int w = blockIdx.x;  // (head of group, row)
  const int hl = w / a.M, i = w % a.M, h = g * G + hl;
  for (int c = threadIdx.x; c < a.hd; c += blockDim.x) {
    float o = Oh[((size_t)h * a.M + i) * a.hd + c];
    for (int t = 0; t < K1n; ++t) {
      const int r = a.chain[(size_t)i * K1n + t];
      if (r >= 0) o += Pc[((size_t)h * a.M + i) * K1n + t] * Vr[((size_t)r * a.nkv + g) * a.hd + c];
    }
    O[(size_t)i * a.nq * a.hd + h * a.hd + c] = o;
  }
}

// ---- attention backward ------------------------------------------------------------
// Dv[h][i] = dO . O (the softmax backward's row term), dOh head-major copy of dO
// tf32: dOh is stored rounded to TF32 (D uses the fp32 values)
__global__ void attn_bwd_prep_kernel(TrainAttn a, const float* dO, const float* O, float* dOh,
                                     float* Dv, bool tf32) {
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= a.nq * a.M) return;
  const int h = w / a.M, i = w % a.M;
  const size_t src = (size_t)i * a.nq * a.hd + h * a.hd;
  float s = 0.f;
  for (int c = lane; c < a.hd; c += 32) {
    const float x = dO[src + c];
    dOh[((size_t)h * a.M + i) * a.hd + c] = tf32 ? round_tf32(x) : x;
    s += x * O[src + c];
  }
  s = warp_sum(s);
  if (lane == 0) Dv[(size_t)h * a.M + i] = s;
}

// One warp per (head of group g, row): the prefix probabilities P1 = exp(S1 - lse) (in
// place over the recomputed scores) and dS1 = P1 (dP1 - D) scale (in place over dP1),
// unless S1 is null; the chain's scores, probabilities and dS give dQh's initial value
// (the prefix part is added after: the GEMM dS1 K1 or the fused dQ kernel) and are added
// into the chain rows' dK / dV.
__global__ void attn_bwd_ds_kernel(TrainAttn a, int g, float* S1, float* dP1, const float* lse,
                                   const float* Dv, const float* Qh, const float* Kr,
                                   const float* Vr, const float* dOh, float* dQh, float* dKr,
                                   float* dVr) {
  const int G = a.nq / a.nkv, lane = threadIdx.x & 31, K1n = a.K - 1;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= G * a.M) return;
  const int hl = w / a.M, i = w % a.M, h = g * G + hl;
  const int anc = anchor_of(a.row_p[i], a.row_d[i], a.n, a.K);
  const float L = lse[(size_t)h * a.M + i], D = Dv[(size_t)h * a.M + i];
  if (S1) {  // without the dense matrices the fused kernels handle the prefix
    float* srow = S1 + ((size_t)hl * a.M + i) * a.n;
    float* drow = dP1 + ((size_t)hl * a.M + i) * a.n;
    for (int j = lane; j < a.n; j += 32) {
      float pr = 0.f, ds = 0.f;
      if (j <= anc) {
        pr = expf(srow[j] - L);
        ds = pr * (drow[j] - D) * a.scale;
      }
      srow[j] = pr;
      drow[j] = ds;
    }
  }
  const float* q = Qh + ((size_t)h * a.M + i) * a.hd;
  const float* dO = dOh + ((size_t)h * a.M + i) * a.hd;
  float* dq = dQh + ((size_t)h * a.M + i) * a.hd;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // head_dim <= 128: four dims per lane
  for (int t = 0; t < K1n; ++t) {
    const int r = a.chain[(size_t)i * K1n + t];
    if (r < 0) continue;  // warp-uniform
    const float* kr = Kr + ((size_t)r * a.nkv + g) * a.hd;
    const float* vr = Vr + ((size_t)r * a.nkv + g) * a.hd;
    const float s = wdot(q, kr, a.hd, lane) * a.scale;
    const float pr = expf(s - L);
    const float dp = wdot(dO, vr, a.hd, lane);
    const float ds = pr * (dp - D) * a.scale;
    for (int c = lane, u = 0; c < a.hd; c += 32, ++u) {
      acc[u] += ds * kr[c];
      atomicAdd(dKr + ((size_t)r * a.nkv + g) * a.hd + c, ds * q[c]);
      atomicAdd(dVr + ((size_t)r * a.nkv + g) * a.hd + c, pr * dO[c]);
    }
  }
  for (int c = lane, u = 0; c < a.hd; c += 32, ++u) dq[c] = acc[u];
}

// The chain part of the backward when the prefix part runs on the fused kernels: one
// warp per (kv head g, row i) walks the G q heads of the group; per head the chain keys'
// scores are recomputed, dQ's chain part is stored (the prefix part is added later), and
// each chain key's dK / dV is summed over the G heads in registers before one atomic add
// per element (G times fewer atomics than one warp per head).
template <int HD>
__global__ void __launch_bounds__(256) attn_bwd_chain_kernel(TrainAttn a, const float* lse,
                                                             const float* Dv, const float* Qh,
                                                             const float* Kr, const float* Vr,
                                                             const float* dOh, float* dQh,
                                                             float* dKr, float* dVr) {
  constexpr int U = HD / 32;
  constexpr int CMAX = 15;  // K <= 16: at most 15 chain keys per row
  const int G = a.nq / a.nkv, lane = threadIdx.x & 31, K1n = a.K - 1;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= a.nkv * a.M) return;
  const int g = w / a.M, i = w - g * a.M;
  int rr[CMAX];
  float dk[CMAX][U], dv[CMAX][U];
#pragma unroll
  for (int t = 0; t < CMAX; ++t) {
    rr[t] = t < K1n ? a.chain[(size_t)i * K1n + t] : -1;
#pragma unroll
    for (int u = 0; u < U; ++u) dk[t][u] = dv[t][u] = 0.f;
  }
  for (int hl = 0; hl < G; ++hl) {
    const int h = g * G + hl;
    const float L = lse[(size_t)h * a.M + i], D = Dv[(size_t)h * a.M + i];
    const float* qrow = Qh + ((size_t)h * a.M + i) * HD;
    const float* orow = dOh + ((size_t)h * a.M + i) * HD;
    float q[U], o[U], dq[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      q[u] = qrow[lane + 32 * u];
      o[u] = orow[lane + 32 * u];
      dq[u] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < CMAX; ++t) {
      if (rr[t] < 0) continue;  // warp-uniform
      const float* kr = Kr + ((size_t)rr[t] * a.nkv + g) * HD;
      const float* vr = Vr + ((size_t)rr[t] * a.nkv + g) * HD;
      float k[U], v[U], sd = 0.f, dd = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        k[u] = kr[lane + 32 * u];
        v[u] = vr[lane + 32 * u];
        sd += q[u] * k[u];
        dd += o[u] * v[u];
      }
      const float pr = expf(warp_sum(sd) * a.scale - L);
      const float ds = pr * (warp_sum(dd) - D) * a.scale;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        dq[u] += ds * k[u];
        dk[t][u] += ds * q[u];
        dv[t][u] += pr * o[u];
      }
    }
    float* dqrow = dQh + ((size_t)h * a.M + i) * HD;
#pragma unroll
    for (int u = 0; u < U; ++u) dqrow[lane + 32 * u] = dq[u];
  }
#pragma unroll
  for (int t = 0; t < CMAX; ++t) {
    if (rr[t] < 0) continue;
    float* gk = dKr + ((size_t)rr[t] * a.nkv + g) * HD;
    float* gv = dVr + ((size_t)rr[t] * a.nkv + g) * HD;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      atomicAdd(gk + lane + 32 * u, dk[t][u]);
      atomicAdd(gv + lane + 32 * u, dv[t][u]);
    }
  }
}

// dK1 / dV1 [nkv][n][hd] (by position) added into the depth-1 rows' dKr / dVr
__global__ void kv1_scatter_kernel(int M, int n, int K, int nkv, int hd, const int* row_p,
                                   const int* row_d, const float* dK1, const float* dV1,
                                   float* dKr, float* dVr) {
  const int i = blockIdx.x;
  const int p = row_p[i], d = row_d[i];
  if (!row_ok(p, d, n, K) || d != 1) return;
  for (int t = threadIdx.x; t < nkv * hd; t += blockDim.x) {
    const int g = t / hd, c = t % hd;
    dKr[(size_t)i * nkv * hd + t] += dK1[((size_t)g * n + p) * hd + c];
    dVr[(size_t)i * nkv * hd + t] += dV1[((size_t)g * n + p) * hd + c];
  }
}

// ---- loss ---------------------------------------------------------------------------
// Per row: lse of the logits, loss_i = lse - logit[label]; the logits become
// dlogits = (softmax - onehot) / M.
__global__ void ce_kernel(int M, int V, float* logits, const int* labels, float* row_loss,
                          unsigned* err) {
  __shared__ float red[32];
  const int i = blockIdx.x;
  float* x = logits + (size_t)i * V;
  float m = -INFINITY;
  for (int j = threadIdx.x; j < V; j += blockDim.x) m = fmaxf(m, x[j]);
  {
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    const float t = ((threadIdx.x & 31) < (blockDim.x >> 5)) ? red[threadIdx.x & 31] : -INFINITY;
    m = warp_max(t);
    __syncthreads();  // red is reused by block_sum
  }
  float s = 0.f;
  for (int j = threadIdx.x; j < V; j += blockDim.x) s += expf(x[j] - m);
  s = block_sum(s, red);
  const float L = m + logf(s);
  int lab = labels[i];
  if (lab < 0 || lab >= V) {
    if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_TOKEN);
    lab = -1;
  }
  const float xl = lab >= 0 ? x[lab] : L;
  __syncthreads();
  for (int j = threadIdx.x; j < V; j += blockDim.x)
    x[j] = (expf(x[j] - L) - (j == lab ? 1.f : 0.f)) / M;
  if (threadIdx.x == 0) row_loss[i] = L - xl;
}

// The same with the row held in registers (V <= 32 * 1024, V % 4 == 0): one pass over the
// logits from memory and one over the result, 1024 threads per row, 8 float4 per thread.
__global__ void __launch_bounds__(1024, 1) ce_reg_kernel(int M, int V, float* logits,
                                                         const int* labels, float* row_loss,
                                                         unsigned* err) {
  constexpr int PER = 8;
  __shared__ float red[32];
  const int i = blockIdx.x;
  float4* x = reinterpret_cast<float4*>(logits + (size_t)i * V);
  const int V4 = V / 4;
  float4 v[PER];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int j = threadIdx.x + k * 1024;
    v[k] = j < V4 ? x[j] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    m = fmaxf(m, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
  }
  {
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = warp_max(red[threadIdx.x & 31]);
    __syncthreads();  // red is reused by block_sum
  }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k)
    sum += (expf(v[k].x - m) + expf(v[k].y - m)) + (expf(v[k].z - m) + expf(v[k].w - m));
  sum = block_sum(sum, red);
  const float L = m + logf(sum);
  int lab = labels[i];
  if (lab < 0 || lab >= V) {
    if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_TOKEN);
    lab = -1;
  }
  const float inv = 1.f / M;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int j = threadIdx.x + k * 1024;
    if (j >= V4) continue;
    const int e = 4 * j;
    float4 o;
    o.x = (expf(v[k].x - L) - (e == lab ? 1.f : 0.f)) * inv;
    o.y = (expf(v[k].y - L) - (e + 1 == lab ? 1.f : 0.f)) * inv;
    o.z = (expf(v[k].z - L) - (e + 2 == lab ? 1.f : 0.f)) * inv;
    o.w = (expf(v[k].w - L) - (e + 3 == lab ? 1.f : 0.f)) * inv;
    if (lab >= e && lab < e + 4) {
      const float xl = lab == e ? v[k].x : lab == e + 1 ? v[k].y : lab == e + 2 ? v[k].z : v[k].w;
      row_loss[i] = L - xl;
    }
    x[j] = o;
  }
  if (lab < 0 && threadIdx.x == 0) row_loss[i] = 0.f;
}

__global__ void mean_kernel(int M, const float* v, float* out) {
  __shared__ float red[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < M; i += blockDim.x) s += v[i];
  s = block_sum(s, red);
  if (threadIdx.x == 0) *out = s / M;
}

// ---- input gradients -----------------------------------------------------------------
// depth-1 rows add their embedding gradient into the token's row
__global__ void embed_grad_kernel(int M, int n, int K, int H, int Vt, const int* row_p,
                                  const int* row_d, const int* tokens, const float* dE,
                                  float* dembed) {
  const int i = blockIdx.x;
  const int p = row_p[i], d = row_d[i];
  if (!row_ok(p, d, n, K) || d != 1) return;
  const int tok = tokens[p];
  if (tok < 0 || tok >= Vt) return;
  for (int h = threadIdx.x; h < H; h += blockDim.x)
    atomicAdd(dembed + (size_t)tok * H + h, dE[(size_t)i * H + h]);
}

__global__ void to_f32_kernel(size_t n, const bf16* src, float* dst) {
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n;
       t += (size_t)gridDim.x * blockDim.x)
    dst[t] = __bfloat162float(src[t]);
}

__global__ void add_kernel(size_t n, const float* a, float* b) {
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n;
       t += (size_t)gridDim.x * blockDim.x)
    b[t] += a[t];
}

unsigned grid_for(size_t n) {
  const size_t b = (n + 255) / 256;
  return (unsigned)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

}  // namespace

void launch_train_inputs(bool bf, int M, int n, int K, int H, const int* row_p,
                         const int* row_d, const int* tokens, const void* hidden,
                         const void* embed, int Vt, const void* emb_mask, const void* h_shared,
                         float* E, float* Hin, unsigned* err, cudaStream_t s) {
  train_inputs_kernel<<<M, 256, 0, s>>>(M, n, K, H, bf, row_p, row_d, tokens, hidden, embed, Vt,
                                        emb_mask, h_shared, E, Hin, err);
}

void launch_rms_fwd(int M, int D, const float* x, int ldx, const float* g, float eps, float* y,
                    int ldy, float* r, cudaStream_t s) {
  rms_fwd_kernel<<<M, 256, 0, s>>>(D, x, ldx, g, eps, y, ldy, r);
}

void launch_rms_bwd(int M, int D, const float* x, int ldx, const float* r, const float* g,
                    const float* dy, int ldy, float* dx, int lddx, bool acc, cudaStream_t s) {
  rms_bwd_kernel<<<M, 256, 0, s>>>(D, x, ldx, r, g, dy, ldy, dx, lddx, acc ? 1 : 0);
}

void launch_colsum(int M, int D, const float* a, int lda, const float* b, int ldb,
                   const float* rs, const int* skip_depth1_rows, float* out, cudaStream_t s) {
  colsum_kernel<<<dim3(cdiv(D, 256), cdiv(M, 64)), 256, 0, s>>>(M, D, a, lda, b, ldb, rs,
                                                                skip_depth1_rows, out);
}

void launch_swiglu_fwd(int M, int I, const float* gu, float* act, cudaStream_t s) {
  swiglu_fwd_kernel<<<grid_for((size_t)M * I), 256, 0, s>>>(M, I, gu, act);
}

void launch_swiglu_bwd(int M, int I, const float* gu, const float* dact, float* dgu,
                       cudaStream_t s) {
  swiglu_bwd_kernel<<<grid_for((size_t)M * I), 256, 0, s>>>(M, I, gu, dact, dgu);
}

void launch_gu_split(int I, int H, const float* dw, float* dgate, float* dup, cudaStream_t s) {
  gu_split_kernel<<<grid_for((size_t)2 * I * H), 256, 0, s>>>(I, H, dw, dgate, dup);
}

void launch_train_rope(int M, int n, int K, int nq, int nkv, int hd, const float* qkv,
                       const int* row_p, const int* row_d, const float2* tab, float* Qh,
                       float* Kr, float* Vr, float* K1, float* V1, bool tf32, cudaStream_t s) {
  train_rope_kernel<<<M, 128, 0, s>>>(M, n, K, nq, nkv, hd, qkv, row_p, row_d, tab, Qh, Kr, Vr,
                                      K1, V1, tf32);
}

void launch_train_rope_bwd(int M, int n, int K, int nq, int nkv, int hd, const float* dQh,
                           const float* dKr, const float* dVr, const int* row_p,
                           const int* row_d, const float2* tab, float* dqkv, cudaStream_t s) {
  train_rope_bwd_kernel<<<M, 128, 0, s>>>(M, n, K, nq, nkv, hd, dQh, dKr, dVr, row_p, row_d, tab,
                                          dqkv);
}

void launch_chain(int M, int n, int K, int Kmax, const int* row_p, const int* row_d,
                  const int* row_index, int* chain, cudaStream_t s) {
  chain_kernel<<<cdiv(M, 256), 256, 0, s>>>(M, n, K, Kmax, row_p, row_d, row_index, chain);
}

void launch_attn_fwd_softmax(const TrainAttn& a, int g, float* S1, const float* Qh,
                             const float* Kr, float* Pc, float* lse, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  attn_fwd_softmax_kernel<<<cdiv(G * a.M, 8), 256, 0, s>>>(a, g, S1, Qh, Kr, Pc, lse);
}

void launch_attn_fwd_out(const TrainAttn& a, int g, const float* Oh, const float* Pc,
                         const float* Vr, float* O, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  attn_fwd_out_kernel<<<G * a.M, 64, 0, s>>>(a, g, Oh, Pc, Vr, O);
}

void launch_attn_bwd_prep(const TrainAttn& a, const float* dO, const float* O, float* dOh,
                          float* Dv, bool tf32, cudaStream_t s) {
  attn_bwd_prep_kernel<<<cdiv(a.nq * a.M, 8), 256, 0, s>>>(a, dO, O, dOh, Dv, tf32);
}

void launch_attn_bwd_ds(const TrainAttn& a, int g, float* S1, float* dP1, const float* lse,
                        const float* Dv, const float* Qh, const float* Kr, const float* Vr,
                        const float* dOh, float* dQh, float* dKr, float* dVr, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  attn_bwd_ds_kernel<<<cdiv(G * a.M, 8), 256, 0, s>>>(a, g, S1, dP1, lse, Dv, Qh, Kr, Vr, dOh,
                                                      dQh, dKr, dVr);
}

bool launch_attn_bwd_chain(const TrainAttn& a, const float* lse, const float* Dv,
                           const float* Qh, const float* Kr, const float* Vr, const float* dOh,
                           float* dQh, float* dKr, float* dVr, cudaStream_t s) {
  if (a.K > 16 || (a.hd != 64 && a.hd != 128)) return false;
  const int blocks = cdiv(a.nkv * a.M, 8);
  if (a.hd == 64)
    attn_bwd_chain_kernel<64><<<blocks, 256, 0, s>>>(a, lse, Dv, Qh, Kr, Vr, dOh, dQh, dKr, dVr);
  else
    attn_bwd_chain_kernel<128><<<blocks, 256, 0, s>>>(a, lse, Dv, Qh, Kr, Vr, dOh, dQh, dKr, dVr);
  return true;
}

void launch_kv1_scatter(int M, int n, int K, int nkv, int hd, const int* row_p, const int* row_d,
                        const float* dK1, const float* dV1, float* dKr, float* dVr,
                        cudaStream_t s) {
  kv1_scatter_kernel<<<M, 128, 0, s>>>(M, n, K, nkv, hd, row_p, row_d, dK1, dV1, dKr, dVr);
}

void launch_ce(int M, int V, float* logits, const int* labels, float* row_loss, float* loss,
               unsigned* err, cudaStream_t s) {
  if (V % 4 == 0 && V <= 32 * 1024)
    ce_reg_kernel<<<M, 1024, 0, s>>>(M, V, logits, labels, row_loss, err);
  else
    ce_kernel<<<M, 256, 0, s>>>(M, V, logits, labels, row_loss, err);
  mean_kernel<<<1, 1024, 0, s>>>(M, row_loss, loss);
}

void launch_embed_grad(int M, int n, int K, int H, int Vt, const int* row_p, const int* row_d,
                       const int* tokens, const float* dE, float* dembed, cudaStream_t s) {
  embed_grad_kernel<<<M, 256, 0, s>>>(M, n, K, H, Vt, row_p, row_d, tokens, dE, dembed);
}

void launch_to_f32(size_t n, const void* src_bf16, float* dst, cudaStream_t s) {
  to_f32_kernel<<<grid_for(n), 256, 0, s>>>(n, (const bf16*)src_bf16, dst);
}

void launch_add(size_t n, const float* a, float* b, cudaStream_t s) {
  add_kernel<<<grid_for(n), 256, 0, s>>>(n, a, b);
}

}  // namespace peagle
