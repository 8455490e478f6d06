// CUDA-core kernels of the P-EAGLE draft pass: input fusion, RMSNorm, split-KV decode
// attention with the causal draft block, the training-style masked attention, greedy
// verification, KV commit, argmax decode, and the fp32 FFMA GEMM used by the fp32
// drafter (whose 1e-4 logit tolerance rules out TF32 tensor cores).
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "kernels.h"
#include "attn_decode.cuh"
#include "tc_ptx.cuh"

namespace peagle {

// =====================================================================================
// FFMA GEMM (fp32 path): one warp per output feature, lanes split the reduction.
// =====================================================================================
template <typename T>
__device__ __forceinline__ void load4(const T* p, float* v);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* v) {
  float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <>
__device__ __forceinline__ void load4<bf16>(const bf16* p, float* v) {
  uint2 t = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&t.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&t.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  v[0] = fa.x; v[1] = fa.y; v[2] = fb.x; v[3] = fb.y;
}

// A 16-byte piece as fp32: 8 bf16 or 4 floats.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& q, float* v);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& q, float* v) {
  v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
  v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
}
template <>
__device__ __forceinline__ void unpack16<bf16>(const uint4& q, float* v) {
  const unsigned w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ W,
                                                        const T* __restrict__ X, int ldx,
                                                        float* __restrict__ Y, int ldy,
                                                        int Nout, int Kd, int R) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * 8 + warp;
  if (m >= Nout) return;
  const T* w = W + (size_t)m * Kd;
  for (int r0 = 0; r0 < R; r0 += 8) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int k = lane * 4; k < Kd; k += 128) {
      float wv[4];
      load4<T>(w + k, wv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (r0 + i < R) {
          float xv[4];
          load4<T>(X + (size_t)(r0 + i) * ldx + k, xv);
          acc[i] = fmaf(wv[0], xv[0], acc[i]);
          acc[i] = fmaf(wv[1], xv[1], acc[i]);
          acc[i] = fmaf(wv[2], xv[2], acc[i]);
          acc[i] = fmaf(wv[3], xv[3], acc[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float s = warp_sum(acc[i]);
      if (lane == 0 && r0 + i < R) Y[(size_t)(r0 + i) * ldy + m] = s;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) epilogue_kernel(const float* __restrict__ Y, int ldy,
                                                       EpiArgs a) {
  const int m0 = blockIdx.x * 128;
  epilogue_tile<T>(a, Y + m0, ldy, a.in_split ? a.R : -1, m0, 0, a.R, threadIdx.x, blockDim.x);
}

void launch_gemm_simt(bool bf16m, const void* W, const void* X, int ldx, float* Y, int ldy,
                      int Nout, int Kd, int R, const EpiArgs& epi, cudaStream_t s) {
  (void)bf16m;  // fp32 drafters only: bf16 projections run on the tensor cores
  dim3 g(cdiv(Nout, 8));
  gemm_simt_kernel<float><<<g, 256, 0, s>>>((const float*)W, (const float*)X, ldx, Y, ldy, Nout, Kd, R);
  dim3 ge(cdiv(Nout, 128));
  epilogue_kernel<float><<<ge, 256, 0, s>>>(Y, ldy, epi);
}

// =====================================================================================
// Input fusion: row inputs of the NTP / MTP positions and the 2H first-layer input.
//   mode 0 (draft pass): row r = b*K + j; j == 0 -> (embed[tokens[b]], F[b]);
//                        j >= 1 -> (emb_mask, f_shared)
//   mode 1 (training forward): row r = (p, d); d == 1 -> (embed[tokens[p]], F[p]);
//                        d >= 2 -> (emb_mask, f_shared)
// X0[r] = [RMSNorm(e) * g_in || RMSNorm(f) * g_hid]; res[r] = f; keys[r] = 0.
// F (the fc output, fixed point) is cleared after use so the next fc launch can
// accumulate into it; each F row is read by exactly one CTA.
// =====================================================================================
constexpr int ROW_THREADS = 512;  // one CTA per row; each thread keeps NPT row elements

template <typename T, int NPT>
__global__ void __launch_bounds__(ROW_THREADS) input_fusion_kernel(
    int mode, int K, int n_src, int H, const T* __restrict__ embed, int Vt,
    const T* __restrict__ emb_mask,
    fx_t* __restrict__ F, const fx_t* __restrict__ f_shared, const int* __restrict__ tokens,
    const int* __restrict__ row_p, const int* __restrict__ row_d, const T* __restrict__ g_in,
    const T* __restrict__ g_hid, float eps, int split, T* __restrict__ X0,
    fx_t* __restrict__ res, unsigned long long* __restrict__ keys, const int* __restrict__ seq_lens,
    int* __restrict__ row_pos_out, unsigned* err) {
  __shared__ float red[32];
  pdl_enter();
  const int r = blockIdx.x;
  const int R = gridDim.x;
  bool ntp;
  int src;  // request (mode 0) or position (mode 1)
  if (mode == 0) {
    src = r / K;
    ntp = (r - src * K) == 0;
  } else if (mode == 2) {  // catch-up: row r has its own token and fc row
    src = r;
    ntp = true;
  } else {
    src = row_p[r];
    ntp = row_d[r] == 1;
    if (src < 0 || src >= n_src) {  // outside the contract: BAD_ROW, use the MTP inputs
      if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_ROW);
      ntp = false;
    }
  }
  const T* e;
  fx_t* f;
  if (ntp) {
    int tok = tokens[src];
    if (tok < 0 || tok >= Vt) {
      if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_TOKEN);
      tok = 0;
    }
    e = embed + (size_t)tok * H;
    f = F + (size_t)src * H;
  } else {
    e = emb_mask;
    f = const_cast<fx_t*>(f_shared);
  }
  // the whole row in registers: every load of the row is issued in one round
  float ev[NPT], gi[NPT], gh[NPT];
  fx_t fq[NPT];
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    const bool ok = i < H;
    ev[k] = ok ? ld(e + i) : 0.f;
    fq[k] = ok ? f[i] : 0;
    gi[k] = ok ? ld(g_in + i) : 0.f;
    gh[k] = ok ? ld(g_hid + i) : 0.f;
  }
  float se = 0.f, sf = 0.f;
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    const float fv = from_fx(fq[k]);
    se += ev[k] * ev[k];
    sf += fv * fv;
  }
  se = block_sum(se, red);
  __syncthreads();
  sf = block_sum(sf, red);
  const float ie = rsqrtf(se / H + eps), ifv = rsqrtf(sf / H + eps);
  fx_t* rs = res + (size_t)r * H;
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i >= H) continue;
    store_act<T>(X0, 2 * H, r, R, split, i, ev[k] * ie * gi[k]);
    store_act<T>(X0, 2 * H, r, R, split, H + i, from_fx(fq[k]) * ifv * gh[k]);
    rs[i] = fq[k];
    // the fc output row of an NTP row is read only here: clear it for the next
    // accumulation (this thread's own elements, already loaded)
    if (ntp) f[i] = 0;
  }
  if (threadIdx.x == 0 && keys) keys[r] = 0ull;
  if (threadIdx.x == 0 && mode != 1 && row_pos_out) row_pos_out[r] = seq_lens[r / K] + r % K;
}

template <typename T>
static void input_fusion_dispatch(int npt, dim3 g, cudaStream_t s, int mode, int K, int n_src,
                                  int H, const T* embed, int Vt, const T* emb_mask, fx_t* F,
                                  const fx_t* f_shared, const int* tokens, const int* row_p,
                                  const int* row_d, const T* g_in, const T* g_hid, float eps,
                                  int split, T* X0, fx_t* res, unsigned long long* keys,
                                  const int* seq_lens, int* row_pos, unsigned* err) {
#define PEAGLE_IF_CASE(N)                                                                     \
  case N:                                                                                     \
    launch_pdl(input_fusion_kernel<T, N>, g, dim3(ROW_THREADS), 0, s, mode, K, n_src, H, embed, \
               Vt, emb_mask, F, f_shared, tokens, row_p, row_d, g_in, g_hid, eps, split, X0,  \
               res, keys, seq_lens, row_pos, err);                                            \
    break;
  switch (npt) {
    PEAGLE_IF_CASE(1)
    PEAGLE_IF_CASE(2)
    PEAGLE_IF_CASE(4)
    PEAGLE_IF_CASE(8)
    PEAGLE_IF_CASE(16)
    default:
      PEAGLE_IF_CASE(32)
  }
#undef PEAGLE_IF_CASE
}

static int row_npt(int H) {
  int npt = 1;
  while (npt * ROW_THREADS < H) npt <<= 1;
  return npt;
}

void launch_input_fusion(bool bf16m, int mode, int R, int K, int n_src, int H, const void* embed,
                         int Vt,
                         const void* emb_mask, fx_t* F, const fx_t* f_shared,
                         const int* tokens, const int* row_p, const int* row_d,
                         const void* g_in, const void* g_hid, float eps, int split, void* X0,
                         fx_t* res, unsigned long long* keys, const int* seq_lens, int* row_pos,
                         unsigned* err, cudaStream_t s) {
  const int npt = row_npt(H);
  if (bf16m)
    input_fusion_dispatch<bf16>(npt, dim3(R), s, mode, K, n_src, H, (const bf16*)embed, Vt,
                                (const bf16*)emb_mask, F, f_shared, tokens, row_p, row_d,
                                (const bf16*)g_in, (const bf16*)g_hid, eps, split, (bf16*)X0, res,
                                keys, seq_lens, row_pos, err);
  else
    input_fusion_dispatch<float>(npt, dim3(R), s, mode, K, n_src, H, (const float*)embed, Vt,
                                 (const float*)emb_mask, F, f_shared, tokens, row_p, row_d,
                                 (const float*)g_in, (const float*)g_hid, eps, 0, (float*)X0, res,
                                 keys, seq_lens, row_pos, err);
}

// =====================================================================================
// RMSNorm of the fp32 residual stream into the next projection's input dtype.
// =====================================================================================
template <typename T, int NPT>
__global__ void __launch_bounds__(ROW_THREADS) rmsnorm_kernel(int H, const fx_t* __restrict__ res,
                                                              const T* __restrict__ gamma,
                                                              float eps, int split,
                                                              T* __restrict__ out) {
  __shared__ float red[32];
  pdl_enter();
  const int r = blockIdx.x;
  const fx_t* x = res + (size_t)r * H;
  float v[NPT], g[NPT];
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    v[k] = i < H ? from_fx(x[i]) : 0.f;
    g[k] = i < H ? ld(gamma + i) : 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < NPT; ++k) ss += v[k] * v[k];
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / H + eps);
#pragma unroll
  for (int k = 0; k < NPT; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < H) store_act<T>(out, H, r, gridDim.x, split, i, v[k] * inv * g[k]);
  }
}

// bf16 variant with 16-byte accesses: 128 threads per row, each owning G groups of 8
// consecutive features (eight fixed-point values in, eight bf16 hi and lo parts out).
template <int G>
__global__ void __launch_bounds__(128) rmsnorm_v8_kernel(int H, const fx_t* __restrict__ res,
                                                         const bf16* __restrict__ gamma,
                                                         float eps, int split,
                                                         bf16* __restrict__ out) {
  __shared__ float red[32];
  pdl_enter();
  const int r = blockIdx.x, R = gridDim.x;
  const int ng = H >> 3;
  const longlong2* x = (const longlong2*)(res + (size_t)r * H);
  float v[G][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int gi = threadIdx.x + k * 128;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const longlong2 q = gi < ng ? x[gi * 4 + u] : make_longlong2(0, 0);
      v[k][2 * u] = from_fx(q.x);
      v[k][2 * u + 1] = from_fx(q.y);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += v[k][e] * v[k][e];
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / H + eps);
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int gi = threadIdx.x + k * 128;
    if (gi >= ng) break;
    const uint4 gw = *(const uint4*)(gamma + gi * 8);
    const bf16* gb = (const bf16*)&gw;
    uint32_t wh[4], wl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float y0 = v[k][2 * u] * inv * __bfloat162float(gb[2 * u]);
      const float y1 = v[k][2 * u + 1] * inv * __bfloat162float(gb[2 * u + 1]);
      const bf16 h0 = __float2bfloat16_rn(y0), h1 = __float2bfloat16_rn(y1);
      const bf16 l0 = __float2bfloat16_rn(y0 - __bfloat162float(h0));
      const bf16 l1 = __float2bfloat16_rn(y1 - __bfloat162float(h1));
      wh[u] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      wl[u] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    *(uint4*)(out + (size_t)r * H + gi * 8) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    if (split)
      *(uint4*)(out + (size_t)(r + R) * H + gi * 8) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
}

// Fixed-point q / k / v of one layer (the additive QKV epilogue's sums) -> fp32 queries
// [R][nq hd] and the bf16 KV cache slot row_pos[r] of request r / K; the accumulators are
// cleared for the next layer.  A row without a cache slot raises KV_OVERFLOW and keeps
// its query.  Thread = two neighbouring features of row blockIdx.y (16-byte loads; a pair
// never straddles q / k / v or a head, all widths being even).
__global__ void __launch_bounds__(256) qkv_finalize_kernel(int K, int nq, int nkv, int hd, int cap,
                                                           fx_t* q_fx, fx_t* kv_fx, float* Qf,
                                                           bf16* kc, bf16* vc,
                                                           const int* row_pos, unsigned* err) {
  pdl_enter();
  const int r = blockIdx.y;
  const int qw = nq * hd, kvw = nkv * hd;
  const int e = 2 * (int)(blockIdx.x * blockDim.x + threadIdx.x);
  if (e >= qw + 2 * kvw) return;
  if (e < qw) {
    longlong2* src = (longlong2*)(q_fx + (size_t)r * qw + e);
    const longlong2 v = *src;
    *src = make_longlong2(0, 0);
    *(float2*)(Qf + (size_t)r * qw + e) = make_float2(from_fx(v.x), from_fx(v.y));
    return;
  }
  const int rem = e - qw;  // keys [0, kvw), values [kvw, 2 kvw)
  longlong2* src = (longlong2*)(kv_fx + (size_t)r * 2 * kvw + rem);
  const longlong2 v = *src;
  *src = make_longlong2(0, 0);
  const int pos = row_pos[r];
  if (pos < 0 || pos >= cap) {
    if (rem == 0) raise_error(err, PEAGLE_DEV_KV_OVERFLOW);
    return;
  }
  const int sec = rem >= kvw ? 1 : 0, gk = rem - sec * kvw;
  const int g = gk / hd, i = gk - g * hd;
  bf16* dst = (sec ? vc : kc) + (((size_t)(r / K) * nkv + g) * cap + pos) * hd + i;
  *(__nv_bfloat162*)dst = __floats2bfloat162_rn(from_fx(v.x), from_fx(v.y));
}

void launch_qkv_finalize(int R, int K, int nq, int nkv, int hd, int cap, fx_t* q_fx, fx_t* kv_fx,
                         float* Qf, void* kc, void* vc, const int* row_pos, unsigned* err,
                         cudaStream_t s) {
  const int pairs = (nq + 2 * nkv) * hd / 2;
  launch_pdl(qkv_finalize_kernel, dim3((unsigned)cdiv(pairs, 256), (unsigned)R), dim3(256), 0, s, K,
             nq, nkv, hd, cap, q_fx, kv_fx, Qf, (bf16*)kc, (bf16*)vc, row_pos, err);
}

void launch_rmsnorm(bool bf16m, int R, int H, const fx_t* res, const void* gamma, float eps,
                    int split, void* out, cudaStream_t s) {
  if (bf16m && H % 8 == 0 && H <= 16 * 128 * 8) {
    const int G = (H / 8 + 127) / 128;
#define PEAGLE_RMS8_CASE(N)                                                              \
  case N:                                                                                \
    launch_pdl(rmsnorm_v8_kernel<N>, dim3(R), dim3(128), 0, s, H, res, (const bf16*)gamma, \
               eps, split, (bf16*)out);                                                  \
    return;
    switch (G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16) {
      PEAGLE_RMS8_CASE(2)
      PEAGLE_RMS8_CASE(4)
      PEAGLE_RMS8_CASE(8)
      PEAGLE_RMS8_CASE(16)
    }
#undef PEAGLE_RMS8_CASE
  }
  const int npt = row_npt(H);
#define PEAGLE_RMS_CASE(N)                                                                 \
  case N:                                                                                  \
    if (bf16m)                                                                             \
      launch_pdl(rmsnorm_kernel<bf16, N>, dim3(R), dim3(ROW_THREADS), 0, s, H, res,         \
                 (const bf16*)gamma, eps, split, (bf16*)out);                              \
    else                                                                                   \
      rmsnorm_kernel<float, N><<<R, ROW_THREADS, 0, s>>>(H, res, (const float*)gamma, eps, \
                                                         0, (float*)out);                  \
    break;
  switch (npt) {
    PEAGLE_RMS_CASE(1)
    PEAGLE_RMS_CASE(2)
    PEAGLE_RMS_CASE(4)
    PEAGLE_RMS_CASE(8)
    PEAGLE_RMS_CASE(16)
    default:
      PEAGLE_RMS_CASE(32)
  }
#undef PEAGLE_RMS_CASE
}

// =====================================================================================
// Split-KV decode attention with GQA and the causal draft block.
// CTA (chunk c, kv head g, request b) handles the K*G query rows that read kv head g;
// keys are cache slots [c*chunk, min((c+1)*chunk, L+K)) where L = seq_lens[b] and the
// draft rows' keys already sit in slots L .. L+K-1.  Row j sees keys 0 .. L+j.
// Each CTA writes (o, m, l) partials; the last CTA of (b, g) (atomic counter, no
// waiting) merges the partials in chunk order and writes O.
// =====================================================================================
constexpr int ATT_MAX_ROWS = 128;

template <typename T, int HD>
__global__ void __launch_bounds__(256) attn_decode_kernel(AttnArgs a) {
  constexpr int E = HD / 32;          // output dims per lane
  constexpr int RPW = ATT_MAX_ROWS / 8;  // max rows per warp
  extern __shared__ float smem[];
  pdl_enter();
  const int b = blockIdx.z, g = blockIdx.y, c = blockIdx.x;
  const int G = a.nq / a.nkv;
  const int rows = a.K * G;
  const int L = a.seq_lens[b];
  int first, total;
  attn_span(a, L, &first, &total);
  const int kbeg = first + c * a.chunk;
  if (kbeg >= total || L < 0) return;
  const int kend = min(total, kbeg + a.chunk);
  float* qs = smem;                       // [rows][HD]
  float* ks = qs + rows * HD;             // [32][HD + 1]
  float* vs = ks + 32 * (HD + 1);         // [32][HD]
  __shared__ int s_last;

  const float* qg = (const float*)a.q;
  for (int idx = threadIdx.x; idx < rows * HD; idx += blockDim.x) {
    int rr = idx / HD, d = idx - rr * HD;
    int j = rr / G, h = g * G + (rr - j * G);
    qs[idx] = qg[((size_t)(b * a.K + j) * a.nq + h) * HD + d] * a.scale;
  }
  const size_t head_off = ((size_t)b * a.nkv + g) * a.cap * HD;
  const T* kc = (const T*)a.kc + head_off;
  const T* vc = (const T*)a.vc + head_off;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m_i[RPW], l_i[RPW], o_i[RPW][E];
#pragma unroll
  for (int t = 0; t < RPW; ++t) {
    m_i[t] = -INFINITY;
    l_i[t] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o_i[t][e] = 0.f;
  }
  for (int t0 = kbeg; t0 < kend; t0 += 32) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * HD; idx += blockDim.x) {
      int kk = idx / HD, d = idx - kk * HD;
      int kp = t0 + kk;
      float kv = 0.f, vv = 0.f;
      if (kp < kend) {
        kv = ld(kc + (size_t)kp * HD + d);
        vv = ld(vc + (size_t)kp * HD + d);
      }
      ks[kk * (HD + 1) + d] = kv;
      vs[kk * HD + d] = vv;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
      const int rr = warp + 8 * t;
      if (rr >= rows) break;
      const int j = rr / G;
      const int kp = t0 + lane;
      const bool valid = kp < kend && kp <= L + j && (a.window <= 0 || kp > L + j - a.window);
      float s = 0.f;
      const float* q = qs + rr * HD;
      const float* kr = ks + lane * (HD + 1);
#pragma unroll 16
      for (int d = 0; d < HD; ++d) s = fmaf(q[d], kr[d], s);
      s = valid ? s : -INFINITY;
      const float tmax = warp_max(s);
      const float m_new = fmaxf(m_i[t], tmax);
      if (m_new == -INFINITY) continue;
      const float p = valid ? expf(s - m_new) : 0.f;
      const float corr = (m_i[t] == -INFINITY) ? 0.f : expf(m_i[t] - m_new);
      l_i[t] = l_i[t] * corr + warp_sum(p);
#pragma unroll
      for (int e = 0; e < E; ++e) o_i[t][e] *= corr;
      for (int kk = 0; kk < 32; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
        for (int e = 0; e < E; ++e) o_i[t][e] = fmaf(pk, vs[kk * HD + lane + 32 * e], o_i[t][e]);
      }
      m_i[t] = m_new;
    }
  }
  // partials: [b][g][c][rr][HD + 2]
  float* part = a.part + (((size_t)b * a.nkv + g) * a.nchunk + c) * rows * (HD + 2);
#pragma unroll
  for (int t = 0; t < RPW; ++t) {
    const int rr = warp + 8 * t;
    if (rr >= rows) break;
    float* pr = part + (size_t)rr * (HD + 2);
#pragma unroll
    for (int e = 0; e < E; ++e) pr[lane + 32 * e] = o_i[t][e];
    if (lane == 0) {
      pr[HD] = m_i[t];
      pr[HD + 1] = l_i[t];
    }
  }
  __syncthreads();
  const int nvalid = attn_nvalid(a, first, total);
  if (threadIdx.x == 0) {
    unsigned prev = atom_add_acq_rel(a.counters + b * a.nkv + g, 1u);
    s_last = (prev == (unsigned)(nvalid - 1));
  }
  __syncthreads();
  if (!s_last) return;
  attn_merge_rows<T, HD>(a, b, g, rows, nvalid, warp, rows, lane, 8);
  if (threadIdx.x == 0) a.counters[b * a.nkv + g] = 0u;
}


template <int HD>
__global__ void __launch_bounds__(256) attn_mma_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm_raw[];
  pdl_enter();
  attn_mma_item<HD, 2>(a, blockIdx.z, blockIdx.y, blockIdx.x, threadIdx.x, blockDim.x, sm_raw,
                       []() { __syncthreads(); });
}

// Merge of the split-KV partials as its own grid: warp w of CTA (x, g, b) merges query
// row 4x + w of (request b, kv head g) over the chunks in order, so the merge is spread
// over rows x heads x requests warps instead of one CTA per head.
template <typename T, int HD>
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnArgs a) {
  pdl_enter();
  const int b = blockIdx.z, g = blockIdx.y;
  const int rows = a.K * (a.nq / a.nkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = blockIdx.x * 4 + warp;
  const int L = a.seq_lens[b];
  int first, total;
  attn_span(a, L, &first, &total);
  if (rr >= rows || L < 0 || total <= first) return;
  attn_merge_rows<T, HD>(a, b, g, rows, attn_nvalid(a, first, total), rr, rr + 1, lane);
}

template <int HD>
static void attn_mma_launch(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.K * (a.nq / a.nkv);
  const int warps = (rows + 15) / 16;
  const size_t sm = (size_t)4 * MMA_KT * HD * 2;
  smem_optin((const void*)attn_mma_kernel<HD>, 100 * 1024);
  dim3 grid(a.nchunk, a.nkv, a.B);
  launch_pdl(attn_mma_kernel<HD>, grid, dim3(32 * warps), sm, s, a);
  launch_pdl(attn_merge_kernel<bf16, HD>, dim3(cdiv(rows, 4), a.nkv, a.B), dim3(128), 0, s, a);
}

template <typename T, int HD>
static void attn_launch(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.K * (a.nq / a.nkv);
  size_t sm = (size_t)(rows * HD + 32 * (HD + 1) + 32 * HD) * sizeof(float);
  smem_optin((const void*)attn_decode_kernel<T, HD>, 200 * 1024);
  dim3 grid(a.nchunk, a.nkv, a.B);
  launch_pdl(attn_decode_kernel<T, HD>, grid, dim3(256), sm, s, a);
}

void launch_attention_decode(bool bf16m, const AttnArgs& a, cudaStream_t s) {
  if (bf16m) {
    if (a.hd == 64) attn_mma_launch<64>(a, s); else attn_mma_launch<128>(a, s);
  } else {
    if (a.hd == 64) attn_launch<float, 64>(a, s); else attn_launch<float, 128>(a, s);
  }
}

// =====================================================================================
// Training-style masked attention (one warp per (row, q head)).  Keys of row (p, d):
// the depth-1 rows at positions 0 .. p-d+1 (gathered by position into k1/v1) and its
// chain rows (p-j, d-j), j = 0 .. d-2 (looked up in row_index).
// =====================================================================================
template <typename T, int HD>
__global__ void __launch_bounds__(256) masked_attn_kernel(MaskedAttnArgs a) {
  constexpr int E = HD / 32;
  __shared__ float qs[8][HD];
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long gw = (long)blockIdx.x * 8 + warp;
  if (gw >= (long)a.M * a.nq) return;
  const int i = (int)(gw / a.nq), h = (int)(gw - (long)i * a.nq);
  const int G = a.nq / a.nkv, g = h / G;
  const int p = a.row_p[i], d = a.row_d[i];
  const int anchor = p - d + 1;
  if (p < 0 || p >= a.n || d < 1 || d > a.Kmax || anchor < 0) {
    for (int t = lane; t < HD; t += 32)
      store_act<T>((T*)a.o, (size_t)a.nq * HD, i, a.M, a.split, h * HD + t, 0.f);
    return;  // outside the contract (reported as BAD_ROW by the row check)
  }
  const float* q = (const float*)a.q + ((size_t)i * a.nq + h) * HD;
  for (int t = lane; t < HD; t += 32) qs[warp][t] = q[t] * a.scale;
  __syncwarp();
  const int n_base = (anchor >= 0) ? anchor + 1 : 0;
  const int n_keys = n_base + max(d - 1, 0);
  float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  const T* K1 = (const T*)a.k1;
  const T* V1 = (const T*)a.v1;
  const T* KA = (const T*)a.k;
  const T* VA = (const T*)a.v;
  for (int t0 = 0; t0 < n_keys; t0 += 32) {
    const int kk = t0 + lane;
    const T* kr = nullptr;
    bool valid = kk < n_keys;
    if (valid) {
      if (kk < n_base) {
        kr = K1 + ((size_t)kk * a.nkv + g) * HD;
      } else {
        const int jj = kk - n_base;  // chain row (p - jj, d - jj), jj = 0 .. d-2
        const int ri = a.row_index[(size_t)(p - jj) * (a.Kmax + 1) + (d - jj)];
        if (ri < 0) valid = false; else kr = KA + ((size_t)ri * a.nkv + g) * HD;
      }
    }
    float s = -INFINITY;
    if (valid) {
      s = 0.f;
#pragma unroll 16
      for (int t = 0; t < HD; ++t) s = fmaf(qs[warp][t], ld(kr + t), s);
    }
    const float tmax = warp_max(s);
    const float m_new = fmaxf(m, tmax);
    if (m_new == -INFINITY) continue;
    const float pr = valid ? expf(s - m_new) : 0.f;
    const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
    l = l * corr + warp_sum(pr);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= corr;
    const int cnt = min(32, n_keys - t0);
    for (int u = 0; u < cnt; ++u) {
      const float pu = __shfl_sync(0xffffffffu, pr, u);
      const int ku = t0 + u;
      const T* vr;
      if (ku < n_base) {
        vr = V1 + ((size_t)ku * a.nkv + g) * HD;
      } else {
        const int jj = ku - n_base;
        const int ri = a.row_index[(size_t)(p - jj) * (a.Kmax + 1) + (d - jj)];
        if (ri < 0) continue;
        vr = VA + ((size_t)ri * a.nkv + g) * HD;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf(pu, ld(vr + lane + 32 * e), o[e]);
    }
    m = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e)
    store_act<T>((T*)a.o, (size_t)a.nq * HD, i, a.M, a.split, h * HD + lane + 32 * e, o[e] * inv);
}

// =====================================================================================
// Training-style masked attention on tensor cores (mma.sync m16n8k16, bf16 hi/lo parts
// of Q and P, fp32 accumulation, online softmax in the log2 domain).  A CTA serves a
// block of MASK_QROWS(G) consecutive rows for kv head g; its 64 MMA rows are the
// (row, q head of group g) pairs.  Keys arrive as two runs of 64-key tiles:
//   A  depth-1 rows by position, 0 .. the largest anchor p-d+1 of the block; row i sees
//      position p' when p' <= p_i - d_i + 1
//   B  all rows from the first row at position (smallest anchor + 1) to the block's
//      last row; row i sees row (p', d') when d' >= 2, p' - d' = p_i - d_i, d' <= d_i
//      (its chain rows (p_i - j, d_i - j), itself included)
// Together the two runs hold every key the mask allows, each once (a depth-1 key is
// only ever seen through run A).  Blocks run last-first: later rows have the longest
// prefixes, so the long CTAs start in the first wave.
// =====================================================================================
constexpr int MASK_MMA_ROWS = 64;  // 4 warps x 16

template <int HD>
__global__ void __launch_bounds__(128) masked_attn_mma_kernel(MaskedAttnArgs a) {
  constexpr int ROWB = HD * 2;
  constexpr int CH = ROWB / 16;
  constexpr int TILEB = MMA_KT * ROWB;
  constexpr int ND = HD / 8;
  constexpr int KS = HD / 16;
  extern __shared__ __align__(128) uint8_t sm_raw[];
  __shared__ int s_kp[2][MMA_KT], s_kd[2][MMA_KT];
  __shared__ int s_aend, s_amin, s_jb0;
  pdl_enter();
  const int G = a.nq / a.nkv;
  const int QR = MASK_MMA_ROWS / G;
  const int i0 = (int)(gridDim.x - 1 - blockIdx.x) * QR;
  const int g = blockIdx.y;
  const int iend = min(a.M, i0 + QR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  auto row_ok = [&](int p, int d) {
    return p >= 0 && p < a.n && d >= 1 && d <= a.Kmax && p - d + 1 >= 0;
  };
  if (threadIdx.x == 0) {
    s_aend = -1;
    s_amin = 0x7fffffff;
  }
  __syncthreads();
  if ((int)threadIdx.x < iend - i0) {
    const int p = a.row_p[i0 + threadIdx.x], d = a.row_d[i0 + threadIdx.x];
    if (row_ok(p, d)) {
      atomicMax(&s_aend, p - d + 1);
      atomicMin(&s_amin, p - d + 1);
    }
  }
  __syncthreads();
  const int a_end = s_aend;
  if (threadIdx.x == 0) {
    // run B starts at the first row whose position exceeds the smallest anchor
    // (rows are p-major; a violated order is reported by the row check and only
    // changes which in-range rows are read)
    int lo = 0, hi = iend;
    const int P0 = s_amin + 1;
    if (a_end >= 0) {
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a.row_p[mid] < P0) lo = mid + 1; else hi = mid;
      }
    } else {
      lo = iend;
    }
    s_jb0 = lo;
  }
  __syncthreads();
  const int jb0 = s_jb0;
  const int ntA = a_end >= 0 ? a_end / MMA_KT + 1 : 0;
  const int ntB = (iend - jb0 + MMA_KT - 1) / MMA_KT;
  const int ntile = ntA + ntB;

  const bf16* K1 = (const bf16*)a.k1 + (size_t)g * HD;
  const bf16* V1 = (const bf16*)a.v1 + (size_t)g * HD;
  const bf16* KR = (const bf16*)a.k + (size_t)g * HD;
  const bf16* VR = (const bf16*)a.v + (size_t)g * HD;
  const size_t kstride = (size_t)a.nkv * HD;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm_raw);
  auto tile_k = [&](int buf) { return sbase + (uint32_t)(buf * 2 * TILEB); };
  auto tile_v = [&](int buf) { return sbase + (uint32_t)(buf * 2 * TILEB + TILEB); };
  auto load_tile = [&](int buf, int it) {
    const bool runA = it < ntA;
    const int t0 = runA ? it * MMA_KT : jb0 + (it - ntA) * MMA_KT;
    const int lim = runA ? a_end + 1 : iend;  // exclusive end of the run
    const bf16* ks = runA ? K1 : KR;
    const bf16* vs = runA ? V1 : VR;
    for (int idx = threadIdx.x; idx < MMA_KT * CH; idx += blockDim.x) {
      const int r = idx / CH, ch = idx - r * CH;
      const int key = t0 + r;
      const bool ok = key < lim;
      const size_t off = (size_t)(ok ? key : t0) * kstride + ch * 8;
      const uint32_t so = (uint32_t)(r * ROWB + ((ch ^ (r & 7)) * 16));
      cp_async16(tile_k(buf) + so, ks + off, ok ? 16 : 0);
      cp_async16(tile_v(buf) + so, vs + off, ok ? 16 : 0);
    }
    if (!runA && threadIdx.x < MMA_KT) {
      const int key = t0 + threadIdx.x;
      const bool ok = key < lim;
      s_kp[buf][threadIdx.x] = ok ? a.row_p[key] : 0;
      s_kd[buf][threadIdx.x] = ok ? a.row_d[key] : 0;
    }
    cp_async_commit();
  };
  if (ntile > 0) load_tile(0, 0);

  // this thread's two MMA rows: (query row, q head) and its mask parameters
  const float qscale = a.scale * 1.4426950408889634f;
  const int r0 = warp * 16 + gq, r1 = r0 + 8;
  const int qi0 = i0 + r0 / G, qi1 = i0 + r1 / G;
  const bool in0 = r0 < QR * G && qi0 < iend, in1 = r1 < QR * G && qi1 < iend;
  const int h0 = g * G + r0 % G, h1 = g * G + r1 % G;
  int lim0 = -1, lim1 = -1, dg0 = 0, dg1 = 0, dd0 = 0, dd1 = 0;  // anchor, p - d, d
  if (in0) {
    const int p = a.row_p[qi0], d = a.row_d[qi0];
    if (row_ok(p, d)) { lim0 = p - d + 1; dg0 = p - d; dd0 = d; }
  }
  if (in1) {
    const int p = a.row_p[qi1], d = a.row_d[qi1];
    if (row_ok(p, d)) { lim1 = p - d + 1; dg1 = p - d; dd1 = d; }
  }
  const float* qg = (const float*)a.q;
  const float* q0 = qg + ((size_t)(in0 ? qi0 : 0) * a.nq + h0) * HD;
  const float* q1 = qg + ((size_t)(in1 ? qi1 : 0) * a.nq + h1) * HD;
  uint32_t qa[KS][4];  // bf16 queries (the scale is applied to the scores)
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int d0 = ks * 16 + 2 * tq, d1 = d0 + 8;
    float x[8];
    x[0] = in0 ? q0[d0] : 0.f;
    x[1] = in0 ? q0[d0 + 1] : 0.f;
    x[2] = in1 ? q1[d0] : 0.f;
    x[3] = in1 ? q1[d0 + 1] : 0.f;
    x[4] = in0 ? q0[d1] : 0.f;
    x[5] = in0 ? q0[d1 + 1] : 0.f;
    x[6] = in1 ? q1[d1] : 0.f;
    x[7] = in1 ? q1[d1 + 1] : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) qa[ks][u] = pack_bf16(x[2 * u], x[2 * u + 1]);
  }
  float o[ND][4];
#pragma unroll
  for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const bool active = warp * 16 < QR * G && i0 + (warp * 16) / G < iend;

  for (int it = 0; it < ntile; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntile) {
      load_tile(buf ^ 1, it + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (active) {
      float sc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int mat = lane >> 3, rr = lane & 7;
          const int key = np * 16 + ((mat >> 1) << 3) + rr;
          const int ch = ks * 2 + (mat & 1);
          const uint32_t addr = tile_k(buf) + (uint32_t)(key * ROWB + ((ch ^ (key & 7)) * 16));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma16816(sc[2 * np], qa[ks], b0, b1);
          mma16816(sc[2 * np + 1], qa[ks], b2, b3);
        }
      }
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        sc[n][0] *= qscale;
        sc[n][1] *= qscale;
        sc[n][2] *= qscale;
        sc[n][3] *= qscale;
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (it < ntA) {
        const int t0 = it * MMA_KT;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int kp = t0 + n * 8 + 2 * tq;
          sc[n][0] = kp <= lim0 ? sc[n][0] : -INFINITY;
          sc[n][1] = kp + 1 <= lim0 ? sc[n][1] : -INFINITY;
          sc[n][2] = kp <= lim1 ? sc[n][2] : -INFINITY;
          sc[n][3] = kp + 1 <= lim1 ? sc[n][3] : -INFINITY;
        }
      } else {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kk = n * 8 + 2 * tq + e;
            const int kp = s_kp[buf][kk], kd = s_kd[buf][kk];
            const bool c0 = kd >= 2 && kp - kd == dg0 && kd <= dd0;
            const bool c1 = kd >= 2 && kp - kd == dg1 && kd <= dd1;
            sc[n][e] = c0 ? sc[n][e] : -INFINITY;
            sc[n][2 + e] = c1 ? sc[n][2 + e] : -INFINITY;
          }
        }
      }
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float cr0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - base0);
      const float cr1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - base1);
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        // probabilities rounded to bf16 once: the PV product and the row sum use the same
        sc[n][0] = bf16r(exp2f(sc[n][0] - base0));
        sc[n][1] = bf16r(exp2f(sc[n][1] - base0));
        sc[n][2] = bf16r(exp2f(sc[n][2] - base1));
        sc[n][3] = bf16r(exp2f(sc[n][3] - base1));
        ps0 += sc[n][0] + sc[n][1];
        ps1 += sc[n][2] + sc[n][3];
      }
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
      l0 = l0 * cr0 + ps0;
      l1 = l1 * cr1 + ps1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int n = 0; n < ND; ++n) {
        o[n][0] *= cr0;
        o[n][1] *= cr0;
        o[n][2] *= cr1;
        o[n][3] *= cr1;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4];
        ph[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        ph[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        ph[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        ph[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < ND / 2; ++dp) {
          const int mat = lane >> 3, rr = lane & 7;
          const int key = kk * 16 + ((mat & 1) << 3) + rr;
          const int ch = dp * 2 + (mat >> 1);
          const uint32_t addr = tile_v(buf) + (uint32_t)(key * ROWB + ((ch ^ (key & 7)) * 16));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma16816(o[2 * dp], ph, b0, b1);
          mma16816(o[2 * dp + 1], ph, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  // normalised output (rows outside the contract see no key and store zeros)
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  bf16* out = (bf16*)a.o;
  const size_t ld = (size_t)a.nq * HD;
#pragma unroll
  for (int n = 0; n < ND; ++n) {
    const int d = n * 8 + 2 * tq;
    if (in0) {
      store_act<bf16>(out, ld, qi0, a.M, a.split, h0 * HD + d, o[n][0] * inv0);
      store_act<bf16>(out, ld, qi0, a.M, a.split, h0 * HD + d + 1, o[n][1] * inv0);
    }
    if (in1) {
      store_act<bf16>(out, ld, qi1, a.M, a.split, h1 * HD + d, o[n][2] * inv1);
      store_act<bf16>(out, ld, qi1, a.M, a.split, h1 * HD + d + 1, o[n][3] * inv1);
    }
  }
}

template <int HD>
static void masked_mma_launch(const MaskedAttnArgs& a, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  const int QR = MASK_MMA_ROWS / G;
  const size_t sm = (size_t)4 * MMA_KT * HD * 2;
  smem_optin((const void*)masked_attn_mma_kernel<HD>, (int)sm);
  dim3 grid((unsigned)cdiv(a.M, QR), (unsigned)a.nkv);
  launch_pdl(masked_attn_mma_kernel<HD>, grid, dim3(128), sm, s, a);
}

void launch_masked_attention(bool bf16m, const MaskedAttnArgs& a, cudaStream_t s) {
  const long warps = (long)a.M * a.nq;
  dim3 grid((unsigned)((warps + 7) / 8));
  if (bf16m) {
    if (a.hd == 64) masked_mma_launch<64>(a, s); else masked_mma_launch<128>(a, s);
  } else {
    if (a.hd == 64) masked_attn_kernel<float, 64><<<grid, 256, 0, s>>>(a);
    else masked_attn_kernel<float, 128><<<grid, 256, 0, s>>>(a);
  }
}

// Row table of the training-style forward: row_index[p * (Kmax+1) + d] = row of (p, d).
// Checks each row against the contract (0 <= p < n, 1 <= d <= K, p-d+1 >= 0, strictly
// increasing p-major order, chain parent present) and raises BAD_ROW otherwise.
__global__ void rows_fill_kernel(int total, int* row_index) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x)
    row_index[i] = -1;
}
__global__ void rows_scatter_kernel(int M, int n, int K, int Kmax, const int* row_p,
                                   const int* row_d, int* row_index, unsigned* err) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < M; i += gridDim.x * blockDim.x) {
    const int p = row_p[i], d = row_d[i];
    bool ok = p >= 0 && p < n && d >= 1 && d <= K && p - d + 1 >= 0;
    if (ok && i > 0) {
      const int pp = row_p[i - 1], dp = row_d[i - 1];
      ok = (pp < p) || (pp == p && dp < d);
    }
    if (ok) row_index[(size_t)p * (Kmax + 1) + d] = i; else raise_error(err, PEAGLE_DEV_BAD_ROW);
  }
}
__global__ void rows_check_kernel(int M, int n, int Kmax, const int* row_p, const int* row_d,
                                  const int* row_index, unsigned* err) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < M; i += gridDim.x * blockDim.x) {
    const int p = row_p[i], d = row_d[i];
    // dependency closure: (p-1, d-1) for d >= 2 (its chain down to the anchor row), and
    // (p-1, 1) for d = 1 (so every depth-1 row up to each anchor is present)
    if (p >= 1 && p <= n && d >= 1 && d <= Kmax) {
      const int dp = d >= 2 ? d - 1 : 1;
      if (row_index[(size_t)(p - 1) * (Kmax + 1) + dp] < 0) raise_error(err, PEAGLE_DEV_BAD_ROW);
    }
  }
}

void launch_rows_prepare(int M, int n, int K, int Kmax, const int* row_p, const int* row_d,
                         int* row_index, unsigned* err, cudaStream_t s) {
  const int total = n * (Kmax + 1);
  rows_fill_kernel<<<cdiv(total, 256) < 1024 ? cdiv(total, 256) : 1024, 256, 0, s>>>(total, row_index);
  const int gb = cdiv(M, 256) < 1024 ? cdiv(M, 256) : 1024;
  rows_scatter_kernel<<<gb > 0 ? gb : 1, 256, 0, s>>>(M, n, K, Kmax, row_p, row_d, row_index, err);
  rows_check_kernel<<<gb > 0 ? gb : 1, 256, 0, s>>>(M, n, Kmax, row_p, row_d, row_index, err);
}

// =====================================================================================
// Argmax decode: key -> draft index -> target id via d2t; resets the key.
// =====================================================================================
__global__ void argmax_decode_kernel(int R, unsigned long long* keys, const int* d2t, int* out) {
  pdl_enter();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int idx = argmax_key_index(keys[r]);
  if (out) out[r] = d2t ? idx + d2t[idx] : idx;
  keys[r] = 0ull;
}

void launch_argmax_decode(int R, unsigned long long* keys, const int* d2t, int* out,
                          cudaStream_t s) {
  launch_pdl(argmax_decode_kernel, dim3(cdiv(R, 128)), dim3(128), 0, s, R, keys, d2t, out);
}

// =====================================================================================
// Efficient LM head ("EAGLE-4", "EAGLE-4 overview": a rank-128 projection scores the
// vocabulary, the full head scores the best candidates).
// =====================================================================================
// Orderable 32-bit image of a score: larger score, larger key; +0 and -0 map together.
__device__ __forceinline__ unsigned score_key(float v) {
  if (v == 0.f) v = 0.f;
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Histogram of the scores' first radix digit (key bits 31..21, 2048 buckets) per draft
// row, counted in shared memory by the scoring kernels (two 16-bit counters per word, so
// 8 draft rows fit in 32 KB) and added into the global [R][2048] histogram that the top-k
// selection starts from.
constexpr int HS_ROWS = 8;
__device__ __forceinline__ void hs_add(unsigned* sh, int rr, float v) {
  const unsigned b = score_key(v) >> 21;
  atomicAdd(&sh[rr * 1024 + (b >> 1)], (b & 1u) ? 65536u : 1u);
}
__device__ __forceinline__ void hs_clear(unsigned* sh) {
  for (int i = threadIdx.x; i < HS_ROWS * 1024; i += blockDim.x) sh[i] = 0u;
}
__device__ __forceinline__ void hs_flush(const unsigned* sh, int r0, int R, unsigned* hist) {
  for (int i = threadIdx.x; i < HS_ROWS * 1024; i += blockDim.x) {
    const unsigned w = sh[i];
    const int rr = i >> 10;
    if (w == 0u || r0 + rr >= R) continue;
    unsigned* h = hist + (size_t)(r0 + rr) * 2048 + 2 * (i & 1023);
    if (w & 0xFFFFu) atomicAdd(h, w & 0xFFFFu);
    if (w >> 16) atomicAdd(h + 1, w >> 16);
  }
}

// Rank-r scores of the whole draft vocabulary, fp32 weights, on the CUDA cores:
//   approx[row][v] = lm_score[v] . z[row],  z = the fixed-point rank-r projection [R][r].
// A vocabulary row is r elements in 16-byte pieces; a group of LPR lanes holds one row
// (CPL pieces per lane), so a warp scores 32 / LPR rows per step.  Draft rows are taken
// RC at a time with their z pieces in registers.  The group's partial sums are combined
// by a reduce-scatter over shuffles: each halving step trades half of the RC sums with
// the partner lane, so after log2(RC) steps a lane holds one draft row's sum, and plain
// shuffle adds finish it.
template <int RANK>
__global__ void __launch_bounds__(256) head_score_f32_kernel(int R, int Vd,
                                                             const fx_t* __restrict__ zfx,
                                                             const float* __restrict__ score,
                                                             float* __restrict__ approx,
                                                             unsigned* __restrict__ hist) {
  constexpr int E = 4;                         // elements per piece
  constexpr int P = RANK / E;                  // pieces per vocabulary row
  constexpr int CPL = P > 32 ? P / 32 : 1;     // pieces per lane
  constexpr int LPR = P / CPL;                 // lanes per vocabulary row (16 or 32)
  constexpr int RPW = 32 / LPR;                // vocabulary rows per warp step
  constexpr int RC = HS_ROWS / CPL;            // draft rows per sweep (<= LPR)
  static_assert(RC <= LPR, "reduce-scatter needs a lane per draft row");
  __shared__ unsigned sh[HS_ROWS * 1024];
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, pl = lane % LPR;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int stride = gridDim.x * 8 * RPW;
  // the draft row whose sum this lane ends with, and whether it stores it
  int mine = 0;
#pragma unroll
  for (int o = LPR / 2, cnt = RC; cnt > 1; o >>= 1, cnt >>= 1) mine += (pl & o) ? cnt / 2 : 0;
  const bool writer = (pl & (LPR / RC - 1)) == 0;
  for (int r0 = 0; r0 < R; r0 += RC) {
    hs_clear(sh);
    float z[RC][CPL][E];
#pragma unroll
    for (int rr = 0; rr < RC; ++rr)
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const fx_t* zp = zfx + (size_t)(r0 + rr) * RANK + (pl + c * LPR) * E;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          longlong2 q = make_longlong2(0, 0);
          if (r0 + rr < R) q = *reinterpret_cast<const longlong2*>(zp + e);
          z[rr][c][e] = from_fx(q.x);
          z[rr][c][e + 1] = from_fx(q.y);
        }
      }
    __syncthreads();
    // the loop bound is the warp's first row, so every lane takes the same steps
    for (int w0 = gw * RPW; w0 < Vd; w0 += stride) {
      const int v = w0 + sub;
      float w[CPL][E];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float4 q = v < Vd ? *reinterpret_cast<const float4*>(score + (size_t)v * RANK +
                                                                   (pl + c * LPR) * E)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        w[c][0] = q.x; w[c][1] = q.y; w[c][2] = q.z; w[c][3] = q.w;
      }
      float acc[RC];
#pragma unroll
      for (int rr = 0; rr < RC; ++rr) {
        float a = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
          for (int e = 0; e < E; ++e) a = fmaf(w[c][e], z[rr][c][e], a);
        acc[rr] = a;
      }
#pragma unroll
      for (int o = LPR / 2, cnt = RC; o > 0; o >>= 1, cnt = cnt > 1 ? cnt >> 1 : 1) {
        const bool upper = (pl & o) != 0;
#pragma unroll
        for (int i = 0; i < (cnt > 1 ? cnt / 2 : 1); ++i) {
          const float send = cnt > 1 ? (upper ? acc[i] : acc[i + cnt / 2]) : acc[0];
          const float keep = cnt > 1 ? (upper ? acc[i + cnt / 2] : acc[i]) : acc[0];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      if (writer && v < Vd && r0 + mine < R) {
        approx[(size_t)(r0 + mine) * Vd + v] = acc[0];
        hs_add(sh, mine, acc[0]);
      }
    }
    __syncthreads();
    hs_flush(sh, r0, R, hist);
    __syncthreads();
  }
}

// Rank-r scores, bf16 weights, on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
// A = 16 vocabulary rows of lm_score, B = 8 draft rows of z as bf16 hi + lo parts (z to
// about 16 significant bits), C = the 16 x 8 scores.  A dot product may run over k in any
// order that A and B share, so each lane takes 16 contiguous bytes of its two A rows per
// 32-wide k chunk (two MMA k-steps) and z at the same k.
// Each CTA streams lm_score through a ring of HS_STAGES shared-memory stages of 32 KB
// (stages dealt to the CTAs in turn): one producer thread issues a bulk copy per stage
// (completion on the stage's `full` mbarrier, L2 evict-last), eight consumer warps take
// one 16-row tile each per turn and release it on the stage's `empty` mbarrier.  Waits
// are bounded: a wait that gives up raises PEAGLE_DEV_TIMEOUT and every role leaves its
// loop.
constexpr int HS_WARPS = 8;
constexpr int HS_THREADS = 32 * (HS_WARPS + 1);
constexpr int HS_STAGES = 4;
constexpr int HS_STAGE_BYTES = 32 * 1024;

template <int RANK>
__global__ void __launch_bounds__(HS_THREADS, 1) head_score_mma_kernel(
    int R, int Vd, const fx_t* __restrict__ zfx, const bf16* __restrict__ score,
    float* __restrict__ approx, unsigned* __restrict__ hist, unsigned* err) {
  constexpr int KC = RANK / 32;                // 32-wide k chunks
  constexpr int AG = KC < 4 ? KC : 4;          // chunks of A read together
  constexpr int ROW_B = RANK * 2;
  constexpr int TILE_B = 16 * ROW_B;
  constexpr int TPS = HS_STAGE_BYTES / TILE_B; // tiles per stage
  static_assert(TPS >= 1, "a stage holds a tile");
  extern __shared__ __align__(128) uint8_t hs_ring[];
  __shared__ unsigned sh[HS_ROWS * 1024];
  __shared__ uint64_t full[HS_STAGES], empty[HS_STAGES];
  __shared__ int abort_flag;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, g = lane >> 2, q = lane & 3;
  // fills of TPS tiles are dealt to the CTAs in turn, so at any moment the grid reads one
  // contiguous window of lm_score (spread over every memory channel)
  const int tiles = (Vd + 15) / 16;
  const int fills = (tiles + TPS - 1) / TPS;
  const int nfill = fills > (int)blockIdx.x ? (fills - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int nt = nfill * TPS;  // CTA-local tile slots (slots past the vocabulary are skipped)
  if (t == 0) {
    for (int i = 0; i < HS_STAGES; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], TPS);
    }
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  pdl_enter();
  for (int r0 = 0, sweep = 0; r0 < R; r0 += HS_ROWS, ++sweep) {
    const int fbase = sweep * nfill;  // fills of earlier sweeps (barrier phases run on)
    hs_clear(sh);
    __syncthreads();
    if (warp == HS_WARPS) {
      if (lane == 0) {
        // the scoring factor is small next to the pass's weights, which stream through L2
        // with evict-first: keep it resident from one pass to the next
        const uint64_t pol = tc::policy_evict_last();
        int issued = 0;
        for (int f = 0; f < nfill && !abort_flag; ++f) {
          const int F = fbase + f, st = F % HS_STAGES;
          if (F >= HS_STAGES && !tc::mbar_wait(&empty[st], ((F / HS_STAGES) - 1) & 1, &abort_flag)) {
            raise_error(err, PEAGLE_DEV_TIMEOUT);
            abort_flag = 1;
            break;
          }
          const int t0 = (f * (int)gridDim.x + (int)blockIdx.x) * TPS;
          const int ft = tiles - t0 < TPS ? tiles - t0 : TPS;  // tiles in this fill
          const int rows = (Vd - 16 * t0) < 16 * ft ? Vd - 16 * t0 : 16 * ft;
          const uint32_t bytes = (uint32_t)rows * ROW_B;
          tc::mbar_expect_tx(&full[st], bytes);
          tc::bulk_load(hs_ring + (size_t)st * HS_STAGE_BYTES, score + (size_t)t0 * 16 * RANK, bytes,
                        &full[st], pol);
          ++issued;
          // slots of a short last fill are released at once
          for (int i = ft; i < TPS; ++i) tc::mbar_arrive(&empty[st]);
        }
        if (abort_flag) {  // let the copies in flight land before the CTA exits
          for (int f = issued > HS_STAGES ? issued - HS_STAGES : 0; f < issued; ++f) {
            const int F = fbase + f;
            tc::mbar_wait(&full[F % HS_STAGES], (F / HS_STAGES) & 1, &abort_flag, 100000000ull);
          }
        }
      }
    } else {
      // B fragments: k-step s of chunk c takes k = 32c + 8q + 4s + {0,1} (b0), {2,3} (b1)
      uint32_t bh[KC][2][2], bl[KC][2][2];
#pragma unroll
      for (int c = 0; c < KC; ++c)
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float z0 = 0.f, z1 = 0.f;
            if (r0 + g < R) {
              const longlong2 zz = *reinterpret_cast<const longlong2*>(
                  zfx + (size_t)(r0 + g) * RANK + 32 * c + 8 * q + 4 * s2 + 2 * j);
              z0 = from_fx(zz.x);
              z1 = from_fx(zz.y);
            }
            split2(z0, z1, bh[c][s2][j], bl[c][s2][j]);
          }
      for (int j = warp; j < nt; j += HS_WARPS) {
        const int tg = ((j / TPS) * (int)gridDim.x + (int)blockIdx.x) * TPS + j % TPS;
        if (tg >= tiles) continue;  // released by the producer
        const int F = fbase + j / TPS, st = F % HS_STAGES;
        if (!tc::mbar_wait(&full[st], (F / HS_STAGES) & 1, &abort_flag)) {
          raise_error(err, PEAGLE_DEV_TIMEOUT);
          abort_flag = 1;
          break;
        }
        const uint8_t* tile = hs_ring + (size_t)st * HS_STAGE_BYTES + (size_t)(j % TPS) * TILE_B;
        const int va = tg * 16 + g, vb = va + 8;
        // hi and lo products and the two k-steps of a chunk accumulate separately
        float acc[2][2][4] = {};
#pragma unroll
        for (int c0 = 0; c0 < KC; c0 += AG) {
          uint4 qa[AG], qb[AG];
#pragma unroll
          for (int c = 0; c < AG; ++c) {
            const int off = 64 * (c0 + c) + 16 * q;
            qa[c] = va < Vd ? *reinterpret_cast<const uint4*>(tile + g * ROW_B + off)
                            : make_uint4(0u, 0u, 0u, 0u);
            qb[c] = vb < Vd ? *reinterpret_cast<const uint4*>(tile + (g + 8) * ROW_B + off)
                            : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int c = 0; c < AG; ++c) {
            const uint32_t wa[4] = {qa[c].x, qa[c].y, qa[c].z, qa[c].w};
            const uint32_t wb[4] = {qb[c].x, qb[c].y, qb[c].z, qb[c].w};
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
              // A: (row g, k 2q, 2q+1) = elements 4s, 4s+1 of the piece; (row g, k 2q+8,
              // 2q+9) = elements 4s+2, 4s+3; rows g+8 likewise from the second row
              const uint32_t af[4] = {wa[2 * s2], wb[2 * s2], wa[2 * s2 + 1], wb[2 * s2 + 1]};
              mma16816(acc[0][s2], af, bh[c0 + c][s2][0], bh[c0 + c][s2][1]);
              mma16816(acc[1][s2], af, bl[c0 + c][s2][0], bl[c0 + c][s2][1]);
            }
          }
        }
        // the products depend on every shared-memory read of the tile: release it
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st]);
        // acc[.][.] = (va, draft 2q), (va, 2q + 1), (vb, 2q), (vb, 2q + 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = 2 * q + (e & 1), v = (e < 2) ? va : vb;
          const float x = (acc[0][0][e] + acc[0][1][e]) + (acc[1][0][e] + acc[1][1][e]);
          if (r0 + rr < R && v < Vd) {
            approx[(size_t)(r0 + rr) * Vd + v] = x;
            hs_add(sh, rr, x);
          }
        }
      }
    }
    __syncthreads();
    if (abort_flag) return;
    hs_flush(sh, r0, R, hist);
  }
}

template <int RANK>
static void head_score_mma_launch(int blocks, cudaStream_t s, int R, int Vd, const fx_t* zfx,
                                  const bf16* score, float* approx, unsigned* hist,
                                  unsigned* err) {
  const size_t smem = (size_t)HS_STAGES * HS_STAGE_BYTES;
  smem_optin((const void*)head_score_mma_kernel<RANK>, (int)smem);
  launch_pdl(head_score_mma_kernel<RANK>, dim3(blocks), dim3(HS_THREADS), smem, s, R, Vd, zfx,
             score, approx, hist, err);
}

template <typename KernelT, typename T>
static void head_score_go(KernelT kern, int blocks, cudaStream_t s, int R, int Vd,
                          const fx_t* zfx, const T* score, float* approx, unsigned* hist) {
  launch_pdl(kern, dim3(blocks), dim3(256), 0, s, R, Vd, zfx, score, approx, hist);
}

void launch_head_score(bool bf16m, int R, int r, int Vd, const fx_t* zfx, const void* score,
                       float* approx, unsigned* hist, unsigned* err, int num_sms, cudaStream_t s) {
  if (bf16m) {
    // one CTA per SM
    int blocks = cdiv(Vd, 16 * 8);
    if (blocks > num_sms) blocks = num_sms;
    const bf16* w = (const bf16*)score;
    if (r == 64) head_score_mma_launch<64>(blocks, s, R, Vd, zfx, w, approx, hist, err);
    else if (r == 128) head_score_mma_launch<128>(blocks, s, R, Vd, zfx, w, approx, hist, err);
    else if (r == 256) head_score_mma_launch<256>(blocks, s, R, Vd, zfx, w, approx, hist, err);
    else head_score_mma_launch<512>(blocks, s, R, Vd, zfx, w, approx, hist, err);
    return;
  }
  // CUDA cores: vocabulary rows a CTA scores per step: 8 warps x (512 bytes / row bytes)
  const int per_cta = 8 * (r * 4 < 512 ? 512 / (r * 4) : 1);
  int blocks = cdiv(Vd, per_cta * 2);
  if (blocks > 2 * num_sms) blocks = 2 * num_sms;
  const float* w = (const float*)score;
  if (r == 64) head_score_go(head_score_f32_kernel<64>, blocks, s, R, Vd, zfx, w, approx, hist);
  else if (r == 128) head_score_go(head_score_f32_kernel<128>, blocks, s, R, Vd, zfx, w, approx, hist);
  else if (r == 256) head_score_go(head_score_f32_kernel<256>, blocks, s, R, Vd, zfx, w, approx, hist);
  else head_score_go(head_score_f32_kernel<512>, blocks, s, R, Vd, zfx, w, approx, hist);
}

// Top-k of each row of scores [R][n], largest first, ties to the lower index, from the
// first-digit histograms the scoring kernel left.  Keys are the scores' orderable 32-bit
// images, selected by radix digits of 11, 11 and 10 bits.  A grid of S slices per row:
// every CTA finds the boundary bucket of the first digit (the one holding the k-th
// largest key) and gathers its slice's keys at or above it (a few hundred per row for
// smooth scores) into a global list; the last CTA of the row to finish loads the list
// into shared memory and resolves the other two digits and the ties there.  Rows whose
// list does not fit are resolved by that CTA over global memory instead, with the ties
// taken in index order.  cand[row][0 .. k) = the chosen indices (any order).  The last
// CTA also clears the row's histogram, list counters and fixed-point projection for the
// next pass.
constexpr int TS_THREADS = 512;
constexpr int TK_CAP = 4096;

struct TopkSmem {
  unsigned hist[2048];
  unsigned lkey[TK_CAP];
  int lidx[TK_CAP];
  unsigned wsum[32];
  unsigned digit, above, nout;
  int last;
};

// The bucket of h[2048] holding the need-th largest key (counted from the top) ->
// S.digit, and the number of keys in the buckets above it -> S.above.
__device__ void tk_find(TopkSmem& S, const unsigned* h, unsigned need) {
  constexpr int BPT = 2048 / TS_THREADS;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  unsigned c[BPT], sum = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    c[j] = h[2047 - BPT * t - j];
    sum += c[j];
  }
  unsigned inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) S.wsum[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const unsigned w = lane < TS_THREADS / 32 ? S.wsum[lane] : 0u;
    unsigned winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += y;
    }
    if (lane < TS_THREADS / 32) S.wsum[lane] = winc - w;
  }
  __syncthreads();
  unsigned run = S.wsum[wid] + inc - sum;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    if (run < need && run + c[j] >= need) {
      S.digit = (unsigned)(2047 - BPT * t - j);
      S.above = run;
    }
    run += c[j];
  }
  __syncthreads();
}

__device__ __forceinline__ void tk_clear(TopkSmem& S) {
  for (int i = threadIdx.x; i < 2048; i += TS_THREADS) S.hist[i] = 0u;
  __syncthreads();
}

// f(key, index) over scores x[beg, end) in global memory
template <typename F>
__device__ __forceinline__ void tk_row(const float* __restrict__ x, int beg, int end, F f) {
  for (int i = beg + threadIdx.x; i < end; i += TS_THREADS) f(score_key(x[i]), i);
}

// Refine the boundary digit d1 (bits 31..21, need1 keys still wanted in it) to the k-th
// key over `each` (a source of (key, index)); returns the key, *need = how many of the
// keys equal to it are taken, *ties = how many there are.
template <typename Each>
__device__ unsigned tk_refine(TopkSmem& S, Each each, unsigned d1, unsigned need1,
                              unsigned* need, unsigned* ties) {
  tk_clear(S);
  each([&](unsigned u, int) {
    if ((u >> 21) == d1) atomicAdd(&S.hist[(u >> 10) & 2047u], 1u);
  });
  __syncthreads();
  tk_find(S, S.hist, need1);
  const unsigned d2 = S.digit, need2 = need1 - S.above;
  const unsigned p22 = (d1 << 11) | d2;
  __syncthreads();
  tk_clear(S);
  each([&](unsigned u, int) {
    if ((u >> 10) == p22) atomicAdd(&S.hist[u & 1023u], 1u);
  });
  __syncthreads();
  tk_find(S, S.hist, need2);
  const unsigned d3 = S.digit;
  *need = need2 - S.above;
  *ties = S.hist[d3];
  return (p22 << 10) | d3;
}

__global__ void __launch_bounds__(TS_THREADS) topk_select_kernel(
    int n, int k, const float* __restrict__ score, unsigned* __restrict__ hist,
    unsigned* __restrict__ gcount, unsigned* __restrict__ gdone, unsigned* __restrict__ gkey,
    int* __restrict__ gidx, int* __restrict__ cand, fx_t* __restrict__ zfx, int zn) {
  __shared__ TopkSmem S;
  pdl_enter();
  const int row = blockIdx.y, t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const float* x = score + (size_t)row * n;
  unsigned* hrow = hist + (size_t)row * 2048;
  for (int i = t; i < 2048; i += TS_THREADS) S.hist[i] = __ldcg(hrow + i);
  if (t == 0) S.nout = 0;
  __syncthreads();
  tk_find(S, S.hist, (unsigned)k);
  const unsigned d1 = S.digit, above1 = S.above;
  const unsigned m = above1 + S.hist[d1];  // keys with digit >= d1
  const unsigned need1 = (unsigned)k - above1;
  {
    const int chunk = cdiv(n, gridDim.x);
    const int beg = blockIdx.x * chunk, end = min(n, beg + chunk);
    unsigned* lk = gkey + (size_t)row * TK_CAP;
    int* li = gidx + (size_t)row * TK_CAP;
    tk_row(x, beg, end, [&](unsigned u, int i) {
      if ((u >> 21) >= d1) {
        const unsigned p = atomicAdd(gcount + row, 1u);
        if (p < (unsigned)TK_CAP) {
          lk[p] = u;
          li[p] = i;
        }
      }
    });
  }
  __syncthreads();
  if (t == 0) S.last = atom_add_acq_rel(gdone + row, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!S.last) return;
  // the last CTA of the row: every slice's keys are in the list
  for (int i = t; i < 2048; i += TS_THREADS) hrow[i] = 0u;
  if (zfx)
    for (int i = t; i < zn; i += TS_THREADS) zfx[(size_t)row * zn + i] = 0;
  int* out = cand + (size_t)row * k;
  unsigned need, ties, kth;
  if (m <= (unsigned)TK_CAP) {
    for (int i = t; i < (int)m; i += TS_THREADS) {
      S.lkey[i] = __ldcg(gkey + (size_t)row * TK_CAP + i);
      S.lidx[i] = __ldcg(gidx + (size_t)row * TK_CAP + i);
    }
    __syncthreads();
    auto each = [&](auto f) {
      for (int i = threadIdx.x; i < (int)m; i += TS_THREADS) f(S.lkey[i], S.lidx[i]);
    };
    kth = tk_refine(S, each, d1, need1, &need, &ties);
    for (int i = t; i < (int)m; i += TS_THREADS) {
      const unsigned u = S.lkey[i];
      bool take = u > kth;
      if (u == kth) {
        if (need == ties) {
          take = true;
        } else {  // the `need` lowest indices among the ties
          const int me = S.lidx[i];
          unsigned rank = 0;
          for (int j = 0; j < (int)m; ++j) rank += (S.lkey[j] == kth && S.lidx[j] < me);
          take = rank < need;
        }
      }
      if (take) out[atomicAdd(&S.nout, 1u)] = S.lidx[i];
    }
  } else {
    auto each = [&](auto f) { tk_row(x, 0, n, f); };
    kth = tk_refine(S, each, d1, need1, &need, &ties);
    tk_row(x, 0, n, [&](unsigned u, int i) {
      if (u > kth || (u == kth && need == ties)) out[atomicAdd(&S.nout, 1u)] = i;
    });
    if (need != ties) {
      __syncthreads();
      const unsigned base = S.nout;  // = k - need
      unsigned taken = 0;
      for (int i0 = 0; i0 < n && taken < need; i0 += TS_THREADS) {
        const int i = i0 + t;
        const bool eq = i < n && score_key(x[i]) == kth;
        const unsigned bal = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) S.wsum[wid] = __popc(bal);
        __syncthreads();
        unsigned before = 0, total = 0;
        for (int w = 0; w < TS_THREADS / 32; ++w) {
          const unsigned c = S.wsum[w];
          if (w < wid) before += c;
          total += c;
        }
        const unsigned rank = taken + before + __popc(bal & ((1u << lane) - 1u));
        if (eq && rank < need) out[base + rank] = i;
        taken += total;
        __syncthreads();
      }
    }
  }
  if (t == 0) {
    gcount[row] = 0u;
    gdone[row] = 0u;
  }
}

void launch_topk(int R, int n, int k, const float* score, unsigned* hist, unsigned* gcount,
                 unsigned* gdone, unsigned* gkey, int* gidx, int* cand, fx_t* zfx, int zn,
                 int num_sms, cudaStream_t s) {
  // slices per row: about two CTAs per SM over all rows, at least 512 keys a slice
  int S = 2 * num_sms / R;
  if (S > cdiv(n, 512)) S = cdiv(n, 512);
  if (S > 64) S = 64;
  if (S < 1) S = 1;
  launch_pdl(topk_select_kernel, dim3(S, R), dim3(TS_THREADS), 0, s, n, k, score, hist, gcount,
             gdone, gkey, gidx, cand, zfx, zn);
}

// Exact logits of the candidates: a CTA per (row, 8 candidates), the row's head input
// (hi + lo parts) staged once in shared memory as fp32, a warp per candidate streaming
// its head row in 16-byte pieces, an argmax key per row (ties: lower index) and, when
// asked, the logit.  The last CTA to finish decodes every row's argmax (token id through
// d2t) and clears the keys and its counter for the next pass.
template <typename T>
__global__ void __launch_bounds__(256) cand_head_kernel(int R, int H, int k,
                                                        const int* __restrict__ cand,
                                                        const T* __restrict__ head,
                                                        const T* __restrict__ y, int split,
                                                        unsigned long long* keys, float* logits,
                                                        int Vd, const int* __restrict__ d2t,
                                                        int* __restrict__ out,
                                                        unsigned* done) {
  constexpr int E = 16 / sizeof(T);
  extern __shared__ float ys[];
  __shared__ bool s_last;
  pdl_enter();
  const int t = threadIdx.x, lane = t & 31;
  const int row = blockIdx.y;
  const T* yh = y + (size_t)row * H;
  const T* yl = y + (size_t)(row + R) * H;
  for (int i = t; i < H; i += 256) ys[i] = to_f32(yh[i]) + (split ? to_f32(yl[i]) : 0.f);
  __syncthreads();
  const int j = blockIdx.x * 8 + (t >> 5);
  if (j < k) {
    const int c = cand[(size_t)row * k + j];
    const uint4* hr = reinterpret_cast<const uint4*>(head + (size_t)c * H);
    const int np = H / E;
    constexpr int NB = 12;  // pieces in flight per lane (a 2880-wide bf16 row in one batch)
    float acc = 0.f;
    for (int p0 = lane; p0 < np; p0 += 32 * NB) {
      uint4 q[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b)
        q[b] = p0 + 32 * b < np ? hr[p0 + 32 * b] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int p = p0 + 32 * b;
        if (p < np) {
          float w[E];
          unpack16<T>(q[b], w);
#pragma unroll
          for (int e = 0; e < E; ++e) acc = fmaf(w[e], ys[p * E + e], acc);
        }
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      atomicMax(keys + row, argmax_key(acc, c));
      if (logits) logits[(size_t)row * Vd + c] = acc;
    }
  }
  __syncthreads();
  if (t == 0) s_last = atom_add_acq_rel(done, 1u) == gridDim.x * gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  for (int rr = t; rr < R; rr += 256) {
    const int idx = argmax_key_index(__ldcg(keys + rr));
    if (out) out[rr] = d2t ? idx + d2t[idx] : idx;
    keys[rr] = 0ull;
  }
  if (t == 0) *done = 0u;
}

__global__ void fill_kernel(size_t n, float v, float* p) {
  pdl_enter();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

void launch_cand_head(bool bf16m, int R, int H, int k, const int* cand, const void* head,
                      const void* y, int split, unsigned long long* keys, float* logits, int Vd,
                      const int* d2t, int* out, unsigned* done, cudaStream_t s) {
  if (logits) {
    const size_t n = (size_t)R * Vd;
    const size_t nb = (n + 255) / 256;
    launch_pdl(fill_kernel, dim3(nb < 1024 ? (unsigned)nb : 1024u), dim3(256), 0, s, n,
               -INFINITY, logits);
  }
  const dim3 grid(cdiv(k, 8), R);
  const size_t smem = (size_t)H * 4;
  if (bf16m)
    launch_pdl(cand_head_kernel<bf16>, grid, dim3(256), smem, s, R, H, k, cand,
               (const bf16*)head, (const bf16*)y, split, keys, logits, Vd, d2t, out, done);
  else
    launch_pdl(cand_head_kernel<float>, grid, dim3(256), smem, s, R, H, k, cand,
               (const float*)head, (const float*)y, 0, keys, logits, Vd, d2t, out, done);
}

// =====================================================================================
// Greedy verification ("EAGLE-4 overview"): longest agreeing prefix + bonus token.
// =====================================================================================
__global__ void verify_kernel(int B, int K, const int* __restrict__ draft,
                              const int* __restrict__ tgt, int* __restrict__ acc,
                              int* __restrict__ bonus) {
  pdl_enter();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int* d = draft + (size_t)b * K;
  const int* t = tgt + (size_t)b * (K + 1);
  int m = 0;
  while (m < K && d[m] == t[m]) ++m;
  acc[b] = m;
  bonus[b] = t[m];
}

void launch_verify(int B, int K, const int* draft, const int* tgt, int* acc, int* bonus,
                   cudaStream_t s) {
  launch_pdl(verify_kernel, dim3(cdiv(B, 128)), dim3(128), 0, s, B, K, draft, tgt, acc, bonus);
}

// =====================================================================================
// KV commit: one CTA per request copies (optionally) the accepted rows of every layer
// into slots seq_lens[b] .. and then advances seq_lens[b].
// =====================================================================================
template <typename T>
__global__ void __launch_bounds__(256) append_kv_kernel(int N, int nkv, int hd, int cap,
                                                        int batch_slots, T* kc, T* vc,
                                                        int* seq_lens, const int* n_commit,
                                                        int n_extra, const T* k_rows,
                                                        const T* v_rows, int n_max, int B,
                                                        unsigned* err) {
  pdl_enter();
  const int b = blockIdx.x;
  const int L = seq_lens[b];
  const int n = n_commit[b] + n_extra;
  if (n < 0 || n > n_max) {
    if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_COMMIT);
    return;
  }
  if (L < 0 || L + n > cap) {
    if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_KV_OVERFLOW);
    return;
  }
  if (k_rows) {
    const size_t per_row = (size_t)nkv * hd;
    const size_t total = (size_t)N * n * per_row;
    for (size_t idx = threadIdx.x; idx < total; idx += blockDim.x) {
      const int layer = (int)(idx / (n * per_row));
      const size_t rem = idx - (size_t)layer * n * per_row;
      const int i = (int)(rem / per_row);
      const size_t rem2 = rem - (size_t)i * per_row;
      const int g = (int)(rem2 / hd), d = (int)(rem2 - (size_t)g * hd);
      const size_t src = ((((size_t)layer * B + b) * n_max + i) * nkv + g) * hd + d;
      const size_t dst = ((((size_t)layer * batch_slots + b) * nkv + g) * cap + (L + i)) * hd + d;
      kc[dst] = k_rows[src];
      vc[dst] = v_rows[src];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) seq_lens[b] = L + n;
}

void launch_append_kv(bool bf16m, int B, int N, int nkv, int hd, int cap, void* kc, void* vc,
                      int* seq_lens, const int* n_commit, int n_extra, const void* k_rows,
                      const void* v_rows, int n_max, int batch_slots, unsigned* err,
                      cudaStream_t s) {
  if (bf16m)
    launch_pdl(append_kv_kernel<bf16>, dim3(B), dim3(256), 0, s, N, nkv, hd, cap, batch_slots,
               (bf16*)kc, (bf16*)vc, seq_lens, n_commit, n_extra, (const bf16*)k_rows,
               (const bf16*)v_rows, n_max, B, err);
  else
    append_kv_kernel<float><<<B, 256, 0, s>>>(N, nkv, hd, cap, batch_slots, (float*)kc, (float*)vc,
        seq_lens, n_commit, n_extra, (const float*)k_rows, (const float*)v_rows, n_max, B, err);
}

}  // namespace peagle

// =====================================================================================
// peagle_decode_attention_static: the split-KV decode attention for callers that cannot
// allocate device memory.  Its split-KV partial results live in the file-scope array
// below (PEAGLE_STATIC_ATTN_SCRATCH_BYTES, held by every GPU that loads the library until
// the process exits) instead of a context workspace.
// =====================================================================================
namespace peagle {

static __device__ __align__(256) float g_static_attn_scratch[PEAGLE_STATIC_ATTN_SCRATCH_BYTES /
                                                             sizeof(float)];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
float* g_static_ptr[kMaxDevices] = {};   // device address of the array, per device

// Device address of the scratch array on the current device (looked up once per device:
// in host code the array's name is only a host-side stand-in).
int static_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PEAGLE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_attn_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "peagle: cudaGetSymbolAddress(static attention scratch) failed: %s\n",
              cudaGetErrorString(e));
      return PEAGLE_ERR_CUDA;
    }
    g_static_ptr[dev] = (float*)p;
  }
  if (smem_optin((const void*)attn_mma_kernel<64>, 100 * 1024) != cudaSuccess ||
      smem_optin((const void*)attn_mma_kernel<128>, 100 * 1024) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  *out = g_static_ptr[dev];
  return PEAGLE_OK;
}

template <int HD>
cudaError_t static_attn_launch(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.K * (a.nq / a.nkv);
  const int warps = (rows + 15) / 16;
  const size_t sm = (size_t)4 * MMA_KT * HD * 2;
  cudaError_t e = launch_pdl(attn_mma_kernel<HD>, dim3(a.nchunk, a.nkv, a.B), dim3(32 * warps),
                             sm, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_merge_kernel<float, HD>, dim3(cdiv(rows, 4), a.nkv, a.B), dim3(128), 0,
                    s, a);
}
}  // namespace

}  // namespace peagle

extern "C" int peagle_decode_attention_static(int32_t batch, int32_t K, int32_t n_q_heads,
                                              int32_t n_kv_heads, int32_t head_dim,
                                              const float* q, const void* k_cache,
                                              const void* v_cache, int32_t capacity,
                                              const int32_t* seq_lens, float* out, void* stream) {
  using namespace peagle;
  if (batch < 1 || K < 1 || n_q_heads < 1 || n_kv_heads < 1 || capacity < K || !q || !k_cache ||
      !v_cache || !seq_lens || !out)
    return PEAGLE_ERR_INVALID;
  if ((head_dim != 64 && head_dim != 128) || n_q_heads % n_kv_heads) return PEAGLE_ERR_UNSUPPORTED;
  const int G = n_q_heads / n_kv_heads;
  const int rows = K * G;
  if (rows > ATT_MAX_ROWS) return PEAGLE_ERR_UNSUPPORTED;
  int num_sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  // split plan: about two CTAs per SM, chunks of whole 64-key tiles, at most 64 chunks;
  // fewer, longer chunks if the partials would not fit the static array
  const size_t per_chunk = (size_t)batch * n_kv_heads * rows * (head_dim + 2) * sizeof(float);
  const size_t max_chunks = PEAGLE_STATIC_ATTN_SCRATCH_BYTES / per_chunk;
  if (max_chunks < 1) {
    fprintf(stderr,
            "peagle_decode_attention_static: batch %d x kv heads %d x rows %d needs %zu bytes "
            "of scratch per chunk, more than the %u-byte static array\n",
            batch, n_kv_heads, rows, per_chunk, (unsigned)PEAGLE_STATIC_ATTN_SCRATCH_BYTES);
    return PEAGLE_ERR_CAPACITY;
  }
  const long long units = (long long)batch * n_kv_heads;
  long long want = (2LL * num_sms + units - 1) / units;
  if (want < 1) want = 1;
  if (want > 64) want = 64;
  if ((unsigned long long)want > max_chunks) want = (long long)max_chunks;
  // whole 64-key tiles per chunk; chunk >= capacity / want, so at most `want` chunks
  const long long chunk64 = ((capacity + want - 1) / want + 63) / 64 * 64;
  if (chunk64 > 0x7fffffffLL) return PEAGLE_ERR_UNSUPPORTED;
  const int chunk = (int)chunk64;
  const int nchunk = (int)((capacity + chunk64 - 1) / chunk64);
  float* scratch = nullptr;
  int r = static_scratch(&scratch);
  if (r != PEAGLE_OK) return r;
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.kc = k_cache;
  a.vc = v_cache;
  a.seq_lens = seq_lens;
  a.o = out;
  a.split = 0;
  a.part = scratch;  // every element read by the merge is written first: no clearing needed
  a.counters = nullptr;
  a.B = batch;
  a.K = K;
  a.nq = n_q_heads;
  a.nkv = n_kv_heads;
  a.hd = head_dim;
  a.cap = capacity;
  a.chunk = chunk;
  a.nchunk = nchunk;
  a.scale = 1.f / sqrtf((float)head_dim);
  a.err = nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = head_dim == 64 ? static_attn_launch<64>(a, s) : static_attn_launch<128>(a, s);
  if (e != cudaSuccess) {
    fprintf(stderr, "peagle_decode_attention_static: launch failed: %s\n", cudaGetErrorString(e));
    return PEAGLE_ERR_CUDA;
  }
  return PEAGLE_OK;
}
