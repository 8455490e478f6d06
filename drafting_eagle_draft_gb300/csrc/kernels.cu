// CUDA-core kernels of the P-EAGLE draft pass: input fusion, RMSNorm, split-KV decode
// attention with the causal draft block, the training-style masked attention, greedy
// verification, KV commit, argmax decode, and the fp32 FFMA GEMM used by the fp32
// drafter (whose 1e-4 logit tolerance rules out TF32 tensor cores).
#include "kernels.h"

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
// =====================================================================================
template <typename T>
__global__ void __launch_bounds__(256) input_fusion_kernel(
    int mode, int K, int n_src, int H, const T* __restrict__ embed, int Vt,
    const T* __restrict__ emb_mask,
    const float* __restrict__ F, const float* __restrict__ f_shared, const int* __restrict__ tokens,
    const int* __restrict__ row_p, const int* __restrict__ row_d, const T* __restrict__ g_in,
    const T* __restrict__ g_hid, float eps, int split, T* __restrict__ X0,
    float* __restrict__ res, unsigned long long* __restrict__ keys, unsigned* err) {
  __shared__ float red[32];
  pdl_enter();
  const int r = blockIdx.x;
  const int R = gridDim.x;
  bool ntp;
  int src;  // request (mode 0) or position (mode 1)
  if (mode == 0) {
    src = r / K;
    ntp = (r - src * K) == 0;
  } else {
    src = row_p[r];
    ntp = row_d[r] == 1;
    if (src < 0 || src >= n_src) {  // outside the contract: BAD_ROW, use the MTP inputs
      if (threadIdx.x == 0) raise_error(err, PEAGLE_DEV_BAD_ROW);
      ntp = false;
    }
  }
  const T* e;
  const float* f;
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
    f = f_shared;
  }
  float se = 0.f, sf = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    float ev = ld(e + i), fv = f[i];
    se += ev * ev;
    sf += fv * fv;
  }
  se = block_sum(se, red);
  __syncthreads();
  sf = block_sum(sf, red);
  const float ie = rsqrtf(se / H + eps), ifv = rsqrtf(sf / H + eps);
  float* rs = res + (size_t)r * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    float fv = f[i];
    store_act<T>(X0, 2 * H, r, R, split, i, ld(e + i) * ie * ld(g_in + i));
    store_act<T>(X0, 2 * H, r, R, split, H + i, fv * ifv * ld(g_hid + i));
    rs[i] = fv;
  }
  if (threadIdx.x == 0 && keys) keys[r] = 0ull;
}

void launch_input_fusion(bool bf16m, int mode, int R, int K, int n_src, int H, const void* embed,
                         int Vt,
                         const void* emb_mask, const float* F, const float* f_shared,
                         const int* tokens, const int* row_p, const int* row_d,
                         const void* g_in, const void* g_hid, float eps, int split, void* X0,
                         float* res, unsigned long long* keys, unsigned* err, cudaStream_t s) {
  if (bf16m)
    launch_pdl(input_fusion_kernel<bf16>, dim3(R), dim3(256), 0, s, mode, K, n_src, H,
               (const bf16*)embed, Vt, (const bf16*)emb_mask, F, f_shared, tokens, row_p, row_d,
               (const bf16*)g_in, (const bf16*)g_hid, eps, split, (bf16*)X0, res, keys, err);
  else
    input_fusion_kernel<float><<<R, 256, 0, s>>>(mode, K, n_src, H, (const float*)embed, Vt,
        (const float*)emb_mask, F, f_shared, tokens, row_p, row_d, (const float*)g_in,
        (const float*)g_hid, eps, 0, (float*)X0, res, keys, err);
}

// =====================================================================================
// RMSNorm of the fp32 residual stream into the next projection's input dtype.
// =====================================================================================
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(int H, const float* __restrict__ res,
                                                      const T* __restrict__ gamma, float eps,
                                                      int split, T* __restrict__ out) {
  __shared__ float red[32];
  pdl_enter();
  const int r = blockIdx.x;
  const float* x = res + (size_t)r * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) ss += x[i] * x[i];
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / H + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    store_act<T>(out, H, r, gridDim.x, split, i, x[i] * inv * ld(gamma + i));
}

void launch_rmsnorm(bool bf16m, int R, int H, const float* res, const void* gamma, float eps,
                    int split, void* out, cudaStream_t s) {
  if (bf16m)
    launch_pdl(rmsnorm_kernel<bf16>, dim3(R), dim3(256), 0, s, H, res, (const bf16*)gamma, eps,
               split, (bf16*)out);
  else
    rmsnorm_kernel<float><<<R, 256, 0, s>>>(H, res, (const float*)gamma, eps, 0, (float*)out);
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
  int total = L + a.K;
  if (total > a.cap) total = a.cap;  // overflow is reported by the QKV epilogue
  const int kbeg = c * a.chunk;
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
      const bool valid = kp < kend && kp <= L + j;
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
  __threadfence();
  __syncthreads();
  const int nvalid = cdiv(total, a.chunk);
  if (threadIdx.x == 0) {
    unsigned prev = atomicAdd(a.counters + b * a.nkv + g, 1u);
    s_last = (prev == (unsigned)(nvalid - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pbase = a.part + ((size_t)b * a.nkv + g) * a.nchunk * rows * (HD + 2);
  T* og = (T*)a.o;
  for (int rr = warp; rr < rows; rr += 8) {
    // chunk statistics in parallel: lane c holds chunks c and c + 32 (nchunk <= 64)
    float mc[2], lc[2], wc[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int cc = lane + 32 * t;
      mc[t] = -INFINITY;
      lc[t] = 0.f;
      if (cc < nvalid) {
        const float* pr = pbase + ((size_t)cc * rows + rr) * (HD + 2);
        mc[t] = __ldcg(pr + HD);
        lc[t] = __ldcg(pr + HD + 1);
      }
    }
    const float M = warp_max(fmaxf(mc[0], mc[1]));
#pragma unroll
    for (int t = 0; t < 2; ++t) wc[t] = (mc[t] == -INFINITY) ? 0.f : expf(mc[t] - M);
    const float Ls = warp_sum(lc[0] * wc[0] + lc[1] * wc[1]);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int cc = 0; cc < nvalid; ++cc) {
      const float w = __shfl_sync(0xffffffffu, cc < 32 ? wc[0] : wc[1], cc & 31);
      const float* pr = pbase + ((size_t)cc * rows + rr) * (HD + 2);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(__ldcg(pr + lane + 32 * e), w, acc[e]);
    }
    const int j = rr / G, h = g * G + (rr - j * G);
    const float inv = 1.f / Ls;
#pragma unroll
    for (int e = 0; e < E; ++e)
      store_act<T>(og, (size_t)a.nq * HD, b * a.K + j, a.B * a.K, a.split, h * HD + lane + 32 * e,
                   acc[e] * inv);
  }
  if (threadIdx.x == 0) a.counters[b * a.nkv + g] = 0u;
}

template <typename T, int HD>
static void attn_launch(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.K * (a.nq / a.nkv);
  size_t sm = (size_t)(rows * HD + 32 * (HD + 1) + 32 * HD) * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(attn_decode_kernel<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         200 * 1024);
    attr_set = true;
  }
  dim3 grid(a.nchunk, a.nkv, a.B);
  launch_pdl(attn_decode_kernel<T, HD>, grid, dim3(256), sm, s, a);
}

void launch_attention_decode(bool bf16m, const AttnArgs& a, cudaStream_t s) {
  if (bf16m) {
    if (a.hd == 64) attn_launch<bf16, 64>(a, s); else attn_launch<bf16, 128>(a, s);
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

void launch_masked_attention(bool bf16m, const MaskedAttnArgs& a, cudaStream_t s) {
  const long warps = (long)a.M * a.nq;
  dim3 grid((unsigned)((warps + 7) / 8));
  if (bf16m) {
    if (a.hd == 64) launch_pdl(masked_attn_kernel<bf16, 64>, grid, dim3(256), 0, s, a);
    else launch_pdl(masked_attn_kernel<bf16, 128>, grid, dim3(256), 0, s, a);
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
__global__ void rows_check_kernel(int M, int Kmax, const int* row_p, const int* row_d,
                                  const int* row_index, unsigned* err) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < M; i += gridDim.x * blockDim.x) {
    const int p = row_p[i], d = row_d[i];
    if (d >= 2 && p >= 1 && d <= Kmax + 1) {
      if (row_index[(size_t)(p - 1) * (Kmax + 1) + (d - 1)] < 0) raise_error(err, PEAGLE_DEV_BAD_ROW);
    }
  }
}

void launch_rows_prepare(int M, int n, int K, int Kmax, const int* row_p, const int* row_d,
                         int* row_index, unsigned* err, cudaStream_t s) {
  const int total = n * (Kmax + 1);
  rows_fill_kernel<<<cdiv(total, 256) < 1024 ? cdiv(total, 256) : 1024, 256, 0, s>>>(total, row_index);
  const int gb = cdiv(M, 256) < 1024 ? cdiv(M, 256) : 1024;
  rows_scatter_kernel<<<gb > 0 ? gb : 1, 256, 0, s>>>(M, n, K, Kmax, row_p, row_d, row_index, err);
  rows_check_kernel<<<gb > 0 ? gb : 1, 256, 0, s>>>(M, Kmax, row_p, row_d, row_index, err);
}

// =====================================================================================
// Argmax decode: key -> draft index -> target id via d2t; resets the key.
// =====================================================================================
__global__ void argmax_decode_kernel(int R, unsigned long long* keys, const int* d2t, int* out) {
  pdl_enter();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int idx = argmax_key_index(keys[r]);
  out[r] = d2t ? idx + d2t[idx] : idx;
  keys[r] = 0ull;
}

void launch_argmax_decode(int R, unsigned long long* keys, const int* d2t, int* out,
                          cudaStream_t s) {
  launch_pdl(argmax_decode_kernel, dim3(cdiv(R, 128)), dim3(128), 0, s, R, keys, d2t, out);
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
