// Fused backward of the training step's depth-1 prefix attention on TF32 tensor cores
// (mma.sync m16n8k8), for bf16 drafters: the probabilities are recomputed from the
// forward's log-sum-exp, so the dense [rows x positions] score matrices never exist.
// ("P-EAGLE: Parallel-Drafting EAGLE with Scalable Training", section 3: the drafter is
// trained over the n x K rows; "Speeding LLM inference with P-EAGLE in vLLM/Speculators",
// "Flex-attention mask": row (p, d) sees the depth-1 rows at positions 0 .. p - d + 1.)
//
// For one head h of kv group g, with S = scale * Q K1^T over the visible prefix,
// P = exp(S - lse), dP = dO V1^T, dS = scale * P * (dP - D) (D = dO . O per row):
//   dQ  += dS K1        query-major: attn_bwd_dq_kernel (adds to the chain part)
//   dK1 += dS^T Q,  dV1 += P^T dO   key-major: attn_bwd_dkv_kernel
// A dot product may run over k in any order its two operands share: each lane takes the
// physical elements 2t, 2t + 1 of an 8-wide k step for the logical positions t, t + 4 of
// the fragment, in A and in B alike, so fragments load as float2 and an accumulator
// fragment (columns 2t, 2t + 1) serves directly as the next product's A fragment.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "train_kernels.h"

namespace peagle {

namespace {

constexpr int FA_LD = 72;  // padded row stride (floats) of the shared-memory tiles

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// operands stored already rounded to TF32 (round_tf32_kernel) enter as their bits
__device__ __forceinline__ uint32_t bits(float x) { return __float_as_uint(x); }

__global__ void round_tf32_kernel(size_t n, float* p) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = __uint_as_float(tf32(p[i]));
}

__device__ __forceinline__ void mma_tf32(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte global -> shared copy; zero-filled when !valid
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ int anchor_row(const TrainAttn& a, int i) {
  if (i >= a.M) return -1;
  const int p = a.row_p[i], d = a.row_d[i];
  const bool ok = p >= 0 && p < a.n && d >= 1 && d <= a.K && p - d + 1 >= 0;
  return ok ? p - d + 1 : -1;
}

// 64 rows of 64 floats (K1 / V1 keys, or Q / dO rows) into a padded shared tile
__device__ __forceinline__ void stage64(float* dst, const float* src, int row0, int nrows,
                                        int tid, int nthr) {
  for (int c = tid; c < 64 * 16; c += nthr) {
    const int r = c >> 4, q = c & 15;
    const bool v = row0 + r < nrows;
    cp16(dst + r * FA_LD + q * 4, src + (size_t)(v ? row0 + r : 0) * 64 + q * 4, v);
  }
}

// ---- dQ: one CTA per (16 rows, kv group), one warp per head of the group --------------
// K1 / V1 tiles of 64 keys are staged (double-buffered) up to the largest anchor of the
// 16 rows; each warp keeps its Q and dO rows as A fragments and its dQ in registers, and
// adds dQ into dQh (which holds the chain part).
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(TrainAttn a, const float* Qh,
                                                          const float* dOh, const float* K1,
                                                          const float* V1, const float* lse,
                                                          const float* Dv, float* dQh) {
  extern __shared__ float smem[];  // [2 stages][K, V][64][FA_LD]
  const int G = a.nq / a.nkv, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const int i0 = blockIdx.x * 16;
  const int r0 = i0 + gq, r1 = r0 + 8;
  const int anc0 = anchor_row(a, r0), anc1 = anchor_row(a, r1);
  int amax = max(anc0, anc1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int nkeys = amax + 1;  // the same in every warp
  if (nkeys <= 0) return;
  const int ntiles = (nkeys + 63) / 64;
  const float* K1g = K1 + (size_t)g * a.n * 64;
  const float* V1g = V1 + (size_t)g * a.n * 64;
  const int nthr = blockDim.x;
  stage64(smem, K1g, 0, a.n, threadIdx.x, nthr);
  stage64(smem + 64 * FA_LD, V1g, 0, a.n, threadIdx.x, nthr);
  cp_commit();

  const bool live = warp < G;
  const int h = g * G + (live ? warp : 0);
  uint32_t qa[8][4], oa[8][4];
  float L0 = 0.f, L1 = 0.f, D0 = 0.f, D1 = 0.f;
  {
    const float* q0 = Qh + ((size_t)h * a.M + min(r0, a.M - 1)) * 64;
    const float* q1 = Qh + ((size_t)h * a.M + min(r1, a.M - 1)) * 64;
    const float* o0 = dOh + ((size_t)h * a.M + min(r0, a.M - 1)) * 64;
    const float* o1 = dOh + ((size_t)h * a.M + min(r1, a.M - 1)) * 64;
    const bool v0 = r0 < a.M, v1 = r1 < a.M;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const float2 x0 = v0 ? *reinterpret_cast<const float2*>(q0 + 8 * s + 2 * tq) : make_float2(0.f, 0.f);
      const float2 x1 = v1 ? *reinterpret_cast<const float2*>(q1 + 8 * s + 2 * tq) : make_float2(0.f, 0.f);
      const float2 y0 = v0 ? *reinterpret_cast<const float2*>(o0 + 8 * s + 2 * tq) : make_float2(0.f, 0.f);
      const float2 y1 = v1 ? *reinterpret_cast<const float2*>(o1 + 8 * s + 2 * tq) : make_float2(0.f, 0.f);
      qa[s][0] = bits(x0.x); qa[s][1] = bits(x1.x); qa[s][2] = bits(x0.y); qa[s][3] = bits(x1.y);
      oa[s][0] = bits(y0.x); oa[s][1] = bits(y1.x); oa[s][2] = bits(y0.y); oa[s][3] = bits(y1.y);
    }
    if (v0) { L0 = lse[(size_t)h * a.M + r0]; D0 = Dv[(size_t)h * a.M + r0]; }
    if (v1) { L1 = lse[(size_t)h * a.M + r1]; D1 = Dv[(size_t)h * a.M + r1]; }
  }
  float dq[8][4];
#pragma unroll
  for (int nn = 0; nn < 8; ++nn) dq[nn][0] = dq[nn][1] = dq[nn][2] = dq[nn][3] = 0.f;

  for (int kt = 0; kt < ntiles; ++kt) {
    float* cur = smem + (size_t)(kt & 1) * 2 * 64 * FA_LD;
    if (kt + 1 < ntiles) {
      float* nxt = smem + (size_t)((kt + 1) & 1) * 2 * 64 * FA_LD;
      stage64(nxt, K1g, (kt + 1) * 64, a.n, threadIdx.x, nthr);
      stage64(nxt + 64 * FA_LD, V1g, (kt + 1) * 64, a.n, threadIdx.x, nthr);
      cp_commit();
      cp_wait1();
    } else {
      cp_wait0();
    }
    __syncthreads();
    const float* Ks = cur;
    const float* Vs = cur + 64 * FA_LD;
    if (live) {
#pragma unroll 2
      for (int kk = 0; kk < 8; ++kk) {
        const int kbase = kt * 64 + kk * 8;
        if (kbase > amax) break;  // warp-uniform
        // even and odd k steps accumulate apart: four short dependency chains
        float sc[2][4] = {}, dp[2][4] = {};
        const float* kr = Ks + (kk * 8 + gq) * FA_LD + 2 * tq;
        const float* vr = Vs + (kk * 8 + gq) * FA_LD + 2 * tq;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const float2 kb = *reinterpret_cast<const float2*>(kr + 8 * s);
          const float2 vb = *reinterpret_cast<const float2*>(vr + 8 * s);
          mma_tf32(sc[s & 1], qa[s][0], qa[s][1], qa[s][2], qa[s][3], bits(kb.x), bits(kb.y));
          mma_tf32(dp[s & 1], oa[s][0], oa[s][1], oa[s][2], oa[s][3], bits(vb.x), bits(vb.y));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sc[0][e] += sc[1][e];
          dp[0][e] += dp[1][e];
        }
        // accumulator: (row gq, key 2tq), (gq, 2tq + 1), (gq + 8, 2tq), (gq + 8, 2tq + 1)
        const int k0 = kbase + 2 * tq, k1 = k0 + 1;
        const float p0 = k0 <= anc0 ? expf(sc[0][0] * a.scale - L0) : 0.f;
        const float p1 = k1 <= anc0 ? expf(sc[0][1] * a.scale - L0) : 0.f;
        const float p2 = k0 <= anc1 ? expf(sc[0][2] * a.scale - L1) : 0.f;
        const float p3 = k1 <= anc1 ? expf(sc[0][3] * a.scale - L1) : 0.f;
        const uint32_t d0 = tf32(p0 * (dp[0][0] - D0) * a.scale);
        const uint32_t d1 = tf32(p1 * (dp[0][1] - D0) * a.scale);
        const uint32_t d2 = tf32(p2 * (dp[0][2] - D1) * a.scale);
        const uint32_t d3 = tf32(p3 * (dp[0][3] - D1) * a.scale);
        // dQ += dS K1: A = dS (keys 2tq, 2tq + 1 as k positions tq, tq + 4), B = K1
        const float* kc0 = Ks + (kk * 8 + 2 * tq) * FA_LD + gq;
#pragma unroll
        for (int nn = 0; nn < 8; ++nn)
          mma_tf32(dq[nn], d0, d2, d1, d3, bits(kc0[8 * nn]), bits(kc0[FA_LD + 8 * nn]));
      }
    }
    __syncthreads();  // the stage is refilled next
  }
  if (!live) return;
  float* g0 = dQh + ((size_t)h * a.M + r0) * 64;
  float* g1 = dQh + ((size_t)h * a.M + r1) * 64;
#pragma unroll
  for (int nn = 0; nn < 8; ++nn) {
    const int c = 8 * nn + 2 * tq;
    if (r0 < a.M) { g0[c] += dq[nn][0]; g0[c + 1] += dq[nn][1]; }
    if (r1 < a.M) { g1[c] += dq[nn][2]; g1[c + 1] += dq[nn][3]; }
  }
}

// ---- dK1 / dV1: one CTA per (64 keys, kv group, chunk of rows), one warp per 16 keys ---
// Only rows at positions >= the block's first key can see it (rows are sorted by
// position); they start at the depth-1 row of that position.  Per (16 rows, head) the Q
// and dO rows are staged (double-buffered); each warp keeps its keys' K1 / V1 rows as A
// fragments and its dK1 / dV1 in registers, added into the outputs at the end (chunks of
// rows meet there).
constexpr int DKV_CHUNK = 512;

struct DkvStage {
  float q[16 * FA_LD];
  float o[16 * FA_LD];
  float L[16], D[16];
  int anc[16];
};

__global__ void __launch_bounds__(128, 3) attn_bwd_dkv_kernel(TrainAttn a, const int* row_index,
                                                           int Kmax, const float* Qh,
                                                           const float* dOh, const float* K1,
                                                           const float* V1, const float* lse,
                                                           const float* Dv, float* dK1,
                                                           float* dV1) {
  __shared__ __align__(16) DkvStage st[2];
  const int G = a.nq / a.nkv, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const int k0 = blockIdx.x * 64;
  if (k0 >= a.n) return;
  const int rs = row_index[(size_t)k0 * (Kmax + 1) + 1];
  if (rs < 0) return;  // no depth-1 row at k0: no row sees these keys
  const int rb = rs + blockIdx.z * DKV_CHUNK;
  if (rb >= a.M) return;
  const int re = min(a.M, rb + DKV_CHUNK);
  const int ntile = (re - rb + 15) / 16;
  const int niter = ntile * G;
  const float* K1g = K1 + (size_t)g * a.n * 64;
  const float* V1g = V1 + (size_t)g * a.n * 64;
  const int kw0 = k0 + warp * 16 + gq, kw1 = kw0 + 8;
  uint32_t ka[8][4], va[8][4];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int c = 8 * s + 2 * tq;
    const float2 x0 = kw0 < a.n ? *reinterpret_cast<const float2*>(K1g + (size_t)kw0 * 64 + c) : make_float2(0.f, 0.f);
    const float2 x1 = kw1 < a.n ? *reinterpret_cast<const float2*>(K1g + (size_t)kw1 * 64 + c) : make_float2(0.f, 0.f);
    const float2 y0 = kw0 < a.n ? *reinterpret_cast<const float2*>(V1g + (size_t)kw0 * 64 + c) : make_float2(0.f, 0.f);
    const float2 y1 = kw1 < a.n ? *reinterpret_cast<const float2*>(V1g + (size_t)kw1 * 64 + c) : make_float2(0.f, 0.f);
    ka[s][0] = bits(x0.x); ka[s][1] = bits(x1.x); ka[s][2] = bits(x0.y); ka[s][3] = bits(x1.y);
    va[s][0] = bits(y0.x); va[s][1] = bits(y1.x); va[s][2] = bits(y0.y); va[s][3] = bits(y1.y);
  }
  float dk[8][4], dv[8][4];
#pragma unroll
  for (int nn = 0; nn < 8; ++nn)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[nn][e] = dv[nn][e] = 0.f;

  // stage iteration it = (16-row tile, head) into buffer b
  auto stage = [&](int it, int b) {
    const int i0 = rb + (it / G) * 16, h = g * G + it % G;
    for (int c = threadIdx.x; c < 16 * 16 * 2; c += 128) {
      const int which = c >> 8, r = (c >> 4) & 15, q = c & 15;
      const int i = i0 + r;
      const bool v = i < re;
      const float* src = (which ? dOh : Qh) + ((size_t)h * a.M + (v ? i : 0)) * 64 + q * 4;
      cp16((which ? st[b].o : st[b].q) + r * FA_LD + q * 4, src, v);
    }
    if (threadIdx.x < 16) {
      const int i = i0 + threadIdx.x;
      const bool v = i < re;
      st[b].L[threadIdx.x] = v ? lse[(size_t)h * a.M + i] : 0.f;
      st[b].D[threadIdx.x] = v ? Dv[(size_t)h * a.M + i] : 0.f;
      st[b].anc[threadIdx.x] = v ? anchor_row(a, i) : -1;
    }
    cp_commit();
  };
  stage(0, 0);
  for (int it = 0; it < niter; ++it) {
    const int b = it & 1;
    if (it + 1 < niter) {
      stage(it + 1, b ^ 1);
      cp_wait1();
    } else {
      cp_wait0();
    }
    __syncthreads();
    const DkvStage& S = st[b];
    // even and odd k steps accumulate apart: eight short dependency chains
    float sT[2][4], dpT[2][4], sT2[2][4], dpT2[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sT[j][e] = dpT[j][e] = sT2[j][e] = dpT2[j][e] = 0.f;
      const float* qr = S.q + (8 * j + gq) * FA_LD + 2 * tq;
      const float* orow = S.o + (8 * j + gq) * FA_LD + 2 * tq;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float2 qb = *reinterpret_cast<const float2*>(qr + 8 * s);
        const float2 ob = *reinterpret_cast<const float2*>(orow + 8 * s);
        mma_tf32((s & 1) ? sT2[j] : sT[j], ka[s][0], ka[s][1], ka[s][2], ka[s][3], bits(qb.x),
                 bits(qb.y));
        mma_tf32((s & 1) ? dpT2[j] : dpT[j], va[s][0], va[s][1], va[s][2], va[s][3], bits(ob.x),
                 bits(ob.y));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sT[j][e] += sT2[j][e];
        dpT[j][e] += dpT2[j][e];
      }
    }
    // accumulator j: (key kw0, row 8j + 2tq), (kw0, 8j + 2tq + 1), (kw1, 8j + 2tq), (kw1, +1)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int ra = 8 * j + 2 * tq, rb2 = ra + 1;
      const int aa = S.anc[ra], ab = S.anc[rb2];
      const float La = S.L[ra], Lb = S.L[rb2], Da = S.D[ra], Db = S.D[rb2];
      const float p0 = kw0 <= aa ? expf(sT[j][0] * a.scale - La) : 0.f;
      const float p1 = kw0 <= ab ? expf(sT[j][1] * a.scale - Lb) : 0.f;
      const float p2 = kw1 <= aa ? expf(sT[j][2] * a.scale - La) : 0.f;
      const float p3 = kw1 <= ab ? expf(sT[j][3] * a.scale - Lb) : 0.f;
      const uint32_t P0 = tf32(p0), P1 = tf32(p1), P2 = tf32(p2), P3 = tf32(p3);
      const uint32_t d0 = tf32(p0 * (dpT[j][0] - Da) * a.scale);
      const uint32_t d1 = tf32(p1 * (dpT[j][1] - Db) * a.scale);
      const uint32_t d2 = tf32(p2 * (dpT[j][2] - Da) * a.scale);
      const uint32_t d3 = tf32(p3 * (dpT[j][3] - Db) * a.scale);
      // A = P^T / dS^T over the rows ra, rb2 of this k step (k positions tq, tq + 4)
      const float* o0 = S.o + ra * FA_LD + gq;
      const float* q0 = S.q + ra * FA_LD + gq;
#pragma unroll
      for (int nn = 0; nn < 8; ++nn) {
        mma_tf32(dv[nn], P0, P2, P1, P3, bits(o0[8 * nn]), bits(o0[FA_LD + 8 * nn]));
        mma_tf32(dk[nn], d0, d2, d1, d3, bits(q0[8 * nn]), bits(q0[FA_LD + 8 * nn]));
      }
    }
    __syncthreads();  // the buffer is refilled next
  }
  float* gk = dK1 + (size_t)g * a.n * 64;
  float* gv = dV1 + (size_t)g * a.n * 64;
#pragma unroll
  for (int nn = 0; nn < 8; ++nn) {
    const int c = 8 * nn + 2 * tq;
    if (kw0 < a.n) {
      atomicAdd(gk + (size_t)kw0 * 64 + c, dk[nn][0]);
      atomicAdd(gk + (size_t)kw0 * 64 + c + 1, dk[nn][1]);
      atomicAdd(gv + (size_t)kw0 * 64 + c, dv[nn][0]);
      atomicAdd(gv + (size_t)kw0 * 64 + c + 1, dv[nn][1]);
    }
    if (kw1 < a.n) {
      atomicAdd(gk + (size_t)kw1 * 64 + c, dk[nn][2]);
      atomicAdd(gk + (size_t)kw1 * 64 + c + 1, dk[nn][3]);
      atomicAdd(gv + (size_t)kw1 * 64 + c, dv[nn][2]);
      atomicAdd(gv + (size_t)kw1 * 64 + c + 1, dv[nn][3]);
    }
  }
}

}  // namespace

bool attn_bwd_fused_ok(const TrainAttn& a) {
  const int G = a.nq / a.nkv;
  return a.hd == 64 && G >= 1 && G <= 8;
}

void launch_attn_bwd_fused(const TrainAttn& a, const int* row_index, int Kmax, const float* Qh,
                           const float* dOh, const float* K1, const float* V1,
                           const float* lse, const float* Dv, float* dQh, float* dK1,
                           float* dV1, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  const size_t smem = (size_t)2 * 2 * 64 * FA_LD * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr_set = true;
  }
  // the stored operands are rounded to TF32 once here, not per use in the products
  for (float* p : {(float*)Qh, (float*)dOh}) round_tf32_kernel<<<1024, 256, 0, s>>>((size_t)a.nq * a.M * 64, p);
  for (float* p : {(float*)K1, (float*)V1}) round_tf32_kernel<<<256, 256, 0, s>>>((size_t)a.nkv * a.n * 64, p);
  attn_bwd_dq_kernel<<<dim3((a.M + 15) / 16, a.nkv), 32 * G, smem, s>>>(a, Qh, dOh, K1, V1, lse,
                                                                       Dv, dQh);
  attn_bwd_dkv_kernel<<<dim3((a.n + 63) / 64, a.nkv, (a.M + DKV_CHUNK - 1) / DKV_CHUNK), 128, 0,
                        s>>>(a, row_index, Kmax, Qh, dOh, K1, V1, lse, Dv, dK1, dV1);
}

}  // namespace peagle
