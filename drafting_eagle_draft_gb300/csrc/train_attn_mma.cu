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
// Column swizzle of the tiles: rows with bit 2 set hold their 8-float column groups in
// swapped pairs (column c stored at c ^ 8).  Fragments read the tiles two ways: float2
// along a row (rows gq, columns 2tq + 8s), conflict-free with the 72-float stride alone,
// and single floats down rows (rows 2tq, 2tq + 1, columns gq + 8n), where rows 0 and 4
// (and 2 and 6) would share banks; the swizzle moves one of each pair by eight banks.
__device__ __forceinline__ int fa_sw(int row) { return (row >> 2) & 1; }
// Column group g of a row with swizzle bit b lives at group g ^ b: from a pointer p to the
// row's group-0 position, group g is at (g even ? p + 8b : p - 8b) + 8g, so unrolled loops
// keep two base pointers and constant offsets.
__device__ __forceinline__ const float* fa_even(const float* p, int b) { return p + 8 * b; }
__device__ __forceinline__ const float* fa_odd(const float* p, int b) { return p - 8 * b; }

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// operands stored already rounded to TF32 by their producers (the RoPE kernel for Q, K1 and
// V1, the backward's preparation kernel for dO) enter as their bits
__device__ __forceinline__ uint32_t bits(float x) { return __float_as_uint(x); }

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
    cp16(dst + r * FA_LD + 4 * (q ^ (fa_sw(r) << 1)), src + (size_t)(v ? row0 + r : 0) * 64 + q * 4,
         v);
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
        const int bg = fa_sw(gq);
        const float *kre = fa_even(kr, bg), *kro = fa_odd(kr, bg);
        const float *vre = fa_even(vr, bg), *vro = fa_odd(vr, bg);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const float2 kb = *reinterpret_cast<const float2*>(((s & 1) ? kro : kre) + 8 * s);
          const float2 vb = *reinterpret_cast<const float2*>(((s & 1) ? vro : vre) + 8 * s);
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
        const int bt = fa_sw(2 * tq);
        const float *kce = fa_even(kc0, bt), *kco = fa_odd(kc0, bt);
#pragma unroll
        for (int nn = 0; nn < 8; ++nn) {
          const float* kc = (nn & 1) ? kco : kce;
          mma_tf32(dq[nn], d0, d2, d1, d3, bits(kc[8 * nn]), bits(kc[FA_LD + 8 * nn]));
        }
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
      cp16((which ? st[b].o : st[b].q) + r * FA_LD + 4 * (q ^ (fa_sw(r) << 1)), src, v);
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
      const int bg = fa_sw(gq);
      const float *qre = fa_even(qr, bg), *qro = fa_odd(qr, bg);
      const float *ore = fa_even(orow, bg), *oro = fa_odd(orow, bg);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float2 qb = *reinterpret_cast<const float2*>(((s & 1) ? qro : qre) + 8 * s);
        const float2 ob = *reinterpret_cast<const float2*>(((s & 1) ? oro : ore) + 8 * s);
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
      const int bt = fa_sw(ra);
      const float *o0e = fa_even(o0, bt), *o0o = fa_odd(o0, bt);
      const float *q0e = fa_even(q0, bt), *q0o = fa_odd(q0, bt);
#pragma unroll
      for (int nn = 0; nn < 8; ++nn) {
        const float* ob = (nn & 1) ? o0o : o0e;
        const float* qb = (nn & 1) ? q0o : q0e;
        mma_tf32(dv[nn], P0, P2, P1, P3, bits(ob[8 * nn]), bits(ob[FA_LD + 8 * nn]));
        mma_tf32(dk[nn], d0, d2, d1, d3, bits(qb[8 * nn]), bits(qb[FA_LD + 8 * nn]));
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

// ---- forward: one CTA per (16 rows, kv group), one warp per head --------------------
// Online softmax over the depth-1 prefix (K1 / V1 tiles of 64 keys staged as in the dQ
// kernel): per tile the scores of the warp's 16 rows, the running row max m and sum l
// (each row's four lanes reduce with shuffles), the accumulator O rescaled and P V added.
// Writes the unnormalised prefix O (per-head rows) and m, l; attn_fwd_combine_kernel then
// adds the chain keys and normalises.
__global__ void __launch_bounds__(256) attn_fwd_prefix_kernel(TrainAttn a, const float* Qh,
                                                              const float* K1, const float* V1,
                                                              float* Op, float* mrow,
                                                              float* lrow) {
  extern __shared__ float smem[];  // [2 stages][K, V][64][FA_LD]
  const int G = a.nq / a.nkv, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const int i0 = blockIdx.x * 16;
  const int r0 = i0 + gq, r1 = r0 + 8;
  const int anc0 = anchor_row(a, r0), anc1 = anchor_row(a, r1);
  int amax = max(anc0, anc1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const bool live = warp < G;
  const int h = g * G + (live ? warp : 0);
  const int ntiles = (amax + 64) / 64;  // 0 when no row sees a key
  const float* K1g = K1 + (size_t)g * a.n * 64;
  const float* V1g = V1 + (size_t)g * a.n * 64;
  const int nthr = blockDim.x;
  if (ntiles > 0) {
    stage64(smem, K1g, 0, a.n, threadIdx.x, nthr);
    stage64(smem + 64 * FA_LD, V1g, 0, a.n, threadIdx.x, nthr);
    cp_commit();
  }
  uint32_t qa[8][4];
  {
    const float* q0 = Qh + ((size_t)h * a.M + min(r0, a.M - 1)) * 64;
    const float* q1 = Qh + ((size_t)h * a.M + min(r1, a.M - 1)) * 64;
    const bool v0 = r0 < a.M, v1 = r1 < a.M;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const float2 x0 = v0 ? *reinterpret_cast<const float2*>(q0 + 8 * s + 2 * tq) : make_float2(0.f, 0.f);
      const float2 x1 = v1 ? *reinterpret_cast<const float2*>(q1 + 8 * s + 2 * tq) : make_float2(0.f, 0.f);
      qa[s][0] = bits(x0.x); qa[s][1] = bits(x1.x); qa[s][2] = bits(x0.y); qa[s][3] = bits(x1.y);
    }
  }
  float o[8][4];
#pragma unroll
  for (int nn = 0; nn < 8; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq, gq + 8
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
      // scores of the tile's 64 keys: 8 groups of 8 (even / odd k steps apart)
      float sc[8][4];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        float e[2][4] = {};
        const float* kr = Ks + (kk * 8 + gq) * FA_LD + 2 * tq;
        const int bg = fa_sw(gq);
        const float *kre = fa_even(kr, bg), *kro = fa_odd(kr, bg);
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
          const float2 kb = *reinterpret_cast<const float2*>(((s2 & 1) ? kro : kre) + 8 * s2);
          mma_tf32(e[s2 & 1], qa[s2][0], qa[s2][1], qa[s2][2], qa[s2][3], bits(kb.x), bits(kb.y));
        }
        const int k0 = kt * 64 + kk * 8 + 2 * tq, k1 = k0 + 1;
        sc[kk][0] = k0 <= anc0 ? (e[0][0] + e[1][0]) * a.scale : -INFINITY;
        sc[kk][1] = k1 <= anc0 ? (e[0][1] + e[1][1]) * a.scale : -INFINITY;
        sc[kk][2] = k0 <= anc1 ? (e[0][2] + e[1][2]) * a.scale : -INFINITY;
        sc[kk][3] = k1 <= anc1 ? (e[0][3] + e[1][3]) * a.scale : -INFINITY;
      }
      float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        t0 = fmaxf(t0, fmaxf(sc[kk][0], sc[kk][1]));
        t1 = fmaxf(t1, fmaxf(sc[kk][2], sc[kk][3]));
      }
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, 1));
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, 2));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, 1));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, 2));
      const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
      // rescale what was accumulated (no key yet: nothing to rescale)
      const float f0 = n0 == -INFINITY ? 1.f : expf(m0 - n0);
      const float f1 = n1 == -INFINITY ? 1.f : expf(m1 - n1);
#pragma unroll
      for (int nn = 0; nn < 8; ++nn) {
        o[nn][0] *= f0; o[nn][1] *= f0;
        o[nn][2] *= f1; o[nn][3] *= f1;
      }
      l0 *= f0;
      l1 *= f1;
      m0 = n0;
      m1 = n1;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const float p0 = sc[kk][0] == -INFINITY ? 0.f : expf(sc[kk][0] - n0);
        const float p1 = sc[kk][1] == -INFINITY ? 0.f : expf(sc[kk][1] - n0);
        const float p2 = sc[kk][2] == -INFINITY ? 0.f : expf(sc[kk][2] - n1);
        const float p3 = sc[kk][3] == -INFINITY ? 0.f : expf(sc[kk][3] - n1);
        s0 += p0 + p1;
        s1 += p2 + p3;
        // O += P V over these 8 keys: A = P (keys 2tq, 2tq + 1 as k positions tq, tq + 4)
        const float* vc = Vs + (kk * 8 + 2 * tq) * FA_LD + gq;
        const int bt = fa_sw(2 * tq);
        const float *vce = fa_even(vc, bt), *vco = fa_odd(vc, bt);
        const uint32_t P0 = tf32(p0), P1 = tf32(p1), P2 = tf32(p2), P3 = tf32(p3);
#pragma unroll
        for (int nn = 0; nn < 8; ++nn) {
          const float* vb = (nn & 1) ? vco : vce;
          mma_tf32(o[nn], P0, P2, P1, P3, bits(vb[8 * nn]), bits(vb[FA_LD + 8 * nn]));
        }
      }
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      l0 += s0;
      l1 += s1;
    }
    __syncthreads();
  }
  if (!live) return;
  float* g0 = Op + ((size_t)h * a.M + r0) * 64;
  float* g1 = Op + ((size_t)h * a.M + r1) * 64;
#pragma unroll
  for (int nn = 0; nn < 8; ++nn) {
    const int c = 8 * nn + 2 * tq;
    if (r0 < a.M) { g0[c] = o[nn][0]; g0[c + 1] = o[nn][1]; }
    if (r1 < a.M) { g1[c] = o[nn][2]; g1[c + 1] = o[nn][3]; }
  }
  if (tq == 0) {
    if (r0 < a.M) { mrow[(size_t)h * a.M + r0] = m0; lrow[(size_t)h * a.M + r0] = l0; }
    if (r1 < a.M) { mrow[(size_t)h * a.M + r1] = m1; lrow[(size_t)h * a.M + r1] = l1; }
  }
}

// One warp per (head, row): the chain keys' scores join the prefix's running max and sum;
// lse, the chain probabilities Pc and the normalised output row O [M][nq hd].
__global__ void attn_fwd_combine_kernel(TrainAttn a, const float* Qh, const float* Kr,
                                        const float* Vr, const float* Op, const float* mrow,
                                        const float* lrow, float* Pc, float* lse, float* O) {
  const int lane = threadIdx.x & 31, G = a.nq / a.nkv, K1n = a.K - 1;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= a.nq * a.M) return;
  const int h = w / a.M, i = w % a.M, g = h / G;
  const float* q = Qh + ((size_t)h * a.M + i) * 64;
  float cs[16];
  float m = mrow[(size_t)h * a.M + i];
  const float mp = m;
  for (int t = 0; t < K1n; ++t) {
    const int r = a.chain[(size_t)i * K1n + t];
    float sv = -INFINITY;
    if (r >= 0) {
      const float* kr = Kr + ((size_t)r * a.nkv + g) * 64;
      float d = q[lane] * kr[lane] + q[lane + 32] * kr[lane + 32];
      d = warp_sum(d);
      sv = d * a.scale;
    }
    cs[t] = sv;
    m = fmaxf(m, sv);
  }
  const float fp = (mp == -INFINITY) ? 0.f : expf(mp - m);
  float l = lrow[(size_t)h * a.M + i] * fp;
  for (int t = 0; t < K1n; ++t) l += cs[t] == -INFINITY ? 0.f : expf(cs[t] - m);
  const float L = (l > 0.f) ? m + logf(l) : 0.f;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float o0 = Op[((size_t)h * a.M + i) * 64 + lane] * fp;
  float o1 = Op[((size_t)h * a.M + i) * 64 + lane + 32] * fp;
  for (int t = 0; t < K1n; ++t) {
    const int r = a.chain[(size_t)i * K1n + t];
    if (r < 0) continue;
    const float pw = expf(cs[t] - m);
    const float* vr = Vr + ((size_t)r * a.nkv + g) * 64;
    o0 += pw * vr[lane];
    o1 += pw * vr[lane + 32];
  }
  float* orow = O + (size_t)i * a.nq * 64 + h * 64;
  orow[lane] = o0 * inv;
  orow[lane + 32] = o1 * inv;
  if (lane < K1n)
    Pc[((size_t)h * a.M + i) * K1n + lane] = cs[lane] == -INFINITY ? 0.f : expf(cs[lane] - L);
  if (lane == 0) lse[(size_t)h * a.M + i] = L;
}

}  // namespace

bool attn_bwd_fused_ok(const TrainAttn& a) {
  const int G = a.nq / a.nkv;
  return a.hd == 64 && G >= 1 && G <= 8;
}

int launch_attn_fwd_fused(const TrainAttn& a, float* Qh, const float* Kr, const float* Vr,
                          float* K1, float* V1, float* Op, float* mrow, float* lrow, float* Pc,
                          float* lse, float* O, const TrainAttnTc* tcx, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  if (tcx && attn_tc_ok(a)) {
    const int r = launch_attn_fwd_prefix_tc(a, *tcx, Qh, K1, V1, Op, mrow, lrow, s);
    if (r != PEAGLE_OK) return r;
  } else {
    const size_t smem = (size_t)2 * 2 * 64 * FA_LD * sizeof(float);
    if (smem_optin((const void*)attn_fwd_prefix_kernel, (int)smem) != cudaSuccess)
      return PEAGLE_ERR_CUDA;
    attn_fwd_prefix_kernel<<<dim3((a.M + 15) / 16, a.nkv), 32 * G, smem, s>>>(a, Qh, K1, V1, Op,
                                                                             mrow, lrow);
  }
  attn_fwd_combine_kernel<<<(a.nq * a.M + 7) / 8, 256, 0, s>>>(a, Qh, Kr, Vr, Op, mrow, lrow, Pc,
                                                              lse, O);
  return PEAGLE_OK;
}

int launch_attn_bwd_fused(const TrainAttn& a, const int* row_index, int Kmax, const float* Qh,
                          const float* dOh, const float* K1, const float* V1,
                          const float* lse, const float* Dv, float* dQh, float* dK1,
                          float* dV1, const TrainAttnTc* tcx, cudaStream_t s) {
  const int G = a.nq / a.nkv;
  const size_t smem = (size_t)2 * 2 * 64 * FA_LD * sizeof(float);
  if (tcx && attn_tc_ok(a)) {
    const int r = launch_attn_bwd_dq_tc(a, *tcx, Qh, dOh, K1, V1, lse, Dv, dQh, s);
    if (r != PEAGLE_OK) return r;
  } else {
    if (smem_optin((const void*)attn_bwd_dq_kernel, (int)smem) != cudaSuccess)
      return PEAGLE_ERR_CUDA;
    attn_bwd_dq_kernel<<<dim3((a.M + 15) / 16, a.nkv), 32 * G, smem, s>>>(a, Qh, dOh, K1, V1,
                                                                         lse, Dv, dQh);
  }
  if (tcx && attn_tc_ok(a) && tcx->qT) {
    const int r = launch_attn_bwd_dkv_tc(a, *tcx, row_index, Kmax, Qh, dOh, K1, V1, lse, Dv,
                                         dK1, dV1, s);
    if (r != PEAGLE_OK) return r;
  } else {
    attn_bwd_dkv_kernel<<<dim3((a.n + 63) / 64, a.nkv, (a.M + DKV_CHUNK - 1) / DKV_CHUNK), 128,
                          0, s>>>(a, row_index, Kmax, Qh, dOh, K1, V1, lse, Dv, dK1, dV1);
  }
  return PEAGLE_OK;
}

}  // namespace peagle
