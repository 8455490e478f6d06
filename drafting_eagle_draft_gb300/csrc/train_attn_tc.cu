// The training step's depth-1 prefix attention on the 5th-generation tensor cores
// (tcgen05.mma kind::tf32, fp32 accumulators in tensor memory), head_dim 64.
// ("P-EAGLE: Parallel-Drafting EAGLE with Scalable Training", section 3: the drafter is
// trained over the n x K rows; "Speeding LLM inference with P-EAGLE in vLLM/Speculators",
// "Flex-attention mask": row (p, d) sees the depth-1 rows at positions 0 .. p - d + 1, its
// anchor.)
//
// Forward: a CTA serves 128 MMA rows, the (query row, q head) pairs of 128 / G consecutive
// rows for the G q heads of kv head g (MMA row t = head (t / Rq), row i0 + t % Rq), and
// walks the keys 0 .. the rows' largest anchor in tiles of 32:
//   S = Q K1^T     M = 128, N = 32, K = 64 (two tensor-memory buffers: S of tile t + 2 is
//                  computed while tile t + 1's softmax runs)
//   softmax        warps 0-3, one thread per MMA row: tcgen05.ld of its 32 scores, the
//                  anchor mask, the running max (log2 domain; the reference max moves only
//                  when a tile's max exceeds it by more than 8, so the output is rarely
//                  rescaled) and sum; the probabilities, rounded to TF32, go to one of two
//                  shared-memory tiles
//   O += P V1      M = 128, N = 64, K = 32 keys: B is V1 transposed ([64][n]), K-major
// Warp 4 issues the MMAs, warp 5 the TMA loads (queries once; K1 tiles in a 3-stage ring,
// V1^T tiles in a 2-stage ring); the roles hand over through mbarriers only.  The output
// is the unnormalised prefix O with the row max (natural-log domain) and sum, as the
// mma.sync kernel writes them; the chain keys join afterwards.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "gemm_tc.h"
#include "gemm_tf32.h"
#include "tc_ptx.cuh"
#include "train_kernels.h"

namespace peagle {

namespace {

constexpr int AT_THREADS = 224;
constexpr int AT_KT = 32;          // keys per tile
constexpr int AT_KST = 3;          // K1 ring stages
constexpr int AT_VST = 2;          // V1^T ring stages
constexpr int AT_Q = 2 * 16384;    // 128 rows x 64 fp32: two k-blocks of 128 rows x 128 B
constexpr int AT_P = 16384;        // 128 rows x 32 fp32 probabilities (one k-block)
constexpr int AT_K = 2 * 4096;     // 32 keys x 64 fp32: two k-blocks of 32 rows x 128 B
constexpr int AT_V = 8192;         // V^T: 64 head dims x 32 keys (one k-block)
constexpr uint64_t AT_WAIT_NS = 2000000000ull;
constexpr uint64_t AT_DRAIN_NS = 10000000ull;

size_t at_fwd_smem() {
  return 1024 + AT_Q + 2 * AT_P + (size_t)AT_KST * AT_K + (size_t)AT_VST * AT_V;
}

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// 2^x (the SFU's approximation; relative error about 2^-22, below TF32's rounding)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16-byte chunk c of row r of a 128-byte-swizzled K-major tile (1024-byte aligned base)
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

struct AtFwdArgs {
  int M, n, K, G, Rq;
  float scale_log2;  // softmax scale * log2(e)
  const int* row_p;
  const int* row_d;
  float* Op;
  float* mrow;
  float* lrow;
  unsigned* err;
};

__device__ __forceinline__ int at_anchor(const AtFwdArgs& a, int i) {
  if (i >= a.M) return -1;
  const int p = a.row_p[i], d = a.row_d[i];
  const bool ok = p >= 0 && p < a.n && d >= 1 && d <= a.K && p - d + 1 >= 0;
  return ok ? p - d + 1 : -1;
}

__global__ void __launch_bounds__(AT_THREADS, 2)
    attn_fwd_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmVt, AtFwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sP = sQ + AT_Q;          // two tiles
  uint8_t* sK = sP + 2 * AT_P;
  uint8_t* sV = sK + AT_KST * AT_K;
  __shared__ uint64_t q_full, k_full[AT_KST], k_empty[AT_KST], v_full[AT_VST], v_empty[AT_VST];
  __shared__ uint64_t s_full[2], p_full[2], pv_done[2], fin;
  __shared__ uint32_t s_tmem;
  __shared__ int s_amax;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int blk = gridDim.x - 1 - blockIdx.x;  // row blocks with the most keys start first
  const int i0 = blk * a.Rq;
  if (tid == 0) {
    s_amax = -1;
    s_abort = 0;
    tc::mbar_init(&q_full, 1);
    for (int k = 0; k < AT_KST; ++k) {
      tc::mbar_init(&k_full[k], 1);
      tc::mbar_init(&k_empty[k], 1);
    }
    for (int k = 0; k < AT_VST; ++k) {
      tc::mbar_init(&v_full[k], 1);
      tc::mbar_init(&v_empty[k], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&s_full[b], 1);
      tc::mbar_init(&p_full[b], 4);  // one arrival per softmax warp
      tc::mbar_init(&pv_done[b], 1);
    }
    tc::mbar_init(&fin, 1);
    tc::fence_barrier_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(&s_tmem, 128u);
    tc::tmem_relinquish();
  }
  // softmax thread t: MMA row t = (head t / Rq, query row i0 + t % Rq)
  const int hl = tid < 128 ? tid / a.Rq : 0, r = tid < 128 ? tid - hl * a.Rq : 0;
  const int i = i0 + r, h = g * a.G + hl;
  const int anc = tid < 128 ? at_anchor(a, i) : -1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (anc >= 0) atomicMax(&s_amax, anc);
  __syncthreads();
  const int T = s_amax >= 0 ? s_amax / AT_KT + 1 : 0;
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem, tO = tmem + 64;  // S buffers at columns 0 / 32, O at 64
  auto fail = [&]() {
    if (!s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
    s_abort = 1;
  };

  if (warp >= 5) {
    // ---- TMA producers: warp 5 the queries and the K1 ring, warp 6 the V1^T ring (apart,
    // so that neither ring's wait holds the other's loads back)
    if (lane == 0 && T > 0) {
      const uint64_t pol = tc::policy_evict_last();
      int issued = 0;
      if (warp == 5) {
        const int krow0 = g * a.n;  // K1 viewed as [nkv n][64]
        tc::mbar_expect_tx(&q_full, (uint32_t)AT_Q);
        for (int q = 0; q < a.G; ++q)
          for (int kb = 0; kb < 2; ++kb)
            tc::tma_load_2d(sQ + kb * 16384 + q * a.Rq * 128, &tmQ, kb * 32,
                            (g * a.G + q) * a.M + i0, &q_full, pol);
        for (int j = 0; j < T; ++j, ++issued) {
          const int ks = j % AT_KST;
          if (j >= AT_KST && !tc::mbar_wait(&k_empty[ks], (uint32_t)((j / AT_KST - 1) & 1),
                                            &s_abort, AT_WAIT_NS)) {
            fail();
            break;
          }
          tc::mbar_expect_tx(&k_full[ks], (uint32_t)AT_K);
          tc::tma_load_2d(sK + ks * AT_K, &tmK, 0, krow0 + j * AT_KT, &k_full[ks], pol);
          tc::tma_load_2d(sK + ks * AT_K + 4096, &tmK, 32, krow0 + j * AT_KT, &k_full[ks], pol);
        }
      } else {
        for (int j = 0; j < T; ++j, ++issued) {
          const int vs = j % AT_VST;
          if (j >= AT_VST && !tc::mbar_wait(&v_empty[vs], (uint32_t)((j / AT_VST - 1) & 1),
                                            &s_abort, AT_WAIT_NS)) {
            fail();
            break;
          }
          tc::mbar_expect_tx(&v_full[vs], (uint32_t)AT_V);
          tc::tma_load_2d(sV + vs * AT_V, &tmVt, j * AT_KT, g * 64, &v_full[vs], pol);
        }
      }
      if (s_abort) {  // the loads in flight land (bounded) before the CTA can exit
        int never = 0;
        if (warp == 5) {
          tc::mbar_wait(&q_full, 0u, &never, AT_DRAIN_NS);
          for (int j = (issued > AT_KST ? issued - AT_KST : 0); j < issued; ++j)
            tc::mbar_wait(&k_full[j % AT_KST], (uint32_t)((j / AT_KST) & 1), &never,
                          AT_DRAIN_NS);
        } else {
          for (int j = (issued > AT_VST ? issued - AT_VST : 0); j < issued; ++j)
            tc::mbar_wait(&v_full[j % AT_VST], (uint32_t)((j / AT_VST) & 1), &never,
                          AT_DRAIN_NS);
        }
      }
    }
  } else if (warp == 4) {
    // ---- MMA issuer
    if (lane == 0 && T > 0) {
      const uint32_t idS = tc::idesc_tf32(128, AT_KT), idPV = tc::idesc_tf32(128, 64);
      auto issue_s = [&](int j) -> bool {  // S(j) = Q K1(j)^T into buffer j & 1
        const int ks = j % AT_KST;
        if (!tc::mbar_wait(&k_full[ks], (uint32_t)((j / AT_KST) & 1), &s_abort, AT_WAIT_NS))
          return false;
        tc::fence_after_sync();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(sQ + kb * 16384));
          const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(sK + ks * AT_K + kb * 4096));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_tf32(tS + (uint32_t)((j & 1) * AT_KT), ad + 2 * k, bd + 2 * k, idS,
                         (kb | k) ? 1u : 0u);
        }
        tc::mma_commit(&s_full[j & 1]);
        tc::mma_commit(&k_empty[ks]);
        return true;
      };
      bool ok = tc::mbar_wait(&q_full, 0u, &s_abort, AT_WAIT_NS);
      for (int j = 0; ok && j < 2 && j < T; ++j) ok = issue_s(j);
      for (int t = 0; ok && t < T; ++t) {
        // P(t) written (S(t) read, the output rescaled where needed)
        const int vs = t % AT_VST;
        if (!tc::mbar_wait(&p_full[t & 1], (uint32_t)((t >> 1) & 1), &s_abort, AT_WAIT_NS) ||
            !tc::mbar_wait(&v_full[vs], (uint32_t)((t / AT_VST) & 1), &s_abort, AT_WAIT_NS)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(sP + (t & 1) * AT_P));
        const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(sV + vs * AT_V));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_tf32(tO, ad + 2 * k, bd + 2 * k, idPV, (t > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&pv_done[t & 1]);
        tc::mma_commit(&v_empty[vs]);
        if (t + 2 < T) ok = issue_s(t + 2);
      }
      if (!ok) fail();
      // every MMA issued has completed before tensor memory is freed
      int never = 0;
      tc::mma_commit(&fin);
      tc::mbar_wait(&fin, 0u, &never, AT_DRAIN_NS);
    }
  } else {
    // ---- softmax warps
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_used = -INFINITY, l = 0.f;  // log2 domain
    for (int t = 0; t < T; ++t) {
      if (!tc::mbar_wait(&s_full[t & 1], (uint32_t)((t >> 1) & 1), &s_abort, AT_WAIT_NS))
        fail();
      tc::fence_after_sync();
      float sv[AT_KT];
      tc::tmem_ld32(tS + lane_off + (uint32_t)((t & 1) * AT_KT), sv);
      tc::tmem_ld_wait();
      const int lim = anc - t * AT_KT;  // keys j <= lim of the tile are visible
      if (lim < AT_KT - 1) {
#pragma unroll
        for (int j = 0; j < AT_KT; ++j)
          if (j > lim) sv[j] = -INFINITY;
      }
      // the tile max of the raw scores (the scale is positive), as a tree
      float mx[AT_KT / 2];
#pragma unroll
      for (int j = 0; j < AT_KT / 2; ++j) mx[j] = fmaxf(sv[j], sv[j + AT_KT / 2]);
#pragma unroll
      for (int w = AT_KT / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
      const float tmax = mx[0] * a.scale_log2;
      float fac = 1.f;
      bool resc = false;
      if (tmax > m_used + 8.f) {
        if (m_used != -INFINITY) {
          resc = true;
          fac = ex2(m_used - tmax);
          l *= fac;
        }
        m_used = tmax;
      }
      // masked scores are -inf and give 0; a row with no visible key yet takes 0 as its
      // reference (its scores are all -inf)
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      uint32_t pb[AT_KT];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < AT_KT; ++j) {
        const float p = ex2(fmaf(sv[j], a.scale_log2, -mref));
        ps[j & 3] += p;
        pb[j] = tf32_rna(p);
      }
      l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      // tcgen05.ld / st are warp-wide: the warp rescales when any of its rows must, once
      // PV(t - 1) has completed
      if (__any_sync(0xffffffffu, resc)) {
        if (t > 0 && !tc::mbar_wait(&pv_done[(t - 1) & 1], (uint32_t)(((t - 1) >> 1) & 1),
                                    &s_abort, AT_WAIT_NS))
          fail();
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          float o[32];
          tc::tmem_ld32(tO + lane_off + c, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= fac;
          tc::tmem_st32(tO + lane_off + c, o);
        }
        tc::tmem_st_wait();
      }
      // the probability tile t & 1 is free once PV(t - 2) has completed
      if (t >= 2 && !tc::mbar_wait(&pv_done[t & 1], (uint32_t)(((t - 2) >> 1) & 1), &s_abort,
                                   AT_WAIT_NS))
        fail();
      uint8_t* pt = sP + (t & 1) * AT_P;
#pragma unroll
      for (int c = 0; c < AT_KT / 4; ++c)
        *reinterpret_cast<uint4*>(pt + sw128(tid, c)) =
            make_uint4(pb[4 * c], pb[4 * c + 1], pb[4 * c + 2], pb[4 * c + 3]);
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&p_full[t & 1]);
      if (s_abort) break;
    }
    if (T > 0 && !s_abort &&
        !tc::mbar_wait(&pv_done[(T - 1) & 1], (uint32_t)(((T - 1) >> 1) & 1), &s_abort,
                       AT_WAIT_NS))
      fail();
    const bool ok = !__any_sync(0xffffffffu, s_abort != 0);  // warp-uniform: tcgen05.ld
    tc::fence_after_sync();
    if (ok) {
      float* dst = a.Op + ((size_t)h * a.M + min(i, a.M - 1)) * 64;
      if (T > 0) {
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          float o[32];
          tc::tmem_ld32(tO + lane_off + c, o);
          tc::tmem_ld_wait();
          if (i < a.M) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + c + j) =
                  make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
          }
        }
      } else if (i < a.M) {
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          *reinterpret_cast<float4*>(dst + j) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (i < a.M) {
        a.mrow[(size_t)h * a.M + i] =
            m_used == -INFINITY ? -INFINITY : m_used * 0.69314718055994531f;
        a.lrow[(size_t)h * a.M + i] = l;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 128u);
  }
}

// ---- backward, dQ += dS K1 --------------------------------------------------------------
// Same CTA rows and key tiles as the forward.  Per tile:
//   S = Q K1^T, dP = dO V1^T   M = 128, N = 32, K = 64 (two buffers each)
//   dS                          softmax warps: P = exp(S scale - lse) under the mask,
//                               dS = P (dP - D) scale, rounded to TF32 into one of two tiles
//   dQ += dS K1                 M = 128, N = 64, K = 32 keys: B is K1 transposed
// The prefix part of dQ is then added to dQh (which holds the chain part).
struct AtDqArgs {
  int M, n, K, G, Rq;
  float scale, scale_log2;
  const int* row_p;
  const int* row_d;
  const float* lse;
  const float* Dv;
  float* dQh;
  unsigned* err;
};

constexpr int DQ_KV = 2 * AT_K;  // one stage: K1 tile and V1 tile (both 32 keys x 64)
constexpr int DQ_ST = 3;

size_t at_dq_smem() { return 1024 + 2 * AT_Q + 2 * AT_P + (size_t)DQ_ST * (DQ_KV + AT_V); }

__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmO,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmKt, AtDqArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sO = sQ + AT_Q;           // dO rows
  uint8_t* sD = sO + AT_Q;           // two dS tiles
  uint8_t* sKV = sD + 2 * AT_P;      // stages: K1 tile, V1 tile
  uint8_t* sKt = sKV + DQ_ST * DQ_KV;
  __shared__ uint64_t q_full, kv_full[DQ_ST], kv_empty[DQ_ST], kt_full[DQ_ST], kt_empty[DQ_ST];
  __shared__ uint64_t sd_full[2], ds_full[2], dq_done[2], fin;
  __shared__ uint32_t s_tmem;
  __shared__ int s_amax;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int blk = gridDim.x - 1 - blockIdx.x;
  const int i0 = blk * a.Rq;
  if (tid == 0) {
    s_amax = -1;
    s_abort = 0;
    tc::mbar_init(&q_full, 1);
    for (int k = 0; k < DQ_ST; ++k) {
      tc::mbar_init(&kv_full[k], 1);
      tc::mbar_init(&kv_empty[k], 1);
      tc::mbar_init(&kt_full[k], 1);
      tc::mbar_init(&kt_empty[k], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sd_full[b], 1);
      tc::mbar_init(&ds_full[b], 4);
      tc::mbar_init(&dq_done[b], 1);
    }
    tc::mbar_init(&fin, 1);
    tc::fence_barrier_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(&s_tmem, 256u);
    tc::tmem_relinquish();
  }
  const int hl = tid < 128 ? tid / a.Rq : 0, r = tid < 128 ? tid - hl * a.Rq : 0;
  const int i = i0 + r, h = g * a.G + hl;
  AtFwdArgs geo;  // the anchor rule only reads these fields
  geo.M = a.M;
  geo.n = a.n;
  geo.K = a.K;
  geo.row_p = a.row_p;
  geo.row_d = a.row_d;
  const int anc = tid < 128 ? at_anchor(geo, i) : -1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (anc >= 0) atomicMax(&s_amax, anc);
  __syncthreads();
  const int T = s_amax >= 0 ? s_amax / AT_KT + 1 : 0;
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem, tP = tmem + 64, tQ = tmem + 128;  // S[2], dP[2], dQ
  auto fail = [&]() {
    if (!s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
    s_abort = 1;
  };

  if (warp >= 5) {
    // ---- TMA producers: warp 5 the queries, dO and the K1 / V1 ring, warp 6 the K1^T ring
    if (lane == 0 && T > 0) {
      const uint64_t pol = tc::policy_evict_last();
      const int krow0 = g * a.n;
      int issued = 0;
      if (warp == 5) {
        tc::mbar_expect_tx(&q_full, (uint32_t)(2 * AT_Q));
        for (int q = 0; q < a.G; ++q)
          for (int kb = 0; kb < 2; ++kb) {
            const int y = (g * a.G + q) * a.M + i0;
            tc::tma_load_2d(sQ + kb * 16384 + q * a.Rq * 128, &tmQ, kb * 32, y, &q_full, pol);
            tc::tma_load_2d(sO + kb * 16384 + q * a.Rq * 128, &tmO, kb * 32, y, &q_full, pol);
          }
        for (int j = 0; j < T; ++j, ++issued) {
          const int st = j % DQ_ST;
          if (j >= DQ_ST && !tc::mbar_wait(&kv_empty[st], (uint32_t)((j / DQ_ST - 1) & 1),
                                           &s_abort, AT_WAIT_NS)) {
            fail();
            break;
          }
          uint8_t* dst = sKV + st * DQ_KV;
          tc::mbar_expect_tx(&kv_full[st], (uint32_t)DQ_KV);
          tc::tma_load_2d(dst, &tmK, 0, krow0 + j * AT_KT, &kv_full[st], pol);
          tc::tma_load_2d(dst + 4096, &tmK, 32, krow0 + j * AT_KT, &kv_full[st], pol);
          tc::tma_load_2d(dst + AT_K, &tmV, 0, krow0 + j * AT_KT, &kv_full[st], pol);
          tc::tma_load_2d(dst + AT_K + 4096, &tmV, 32, krow0 + j * AT_KT, &kv_full[st], pol);
        }
      } else {
        for (int j = 0; j < T; ++j, ++issued) {
          const int st = j % DQ_ST;
          if (j >= DQ_ST && !tc::mbar_wait(&kt_empty[st], (uint32_t)((j / DQ_ST - 1) & 1),
                                           &s_abort, AT_WAIT_NS)) {
            fail();
            break;
          }
          tc::mbar_expect_tx(&kt_full[st], (uint32_t)AT_V);
          tc::tma_load_2d(sKt + st * AT_V, &tmKt, j * AT_KT, g * 64, &kt_full[st], pol);
        }
      }
      if (s_abort) {
        int never = 0;
        uint64_t* ring = warp == 5 ? kv_full : kt_full;
        if (warp == 5) tc::mbar_wait(&q_full, 0u, &never, AT_DRAIN_NS);
        for (int j = (issued > DQ_ST ? issued - DQ_ST : 0); j < issued; ++j)
          tc::mbar_wait(&ring[j % DQ_ST], (uint32_t)((j / DQ_ST) & 1), &never, AT_DRAIN_NS);
      }
    }
  } else if (warp == 4) {
    if (lane == 0 && T > 0) {
      const uint32_t idS = tc::idesc_tf32(128, AT_KT), idQ = tc::idesc_tf32(128, 64);
      auto issue_sd = [&](int j) -> bool {  // S(j), dP(j) into buffers j & 1
        const int st = j % DQ_ST;
        if (!tc::mbar_wait(&kv_full[st], (uint32_t)((j / DQ_ST) & 1), &s_abort, AT_WAIT_NS))
          return false;
        tc::fence_after_sync();
        const uint8_t* kv = sKV + st * DQ_KV;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t aq = tc::smem_desc_sw128(tc::smem_u32(sQ + kb * 16384));
          const uint64_t ao = tc::smem_desc_sw128(tc::smem_u32(sO + kb * 16384));
          const uint64_t bk = tc::smem_desc_sw128(tc::smem_u32(kv + kb * 4096));
          const uint64_t bv = tc::smem_desc_sw128(tc::smem_u32(kv + AT_K + kb * 4096));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc::mma_tf32(tS + (uint32_t)((j & 1) * AT_KT), aq + 2 * k, bk + 2 * k, idS,
                         (kb | k) ? 1u : 0u);
            tc::mma_tf32(tP + (uint32_t)((j & 1) * AT_KT), ao + 2 * k, bv + 2 * k, idS,
                         (kb | k) ? 1u : 0u);
          }
        }
        tc::mma_commit(&sd_full[j & 1]);
        tc::mma_commit(&kv_empty[st]);
        return true;
      };
      bool ok = tc::mbar_wait(&q_full, 0u, &s_abort, AT_WAIT_NS);
      for (int j = 0; ok && j < 2 && j < T; ++j) ok = issue_sd(j);
      for (int t = 0; ok && t < T; ++t) {
        const int st = t % DQ_ST;
        if (!tc::mbar_wait(&ds_full[t & 1], (uint32_t)((t >> 1) & 1), &s_abort, AT_WAIT_NS) ||
            !tc::mbar_wait(&kt_full[st], (uint32_t)((t / DQ_ST) & 1), &s_abort, AT_WAIT_NS)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(sD + (t & 1) * AT_P));
        const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(sKt + st * AT_V));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_tf32(tQ, ad + 2 * k, bd + 2 * k, idQ, (t > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&dq_done[t & 1]);
        tc::mma_commit(&kt_empty[st]);
        if (t + 2 < T) ok = issue_sd(t + 2);
      }
      if (!ok) fail();
      int never = 0;
      tc::mma_commit(&fin);
      tc::mbar_wait(&fin, 0u, &never, AT_DRAIN_NS);
    }
  } else {
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const bool row_ok = i < a.M;
    const float L2 = row_ok ? a.lse[(size_t)h * a.M + i] * 1.4426950408889634f : 0.f;
    const float Dr = row_ok ? a.Dv[(size_t)h * a.M + i] : 0.f;
    const float dD = -Dr * a.scale;  // dS = P (dP - D) scale = P (dP scale - D scale)
    for (int t = 0; t < T; ++t) {
      if (!tc::mbar_wait(&sd_full[t & 1], (uint32_t)((t >> 1) & 1), &s_abort, AT_WAIT_NS))
        fail();
      tc::fence_after_sync();
      float sv[AT_KT], pv[AT_KT];
      tc::tmem_ld32(tS + lane_off + (uint32_t)((t & 1) * AT_KT), sv);
      tc::tmem_ld32(tP + lane_off + (uint32_t)((t & 1) * AT_KT), pv);
      tc::tmem_ld_wait();
      const int lim = anc - t * AT_KT;  // keys j <= lim of the tile are visible
      if (lim < AT_KT - 1) {
#pragma unroll
        for (int j = 0; j < AT_KT; ++j)
          if (j > lim) sv[j] = -INFINITY;
      }
      uint32_t db[AT_KT];
#pragma unroll
      for (int j = 0; j < AT_KT; ++j) {
        const float p = ex2(fmaf(sv[j], a.scale_log2, -L2));
        db[j] = tf32_rna(p * fmaf(pv[j], a.scale, dD));
      }
      // the dS tile t & 1 is free once dQ(t - 2) has completed
      if (t >= 2 && !tc::mbar_wait(&dq_done[t & 1], (uint32_t)(((t - 2) >> 1) & 1), &s_abort,
                                   AT_WAIT_NS))
        fail();
      uint8_t* pt = sD + (t & 1) * AT_P;
#pragma unroll
      for (int c = 0; c < AT_KT / 4; ++c)
        *reinterpret_cast<uint4*>(pt + sw128(tid, c)) =
            make_uint4(db[4 * c], db[4 * c + 1], db[4 * c + 2], db[4 * c + 3]);
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ds_full[t & 1]);
      if (s_abort) break;
    }
    if (T > 0 && !s_abort &&
        !tc::mbar_wait(&dq_done[(T - 1) & 1], (uint32_t)(((T - 1) >> 1) & 1), &s_abort,
                       AT_WAIT_NS))
      fail();
    const bool ok = !__any_sync(0xffffffffu, s_abort != 0);
    tc::fence_after_sync();
    if (ok && T > 0) {
      float* dst = a.dQh + ((size_t)h * a.M + min(i, a.M - 1)) * 64;
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        float o[32];
        tc::tmem_ld32(tQ + lane_off + c, o);
        tc::tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 v = *reinterpret_cast<const float4*>(dst + c + j);
            v.x += o[j];
            v.y += o[j + 1];
            v.z += o[j + 2];
            v.w += o[j + 3];
            *reinterpret_cast<float4*>(dst + c + j) = v;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 256u);
  }
}

// ---- backward, dK1 += dS^T Q and dV1 += P^T dO --------------------------------------------
// A CTA holds 128 keys of kv head g (MMA rows = keys; their K1 and V1 rows stay in shared
// memory) and walks a chunk of the rows that can see them, 32 rows of one q head at a time:
//   S^T = K1 Q^T, dP^T = V1 dO^T   M = 128, N = 32, K = 64 (two buffers each)
//   P^T, dS^T                       softmax warps, one thread per key: P = exp(S scale -
//                                   lse) under the mask, dS = P (dP - D) scale, rounded to
//                                   TF32 into one of two tile pairs
//   dV += P^T dO, dK += dS^T Q      M = 128, N = 64, K = 32 rows: B is dO / Q transposed
// At the end each key's dK1 / dV1 row is added into the outputs (chunks of rows meet there).
struct AtDkvArgs {
  int M, n, K, G, Kmax, chunk;
  float scale, scale_log2;
  const int* row_p;
  const int* row_d;
  const int* row_index;
  const float* lse;
  const float* Dv;
  float* dK1;
  float* dV1;
  unsigned* err;
};

constexpr int DK_RT = 32;                   // rows per iteration
constexpr int DK_KV = 2 * 16384;            // 128 keys x 64 fp32 (two k-blocks)
constexpr int DK_A = 2 * (2 * 4096);        // ring A stage: Q tile, dO tile (32 rows x 64)
constexpr int DK_B = 2 * 8192;              // ring B stage: Q^T, dO^T tiles (64 x 32 rows)
constexpr int DK_ST = 2;

size_t at_dkv_smem() { return 1024 + 2 * DK_KV + 4 * AT_P + (size_t)DK_ST * (DK_A + DK_B); }

struct DkRowVals {
  float L2[DK_RT];  // lse log2(e) of the tile's rows (this head)
  float Ds[DK_RT];  // D scale
  int anc[DK_RT];   // anchors (-1: no key visible)
};

__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmO,
                           const __grid_constant__ CUtensorMap tmQt,
                           const __grid_constant__ CUtensorMap tmOt,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, AtDkvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = sm;
  uint8_t* sV = sK + DK_KV;
  uint8_t* sPt = sV + DK_KV;          // two P^T tiles
  uint8_t* sDt = sPt + 2 * AT_P;      // two dS^T tiles
  uint8_t* sA = sDt + 2 * AT_P;       // ring A
  uint8_t* sB = sA + DK_ST * DK_A;    // ring B
  __shared__ DkRowVals rv[DK_ST];
  __shared__ uint64_t kv_full, a_full[DK_ST], a_empty[DK_ST], b_full[DK_ST], b_empty[DK_ST];
  __shared__ uint64_t sd_full[2], ds_full[2], pd_done[2], fin;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = blockIdx.x * 128, g = blockIdx.y;
  if (k0 >= a.n) return;
  const int rs = a.row_index[(size_t)k0 * (a.Kmax + 1) + 1];
  if (rs < 0) return;                     // no depth-1 row at k0: no row sees these keys
  const int rb = (rs & ~3) + blockIdx.z * a.chunk;  // 16-byte aligned for the Q^T boxes
  if (rb >= a.M) return;
  const int re = min(a.M, rb + a.chunk);
  const int nrt = (re - rb + DK_RT - 1) / DK_RT;
  const int T = nrt * a.G;                // iterations: (row tile, head) pairs
  if (tid == 0) {
    s_abort = 0;
    tc::mbar_init(&kv_full, 1);
    for (int k = 0; k < DK_ST; ++k) {
      tc::mbar_init(&a_full[k], 1);
      tc::mbar_init(&a_empty[k], 1);
      tc::mbar_init(&b_full[k], 1);
      tc::mbar_init(&b_empty[k], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sd_full[b], 1);
      tc::mbar_init(&ds_full[b], 4);
      tc::mbar_init(&pd_done[b], 1);
    }
    tc::mbar_init(&fin, 1);
    tc::fence_barrier_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(&s_tmem, 256u);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem, tP = tmem + 64, tV = tmem + 128, tK = tmem + 192;
  auto fail = [&]() {
    if (!s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
    s_abort = 1;
  };
  // iteration t: rows r0 = rb + (t / G) * 32 .., head g * G + t % G
  auto it_row = [&](int t) { return rb + (t / a.G) * DK_RT; };
  auto it_head = [&](int t) { return g * a.G + t % a.G; };

  if (warp == 5) {
    // ---- producer A: the key block's K1 / V1 rows once, then Q / dO tiles
    if (lane == 0) {
      const uint64_t pol = tc::policy_evict_last();
      tc::mbar_expect_tx(&kv_full, (uint32_t)(2 * DK_KV));
      for (int kb = 0; kb < 2; ++kb) {
        tc::tma_load_2d(sK + kb * 16384, &tmK, kb * 32, g * a.n + k0, &kv_full, pol);
        tc::tma_load_2d(sV + kb * 16384, &tmV, kb * 32, g * a.n + k0, &kv_full, pol);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t, ++issued) {
        const int st = t % DK_ST;
        if (t >= DK_ST && !tc::mbar_wait(&a_empty[st], (uint32_t)((t / DK_ST - 1) & 1),
                                         &s_abort, AT_WAIT_NS)) {
          fail();
          break;
        }
        const int y = it_head(t) * a.M + it_row(t);
        uint8_t* dst = sA + st * DK_A;
        tc::mbar_expect_tx(&a_full[st], (uint32_t)DK_A);
        for (int kb = 0; kb < 2; ++kb) {
          tc::tma_load_2d(dst + kb * 4096, &tmQ, kb * 32, y, &a_full[st], pol);
          tc::tma_load_2d(dst + 8192 + kb * 4096, &tmO, kb * 32, y, &a_full[st], pol);
        }
      }
      if (s_abort) {
        int never = 0;
        tc::mbar_wait(&kv_full, 0u, &never, AT_DRAIN_NS);
        for (int j = (issued > DK_ST ? issued - DK_ST : 0); j < issued; ++j)
          tc::mbar_wait(&a_full[j % DK_ST], (uint32_t)((j / DK_ST) & 1), &never, AT_DRAIN_NS);
      }
    }
  } else if (warp == 6) {
    // ---- producer B: the rows' lse / D / anchors (every lane one row), Q^T / dO^T tiles
    const uint64_t pol = tc::policy_evict_last();
    int issued = 0;
    for (int t = 0; t < T; ++t, ++issued) {
      const int st = t % DK_ST;
      bool ok = true;
      if (t >= DK_ST && !tc::mbar_wait(&b_empty[st], (uint32_t)((t / DK_ST - 1) & 1), &s_abort,
                                       AT_WAIT_NS)) {
        fail();
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      const int i = it_row(t) + lane, h = it_head(t);
      int anc = -1;
      if (i < a.M) {
        const int p = a.row_p[i], d = a.row_d[i];
        if (p >= 0 && p < a.n && d >= 1 && d <= a.K && p - d + 1 >= 0) anc = p - d + 1;
      }
      rv[st].anc[lane] = anc;
      rv[st].L2[lane] = i < a.M ? a.lse[(size_t)h * a.M + i] * 1.4426950408889634f : 0.f;
      rv[st].Ds[lane] = i < a.M ? a.Dv[(size_t)h * a.M + i] * a.scale : 0.f;
      __syncwarp();
      if (lane == 0) {
        uint8_t* dst = sB + st * DK_B;
        tc::mbar_expect_tx(&b_full[st], (uint32_t)DK_B);
        tc::tma_load_2d(dst, &tmQt, it_row(t), h * 64, &b_full[st], pol);
        tc::tma_load_2d(dst + 8192, &tmOt, it_row(t), h * 64, &b_full[st], pol);
      }
    }
    if (lane == 0 && s_abort) {
      int never = 0;
      for (int j = (issued > DK_ST ? issued - DK_ST : 0); j < issued; ++j)
        tc::mbar_wait(&b_full[j % DK_ST], (uint32_t)((j / DK_ST) & 1), &never, AT_DRAIN_NS);
    }
  } else if (warp == 4) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc::idesc_tf32(128, DK_RT), idD = tc::idesc_tf32(128, 64);
      auto issue_sd = [&](int j) -> bool {  // S^T(j), dP^T(j) into buffers j & 1
        const int st = j % DK_ST;
        if (!tc::mbar_wait(&a_full[st], (uint32_t)((j / DK_ST) & 1), &s_abort, AT_WAIT_NS))
          return false;
        tc::fence_after_sync();
        const uint8_t* src = sA + st * DK_A;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint64_t ak = tc::smem_desc_sw128(tc::smem_u32(sK + kb * 16384));
          const uint64_t av = tc::smem_desc_sw128(tc::smem_u32(sV + kb * 16384));
          const uint64_t bq = tc::smem_desc_sw128(tc::smem_u32(src + kb * 4096));
          const uint64_t bo = tc::smem_desc_sw128(tc::smem_u32(src + 8192 + kb * 4096));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc::mma_tf32(tS + (uint32_t)((j & 1) * DK_RT), ak + 2 * k, bq + 2 * k, idS,
                         (kb | k) ? 1u : 0u);
            tc::mma_tf32(tP + (uint32_t)((j & 1) * DK_RT), av + 2 * k, bo + 2 * k, idS,
                         (kb | k) ? 1u : 0u);
          }
        }
        tc::mma_commit(&sd_full[j & 1]);
        tc::mma_commit(&a_empty[st]);
        return true;
      };
      bool ok = tc::mbar_wait(&kv_full, 0u, &s_abort, AT_WAIT_NS);
      for (int j = 0; ok && j < 2 && j < T; ++j) ok = issue_sd(j);
      for (int t = 0; ok && t < T; ++t) {
        const int st = t % DK_ST;
        if (!tc::mbar_wait(&ds_full[t & 1], (uint32_t)((t >> 1) & 1), &s_abort, AT_WAIT_NS) ||
            !tc::mbar_wait(&b_full[st], (uint32_t)((t / DK_ST) & 1), &s_abort, AT_WAIT_NS)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint64_t ap = tc::smem_desc_sw128(tc::smem_u32(sPt + (t & 1) * AT_P));
        const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(sDt + (t & 1) * AT_P));
        const uint64_t bo = tc::smem_desc_sw128(tc::smem_u32(sB + st * DK_B + 8192));
        const uint64_t bq = tc::smem_desc_sw128(tc::smem_u32(sB + st * DK_B));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tc::mma_tf32(tV, ap + 2 * k, bo + 2 * k, idD, (t > 0 || k > 0) ? 1u : 0u);
          tc::mma_tf32(tK, ad + 2 * k, bq + 2 * k, idD, (t > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit(&pd_done[t & 1]);
        tc::mma_commit(&b_empty[st]);
        if (t + 2 < T) ok = issue_sd(t + 2);
      }
      if (!ok) fail();
      int never = 0;
      tc::mma_commit(&fin);
      tc::mbar_wait(&fin, 0u, &never, AT_DRAIN_NS);
    }
  } else {
    // ---- softmax warps: thread = key k0 + tid
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int key = k0 + tid;
    for (int t = 0; t < T; ++t) {
      const int st = t % DK_ST;
      if (!tc::mbar_wait(&sd_full[t & 1], (uint32_t)((t >> 1) & 1), &s_abort, AT_WAIT_NS) ||
          !tc::mbar_wait(&b_full[st], (uint32_t)((t / DK_ST) & 1), &s_abort, AT_WAIT_NS))
        fail();
      tc::fence_after_sync();
      float sv[DK_RT], pv[DK_RT];
      tc::tmem_ld32(tS + lane_off + (uint32_t)((t & 1) * DK_RT), sv);
      tc::tmem_ld32(tP + lane_off + (uint32_t)((t & 1) * DK_RT), pv);
      tc::tmem_ld_wait();
      const DkRowVals& R = rv[st];
      uint32_t pb[DK_RT], db[DK_RT];
#pragma unroll
      for (int j = 0; j < DK_RT; ++j) {
        const float p = key <= R.anc[j] ? ex2(fmaf(sv[j], a.scale_log2, -R.L2[j])) : 0.f;
        pb[j] = tf32_rna(p);
        db[j] = tf32_rna(p * fmaf(pv[j], a.scale, -R.Ds[j]));
      }
      // the tiles t & 1 are free once dV / dK(t - 2) have completed
      if (t >= 2 && !tc::mbar_wait(&pd_done[t & 1], (uint32_t)(((t - 2) >> 1) & 1), &s_abort,
                                   AT_WAIT_NS))
        fail();
      uint8_t* pt = sPt + (t & 1) * AT_P;
      uint8_t* dt = sDt + (t & 1) * AT_P;
#pragma unroll
      for (int c = 0; c < DK_RT / 4; ++c) {
        *reinterpret_cast<uint4*>(pt + sw128(tid, c)) =
            make_uint4(pb[4 * c], pb[4 * c + 1], pb[4 * c + 2], pb[4 * c + 3]);
        *reinterpret_cast<uint4*>(dt + sw128(tid, c)) =
            make_uint4(db[4 * c], db[4 * c + 1], db[4 * c + 2], db[4 * c + 3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ds_full[t & 1]);
      if (s_abort) break;
    }
    if (T > 0 && !s_abort &&
        !tc::mbar_wait(&pd_done[(T - 1) & 1], (uint32_t)(((T - 1) >> 1) & 1), &s_abort,
                       AT_WAIT_NS))
      fail();
    const bool ok = !__any_sync(0xffffffffu, s_abort != 0);
    tc::fence_after_sync();
    if (ok && T > 0) {
      float* gk = a.dK1 + ((size_t)g * a.n + min(key, a.n - 1)) * 64;
      float* gv = a.dV1 + ((size_t)g * a.n + min(key, a.n - 1)) * 64;
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        float o[32];
        tc::tmem_ld32(tK + lane_off + c, o);
        tc::tmem_ld_wait();
        if (key < a.n) {
#pragma unroll
          for (int j = 0; j < 32; ++j) atomicAdd(gk + c + j, o[j]);
        }
        tc::tmem_ld32(tV + lane_off + c, o);
        tc::tmem_ld_wait();
        if (key < a.n) {
#pragma unroll
          for (int j = 0; j < 32; ++j) atomicAdd(gv + c + j, o[j]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 256u);
  }
}

}  // namespace

bool attn_tc_ok(const TrainAttn& a) {
  const int G = a.nkv > 0 ? a.nq / a.nkv : 0;
  return a.hd == 64 && (G == 1 || G == 2 || G == 4 || G == 8) && a.nq % a.nkv == 0;
}

int launch_attn_fwd_prefix_tc(const TrainAttn& a, const TrainAttnTc& x, const float* Qh,
                              const float* K1, const float* V1, float* Op, float* mrow,
                              float* lrow, cudaStream_t s) {
  if (!attn_tc_ok(a) || !x.tc || !x.kvT || x.ldn < a.n || (x.ldn & 3)) return PEAGLE_ERR_UNSUPPORTED;
  const int G = a.nq / a.nkv, Rq = 128 / G;
  // V1 [nkv][n][64] -> V1^T [nkv][64][ldn]
  launch_transpose_f32(V1, a.n, 64, 64, x.kvT, x.ldn, s, a.nkv, (size_t)a.n * 64,
                       (size_t)64 * x.ldn);
  CUtensorMap mQ, mK, mV;
  if (!tc_tensor_map_f32(x.tc, &mQ, Qh, a.nq * a.M, 64, 64, Rq) ||
      !tc_tensor_map_f32(x.tc, &mK, K1, a.nkv * a.n, 64, 64, AT_KT) ||
      !tc_tensor_map_f32(x.tc, &mV, x.kvT, a.nkv * 64, a.n, x.ldn, 64))
    return PEAGLE_ERR_UNSUPPORTED;
  AtFwdArgs f;
  f.M = a.M;
  f.n = a.n;
  f.K = a.K;
  f.G = G;
  f.Rq = Rq;
  f.scale_log2 = a.scale * 1.4426950408889634f;
  f.row_p = a.row_p;
  f.row_d = a.row_d;
  f.Op = Op;
  f.mrow = mrow;
  f.lrow = lrow;
  f.err = x.err;
  const size_t smem = at_fwd_smem();
  if (smem_optin((const void*)attn_fwd_prefix_tc_kernel, smem) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  dim3 grid((a.M + Rq - 1) / Rq, a.nkv);
  attn_fwd_prefix_tc_kernel<<<grid, AT_THREADS, smem, s>>>(mQ, mK, mV, f);
  return cudaGetLastError() == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

int launch_attn_bwd_dq_tc(const TrainAttn& a, const TrainAttnTc& x, const float* Qh,
                          const float* dOh, const float* K1, const float* V1, const float* lse,
                          const float* Dv, float* dQh, cudaStream_t s) {
  if (!attn_tc_ok(a) || !x.tc || !x.kvT || x.ldn < a.n || (x.ldn & 3)) return PEAGLE_ERR_UNSUPPORTED;
  const int G = a.nq / a.nkv, Rq = 128 / G;
  // K1 [nkv][n][64] -> K1^T [nkv][64][ldn]
  launch_transpose_f32(K1, a.n, 64, 64, x.kvT, x.ldn, s, a.nkv, (size_t)a.n * 64,
                       (size_t)64 * x.ldn);
  CUtensorMap mQ, mO, mK, mV, mKt;
  if (!tc_tensor_map_f32(x.tc, &mQ, Qh, a.nq * a.M, 64, 64, Rq) ||
      !tc_tensor_map_f32(x.tc, &mO, dOh, a.nq * a.M, 64, 64, Rq) ||
      !tc_tensor_map_f32(x.tc, &mK, K1, a.nkv * a.n, 64, 64, AT_KT) ||
      !tc_tensor_map_f32(x.tc, &mV, V1, a.nkv * a.n, 64, 64, AT_KT) ||
      !tc_tensor_map_f32(x.tc, &mKt, x.kvT, a.nkv * 64, a.n, x.ldn, 64))
    return PEAGLE_ERR_UNSUPPORTED;
  AtDqArgs f;
  f.M = a.M;
  f.n = a.n;
  f.K = a.K;
  f.G = G;
  f.Rq = Rq;
  f.scale = a.scale;
  f.scale_log2 = a.scale * 1.4426950408889634f;
  f.row_p = a.row_p;
  f.row_d = a.row_d;
  f.lse = lse;
  f.Dv = Dv;
  f.dQh = dQh;
  f.err = x.err;
  const size_t smem = at_dq_smem();
  if (smem_optin((const void*)attn_bwd_dq_tc_kernel, smem) != cudaSuccess) return PEAGLE_ERR_CUDA;
  dim3 grid((a.M + Rq - 1) / Rq, a.nkv);
  attn_bwd_dq_tc_kernel<<<grid, AT_THREADS, smem, s>>>(mQ, mO, mK, mV, mKt, f);
  return cudaGetLastError() == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

int launch_attn_bwd_dkv_tc(const TrainAttn& a, const TrainAttnTc& x, const int* row_index,
                           int Kmax, const float* Qh, const float* dOh, const float* K1,
                           const float* V1, const float* lse, const float* Dv, float* dK1,
                           float* dV1, cudaStream_t s) {
  if (!attn_tc_ok(a) || !x.tc || !x.qT || !x.doT || x.ldm < a.M || (x.ldm & 3))
    return PEAGLE_ERR_UNSUPPORTED;
  const int G = a.nq / a.nkv;
  // Q, dO [nq][M][64] -> [nq][64][ldm]
  launch_transpose_f32(Qh, a.M, 64, 64, x.qT, x.ldm, s, a.nq, (size_t)a.M * 64,
                       (size_t)64 * x.ldm);
  launch_transpose_f32(dOh, a.M, 64, 64, x.doT, x.ldm, s, a.nq, (size_t)a.M * 64,
                       (size_t)64 * x.ldm);
  CUtensorMap mQ, mO, mQt, mOt, mK, mV;
  if (!tc_tensor_map_f32(x.tc, &mQ, Qh, a.nq * a.M, 64, 64, DK_RT) ||
      !tc_tensor_map_f32(x.tc, &mO, dOh, a.nq * a.M, 64, 64, DK_RT) ||
      !tc_tensor_map_f32(x.tc, &mQt, x.qT, a.nq * 64, a.M, x.ldm, 64) ||
      !tc_tensor_map_f32(x.tc, &mOt, x.doT, a.nq * 64, a.M, x.ldm, 64) ||
      !tc_tensor_map_f32(x.tc, &mK, K1, a.nkv * a.n, 64, 64, 128) ||
      !tc_tensor_map_f32(x.tc, &mV, V1, a.nkv * a.n, 64, 64, 128))
    return PEAGLE_ERR_UNSUPPORTED;
  AtDkvArgs f;
  f.M = a.M;
  f.n = a.n;
  f.K = a.K;
  f.G = G;
  f.Kmax = Kmax;
  f.chunk = 512;
  f.scale = a.scale;
  f.scale_log2 = a.scale * 1.4426950408889634f;
  f.row_p = a.row_p;
  f.row_d = a.row_d;
  f.row_index = row_index;
  f.lse = lse;
  f.Dv = Dv;
  f.dK1 = dK1;
  f.dV1 = dV1;
  f.err = x.err;
  const size_t smem = at_dkv_smem();
  if (smem_optin((const void*)attn_bwd_dkv_tc_kernel, smem) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  dim3 grid((a.n + 127) / 128, a.nkv, (a.M + f.chunk + 3) / f.chunk);
  attn_bwd_dkv_tc_kernel<<<grid, AT_THREADS, smem, s>>>(mQ, mO, mQt, mOt, mK, mV, f);
  return cudaGetLastError() == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

}  // namespace peagle
