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

constexpr int AT_THREADS = 192;
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

  if (warp == 5) {
    // ---- TMA producer
    if (lane == 0 && T > 0) {
      const uint64_t pol = tc::policy_evict_last();
      const int krow0 = g * a.n;  // K1 viewed as [nkv n][64]
      tc::mbar_expect_tx(&q_full, (uint32_t)AT_Q);
      for (int q = 0; q < a.G; ++q)
        for (int kb = 0; kb < 2; ++kb)
          tc::tma_load_2d(sQ + kb * 16384 + q * a.Rq * 128, &tmQ, kb * 32,
                          (g * a.G + q) * a.M + i0, &q_full, pol);
      int kiss = 0, viss = 0;
      for (int j = 0; j < T; ++j) {
        const int ks = j % AT_KST, vs = j % AT_VST;
        if (j >= AT_KST && !tc::mbar_wait(&k_empty[ks], (uint32_t)((j / AT_KST - 1) & 1),
                                          &s_abort, AT_WAIT_NS)) {
          fail();
          break;
        }
        tc::mbar_expect_tx(&k_full[ks], (uint32_t)AT_K);
        tc::tma_load_2d(sK + ks * AT_K, &tmK, 0, krow0 + j * AT_KT, &k_full[ks], pol);
        tc::tma_load_2d(sK + ks * AT_K + 4096, &tmK, 32, krow0 + j * AT_KT, &k_full[ks], pol);
        ++kiss;
        if (j >= AT_VST && !tc::mbar_wait(&v_empty[vs], (uint32_t)((j / AT_VST - 1) & 1),
                                          &s_abort, AT_WAIT_NS)) {
          fail();
          break;
        }
        tc::mbar_expect_tx(&v_full[vs], (uint32_t)AT_V);
        tc::tma_load_2d(sV + vs * AT_V, &tmVt, j * AT_KT, g * 64, &v_full[vs], pol);
        ++viss;
      }
      if (s_abort) {  // the loads in flight land (bounded) before the CTA can exit
        int never = 0;
        tc::mbar_wait(&q_full, 0u, &never, AT_DRAIN_NS);
        for (int j = (kiss > AT_KST ? kiss - AT_KST : 0); j < kiss; ++j)
          tc::mbar_wait(&k_full[j % AT_KST], (uint32_t)((j / AT_KST) & 1), &never, AT_DRAIN_NS);
        for (int j = (viss > AT_VST ? viss - AT_VST : 0); j < viss; ++j)
          tc::mbar_wait(&v_full[j % AT_VST], (uint32_t)((j / AT_VST) & 1), &never, AT_DRAIN_NS);
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
      const int kbase = t * AT_KT;
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < AT_KT; ++j) {
        sv[j] = kbase + j <= anc ? sv[j] * a.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, sv[j]);
      }
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
      uint32_t pb[AT_KT];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < AT_KT; ++j) {
        const float p = sv[j] == -INFINITY ? 0.f : ex2(sv[j] - m_used);
        psum += p;
        pb[j] = tf32_rna(p);
      }
      l += psum;
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

}  // namespace peagle
