// Training-style masked attention of the parallel drafter on the 5th-generation tensor
// cores ("P-EAGLE: Parallel-Drafting EAGLE with Scalable Training", section 3.1: the
// attention mask of the parallel-prediction forward), head_dim 64.
//
// A CTA serves 128 MMA rows: the (query row, q head) pairs of 128 / G consecutive rows
// for kv head g.  Keys come as 64-key tiles in the two runs of the mask's closed form
// (depth-1 positions 0 .. the block's largest anchor, then the block's chain rows; see
// the tensor-core mma.sync kernel in kernels.cu).  Per tile:
//   S = Q K^T    tcgen05.mma M=128, N=64, K=64, fp32 in tensor memory
//   softmax      one thread per MMA row reads its 64 scores (tcgen05.ld), masks them,
//                updates the running max / sum (log2 domain) and writes its bf16
//                probabilities to shared memory (the next MMA's A operand)
//   O += P V     tcgen05.mma M=128, N=64 (head dims), K=64 keys, V read MN-major
// The output accumulator stays in tensor memory; when a row's reference maximum is raised
// (lazily: only by more than 2^8), its thread rescales the row there (tcgen05.ld / st)
// before the next product.  K and V tiles arrive
// by TMA, two tiles ahead.  Queries and probabilities are rounded to bf16 as in the
// mma.sync kernel, so both kernels compute the same function (exponentials here on the
// SFU, 2^x to about 2^-22 relative, far below the probabilities' bf16 rounding).
#include <cuda.h>
#include <stdio.h>

#include "attn_decode.cuh"
#include "common.cuh"
#include "epilogue.cuh"
#include "gemm_tc.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace peagle {
namespace {

constexpr int MT_KT = 64;           // keys per tile
constexpr int MT_THREADS = 128;     // one thread per MMA row
constexpr int MT_TILE = 64 * 128;   // 64 rows x 64 bf16 (128 B), 128-byte swizzle
constexpr int MT_SMEM = 1024 + 2 * 16384 + 4 * MT_TILE;  // Q, P, K[2], V[2]
constexpr uint64_t MT_WAIT_NS = 2000000000ull;
constexpr int MT_LAZY_LOG2 = 8;  // rescale O only when a row's maximum grows by more than 2^8

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16-byte chunk c of row r of a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(MT_THREADS) masked_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmV1,
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    MaskedAttnArgs a) {
  constexpr int HD = 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = sm;
  uint8_t* sP = sm + 16384;
  uint8_t* sK = sm + 32768;                // 2 tiles
  uint8_t* sV = sK + 2 * MT_TILE;          // 2 tiles
  __shared__ uint64_t kv_full[2], s_done, pv_done;
  __shared__ int s_kp[2][MT_KT], s_kd[2][MT_KT];
  __shared__ int s_aend, s_amin, s_jb0;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  pdl_enter();
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = a.nq / a.nkv;
  const int QR = 128 / G;
  const int i0 = (int)(gridDim.x - 1 - blockIdx.x) * QR;
  const int g = blockIdx.y;
  const int iend = min(a.M, i0 + QR);
  auto row_ok = [&](int p, int d) {
    return p >= 0 && p < a.n && d >= 1 && d <= a.Kmax && p - d + 1 >= 0;
  };
  if (tid == 0) {
    s_aend = -1;
    s_amin = 0x7fffffff;
    s_abort = 0;
    tc::mbar_init(&kv_full[0], 1);
    tc::mbar_init(&kv_full[1], 1);
    tc::mbar_init(&s_done, 1);
    tc::mbar_init(&pv_done, 1);
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&tmK1);
    tc::tma_prefetch_desc(&tmV1);
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, 128);  // S in columns [0, 64), O in [64, 128)
    tc::tmem_relinquish();
  }
  __syncthreads();
  if (tid < iend - i0) {
    const int p = a.row_p[i0 + tid], d = a.row_d[i0 + tid];
    if (row_ok(p, d)) {
      atomicMax(&s_aend, p - d + 1);
      atomicMin(&s_amin, p - d + 1);
    }
  }
  __syncthreads();
  const int a_end = s_aend;
  if (tid == 0) {
    // run B starts at the first row whose position exceeds the smallest anchor
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
  const int ntA = a_end >= 0 ? a_end / MT_KT + 1 : 0;
  const int ntB = (iend - jb0 + MT_KT - 1) / MT_KT;
  const int ntile = ntA + ntB;
  const uint64_t pol = tc::policy_evict_last();  // K / V rows are re-read by many CTAs

  // tile `it` into buffer `buf`: TMA by thread 0; run B's key (p, d) by threads < 64
  auto load_tile = [&](int buf, int it) {
    const bool runA = it < ntA;
    const int t0 = runA ? it * MT_KT : jb0 + (it - ntA) * MT_KT;
    if (tid == 0) {
      tc::mbar_expect_tx(&kv_full[buf], 2 * MT_TILE);
      tc::tma_load_2d(sK + buf * MT_TILE, runA ? &tmK1 : &tmK, g * HD, t0, &kv_full[buf], pol);
      tc::tma_load_2d(sV + buf * MT_TILE, runA ? &tmV1 : &tmV, g * HD, t0, &kv_full[buf], pol);
    }
    if (!runA && tid < MT_KT) {
      const int key = t0 + tid;
      const bool ok = key < iend;
      s_kp[buf][tid] = ok ? a.row_p[key] : 0;
      s_kd[buf][tid] = ok ? a.row_d[key] : 0;
    }
  };

  // this thread's MMA row: query row qi, q head h; its mask parameters
  const int qi = i0 + tid / G, h = g * G + tid % G;
  const bool in = tid < QR * G && qi < iend;
  int lim = -1, dg = 0, dd = 0;  // anchor p - d + 1, chain diagonal p - d, depth d
  if (in) {
    const int p = a.row_p[qi], d = a.row_d[qi];
    if (row_ok(p, d)) {
      lim = p - d + 1;
      dg = p - d;
      dd = d;
    }
  }
  if (a.q_bf16) {
    // queries stored as bf16 by the QKV epilogue: the row's 128 bytes as they are
    const uint4* q =
        (const uint4*)((const bf16*)a.q + ((size_t)(in ? qi : 0) * a.nq + h) * HD);
    uint4 x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = in ? q[c] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < 8; ++c) *(uint4*)(sQ + sw128(tid, c)) = x[c];
  } else {
    // queries (bf16, the scale is applied to the scores) into the A tile of S = Q K^T
    const float4* q = (const float4*)((const float*)a.q + ((size_t)(in ? qi : 0) * a.nq + h) * HD);
    float4 x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) x[u] = in ? q[u] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 lo = x[2 * c], hi = x[2 * c + 1];
      *(uint4*)(sQ + sw128(tid, c)) = make_uint4(pack_bf16(lo.x, lo.y), pack_bf16(lo.z, lo.w),
                                                 pack_bf16(hi.x, hi.y), pack_bf16(hi.z, hi.w));
    }
  }
  if (ntile > 0) load_tile(0, 0);
  if (ntile > 1) load_tile(1, 1);
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem + lane_off, tO = tmem + 64 + lane_off;
  const uint32_t idS = tc::idesc_bf16(128, 64);
  const uint32_t idPV = tc::idesc_bf16(128, 64) | (1u << 16);  // B (V) read MN-major
  const uint64_t dQ = tc::smem_desc_sw128(tc::smem_u32(sQ));
  const uint64_t dP = tc::smem_desc_sw128(tc::smem_u32(sP));
  const float qscale = a.scale * 1.4426950408889634f;
  float m = -INFINITY, l = 0.f;
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
    if (!tc::mbar_wait(bar, parity, &s_abort, MT_WAIT_NS)) s_abort = 1;
  };

  for (int it = 0; it < ntile; ++it) {
    const int buf = it & 1;
    // ---- S = Q K^T (one thread issues)
    if (tid == 0) {
      wait_bar(&kv_full[buf], (uint32_t)(it >> 1) & 1u);
      if (!s_abort) {
        tc::fence_after_sync();
        const uint64_t dK = tc::smem_desc_sw128(tc::smem_u32(sK + buf * MT_TILE));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem, dQ + 2 * k, dK + 2 * k, idS, k > 0 ? 1u : 0u);
        tc::mma_commit(&s_done);
      }
    }
    wait_bar(&s_done, (uint32_t)it & 1u);
    if (s_abort) break;
    tc::fence_after_sync();
    float s[64];
    tc::tmem_ld32(tS, s);
    tc::tmem_ld32(tS + 32, s + 32);
    tc::tmem_ld_wait();
    // ---- mask, scale, online softmax (log2 domain); probabilities rounded to bf16
    float mx = -INFINITY;
    if (it < ntA) {
      const int t0 = it * MT_KT;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        s[j] = (t0 + j <= lim) ? s[j] * qscale : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int kp = s_kp[buf][j], kd = s_kd[buf][j];
        const bool ok = kd >= 2 && kp - kd == dg && kd <= dd;
        s[j] = ok ? s[j] * qscale : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
    }
    // the row's reference maximum m is raised the first time and then only when a tile's
    // maximum exceeds it by more than 2^MT_LAZY_LOG2 (O and l rescaled): probabilities stay
    // within [0, 2^MT_LAZY_LOG2] with the same bf16 relative precision, and O is rarely
    // read back
    float cr = 1.f;
    if (mx > m + (float)MT_LAZY_LOG2 || (m == -INFINITY && mx > -INFINITY)) {
      cr = (m == -INFINITY) ? 0.f : fast_ex2(m - mx);
      m = mx;
    }
    const float base = (m == -INFINITY) ? 0.f : m;
    float ps = 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      s[j] = bf16r(fast_ex2(s[j] - base));  // SFU 2^x (error far below the bf16 rounding)
      ps += s[j];
    }
    l = l * cr + ps;
    // ---- the previous product is done with P, O and its K / V buffer
    if (it > 0) {
      wait_bar(&pv_done, (uint32_t)(it - 1) & 1u);
      if (s_abort) break;
      tc::fence_after_sync();
      if (it + 1 < ntile) load_tile(buf ^ 1, it + 1);
      if (__any_sync(0xffffffffu, cr != 1.f)) {
        float o[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tc::tmem_ld32(tO + 32 * half, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= cr;
          tc::tmem_st32(tO + 32 * half, o);
        }
        tc::tmem_st_wait();
      }
    }
    // ---- P row into the A tile of O += P V
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 w;
      w.x = pack_bf16(s[8 * c + 0], s[8 * c + 1]);
      w.y = pack_bf16(s[8 * c + 2], s[8 * c + 3]);
      w.z = pack_bf16(s[8 * c + 4], s[8 * c + 5]);
      w.w = pack_bf16(s[8 * c + 6], s[8 * c + 7]);
      *(uint4*)(sP + sw128(tid, c)) = w;
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      const uint64_t dV = tc::smem_desc_sw128(tc::smem_u32(sV + buf * MT_TILE));
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_bf16(tmem + 64, dP + 2 * k, dV + 128 * k, idPV, (it > 0 || k > 0) ? 1u : 0u);
      tc::mma_commit(&pv_done);
    }
  }
  // ---- normalised output (rows outside the contract see no key and store zeros)
  if (ntile > 0 && !s_abort) wait_bar(&pv_done, (uint32_t)(ntile - 1) & 1u);
  __syncthreads();
  if (s_abort) {
    if (tid == 0) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
  } else {
    tc::fence_after_sync();
    float o[64];
    if (ntile > 0) {
      tc::tmem_ld32(tO, o);
      tc::tmem_ld32(tO + 32, o + 32);
      tc::tmem_ld_wait();
    }
    if (in) {
      // hi (and lo) bf16 parts, 16 bytes per store
      const float inv = (ntile > 0 && l > 0.f) ? 1.f / l : 0.f;
      const size_t ld = (size_t)a.nq * HD;
      uint4* hi_row = (uint4*)((bf16*)a.o + (size_t)qi * ld + h * HD);
      uint4* lo_row = (uint4*)((bf16*)a.o + (size_t)(qi + a.M) * ld + h * HD);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float v0 = ntile > 0 ? o[8 * c + 2 * u] * inv : 0.f;
          const float v1 = ntile > 0 ? o[8 * c + 2 * u + 1] * inv : 0.f;
          const float h0 = bf16r(v0), h1 = bf16r(v1);
          wh[u] = pack_bf16(h0, h1);
          wl[u] = pack_bf16(v0 - h0, v1 - h1);
        }
        hi_row[c] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        if (a.split) lo_row[c] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 128);
  }
}

}  // namespace

int masked_attn_tc_launch(TcGemmPlan* pl, const MaskedAttnArgs& a, cudaStream_t s) {
  if (!pl || a.hd != 64 || a.nkv <= 0 || a.nq % a.nkv || 128 % (a.nq / a.nkv) || a.M <= 0)
    return PEAGLE_ERR_UNSUPPORTED;
  // K / V rows (all rows, and the depth-1 rows by position) as [rows][nkv * 64] with
  // boxes of 64 rows x one head's 64 columns
  CUtensorMap mk1, mv1, mk, mv;
  const int w = a.nkv * 64;
  if (!tc_tensor_map(pl, &mk1, a.k1, a.n, w, w, 64) ||
      !tc_tensor_map(pl, &mv1, a.v1, a.n, w, w, 64) ||
      !tc_tensor_map(pl, &mk, a.k, a.M, w, w, 64) || !tc_tensor_map(pl, &mv, a.v, a.M, w, w, 64))
    return PEAGLE_ERR_UNSUPPORTED;
  if (smem_optin((const void*)masked_attn_tc_kernel, MT_SMEM) != cudaSuccess)
    return PEAGLE_ERR_CUDA;
  const int QR = 128 / (a.nq / a.nkv);
  dim3 grid((unsigned)((a.M + QR - 1) / QR), (unsigned)a.nkv);
  cudaError_t e = launch_pdl(masked_attn_tc_kernel, grid, dim3(MT_THREADS), (size_t)MT_SMEM, s,
                             mk1, mv1, mk, mv, a);
  return e == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

}  // namespace peagle
