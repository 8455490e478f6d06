// The training step's plain products on the library's own kernels.
//
// bf16 drafters: C = alpha A B^T + beta C on tcgen05 tensor cores, kind::tf32 -- fp32
// operands in memory, rounded to TF32 by the MMA, fp32 accumulation in tensor memory.
// Both operands K-major ([rows][k], 32 fp32 = one 128-byte row per k-block, loaded by TMA
// with 128-byte swizzle); an operand stored the other way round (the backward's dX = dY W
// and dW = dY^T X) is first transposed into a scratch buffer by a tiled transpose kernel,
// and so is one whose row stride is not a multiple of 16 bytes (TMA's rule).
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles: an N = 256 MMA reads 12 KB of
// operands from shared memory per 8-deep k step (the 128 x 128 shape needs 8 KB for half
// the work), so the tensor pipe, not shared-memory bandwidth, sets the pace.  Warp 0 lane
// 0 issues the TMA loads into a 4-stage ring, warp 1 lane 0 the MMAs (4 of K = 8 per
// k-block) into one of two 256-column accumulators, and warps 2-5 read the other
// accumulator back (one output row per thread) and store alpha * acc + beta * C, so a
// tile's epilogue overlaps the next tile's main loop.  Tiles are visited in groups of 16
// row tiles, so the CTAs in flight at any moment share their A and B tiles through L2.
//
// fp32 drafters keep fp32 arithmetic: a tiled CUDA-core GEMM with the same transposes.
#include <cuda.h>
#include <stdio.h>

#include "gemm_tc.h"
#include "gemm_tf32.h"
#include "tc_ptx.cuh"

namespace peagle {

namespace {

constexpr int TF_THREADS = 192;
constexpr int TF_BM = 128, TF_BN = 256;
constexpr int TF_A_TILE = TF_BM * 128;  // bytes of one 128-row x 32-fp32 operand tile
constexpr int TF_B_TILE = TF_BN * 128;  // bytes of one 256-row x 32-fp32 operand tile
constexpr int TF_STAGES = 4;
constexpr int TF_GROUP_M = 16;
constexpr uint64_t TF_WAIT_NS = 2000000000ull;

size_t tf_smem_bytes() {
  return 1024 + (size_t)TF_STAGES * (TF_A_TILE + TF_B_TILE) + (2 * TF_STAGES + 5) * 8 + 16;
}

struct TfArgs {
  int M, N, K, ldc, tiles_m, tiles_n;
  float alpha, beta;
  float* C;
  unsigned* err;
};

// Tile t of the grouped order: groups of TF_GROUP_M row tiles, row tile fastest inside a
// group, so consecutive tiles share their B tile and a group's tiles share A tiles.
__device__ __forceinline__ void tf_tile(const TfArgs& a, int t, int& mi, int& ni) {
  const int per_group = TF_GROUP_M * a.tiles_n;
  const int g = t / per_group;
  const int first = g * TF_GROUP_M;
  const int gm = min(a.tiles_m - first, TF_GROUP_M);
  const int r = t - g * per_group;
  mi = first + r % gm;
  ni = r / gm;
}

__global__ void __launch_bounds__(TF_THREADS, 1)
    tf32_gemm_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                     TfArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = sA + TF_STAGES * TF_A_TILE;
  uint64_t* full = (uint64_t*)(sB + TF_STAGES * TF_B_TILE);
  uint64_t* empty = full + TF_STAGES;
  uint64_t* accf = empty + TF_STAGES;  // [2] accumulator b holds a finished tile
  uint64_t* acce = accf + 2;           // [2] accumulator b was read back (4 warp arrivals)
  uint64_t* fin = acce + 2;            // every MMA issued has completed
  uint32_t* s_tmem = (uint32_t*)(fin + 1);
  volatile int* s_abort = (volatile int*)(s_tmem + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (a.K + 31) / 32;
  const int tiles = a.tiles_m * a.tiles_n;
  if (threadIdx.x == 0) {
    for (int i = 0; i < TF_STAGES; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);
    }
    tc::mbar_init(fin, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(s_tmem, 2u * TF_BN);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = tc::policy_evict_last();
      long long it = 0;  // k-blocks loaded so far (all tiles)
      for (int t = blockIdx.x; t < tiles && !*s_abort; t += gridDim.x) {
        int mi, ni;
        tf_tile(a, t, mi, ni);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = (int)(it % TF_STAGES);
          if (it >= TF_STAGES &&
              !tc::mbar_wait(&empty[st], (uint32_t)(((it / TF_STAGES) - 1) & 1), s_abort,
                             TF_WAIT_NS)) {
            if (!*s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
            *s_abort = 1;
            break;
          }
          tc::mbar_expect_tx(&full[st], (uint32_t)(TF_A_TILE + TF_B_TILE));
          tc::tma_load_2d(sA + (size_t)st * TF_A_TILE, &ma, kb * 32, mi * TF_BM, &full[st], pol);
          tc::tma_load_2d(sB + (size_t)st * TF_B_TILE, &mb, kb * 32, ni * TF_BN, &full[st], pol);
        }
      }
      if (*s_abort) {
        // the loads in flight land (bounded) before the CTA can exit
        int never = 0;
        for (long long q = (it > TF_STAGES ? it - TF_STAGES : 0); q < it; ++q)
          tc::mbar_wait(&full[q % TF_STAGES], (uint32_t)((q / TF_STAGES) & 1), &never,
                        10000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_tf32(TF_BM, TF_BN);
      long long it = 0;
      int j = 0;  // tiles of this CTA
      for (int t = blockIdx.x; t < tiles && !*s_abort; t += gridDim.x, ++j) {
        const int b = j & 1;
        if (j >= 2 &&
            !tc::mbar_wait(&acce[b], (uint32_t)(((j >> 1) - 1) & 1), s_abort, TF_WAIT_NS)) {
          if (!*s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
          *s_abort = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(b * TF_BN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = (int)(it % TF_STAGES);
          if (!tc::mbar_wait(&full[st], (uint32_t)((it / TF_STAGES) & 1), s_abort,
                             TF_WAIT_NS)) {
            if (!*s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
            *s_abort = 1;
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(sA + (size_t)st * TF_A_TILE));
          const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(sB + (size_t)st * TF_B_TILE));
#pragma unroll
          for (int k = 0; k < 4; ++k)  // K = 8 TF32 values (32 bytes) per MMA
            tc::mma_tf32(d, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(&empty[st]);
        }
        if (!ok) break;
        tc::mma_commit(&accf[b]);
      }
      // arrives once every MMA issued above has completed (also after an abort), so that
      // tensor memory is freed only when nothing writes it any more
      tc::mma_commit(fin);
      int never = 0;
      tc::mbar_wait(fin, 0u, &never, 10000000ull);
    }
  } else {
    // epilogue: thread t holds output row (tile row) t = TMEM lane t, 256 columns
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const bool vec = (a.ldc & 3) == 0 && ((uintptr_t)a.C & 15) == 0;
    int j = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++j) {
      const int b = j & 1;
      if (!tc::mbar_wait(&accf[b], (uint32_t)((j >> 1) & 1), s_abort, TF_WAIT_NS)) {
        if (lane == 0 && !*s_abort) raise_error(a.err, PEAGLE_DEV_TIMEOUT);
        *s_abort = 1;
        break;
      }
      tc::fence_after_sync();
      int mi, ni;
      tf_tile(a, t, mi, ni);
      const int m = mi * TF_BM + r;
      const uint32_t tb = tmem + (uint32_t)(b * TF_BN) + ((uint32_t)(quarter * 32) << 16);
      float* crow = a.C + (size_t)m * a.ldc;
      for (int c0 = 0; c0 < TF_BN; c0 += 32) {
        float v[32];
        tc::tmem_ld32(tb + c0, v);
        tc::tmem_ld_wait();
        const int n = ni * TF_BN + c0;
        if (m >= a.M || n >= a.N) continue;
        if (vec && n + 32 <= a.N) {
#pragma unroll
          for (int q = 0; q < 32; q += 4) {
            float4 o = make_float4(a.alpha * v[q], a.alpha * v[q + 1], a.alpha * v[q + 2],
                                   a.alpha * v[q + 3]);
            if (a.beta != 0.f) {
              const float4 c = *(const float4*)(crow + n + q);
              o.x += a.beta * c.x;
              o.y += a.beta * c.y;
              o.z += a.beta * c.z;
              o.w += a.beta * c.w;
            }
            *(float4*)(crow + n + q) = o;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            if (n + q < a.N) {
              float o = a.alpha * v[q];
              if (a.beta != 0.f) o += a.beta * crow[n + q];
              crow[n + q] = o;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acce[b]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2u * TF_BN);
  }
}

// out[c][r] = in[r][c] for r < rows, c < cols: 64 x 64 tiles through shared memory, 16
// elements per thread (coalesced 128-byte rows on both sides; the 65-float row stride
// keeps the column reads free of bank conflicts).
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ in, int rows,
                                                        int cols, int ld_in,
                                                        float* __restrict__ out, int ld_out,
                                                        size_t stride_in, size_t stride_out) {
  __shared__ float t[64][65];
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  in += blockIdx.z * stride_in;  // batch z
  out += blockIdx.z * stride_out;
  const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + ty + 8 * i;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + tx + 32 * h;
      if (r < rows && c < cols) t[ty + 8 * i][tx + 32 * h] = __ldg(in + (size_t)r * ld_in + c);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = c0 + ty + 8 * i;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = r0 + tx + 32 * h;
      if (r < rows && c < cols) out[(size_t)c * ld_out + r] = t[tx + 32 * h][ty + 8 * i];
    }
  }
}

// out[r][c] = in[r][c] into a buffer whose row stride is padded.
__global__ void pack_kernel(const float* __restrict__ in, int rows, int cols, int ld_in,
                            float* __restrict__ out, int ld_out) {
  const size_t total = (size_t)rows * cols;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / cols, c = i - r * cols;
    out[r * ld_out + c] = in[r * ld_in + c];
  }
}

// fp32 drafters: C[m x n] = alpha op(A) op(B) + beta C on the CUDA cores, 64 x 64 tiles,
// 4 x 4 outputs per thread; op(A) is A [m x k] or A^T of A [k x m], op(B) is B [k x n] or
// B^T of B [n x k].
__global__ void __launch_bounds__(256) simt_gemm_kernel(bool ta, bool tb, int m, int n, int k,
                                                       float alpha, const float* __restrict__ A,
                                                       int lda, const float* __restrict__ B,
                                                       int ldb, float beta, float* C, int ldc) {
  __shared__ float sa[16][65];
  __shared__ float sb[16][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int l0 = 0; l0 < k; l0 += 16) {
    for (int e = threadIdx.x; e < 16 * 64; e += 256) {
      const int l = e / 64, q = e % 64;
      const int gi = i0 + q, gj = j0 + q, gl = l0 + l;
      float av = 0.f, bv = 0.f;
      if (gi < m && gl < k) av = ta ? A[(size_t)gl * lda + gi] : A[(size_t)gi * lda + gl];
      if (gj < n && gl < k) bv = tb ? B[(size_t)gj * ldb + gl] : B[(size_t)gl * ldb + gj];
      sa[l][q] = av;
      sb[l][q] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int l = 0; l < 16; ++l) {
      float x[4], y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x[u] = sa[l][ty * 4 + u];
        y[u] = sb[l][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(x[u], y[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= m) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j >= n) continue;
      float o = alpha * acc[u][v];
      if (beta != 0.f) o += beta * C[(size_t)i * ldc + j];
      C[(size_t)i * ldc + j] = o;
    }
  }
}

int cdiv_i(long long a, int b) { return (int)((a + b - 1) / b); }

}  // namespace

void launch_transpose_f32(const float* in, int rows, int cols, int ld_in, float* out, int ld_out,
                          cudaStream_t s, int batch, size_t stride_in, size_t stride_out) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return;
  dim3 grid(cdiv_i(cols, 64), cdiv_i(rows, 64), batch);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(in, rows, cols, ld_in, out, ld_out, stride_in,
                                                stride_out);
}

size_t tf32_scratch_floats(int rows, int cols) {
  return (size_t)rows * (size_t)((cols + 3) / 4 * 4);
}

int train_gemm(const TrainGemmCtx& g, bool ta, bool tb, int m, int n, int k, float alpha,
               const float* A, int lda, const float* B, int ldb, float beta, float* C, int ldc,
               cudaStream_t s) {
  if (m <= 0 || n <= 0) return PEAGLE_OK;
  if (!g.tc) {
    dim3 grid(cdiv_i(n, 64), cdiv_i(m, 64));
    simt_gemm_kernel<<<grid, 256, 0, s>>>(ta, tb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc);
    return cudaGetLastError() == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
  }
  // K-major operands A' [m][k] and B' [n][k] with 16-byte row strides
  auto k_major = [&](const float* X, int ldx, bool stored_k_major, int rows, float* scratch,
                     size_t cap, int* ld_out) -> const float* {
    const bool aligned = (ldx & 3) == 0 && ((uintptr_t)X & 15) == 0;
    if (stored_k_major && aligned) {
      *ld_out = ldx;
      return X;
    }
    const int ld = (k + 3) / 4 * 4;
    if ((size_t)rows * ld > cap) return nullptr;
    if (stored_k_major) {  // [rows][k] with an unaligned stride: copy
      pack_kernel<<<1024, 256, 0, s>>>(X, rows, k, ldx, scratch, ld);
    } else {  // stored [k][rows]: transpose
      launch_transpose_f32(X, k, rows, ldx, scratch, ld, s);
    }
    *ld_out = ld;
    return scratch;
  };
  int lda_k = 0, ldb_k = 0;
  const float* Ak = k_major(A, lda, !ta, m, g.scratch_a, g.scratch_floats, &lda_k);
  const float* Bk = k_major(B, ldb, tb, n, g.scratch_b, g.scratch_floats, &ldb_k);
  if (!Ak || !Bk) return PEAGLE_ERR_CAPACITY;
  CUtensorMap mA, mB;
  if (!tc_tensor_map_f32(g.tc, &mA, Ak, m, k, lda_k, TF_BM) ||
      !tc_tensor_map_f32(g.tc, &mB, Bk, n, k, ldb_k, TF_BN))
    return PEAGLE_ERR_UNSUPPORTED;
  const size_t smem = tf_smem_bytes();
  if (smem_optin((const void*)tf32_gemm_kernel, smem) != cudaSuccess) return PEAGLE_ERR_CUDA;
  TfArgs a;
  a.M = m;
  a.N = n;
  a.K = k;
  a.ldc = ldc;
  a.tiles_m = cdiv_i(m, TF_BM);
  a.tiles_n = cdiv_i(n, TF_BN);
  a.alpha = alpha;
  a.beta = beta;
  a.C = C;
  a.err = g.err;
  const long long tiles = (long long)a.tiles_m * a.tiles_n;
  if (tiles > (1LL << 30)) return PEAGLE_ERR_CAPACITY;
  const int sms = tc_num_sms(g.tc);
  const int grid = (int)(tiles < sms ? tiles : sms);
  tf32_gemm_kernel<<<grid, TF_THREADS, smem, s>>>(mA, mB, a);
  return cudaGetLastError() == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

}  // namespace peagle
