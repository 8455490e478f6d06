// Tensor-core GEMM of the bf16 draft pass on sm_103a: tcgen05.mma with the accumulator
// in tensor memory, operands streamed by TMA into a shared-memory ring, stream-K work
// split, and the pass's fused epilogues.
//
// Y^T = W X^T with W [Nout, Kd] (weights, the MMA's M=128 operand, "swap-AB") and
// X [rows, Kd] (activations, the MMA's N operand).  The decode pass has only batch x K
// rows, so the weight stream is the whole cost: the flattened (tile, k-block) space is
// cut into one equal contiguous range per CTA (stream-K), every SM streams the same
// number of weight bytes, and a tile shared by several CTAs is finished by whichever
// contributor arrives last (atomic counter, no waiting), which adds the fp32 partials in
// contributor order and applies the epilogue.
//
// Split activations: an operand row may be carried as a bf16 hi part and a bf16 lo part
// (x = hi + lo to about 16 significant bits).  Both parts go through the same MMA as
// extra N columns and the epilogue adds their products, so the weights are read once.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA loads, warp 1 lane 0 issues
// tcgen05.mma (and warp 1 owns the TMEM allocation), warps 2-5 drain the accumulator
// (tcgen05.ld), exchange partials and run the epilogue.  Two TMEM accumulators let the
// epilogue of one segment overlap the MMAs of the next.
//
// Programmatic dependent launch: weight tiles do not depend on the previous kernel, so
// the producer issues the first ring's weight loads before griddepcontrol.wait and the
// activation loads after it.
#include <cuda.h>
#include <stdio.h>
#include <stdlib.h>

#include <map>
#include <mutex>
#include <tuple>

#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace peagle {

constexpr int TC_THREADS = 192;  // one epilogue group (decode-sized GEMMs)
constexpr int TC_THREADS2 = 320; // two epilogue groups (large-M GEMMs)
constexpr int A_BYTES = 128 * 128;  // one 128 x 64 bf16 weight tile
// 64-wide k-blocks per stage of the CTA-pair kernel: one tensor load brings two k-blocks of
// a 128-row tile (32 KB), which the TMA units stream faster than twice as many 16 KB loads
constexpr int PAIR_KU = 2;
constexpr int STAGE_F_BYTES = 32 * 128 * 4;

struct TcParams {
  int Nout, Kd;
  int R;        // logical rows
  int split;    // X rows [0,R) hi parts, [R,2R) lo parts
  int additive; // epilogue adds into its destination: no cross-CTA reduction
  int BN;       // MMA N = operand rows per tile
  int rpt;      // logical rows per tile
  int lo_col;   // split: TMEM column of the lo part of tile row 0
  int two_box;  // split with several tiles: hi and lo rows come from two 128-row boxes
  int b_rows;   // operand rows per stage (one box): BN, or 2R when folded
  int mt;       // 128-row weight sub-tiles per tile (1 or 2), all against the same operand
  int fold;     // split single tile: the MMA adds the hi and the lo products into the same
                // R accumulator columns (two MMAs per k-step), so BN = R
  int n_tiles;  // row tiles
  int m_tiles;  // 128-feature weight tiles
  int m_inner;  // tile order: weight tiles vary fastest (the weights are re-read per row
                // tile and must stay in L2), else row tiles vary fastest
  int KB;       // k-blocks of 64
  long long total;  // stream-K iterations: (tiles - dp_waves * G) * KB
  int G;        // CTAs
  int dp_waves; // whole tiles per CTA taken first in waves (tile = w * G + c), before the
                // stream-K split of the remaining tiles
  int stages;
  uint32_t tmem_cols;
  float* ws;          // partial slots [2G][BN][128]
  unsigned* counters; // per tile, zero between launches
  unsigned* err;
};

// Stream-K space: iterations (tile - dp_waves * G) * KB + kb of the tiles left after the
// whole-tile waves; CTA c owns [range_begin(c), range_begin(c + 1)).
__device__ __forceinline__ long long range_begin(long long c, const TcParams& p) {
  return c * p.total / p.G;
}

// This CTA's iterations v = 0 .. n-1: first dp_waves whole tiles (w * G + c), then its
// stream-K range.  Large-M GEMMs get whole-tile waves so that concurrently running CTAs
// work on neighbouring tiles (L2 reuse); decode-sized GEMMs are pure stream-K.
struct Work {
  long long dpv;            // iterations in whole-tile waves
  long long sk_beg, sk_end; // stream-K range
  long long n;
};
__device__ __forceinline__ Work make_work(const TcParams& p, int c) {
  Work w;
  w.dpv = (long long)p.dp_waves * p.KB;
  w.sk_beg = range_begin(c, p);
  w.sk_end = range_begin(c + 1, p);
  w.n = w.dpv + (w.sk_end - w.sk_beg);
  return w;
}
// tile and k-block of iteration v; *seg_end = end of the tile segment containing v
__device__ __forceinline__ int work_tile(const TcParams& p, const Work& w, int c, long long v,
                                         int* kb, long long* seg_end) {
  if (v < w.dpv) {
    const int wv = (int)(v / p.KB);
    *kb = (int)(v - (long long)wv * p.KB);
    if (seg_end) *seg_end = (long long)(wv + 1) * p.KB;
    return wv * p.G + c;
  }
  const long long it = w.sk_beg + (v - w.dpv);
  const int t = (int)(it / p.KB);
  *kb = (int)(it - (long long)t * p.KB);
  if (seg_end) {
    long long e = (long long)(t + 1) * p.KB;
    if (e > w.sk_end) e = w.sk_end;
    *seg_end = w.dpv + (e - w.sk_beg);
  }
  return p.dp_waves * p.G + t;
}
// CTA whose stream-K range contains iteration `it`
__device__ __forceinline__ int owner_of(long long it, const TcParams& p) {
  long long c = it * p.G / p.total;
  while (c + 1 < p.G && range_begin(c + 1, p) <= it) ++c;
  while (c > 0 && range_begin(c, p) > it) --c;
  return (int)c;
}

// named barriers: 1 + g for epilogue group g (128 threads), 3 for all epilogue warps
__device__ __forceinline__ void epi_bar(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}
template <int NEG>
__device__ __forceinline__ void epi_bar_all() {
  if (NEG == 1) asm volatile("bar.sync 1, 128;" ::: "memory");
  else asm volatile("bar.sync 3, %0;" ::"n"(128 * NEG) : "memory");
}

__device__ __forceinline__ int tile_m(int tile, const TcParams& p) {
  return p.m_inner ? tile % p.m_tiles : tile / p.n_tiles;
}
__device__ __forceinline__ int tile_n(int tile, const TcParams& p) {
  return p.m_inner ? tile / p.m_tiles : tile % p.n_tiles;
}

// Activation operand of k-block kb for row tile nt: one box of BN rows, or (split over
// several tiles) the tile's 128 hi rows followed by its 128 lo rows.
__device__ __forceinline__ void load_b(uint8_t* dst, const CUtensorMap* m, int kb, int nt,
                                       uint64_t* bar, uint64_t pol, const TcParams& p) {
  if (p.two_box) {
    tc::tma_load_2d(dst, m, kb * 64, nt * 128, bar, pol);
    tc::tma_load_2d(dst + 128 * 128, m, kb * 64, p.R + nt * 128, bar, pol);
  } else {
    tc::tma_load_2d(dst, m, kb * 64, nt * p.b_rows, bar, pol);
  }
}

// NEG epilogue groups of four warps.  NEG = 1 (decode-sized): two CTAs per SM, so under
// programmatic dependent launch the next projection's CTA starts (and prefetches its
// weights) beside this one.  NEG = 2 (large M, tensor-bound): the two groups drain
// alternate row chunks of a tile, each with its own half of the staging buffer.
template <int NEG>
__global__ void __launch_bounds__(NEG == 1 ? TC_THREADS : TC_THREADS2, NEG == 1 ? 2 : 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const TcParams p, const EpiArgs epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int S = p.stages;
  const int B_BYTES = p.b_rows * 128;
  const int AS_BYTES = p.mt * A_BYTES;  // weight bytes per stage
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)S * AS_BYTES;
  float* stg = (float*)(sB + (size_t)S * B_BYTES);  // [32][128] fp32 epilogue staging
  uint64_t* full = (uint64_t*)((uint8_t*)stg + STAGE_F_BYTES);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint64_t* acce = accf + 2;
  uint32_t* s_tmem = (uint32_t*)(acce + 2);
  volatile int* s_flag = (volatile int*)(s_tmem + 1);
  volatile int* s_abort = s_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&accf[i], 1);
      tc::mbar_init(&acce[i], 128 * NEG);
    }
    *s_abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tc::tmem_alloc(s_tmem, p.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  tc::pdl_launch_dependents();

  const Work wk = make_work(p, c);
  const int KB = p.KB;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // the operand read once streams through L2 (evict first); the one cycled across
      // tiles stays (evict last): activations for decode-sized GEMMs, weights when the
      // weight tiles vary fastest
      const uint64_t pol_w = p.m_inner ? tc::policy_evict_last() : tc::policy_evict_first();
      const uint64_t pol_x = p.m_inner ? tc::policy_evict_first() : tc::policy_evict_last();
      const uint32_t bytes = AS_BYTES + B_BYTES;
      const long long n_it = wk.n;
      const int npre = (int)(n_it < S ? n_it : S);
      for (int i = 0; i < npre; ++i) {
        int kb;
        const int tile = work_tile(p, wk, c, i, &kb, nullptr);
        tc::mbar_expect_tx(&full[i], bytes);
        for (int h = 0; h < p.mt; ++h)
          tc::tma_load_2d(sA + (size_t)i * AS_BYTES + h * A_BYTES, &tmW, kb * 64,
                          (tile_m(tile, p) * p.mt + h) * 128, &full[i], pol_w);
      }
      tc::pdl_wait();
      for (int i = 0; i < npre; ++i) {
        int kb;
        const int tile = work_tile(p, wk, c, i, &kb, nullptr);
        load_b(sB + (size_t)i * B_BYTES, &tmX, kb, tile_n(tile, p), &full[i], pol_x, p);
      }
      int stage = npre % S;
      uint32_t ph = (npre == S) ? 1u : 0u;
      for (long long it = npre; it < n_it; ++it) {
        if (!tc::mbar_wait(&empty[stage], ph ^ 1u, s_abort)) {
          raise_error(p.err, PEAGLE_DEV_TIMEOUT);
          *s_abort = 1;
          break;
        }
        int kb;
        const int tile = work_tile(p, wk, c, it, &kb, nullptr);
        tc::mbar_expect_tx(&full[stage], bytes);
        for (int h = 0; h < p.mt; ++h)
          tc::tma_load_2d(sA + (size_t)stage * AS_BYTES + h * A_BYTES, &tmW, kb * 64,
                          (tile_m(tile, p) * p.mt + h) * 128, &full[stage], pol_w);
        load_b(sB + (size_t)stage * B_BYTES, &tmX, kb, tile_n(tile, p), &full[stage], pol_x, p);
        if (++stage == S) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, p.BN);
      int stage = 0;
      uint32_t ph = 0;
      int seg = 0;
      bool ok = true;
      for (long long it = 0; it < wk.n && ok;) {
        int kb0;
        long long seg_end;
        work_tile(p, wk, c, it, &kb0, &seg_end);
        const int buf = seg & 1;
        const uint32_t use = (uint32_t)(seg >> 1);
        if (!tc::mbar_wait(&acce[buf], (use & 1u) ^ 1u, s_abort)) {
          raise_error(p.err, PEAGLE_DEV_TIMEOUT);
          *s_abort = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(buf * p.mt * p.BN);
        const long long seg_beg = it;
        for (; it < seg_end; ++it) {
          if (!tc::mbar_wait(&full[stage], ph, s_abort)) {
            raise_error(p.err, PEAGLE_DEV_TIMEOUT);
            *s_abort = 1;
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(sB + (size_t)stage * B_BYTES));
          // folded: the lo rows start R rows (R * 128 bytes, whole swizzle atoms) later
          const uint64_t bl = tc::smem_desc_sw128(
              tc::smem_u32(sB + (size_t)stage * B_BYTES + (size_t)p.R * 128));
          for (int h = 0; h < p.mt; ++h) {
            const uint32_t dh = d + (uint32_t)(h * p.BN);
            const uint64_t ah = tc::smem_desc_sw128(
                tc::smem_u32(sA + (size_t)stage * AS_BYTES + (size_t)h * A_BYTES));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              tc::mma_bf16(dh, ah + 2 * k, bd + 2 * k, idesc, (it != seg_beg || k > 0) ? 1u : 0u);
              if (p.fold) tc::mma_bf16(dh, ah + 2 * k, bl + 2 * k, idesc, 1u);
            }
          }
          tc::mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            ph ^= 1u;
          }
        }
        tc::mma_commit(&accf[buf]);
        ++seg;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int eg = (threadIdx.x - 64) >> 7;  // epilogue group
    const int et = (threadIdx.x - 64) & 127; // 0 .. 127 within the group
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int ml = quarter * 32 + lane;      // tile feature = TMEM lane
    const int R = p.R;
    // staging: [32 / NEG rows][128] fp32 per group
    float* gstg = stg + (size_t)eg * (32 / NEG) * 128;
    int seg = 0;
    for (long long it = 0; it < wk.n;) {
      int kb0;
      long long seg_end;
      const int tile = work_tile(p, wk, c, it, &kb0, &seg_end);
      const bool whole = it < wk.dpv;  // a wave tile: this CTA is its only contributor
      it = seg_end;
      const int buf = seg & 1;
      const uint32_t use = (uint32_t)(seg >> 1);
      ++seg;
      // one thread per group observes the accumulator barrier; the group's named barrier
      // publishes the outcome so its warps stay in lock-step even if the wait gives up
      if (et == 0 && !tc::mbar_wait(&accf[buf], use & 1u, s_abort)) {
        raise_error(p.err, PEAGLE_DEV_TIMEOUT);
        *s_abort = 1;
      }
      epi_bar(eg);
      if (*s_abort) break;
      tc::fence_after_sync();
      const int mt = tile_m(tile, p), nt = tile_n(tile, p);
      const int row0 = nt * p.rpt;               // first logical row of this tile
      const int lrows = min(p.rpt, R - row0);    // logical rows in this tile
      const long long t_beg = (long long)(tile - p.dp_waves * p.G) * KB;  // stream-K space
      const int cf = whole ? c : owner_of(t_beg, p);
      const int cl = whole ? c : owner_of(t_beg + KB - 1, p);
      // hi and lo products in separate TMEM columns (split), or summed by the MMA (fold)
      const int sp = (p.split && !p.fold) ? 1 : 0;
      // sub-tile h (128 weight rows) of this tile: TMEM columns [h BN, (h+1) BN) of the buffer
      const uint32_t tb0 =
          tmem + (uint32_t)(buf * p.mt * p.BN) + ((uint32_t)(quarter * 32) << 16);
      // chunking: split tiles take 16 / NEG logical rows per chunk (hi + lo columns), others
      // 32 / NEG; chunk ch belongs to group ch % NEG
      const int step = (sp ? 16 : 32) / NEG;
      const int nch = (lrows + step - 1) / step;
      // sub-tiles holding output features (a last tile may have one past Nout)
      const int nh = min(p.mt, (epi.Nout - mt * p.mt * 128 + 127) / 128);
      if (cf == cl || p.additive) {
        // ---- sole owner, or an additive epilogue (each contributor adds its own partial):
        //      TMEM -> staging -> epilogue.  The fixed-point adds (residual, fc output) are
        //      elementwise: each thread adds its own feature's rows straight from the
        //      registers it loaded, with no staging and no group barrier.
        const bool direct = epi.kind == EPI_RESID || epi.kind == EPI_STORE;
        constexpr int HALF = 16 / NEG;  // TMEM columns per load
        for (int h = 0; h < nh; ++h) {
          const int m0 = (mt * p.mt + h) * 128;
          const uint32_t tb = tb0 + (uint32_t)(h * p.BN);
          const bool last_h = h == nh - 1;
          for (int ch = eg; ch < nch; ch += NEG) {
            const int i0 = ch * step;
            float v[HALF], w[HALF];
#pragma unroll
            for (int j = 0; j < HALF; ++j) w[j] = 0.f;
            if (NEG == 1) {
              tc::tmem_ld16(tb + i0, v);
              if (sp) {
                tc::tmem_ld16(tb + p.lo_col + i0, w);
              } else if (i0 + 16 < p.BN) {
                tc::tmem_ld16(tb + i0 + 16, w);
              }
            } else {
              tc::tmem_ld8(tb + i0, v);
              if (sp) {
                tc::tmem_ld8(tb + p.lo_col + i0, w);
              } else if (i0 + 8 < p.BN) {
                tc::tmem_ld8(tb + i0 + 8, w);
              }
            }
            tc::tmem_ld_wait();
            const bool release = last_h && ch + NEG >= nch;  // group's last TMEM read
            if (direct) {
              if (release) {
                tc::fence_before_sync();
                tc::mbar_arrive(&acce[buf]);
              }
              const int m = m0 + ml;
              const int rc = min(step, lrows - i0);
              fx_t* dst = epi.kind == EPI_STORE ? epi.out_fx : epi.resid;
              const int ldd = epi.kind == EPI_STORE ? epi.out_ld : epi.ld_res;
              if (m < epi.Nout) {
                fx_t* col = dst + (size_t)(row0 + i0) * ldd + m;
#pragma unroll
                for (int j = 0; j < HALF; ++j) {
                  if (sp) {
                    if (j < rc) red_add_fx(col + (size_t)j * ldd, to_fx(v[j] + w[j]));
                  } else {
                    if (j < rc) red_add_fx(col + (size_t)j * ldd, to_fx(v[j]));
                    if (HALF + j < rc) red_add_fx(col + (size_t)(HALF + j) * ldd, to_fx(w[j]));
                  }
                }
              }
              continue;
            }
#pragma unroll
            for (int j = 0; j < HALF; ++j) {
              gstg[j * 128 + ml] = v[j];
              gstg[(HALF + j) * 128 + ml] = w[j];
            }
            if (release) {
              tc::fence_before_sync();
              tc::mbar_arrive(&acce[buf]);
            }
            epi_bar(eg);
            epilogue_tile<bf16>(epi, gstg, 128, sp ? 16 / NEG : -1, m0, row0 + i0,
                                min(step, lrows - i0), et, 128);
            epi_bar(eg);
          }
        }
        if (eg >= nch) {  // a group without a chunk still releases the accumulator
          tc::fence_before_sync();
          tc::mbar_arrive(&acce[buf]);
        }
      } else {
        // ---- shared tile: write this CTA's partial, the last contributor reduces
        const int SW = p.mt * p.BN;  // partial columns: every sub-tile's accumulator
        const int slot = (range_begin(c, p) >= t_beg) ? 2 * c : 2 * c + 1;
        float* wsl = p.ws + (size_t)slot * SW * 128;
        for (int c0 = eg * 16; c0 < SW; c0 += 16 * NEG) {
          float v[16];
          tc::tmem_ld16(tb0 + c0, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) wsl[(size_t)(c0 + j) * 128 + ml] = v[j];
        }
        tc::fence_before_sync();
        tc::mbar_arrive(&acce[buf]);
        epi_bar_all<NEG>();
        if (eg == 0 && et == 0) {
          const unsigned prev = atom_add_acq_rel(p.counters + tile, 1u);
          *s_flag = (prev == (unsigned)(cl - cf)) ? 1 : 0;
        }
        epi_bar_all<NEG>();
        if (*s_flag) {
          // contributor cf's share of this tile is its last segment unless its range starts
          // exactly at the tile; every later contributor's share is its first segment
          const int slot_f = (range_begin(cf, p) == t_beg) ? 2 * cf : 2 * cf + 1;
          constexpr int SR = 32 / NEG;  // staging rows per chunk
          const int half = sp ? SR / 2 : SR;
          for (int h = 0; h < nh; ++h) {
            const int m0 = (mt * p.mt + h) * 128;
            for (int ch = eg; ch < nch; ch += NEG) {
              const int i0 = ch * step;
              // staging rows [0,half) / [half,2 half): hi / lo parts (split) or rows i0..
              int col[SR];
              float acc[SR];
#pragma unroll
              for (int j = 0; j < SR; ++j) {
                if (sp) {
                  const int ii = i0 + (j % half);
                  col[j] = h * p.BN + min((j < half) ? ii : p.lo_col + ii, p.BN - 1);
                } else {
                  col[j] = h * p.BN + min(i0 + j, p.BN - 1);
                }
                acc[j] = 0.f;
              }
              for (int cc = cf; cc <= cl; ++cc) {
                const float* src = p.ws + (size_t)(cc == cf ? slot_f : 2 * cc) * SW * 128 + ml;
#pragma unroll
                for (int j = 0; j < SR; ++j) acc[j] += __ldcg(src + (size_t)col[j] * 128);
              }
#pragma unroll
              for (int j = 0; j < SR; ++j) gstg[j * 128 + ml] = acc[j];
              epi_bar(eg);
              epilogue_tile<bf16>(epi, gstg, 128, sp ? half : -1, m0, row0 + i0,
                                  min(step, lrows - i0), et, 128);
              epi_bar(eg);
            }
          }
          epi_bar_all<NEG>();
          if (eg == 0 && et == 0) p.counters[tile] = 0u;
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, p.tmem_cols);
  }
}

// -------------------------------------------------------------------------------------
// CTA-pair variant for large-M GEMMs (the training-style forward): a cluster of two CTAs
// on neighbouring SMs runs one tcgen05.mma.cta_group::2 of M = 256 weight rows x N = 256
// activation rows.  Each CTA loads its own 128 weight rows and half of the activation
// rows (the hi rows in the even CTA, the lo rows in the odd one, or rows 0-127 / 128-255),
// so a k-block moves 32 KB into each SM instead of 48 KB: the operand stream from L2 is
// what bounds the single-CTA kernel at about half the tensor peak.  The accumulator is
// 128 lanes x 256 columns in each CTA's tensor memory, drained by each CTA's own epilogue.
// Tiles are whole (no stream-K): pair-tile t = wave * pairs + pair.
//
// Hand-offs: both CTAs' loads of a stage complete on the even CTA's stage barrier (the
// pair form of the tensor load), where the single issuing thread waits.  The MMA's commits
// arrive on the stage-free and accumulator-full barriers of both CTAs (multicast); each
// CTA's epilogue releases an accumulator with one arrive per group on the even CTA's
// barrier.
__device__ __forceinline__ int pair_tile_m(int t, const TcParams& p) {
  return p.m_inner ? t % p.m_tiles : t / p.n_tiles;
}
__device__ __forceinline__ int pair_tile_n(int t, const TcParams& p) {
  return p.m_inner ? t / p.m_tiles : t % p.n_tiles;
}

__global__ void __launch_bounds__(TC_THREADS2, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmX, const TcParams p,
                        const EpiArgs epi) {
  constexpr int NEG = 2;
  constexpr int HB = 128 * 128;  // half of the activation rows of a k-block (128 x 64 bf16)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int S = p.stages;
  uint8_t* sA = smem;                                       // [S][PAIR_KU] weight tiles
  uint8_t* sB = sA + (size_t)S * PAIR_KU * A_BYTES;          // [S][PAIR_KU] activation halves
  float* stg = (float*)(sB + (size_t)S * PAIR_KU * HB);  // [NEG][32][128] fp32 epilogue staging
  uint64_t* full = (uint64_t*)((uint8_t*)stg + NEG * STAGE_F_BYTES);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint64_t* acce = accf + 2;
  uint64_t* done_bar = acce + 2;
  uint32_t* s_tmem = (uint32_t*)(done_bar + 1);
  volatile int* s_abort = (volatile int*)(s_tmem + 1);
  __shared__ int s_rpos[NEG][128];  // RoPE positions of the tile's rows, per epilogue group

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const bool lead = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int T = p.m_tiles * p.n_tiles;  // pair-tiles
  const int KB = p.KB;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);  // even CTA: its producer's arrive, both CTAs' bytes
      tc::mbar_init(&empty[i], 1);           // the MMA's multicast commit
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&accf[i], 1);
      tc::mbar_init(&acce[i], 2 * NEG);  // one arrive per epilogue group of each CTA
    }
    tc::mbar_init(done_bar, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmX);
  }
  __syncwarp();
  if (warp == 1) {
    tc::tmem_alloc_pair(s_tmem, p.tmem_cols);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  tc::pdl_launch_dependents();

  // this pair's tiles: t = pair, pair + npairs, ...
  const int my_tiles = pair < T ? (T - 1 - pair) / npairs + 1 : 0;
  const long long n_it = (long long)my_tiles * KB;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = p.m_inner ? tc::policy_evict_last() : tc::policy_evict_first();
      const uint64_t pol_x = p.m_inner ? tc::policy_evict_first() : tc::policy_evict_last();
      // both CTAs' loads count on the even one
      const uint32_t bytes = 2 * PAIR_KU * (A_BYTES + HB);
      const uint32_t lead_full = tc::mapa_shared(full, 0);
      // A and B halves of PAIR_KU k-blocks into this CTA's stage, completing on the even
      // CTA's barrier
      auto load = [&](int st, int kb, int wr, int xr, bool a, bool b) {
        if (a)
          tc::tma_load_3d_pair(sA + (size_t)st * PAIR_KU * A_BYTES, &tmW, 0, wr, kb * PAIR_KU,
                               lead_full + (uint32_t)(st * 8), pol_w);
        if (b)
          tc::tma_load_3d_pair(sB + (size_t)st * PAIR_KU * HB, &tmX, 0, xr, kb * PAIR_KU,
                               lead_full + (uint32_t)(st * 8), pol_x);
      };
      auto coords = [&](long long it, int* kb, int* wrow, int* xrow) {
        const int ti = (int)(it / KB);
        *kb = (int)(it - (long long)ti * KB);
        const int t = pair + ti * npairs;
        const int mt = pair_tile_m(t, p), nt = pair_tile_n(t, p);
        *wrow = (2 * mt + (int)rank) * 128;
        *xrow = p.split ? (rank ? p.R : 0) + nt * 128 : nt * 256 + (int)rank * 128;
      };
      const int npre = (int)(n_it < S ? n_it : S);
      for (int i = 0; i < npre; ++i) {
        int kb, wr, xr;
        coords(i, &kb, &wr, &xr);
        if (lead) tc::mbar_expect_tx(&full[i], bytes);
        load(i, kb, wr, xr, true, false);
      }
      tc::pdl_wait();
      for (int i = 0; i < npre; ++i) {
        int kb, wr, xr;
        coords(i, &kb, &wr, &xr);
        load(i, kb, wr, xr, false, true);
      }
      int stage = npre % S;
      uint32_t ph = (npre == S) ? 1u : 0u;
      for (long long it = npre; it < n_it; ++it) {
        if (!tc::mbar_wait_cluster(&empty[stage], ph ^ 1u, s_abort)) {
          raise_error(p.err, PEAGLE_DEV_TIMEOUT);
          *s_abort = 1;
          break;
        }
        int kb, wr, xr;
        coords(it, &kb, &wr, &xr);
        if (lead) tc::mbar_expect_tx(&full[stage], bytes);
        load(stage, kb, wr, xr, true, true);
        if (++stage == S) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && lead) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      const uint32_t idesc = tc::idesc_bf16(256, 256);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      bool issued = false;
      for (int ti = 0; ti < my_tiles && ok; ++ti) {
        const int buf = ti & 1;
        const uint32_t use = (uint32_t)(ti >> 1);
        if (!tc::mbar_wait_cluster(&acce[buf], (use & 1u) ^ 1u, s_abort)) {
          raise_error(p.err, PEAGLE_DEV_TIMEOUT);
          *s_abort = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(buf * 256);
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait_cluster(&full[stage], ph, s_abort)) {
            raise_error(p.err, PEAGLE_DEV_TIMEOUT);
            *s_abort = 1;
            ok = false;
            break;
          }
          tc::fence_after_sync();
#pragma unroll
          for (int j = 0; j < PAIR_KU; ++j) {
            const uint64_t ad = tc::smem_desc_sw128(
                tc::smem_u32(sA + ((size_t)stage * PAIR_KU + j) * A_BYTES));
            const uint64_t bd =
                tc::smem_desc_sw128(tc::smem_u32(sB + ((size_t)stage * PAIR_KU + j) * HB));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc,
                                (kb > 0 || j > 0 || k > 0) ? 1u : 0u);
          }
          issued = true;
          tc::mma_commit_pair(&empty[stage], (uint16_t)3);
          if (++stage == S) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc::mma_commit_pair(&accf[buf], (uint16_t)3);
      }
      // every MMA (they write both CTAs' tensor memory) is complete before the pair parts
      if (issued) {
        tc::mma_commit_pair(done_bar, (uint16_t)1);
        int never = 0;
        tc::mbar_wait(done_bar, 0, &never, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int eg = (threadIdx.x - 64) >> 7;
    const int et = (threadIdx.x - 64) & 127;
    const int quarter = warp & 3;
    const int ml = quarter * 32 + lane;
    const int R = p.R;
    float* gstg = stg + (size_t)eg * 32 * 128;
    const uint32_t lead_acce = tc::mapa_shared(acce, 0);
    // a RoPE epilogue reads its rows' positions from a table filled while the MMAs run
    const bool pos_tab = epi.row_pos != nullptr && p.rpt <= 128;
    auto release = [&](int buf) {  // this group is done reading accumulator `buf`
      if (lead) tc::mbar_arrive(&acce[buf]);
      else tc::mbar_arrive_remote(lead_acce + (uint32_t)(buf * 8));
    };
    for (int ti = 0; ti < my_tiles; ++ti) {
      const int t = pair + ti * npairs;
      const int buf = ti & 1;
      const uint32_t use = (uint32_t)(ti >> 1);
      const int mt = pair_tile_m(t, p), nt = pair_tile_n(t, p);
      const int m0 = (2 * mt + (int)rank) * 128;
      const int row0 = nt * p.rpt;
      const int lrows = min(p.rpt, R - row0);
      if (pos_tab && et < lrows) s_rpos[eg][et] = epi.row_pos[row0 + et];
      if (et == 0 && !tc::mbar_wait_cluster(&accf[buf], use & 1u, s_abort)) {
        raise_error(p.err, PEAGLE_DEV_TIMEOUT);
        *s_abort = 1;
      }
      epi_bar(eg);
      if (*s_abort) break;
      tc::fence_after_sync();
      const uint32_t tb = tmem + (uint32_t)(buf * 256) + ((uint32_t)(quarter * 32) << 16);
      // chunks of 16 logical rows (hi + lo columns) or 32 rows; chunk ch to group ch % NEG
      const int step = p.split ? 16 : 32;
      const int nch = (lrows + step - 1) / step;
      for (int ch = eg; ch < nch; ch += NEG) {
        const int i0 = ch * step;
        float v[16], w[16];
        tc::tmem_ld16(tb + i0, v);
        tc::tmem_ld16(tb + (p.split ? p.lo_col : 16) + i0, w);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          gstg[j * 128 + ml] = v[j];
          gstg[(16 + j) * 128 + ml] = w[j];
        }
        const bool last = ch + NEG >= nch;
        if (last) tc::fence_before_sync();
        epi_bar(eg);
        if (last && et == 0) release(buf);
        if (m0 < epi.Nout)
          epilogue_tile<bf16>(epi, gstg, 128, p.split ? 16 : -1, m0, row0 + i0,
                              min(step, lrows - i0), et, 128, nullptr,
                              pos_tab ? &s_rpos[eg][i0] : nullptr);
        epi_bar(eg);
      }
      if (eg >= nch && et == 0) release(buf);
    }
  }
  __syncwarp();
  tc::fence_before_sync();
  tc::cluster_sync();  // no CTA leaves while its partner's MMAs or arrivals may target it
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, p.tmem_cols);
  }
}

// =====================================================================================
// host side
// =====================================================================================
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct TcGemmPlan {
  int num_sms;
  bool pair;  // large-M GEMMs on CTA pairs
  int pair_clusters;  // CTA pairs that fit on the GPU at once (a cluster stays in one GPC)
  int fold_mode;      // folded wide tiles: 0 where they pay (the only mode in use)
  int max_bn;
  float* ws;
  unsigned* counters;
  int max_tiles;
  unsigned* err;
  EncodeTiledFn encode;
  std::mutex mu;
  std::map<std::tuple<const void*, int, int, int, int>, CUtensorMap> maps;
};

static bool encode_map(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                       int ld, int box_rows) {
  auto key = std::make_tuple(base, rows, cols, ld, box_rows);
  {
    std::lock_guard<std::mutex> g(p->mu);
    auto itr = p->maps.find(key);
    if (itr != p->maps.end()) {
      *out = itr->second;
      return true;
    }
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = p->encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "peagle: cuTensorMapEncodeTiled failed (%d) rows=%d cols=%d ld=%d box=%d\n",
            (int)r, rows, cols, ld, box_rows);
    return false;
  }
  std::lock_guard<std::mutex> g(p->mu);
  if (p->maps.size() > 4096) p->maps.clear();
  p->maps[key] = *out;
  return true;
}

static size_t smem_bytes_pair(int stages) {
  return 1024 + (size_t)stages * PAIR_KU * (A_BYTES + 128 * 128) + 2 * STAGE_F_BYTES +
         (size_t)(2 * stages + 5) * 8 + 16;
}
// dynamic shared memory of the pair kernel: the 227 KB per-block limit less its 1 KB of
// static RoPE position tables
constexpr size_t PAIR_SMEM_BUDGET = 226 * 1024;
static size_t smem_bytes(int stages, int b_rows, int mt) {
  return 1024 /*align slack*/ + (size_t)stages * (mt * A_BYTES + b_rows * 128) + STAGE_F_BYTES +
         (size_t)(2 * stages + 4) * 8 + 16;
}

bool tc_tensor_map(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                   int ld, int box_rows) {
  return encode_map(p, out, base, rows, cols, ld, box_rows);
}
bool tc_tensor_map_ku(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                      int ld, int box_rows, int ku) {
  // (element within a 64-wide k-block, row, k-block): one box = ku consecutive k-blocks
  // of box_rows rows, each a 128-byte-swizzled [box_rows][64] tile
  if (cols % 64 || ku < 1) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)ku};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = p->encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "peagle: cuTensorMapEncodeTiled (3D) failed (%d) rows=%d cols=%d ld=%d\n",
            (int)r, rows, cols, ld);
    return false;
  }
  return true;
}
bool tc_tensor_map_f32(TcGemmPlan* p, CUtensorMap* out, const void* base, int rows, int cols,
                       int ld, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = p->encode(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "peagle: cuTensorMapEncodeTiled (fp32) failed (%d) rows=%d cols=%d ld=%d\n",
            (int)r, rows, cols, ld);
    return false;
  }
  return true;
}
float* tc_partials(TcGemmPlan* p) { return p->ws; }
int tc_num_sms(TcGemmPlan* p) { return p->num_sms; }
unsigned* tc_tile_counters(TcGemmPlan* p) { return p->counters; }
int tc_max_tiles(TcGemmPlan* p) { return p->max_tiles; }

void tc_destroy(TcGemmPlan* p) {
  if (!p) return;
  if (p->ws) cudaFree(p->ws);
  if (p->counters) cudaFree(p->counters);
  delete p;
}

int tc_create(TcGemmPlan** out, int num_sms, int rows_max, int max_dim, unsigned* err) {
  *out = nullptr;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return PEAGLE_ERR_CUDA;
  TcGemmPlan* p = new TcGemmPlan();
  p->num_sms = num_sms;
  p->encode = (EncodeTiledFn)fn;
  p->err = err;
  p->max_bn = 256;
  p->ws = nullptr;
  p->counters = nullptr;
  const int n_tiles_max = (rows_max + 15) / 16 + 1;
  p->max_tiles = ((max_dim + 127) / 128 + 1) * n_tiles_max;
  if (cudaMalloc(&p->ws, (size_t)2 * num_sms * p->max_bn * 128 * 4) != cudaSuccess ||
      cudaMalloc(&p->counters, (size_t)p->max_tiles * 4) != cudaSuccess ||
      cudaMemset(p->counters, 0, (size_t)p->max_tiles * 4) != cudaSuccess) {
    tc_destroy(p);
    return PEAGLE_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(tc_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)PAIR_SMEM_BUDGET) != cudaSuccess ||
      cudaFuncSetAttribute(tc_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           227 * 1024) != cudaSuccess ||
      cudaFuncSetAttribute(tc_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           227 * 1024) != cudaSuccess) {
    tc_destroy(p);
    return PEAGLE_ERR_CUDA;
  }
  {
    // a persistent grid of pairs must be resident at once: as many pairs as clusters of
    // two fit (each GPC holds an even number of the CTAs), not num_sms / 2
    p->pair = true;
    p->fold_mode = 0;
    p->pair_clusters = 0;
    int stages = 2;
    while (stages < 8 && smem_bytes_pair(stages + 1) <= PAIR_SMEM_BUDGET) ++stages;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(TC_THREADS2);
    cfg.dynamicSmemBytes = smem_bytes_pair(stages);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, tc_gemm_pair_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      nc = 0;
    }
    p->pair_clusters = nc < num_sms / 2 ? nc : num_sms / 2;
  }
  *out = p;
  return PEAGLE_OK;
}

static uint32_t pow2_at_least(uint32_t v) {
  uint32_t r = 32;
  while (r < v) r <<= 1;
  return r;
}

int tc_gemm(TcGemmPlan* pl, const void* W, const void* X, int ldx, int Nout, int Kd, int R,
            const EpiArgs& epi, cudaStream_t s) {
  TcParams p;
  p.Nout = Nout;
  p.Kd = Kd;
  p.R = R;
  p.split = epi.in_split ? 1 : 0;
  p.additive = (epi.kind == EPI_STORE || epi.kind == EPI_RESID || epi.kind == EPI_QKV_FX) ? 1 : 0;
  const int xrows = p.split ? 2 * R : R;
  p.two_box = 0;
  if (p.split && 2 * R <= 240) {
    // one tile: a single box of BN rows holds the hi rows [0,R) and the lo rows [R,2R)
    p.BN = (2 * R + 15) / 16 * 16;
    p.rpt = R;
    p.lo_col = R;
    p.n_tiles = 1;
  } else if (p.split) {
    // 128 logical rows per tile: hi rows in TMEM columns [0,128), lo rows in [128,256)
    p.BN = 256;
    p.rpt = 128;
    p.lo_col = 128;
    p.two_box = 1;
    p.n_tiles = (R + 127) / 128;
  } else {
    p.BN = R <= 256 ? (R + 15) / 16 * 16 : 256;
    p.rpt = p.BN;
    p.lo_col = 0;
    p.n_tiles = (R + p.BN - 1) / p.BN;
  }
  p.KB = Kd / 64;
  p.b_rows = p.BN;
  p.mt = 1;
  p.fold = 0;
  if (pl->pair && p.n_tiles > 1 && Kd % 64 == 0 && pl->pair_clusters > 0) {
    // CTA pairs: pair-tiles of 256 weight rows x (128 logical rows, hi + lo, or 256 rows)
    TcParams q = p;
    q.BN = 256;
    q.rpt = p.split ? 128 : 256;
    q.lo_col = p.split ? 128 : 0;
    q.n_tiles = (R + q.rpt - 1) / q.rpt;
    q.m_tiles = (Nout + 255) / 256;
    const long long wbytes = (long long)Nout * Kd * 2;
    const long long xbytes = (long long)xrows * Kd * 2;
    q.m_inner = wbytes < xbytes ? 1 : 0;
    const long long T = (long long)q.m_tiles * q.n_tiles;
    const int npairs = (int)(T < pl->pair_clusters ? T : pl->pair_clusters);
    q.G = npairs;
    q.dp_waves = 0;
    q.total = 0;
    int stages = 2;
    while (stages < 8 && smem_bytes_pair(stages + 1) <= PAIR_SMEM_BUDGET) ++stages;
    q.stages = stages;
    q.tmem_cols = 512;
    q.ws = pl->ws;
    q.counters = pl->counters;
    q.err = pl->err;
    q.KB = (Kd / 64 + PAIR_KU - 1) / PAIR_KU;  // k-units (the last may read zeros past Kd)
    CUtensorMap mw, mx;
    if (!tc_tensor_map_ku(pl, &mw, W, Nout, Kd, Kd, 128, PAIR_KU)) return PEAGLE_ERR_CUDA;
    if (!tc_tensor_map_ku(pl, &mx, X, xrows, Kd, ldx, 128, PAIR_KU)) return PEAGLE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * npairs);
    cfg.blockDim = dim3(TC_THREADS2);
    cfg.dynamicSmemBytes = smem_bytes_pair(stages);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel, mw, mx, q, epi);
    return e == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
  }
  // A split single tile of 64+ rows (R a multiple of 16, whole 256-row weight blocks):
  // every stage carries 2R operand rows, more bytes than a 128-row weight tile, and the
  // tile traffic through L2 and the TMA units (about 7-8 TB/s in all) bounds the GEMM.
  // Two 128-row weight sub-tiles per tile share each operand stage (32 + 2R/8 KB per
  // stage instead of 16 + 2R/8), and the MMA adds the hi and the lo products into the
  // same R accumulator columns (two MMAs per k-step) so both sub-tiles' accumulators fit
  // in tensor memory twice.  It pays where every CTA streams 20+ k-blocks between
  // epilogues of the residual or SwiGLU form (80 rows: gate/up 79 -> 71 us, down 40 -> 38
  // us per launch); with fewer, or the heavier QKV / LM-head epilogues, the doubled tile
  // gives each epilogue twice the work for the same streaming and loses (QKV 57 -> 73 us).
  const long long fold_iters = (long long)(Nout / 256) * (Kd / 64);
  const bool fold_pays =
      fold_iters >= 20LL * pl->num_sms && (epi.kind == EPI_RESID || epi.kind == EPI_SWIGLU);
  if (p.split && !p.two_box && R >= 64 && R % 16 == 0 && Nout % 256 == 0 &&
      2 * R <= pl->max_bn && pl->fold_mode >= 0 && (fold_pays || pl->fold_mode == 1)) {
    p.fold = 1;
    p.mt = 2;
    p.BN = R;
    p.b_rows = 2 * R;
    p.lo_col = 0;
  }
  // large-M projections are tensor-bound: two epilogue groups keep up with the MMA; a
  // single tile of 128+ operand rows also drains faster with two (ragged batch of 16 x
  // K=5, 80 rows: 1285 -> 1214 us per pass)
  const int neg = (p.n_tiles > 1 || p.b_rows >= 128) ? 2 : 1;
  const int m_tiles = (Nout + 128 * p.mt - 1) / (128 * p.mt);
  const long long tiles = (long long)m_tiles * p.n_tiles;
  p.m_tiles = m_tiles;
  // Concurrent CTAs work on neighbouring tiles: with weight tiles innermost all of W is
  // touched while a few row tiles are live, so W is read from DRAM once if it fits in L2;
  // with row tiles innermost the same holds for the activations.  Cycle the smaller one.
  {
    const long long wbytes = (long long)Nout * Kd * 2;
    const long long xbytes = (long long)xrows * Kd * 2;
    p.m_inner = (p.n_tiles > 1 && wbytes < xbytes) ? 1 : 0;
  }
  if (tiles > pl->max_tiles || Kd % 64) return PEAGLE_ERR_CAPACITY;
  p.G = (int)(tiles * p.KB < pl->num_sms ? tiles * p.KB : pl->num_sms);
  // whole-tile waves first: large-M GEMMs (L2 reuse), and single-tile GEMMs of 64+ rows
  // whose epilogue needs whole tiles (a shared tile costs a partial of BN x 128 fp32 per
  // contributor, 80 KB at 80 rows)
  p.dp_waves = (p.n_tiles > 1 || (!p.additive && p.b_rows >= 128)) ? (int)(tiles / p.G) : 0;
  p.total = (tiles - (long long)p.dp_waves * p.G) * p.KB;
  // shared memory ring: decode-sized tiles keep ~110 KB so a second CTA (the next
  // kernel's, under programmatic dependent launch) fits on the SM; large tiles take more
  const size_t budget = p.fold ? 227 * 1024 : p.b_rows <= 64 ? 112 * 1024 : 220 * 1024;
  int stages = 2;
  while (stages < 12 && smem_bytes(stages + 1, p.b_rows, p.mt) <= budget) ++stages;
  p.stages = stages;

  // single-tile split reads 16-column groups starting at column R + i0, which may run
  // up to 15 columns past the second accumulator: keep that slack allocated
  p.tmem_cols = pow2_at_least(
      (uint32_t)(2 * p.mt * p.BN + ((p.split && !p.two_box && !p.fold) ? 16 : 0)));
  if (p.tmem_cols > 512) return PEAGLE_ERR_CAPACITY;
  p.ws = pl->ws;
  p.counters = pl->counters;
  p.err = pl->err;
  CUtensorMap mw, mx;
  if (!encode_map(pl, &mw, W, Nout, Kd, Kd, 128)) return PEAGLE_ERR_CUDA;
  if (!encode_map(pl, &mx, X, xrows, Kd, ldx, p.two_box ? 128 : p.b_rows)) return PEAGLE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(neg == 1 ? TC_THREADS : TC_THREADS2);
  cfg.dynamicSmemBytes = smem_bytes(stages, p.b_rows, p.mt);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = neg == 1 ? cudaLaunchKernelEx(&cfg, tc_gemm_kernel<1>, mw, mx, p, epi)
                            : cudaLaunchKernelEx(&cfg, tc_gemm_kernel<2>, mw, mx, p, epi);
  return e == cudaSuccess ? PEAGLE_OK : PEAGLE_ERR_CUDA;
}

}  // namespace peagle
