// Split-KV decode attention work items shared by the standalone attention kernels and
// the persistent pass kernel: mma.sync helpers, one (request, kv head, key chunk) item
// and the merge of one query row's chunk partials.
#pragma once

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace peagle {

// =====================================================================================
// Split-KV decode attention on the tensor cores (bf16 caches): mma.sync m16n8k16.
// One warp per 16 query rows (rows = K*G of one kv head, <= 128), CTA = one chunk of
// keys of one (request, kv head).  K/V tiles of 64 keys are double-buffered in shared
// memory by cp.async with a 16-byte XOR swizzle and read with ldmatrix.  Queries and
// softmax probabilities are rounded to bf16 (the probabilities once: the PV product and the
// row sum use the same values); keys and values are the cache's bf16; products accumulate
// in fp32.  Online softmax in the log2 domain; partials and the merge are those of the
// CUDA-core kernel.
// =====================================================================================
// round to the nearest bf16 value, kept in fp32
__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
// 2^x on the SFU (relative error about 2^-22, far below the bf16 rounding that follows)
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// hi/lo bf16 split of a pair of fp32 values
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int MMA_KT = 64;  // keys per tile

// Keys of request b's split-KV items: positions [*first, *total).  total = L + K (capped
// at the cache capacity; overflow is reported by the QKV epilogue).  With a sliding window
// of W positions ("EAGLE-4", "EAGLE-4 overview"), row j sees L + j - W + 1 .. L + j, so
// the items start at row 0's first visible key; item c covers [first + c * chunk, ...).
__device__ __forceinline__ void attn_span(const AttnArgs& a, int L, int* first, int* total) {
  int t = L + a.K;
  if (t > a.cap) t = a.cap;
  int f = 0;
  if (a.window > 0) {
    f = L - a.window + 1;
    if (f < 0) f = 0;
  }
  *first = f;
  *total = t;
}
__device__ __forceinline__ int attn_nvalid(const AttnArgs& a, int first, int total) {
  return total > first ? (total - first + a.chunk - 1) / a.chunk : 0;
}

// One work item: chunk c of (request b, kv head g), run by the nthr threads tid = 0 ..
// nthr-1 of a thread group (>= 32 * ceil(rows / 16)) that synchronises with bar().
__device__ __forceinline__ void cp_async_wait_n(int n) {
  if (n <= 0) cp_async_wait<0>();
  else if (n == 1) cp_async_wait<1>();
  else if (n == 2) cp_async_wait<2>();
  else cp_async_wait<3>();
}

// NBUF K/V tile buffers (<= 4): the loads of up to NBUF tiles are in flight at once.
// QFX: a.q holds the queries as 64-bit fixed point (the persistent pass kernel's sums)
// instead of fp32.
template <int HD, int NBUF, typename Bar, bool QFX = false>
__device__ __forceinline__ void attn_mma_item(const AttnArgs& a, int b, int g, int c, int tid,
                                              int nthr, uint8_t* sm_raw, Bar bar) {
  static_assert(NBUF >= 2 && NBUF <= 4, "1 < NBUF <= 4");
  constexpr int ROWB = HD * 2;           // bytes per key row
  constexpr int CH = ROWB / 16;          // 16-byte chunks per row
  constexpr int TILEB = MMA_KT * ROWB;   // bytes per K (or V) tile
  constexpr int ND = HD / 8;             // output n-tiles
  constexpr int KS = HD / 16;            // k-steps of QK^T
  const int G = a.nq / a.nkv;
  const int rows = a.K * G;
  const int L = a.seq_lens[b];
  int first, total;
  attn_span(a, L, &first, &total);
  const int kbeg = first + c * a.chunk;
  if (kbeg >= total || L < 0) return;
  const int kend = min(total, kbeg + a.chunk);
  const int warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const size_t head_off = ((size_t)b * a.nkv + g) * a.cap * HD;
  const bf16* kc = (const bf16*)a.kc + head_off;
  const bf16* vc = (const bf16*)a.vc + head_off;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm_raw);
  // smem: NBUF x [K tile, V tile]
  auto tile_k = [&](int buf) { return sbase + (uint32_t)(buf * 2 * TILEB); };
  auto tile_v = [&](int buf) { return sbase + (uint32_t)(buf * 2 * TILEB + TILEB); };
  auto load_tile = [&](int buf, int t0) {
    for (int idx = tid; idx < MMA_KT * CH; idx += nthr) {
      const int r = idx / CH, ch = idx - r * CH;
      const int key = t0 + r;
      const bool ok = key < kend;
      const size_t off = (size_t)(ok ? key : kbeg) * HD + ch * 8;
      const uint32_t so = (uint32_t)(r * ROWB + ((ch ^ (r & 7)) * 16));
      cp_async16(tile_k(buf) + so, kc + off, ok ? 16 : 0);
      cp_async16(tile_v(buf) + so, vc + off, ok ? 16 : 0);
    }
    cp_async_commit();
  };
  load_tile(0, kbeg);  // the first K/V tile is in flight while the queries load
  // query fragments of this warp's 16 rows (bf16; the scale is applied in the exponent)
  const float qscale = a.scale * 1.4426950408889634f;
  const int r0 = warp * 16 + gq, r1 = r0 + 8;
  const bool v0 = r0 < rows, v1 = r1 < rows;
  const int j0 = v0 ? r0 / G : 0, j1 = v1 ? r1 / G : 0;
  const size_t qo0 = ((size_t)(b * a.K + j0) * a.nq + g * G + (r0 - j0 * G)) * HD;
  const size_t qo1 = ((size_t)(b * a.K + j1) * a.nq + g * G + (r1 - j1 * G)) * HD;
  auto qv = [&](size_t off) -> float {
    if constexpr (QFX) return from_fx(__ldcg((const fx_t*)a.q + off));
    else return ((const float*)a.q)[off];
  };
  uint32_t qa[KS][4];  // bf16 queries (the scale is applied to the scores)
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int d0 = ks * 16 + 2 * tq, d1 = d0 + 8;
    float x[8];
    x[0] = v0 ? qv(qo0 + d0) : 0.f;
    x[1] = v0 ? qv(qo0 + d0 + 1) : 0.f;
    x[2] = v1 ? qv(qo1 + d0) : 0.f;
    x[3] = v1 ? qv(qo1 + d0 + 1) : 0.f;
    x[4] = v0 ? qv(qo0 + d1) : 0.f;
    x[5] = v0 ? qv(qo0 + d1 + 1) : 0.f;
    x[6] = v1 ? qv(qo1 + d1) : 0.f;
    x[7] = v1 ? qv(qo1 + d1 + 1) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) qa[ks][u] = pack_bf16(x[2 * u], x[2 * u + 1]);
  }
  const int lim0 = L + j0, lim1 = L + j1;  // last visible key of each row
  // first visible key of each row (sliding window), else the start of the context
  const int lo0 = a.window > 0 ? lim0 - a.window + 1 : 0;
  const int lo1 = a.window > 0 ? lim1 - a.window + 1 : 0;
  float o[ND][4];
#pragma unroll
  for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const bool active = warp * 16 < rows;
  const int ntile = (kend - kbeg + MMA_KT - 1) / MMA_KT;
  int loaded = 1;  // tile 0 was issued before the queries
  for (; loaded < ntile && loaded < NBUF; ++loaded) load_tile(loaded, kbeg + loaded * MMA_KT);
  for (int it = 0; it < ntile; ++it) {
    const int buf = it % NBUF;
    const int t0 = kbeg + it * MMA_KT;
    cp_async_wait_n(loaded - 1 - it);  // groups committed after tile it may stay in flight
    bar();
    if (active) {
      // ---- S = Q K^T for 64 keys: 8 n-tiles of 8 keys
      float sc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {  // pairs of key n-tiles
          // matrices: (keys 16np..+7, dims 16ks..+7), (same keys, dims +8),
          //           (keys 16np+8..+15, dims 16ks..), (keys +8, dims +8)
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
      // ---- scale (1/sqrt(hd) and log2 e), mask and online softmax (log2 domain)
      // the mask: only tiles that reach a row's last visible key, the window's first or the
      // chunk's end need it (the raw scores are masked; the scale is applied in the exponent)
      const bool full = v0 && v1 && t0 + MMA_KT <= kend && t0 + MMA_KT - 1 <= min(lim0, lim1) &&
                        t0 >= max(lo0, lo1);
      if (!full) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int kp = t0 + n * 8 + 2 * tq;
          sc[n][0] = (kp < kend && kp <= lim0 && kp >= lo0 && v0) ? sc[n][0] : -INFINITY;
          sc[n][1] = (kp + 1 < kend && kp + 1 <= lim0 && kp + 1 >= lo0 && v0) ? sc[n][1] : -INFINITY;
          sc[n][2] = (kp < kend && kp <= lim1 && kp >= lo1 && v1) ? sc[n][2] : -INFINITY;
          sc[n][3] = (kp + 1 < kend && kp + 1 <= lim1 && kp + 1 >= lo1 && v1) ? sc[n][3] : -INFINITY;
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // running max in the log2 domain of the scaled scores (the scale is positive)
      const float mn0 = fmaxf(m0, mx0 * qscale), mn1 = fmaxf(m1, mx1 * qscale);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float cr0 = (m0 == -INFINITY) ? 0.f : fast_ex2(m0 - base0);
      const float cr1 = (m1 == -INFINITY) ? 0.f : fast_ex2(m1 - base1);
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        // probabilities rounded to bf16 once: the PV product and the row sum use the same
        sc[n][0] = bf16r(fast_ex2(fmaf(sc[n][0], qscale, -base0)));
        sc[n][1] = bf16r(fast_ex2(fmaf(sc[n][1], qscale, -base0)));
        sc[n][2] = bf16r(fast_ex2(fmaf(sc[n][2], qscale, -base1)));
        sc[n][3] = bf16r(fast_ex2(fmaf(sc[n][3], qscale, -base1)));
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
      // ---- O += P V: 4 k-steps of 16 keys
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4];
        ph[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        ph[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        ph[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        ph[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < ND / 2; ++dp) {  // pairs of output n-tiles (16 dims)
          // matrices (trans): (keys 16kk..+7, dims 16dp..+7), (keys +8, same dims),
          //                   (keys 16kk.., dims +8), (keys +8, dims +8)
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
    bar();
    if (loaded < ntile) {  // the buffer just consumed takes the next tile
      load_tile(loaded % NBUF, kbeg + loaded * MMA_KT);
      ++loaded;
    }
  }
  // ---- partials: m and l in natural-log units, o unnormalised
  const int rows_alloc = rows;
  float* part = a.part + (((size_t)b * a.nkv + g) * a.nchunk + c) * rows_alloc * (HD + 2);
  if (active) {
    const float ln2 = 0.6931471805599453f;
#pragma unroll
    for (int n = 0; n < ND; ++n) {
      const int d = n * 8 + 2 * tq;
      if (v0) {
        part[(size_t)r0 * (HD + 2) + d] = o[n][0];
        part[(size_t)r0 * (HD + 2) + d + 1] = o[n][1];
      }
      if (v1) {
        part[(size_t)r1 * (HD + 2) + d] = o[n][2];
        part[(size_t)r1 * (HD + 2) + d + 1] = o[n][3];
      }
    }
    if (tq == 0) {
      if (v0) {
        part[(size_t)r0 * (HD + 2) + HD] = (m0 == -INFINITY) ? -INFINITY : m0 * ln2;
        part[(size_t)r0 * (HD + 2) + HD + 1] = l0;
      }
      if (v1) {
        part[(size_t)r1 * (HD + 2) + HD] = (m1 == -INFINITY) ? -INFINITY : m1 * ln2;
        part[(size_t)r1 * (HD + 2) + HD + 1] = l1;
      }
    }
  }
}


// Merge of the split-KV partials (o unnormalised, m, l per query row and chunk) by the
// last CTA of (request b, kv head g), in chunk order; rows are spread over the warps.
template <typename T, int HD>
__device__ __forceinline__ void attn_merge_rows(const AttnArgs& a, int b, int g, int rows,
                                                int nvalid, int rbeg, int rend, int lane,
                                                int rstep = 1) {
  constexpr int E = HD / 32;
  const int G = a.nq / a.nkv;
  const float* pbase = a.part + ((size_t)b * a.nkv + g) * a.nchunk * rows * (HD + 2);
  T* og = (T*)a.o;
  // the values of the first CB chunks are loaded together with the statistics (one round
  // trip to L2 for up to CB chunks)
  constexpr int CB = 64 / E;
  for (int rr = rbeg; rr < rend; rr += rstep) {
    float pv[CB][E];
#pragma unroll
    for (int cc = 0; cc < CB; ++cc) {
      const float* pr = pbase + ((size_t)cc * rows + rr) * (HD + 2);
#pragma unroll
      for (int e = 0; e < E; ++e) pv[cc][e] = cc < nvalid ? __ldcg(pr + lane + 32 * e) : 0.f;
    }
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
#pragma unroll
    for (int cc = 0; cc < CB; ++cc) {
      const float w = __shfl_sync(0xffffffffu, cc < 32 ? wc[0] : wc[1], cc & 31);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(pv[cc][e], w, acc[e]);
    }
#pragma unroll 8
    for (int cc = CB; cc < nvalid; ++cc) {
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
}

}  // namespace peagle
