// Fused GEMM epilogues of the draft pass.
//
// Every projection of the pass is Y[r, m] = sum_k X[r, k] W[m, k] (nn.Linear) over a
// handful of rows r (batch x K) and a long output dimension m.  The epilogue turns a
// finished 128-feature tile of Y (fp32) into the pass's next tensor, so that Y itself
// never reaches HBM:
//   STORE      fixed-point accumulation (fc projection; fc(h_shared) at create time)
//   QKV_ROPE   RoPE (rotate-half pairs i, i+hd/2) on q and k, then q -> Q [R, nq, hd],
//              k, v -> the drafter KV cache slot of each row (decode) or to per-row
//              K/V arrays (training-style forward)
//   RESID      residual stream += Y (o-proj, down-proj), fixed point
//   SWIGLU     act = silu(gate) * up, with gate/up rows interleaved in 64-row blocks
//   LMHEAD     optional fp32 logits + per-row argmax folded into a 64-bit atomicMax key
//   QKV_FX     RoPE'd q and k, and v, added into fixed-point accumulators (additive form of
//              QKV_ROPE; a later step converts them and writes the KV cache)
// A tile never splits a head (hd in {64, 128}, tiles start at multiples of 128) nor a
// gate/up block, so each epilogue only needs its own tile.  STORE and RESID are additive:
// every split-K contributor adds its own partial with integer atomics (see fx_t), so they
// need no cross-CTA reduction.
#pragma once

#include "common.cuh"

namespace peagle {

enum EpiKind : int {
  EPI_STORE = 0,
  EPI_QKV_ROPE = 1,
  EPI_RESID = 2,
  EPI_SWIGLU = 3,
  EPI_LMHEAD = 4,
  EPI_QKV_FX = 5  // additive QKV: RoPE'd partials added into fixed-point q / k,v buffers
};

struct EpiArgs {
  int kind;
  int R;     // valid (logical) rows
  int Nout;  // valid output features
  int in_split;   // the GEMM's activation operand holds rows [0,R) = bf16 hi parts and
                  // [R,2R) = bf16 lo parts; the epilogue adds the two partial products
  int out_split;  // activation outputs (SWIGLU) are written as hi rows [0,R), lo [R,2R)
  // STORE: fixed-point destination [R, out_ld] (accumulated, zero beforehand)
  fx_t* out_fx;
  int out_ld;
  // RESID: fixed-point residual [R, ld_res]
  fx_t* resid;
  int ld_res;
  // QKV_ROPE
  void* q_out;            // [R, nq*hd]; fp32 when q_f32, else the activation dtype
  int q_f32;
  void* k_dst;            // decode: cache layer base [B][nkv][cap][hd]; rows: [R][nkv][hd]
  void* v_dst;
  void* k1_dst;           // rows mode: depth-1 copy [n][nkv][hd] (may be null)
  void* v1_dst;
  const int* row_pos;     // RoPE position of each row (decode: seq_lens[b] + j, written by
                          // the input-fusion kernel; rows mode: p)
  const int* row_depth;   // rows mode: depth of each row (1-based)
  int n_seq;              // rows mode: sequence length (depth-1 copy bound)
  int decode;             // 1: decode (cache slot = seq_lens[b] + j), 0: rows
  int K;                  // decode: draft depth (rows per request)
  int nq, nkv, hd, cap;
  const float2* rope;     // [max_positions][hd/2] (cos, sin)
  int max_pos;
  // SWIGLU
  void* act_out;          // [R, I] (or [2R, I] when out_split)
  int I;
  // LMHEAD
  float* logits;          // [R, Nout] or null
  unsigned long long* keys;  // [R]
  unsigned* err;
  // QKV_FX: fixed-point accumulators q [R, nq*hd] and k,v [R][2][nkv*hd] (zero beforehand)
  fx_t* q_fx;
  fx_t* kv_fx;
  // deferred RMSNorm: when row_ss is set, the operand rows hold x * gamma and row r's
  // result is scaled by rsqrt(row_ss[r] * ss_inv_n + ss_eps) (row_ss: sum of x^2, fixed
  // point).  Applies to QKV_FX, SWIGLU and LMHEAD.
  const fx_t* row_ss;
  float ss_inv_n, ss_eps;
};

__device__ __forceinline__ float epi_row_scale(const EpiArgs& a, int r) {
  return a.row_ss ? rsqrtf(from_fx(a.row_ss[r]) * a.ss_inv_n + a.ss_eps) : 1.f;
}

// Store an activation that feeds the next projection: a single value, or its bf16
// hi part at row r and the bf16 rounding of the remainder at row r + R.
template <typename T>
__device__ __forceinline__ void store_act(T* base, size_t row_stride, int r, int R, int split,
                                          int col, float v) {
  T hi = from_f32<T>(v);
  base[(size_t)r * row_stride + col] = hi;
  if (split) base[(size_t)(r + R) * row_stride + col] = from_f32<T>(v - to_f32(hi));
}

// Apply the epilogue to rows r0 .. r0+rcount-1 of a 128-feature tile starting at m0.
// The tile value of row r0+i, feature m0+ml is src[i*ld + ml], plus src[(i+lo_off)*ld + ml]
// when lo_off >= 0 (the lo-part product of a split activation operand).
// rscale / rpos (optional, e.g. in shared memory): row r0+i's norm scale and RoPE position
// for i < rcount, gathered by the caller so the loops below issue no dependent loads.
template <typename T>
__device__ __forceinline__ void epilogue_tile(const EpiArgs& a, const float* src, int ld,
                                              int lo_off, int m0, int r0, int rcount, int tid,
                                              int nthr, const float* rscale = nullptr,
                                              const int* rpos = nullptr) {
  const int mcount = min(128, a.Nout - m0);
  auto val = [&](int i, int ml) -> float {
    float v = src[(size_t)i * ld + ml];
    if (lo_off >= 0) v += src[(size_t)(i + lo_off) * ld + ml];
    return v;
  };
  auto rsc = [&](int i) -> float { return rscale ? rscale[i] : epi_row_scale(a, r0 + i); };
  switch (a.kind) {
    case EPI_STORE:
    case EPI_RESID: {
      fx_t* dst = a.kind == EPI_STORE ? a.out_fx : a.resid;
      const int ldd = a.kind == EPI_STORE ? a.out_ld : a.ld_res;
      for (int idx = tid; idx < rcount * 128; idx += nthr) {
        int i = idx >> 7, ml = idx & 127;
        if (ml < mcount) red_add_fx(dst + (size_t)(r0 + i) * ldd + m0 + ml, to_fx(val(i, ml)));
      }
    } break;
    case EPI_SWIGLU: {
      // tile rows [0,64) = gate, [64,128) = up of intermediate features m0/2 + f
      T* act = (T*)a.act_out;
      for (int idx = tid; idx < rcount * 64; idx += nthr) {
        int i = idx >> 6, f = idx & 63;
        const float sc = rsc(i);
        float g = val(i, f) * sc;
        float u = val(i, 64 + f) * sc;
        float s = g / (1.f + expf(-g));
        store_act<T>(act, a.I, r0 + i, a.R, a.out_split, (m0 >> 1) + f, s * u);
      }
    } break;
    case EPI_QKV_ROPE: {
      const int hd = a.hd, half = hd >> 1;
      const int qend = a.nq * hd, kend = (a.nq + a.nkv) * hd;
      // the output of row r, section sec (0 q, 1 k, 2 v), feature m (kv head g, index i
      // within the head): out0 at i, and for q / k the rotated partner out1 at i + half
      auto put = [&](int r, int sec, int m, int g, int i, int pos, int dep, float out0,
                     float out1) {
        if (sec == 0) {
          if (a.q_f32) {
            float* q = (float*)a.q_out + (size_t)r * a.nq * hd + m;
            q[0] = out0;
            q[half] = out1;
          } else {
            T* q = (T*)a.q_out + (size_t)r * a.nq * hd + m;
            q[0] = from_f32<T>(out0);
            q[half] = from_f32<T>(out1);
          }
          return;
        }
        T* dst = (T*)(sec == 1 ? a.k_dst : a.v_dst);
        size_t off;
        if (a.decode)
          off = (((size_t)(r / a.K) * a.nkv + g) * a.cap + pos) * hd + i;
        else
          off = ((size_t)r * a.nkv + g) * hd + i;
        dst[off] = from_f32<T>(out0);
        if (sec == 1) dst[off + half] = from_f32<T>(out1);
        if (!a.decode && dep == 1 && pos >= 0 && pos < a.n_seq) {
          T* d1 = (T*)(sec == 1 ? a.k1_dst : a.v1_dst);
          if (d1) {
            const size_t o1 = ((size_t)pos * a.nkv + g) * hd + i;
            d1[o1] = from_f32<T>(out0);
            if (sec == 1) d1[o1 + half] = from_f32<T>(out1);
          }
        }
      };
      if (nthr == 128 && mcount == 128 && 128 % hd == 0 &&
          (m0 + 128 <= qend || (m0 >= qend && m0 + 128 <= kend))) {
        // A tile of rotated features only (q or k): thread = (rotation pair, row parity),
        // so that every thread works; rows' positions, depths and RoPE factors of a batch
        // are fetched before any of them is used.
        const int sec = m0 < qend ? 0 : 1;
        const int pr = tid & 63, rg = tid >> 6;
        const int i = pr % half;
        const int ml = (pr / half) * hd + i;
        const int m = m0 + ml;
        const int g = sec == 0 ? 0 : (m - qend) / hd;
        constexpr int U = 8;
        for (int t0 = rg; t0 < rcount; t0 += 2 * U) {
          int pos_u[U], dep_u[U];
          float2 cs_u[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int ti = t0 + 2 * u;
            pos_u[u] = ti < rcount ? (rpos ? rpos[ti] : __ldg(a.row_pos + r0 + ti)) : -1;
            dep_u[u] = (ti < rcount && !a.decode && a.row_depth) ? __ldg(a.row_depth + r0 + ti) : 0;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const bool need = pos_u[u] >= 0 && pos_u[u] < a.max_pos;
            cs_u[u] = need ? __ldg(a.rope + (size_t)pos_u[u] * half + i) : make_float2(1.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int ti = t0 + 2 * u;
            if (ti >= rcount) break;
            const int pos = pos_u[u];
            if (a.decode && (pos < 0 || pos >= a.cap)) {
              if (sec == 0 && i == 0 && m == 0) raise_error(a.err, PEAGLE_DEV_KV_OVERFLOW);
              if (sec != 0) continue;  // no cache slot for this row
            }
            const float v0 = val(ti, ml), v1 = val(ti, ml + half);
            put(r0 + ti, sec, m, g, i, pos, dep_u[u], v0 * cs_u[u].x - v1 * cs_u[u].y,
                v1 * cs_u[u].x + v0 * cs_u[u].y);
          }
        }
        break;
      }
      // One output feature per thread (consecutive threads write consecutive features);
      // the rows' positions, depths and RoPE factors of a batch of 16 rows are fetched
      // before any of them is used.
      constexpr int U = 16;
      for (int ml = tid; ml < mcount; ml += nthr) {
        const int m = m0 + ml;
        const int i = m % hd;
        const int sec = (m < qend) ? 0 : (m < kend ? 1 : 2);
        if (sec != 2 && i >= half) continue;  // handled together with its pair partner
        const int g = sec == 0 ? 0 : (m - (sec == 1 ? qend : kend)) / hd;
        for (int t0 = 0; t0 < rcount; t0 += U) {
          int pos_u[U], dep_u[U];
          float2 cs_u[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int ti = t0 + u;
            pos_u[u] = ti < rcount ? (rpos ? rpos[ti] : __ldg(a.row_pos + r0 + ti)) : -1;
            dep_u[u] = (ti < rcount && !a.decode && a.row_depth) ? __ldg(a.row_depth + r0 + ti) : 0;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const bool need = sec != 2 && pos_u[u] >= 0 && pos_u[u] < a.max_pos;
            cs_u[u] = need ? __ldg(a.rope + (size_t)pos_u[u] * half + i) : make_float2(1.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int ti = t0 + u;
            if (ti >= rcount) break;
            const int r = r0 + ti;
            const int pos = pos_u[u];
            if (a.decode && (pos < 0 || pos >= a.cap)) {
              if (sec == 0 && i == 0 && m == 0) raise_error(a.err, PEAGLE_DEV_KV_OVERFLOW);
              if (sec != 0) continue;  // no cache slot for this row
            }
            const float v0 = val(ti, ml);
            float out0, out1 = 0.f;
            if (sec == 2) {
              out0 = v0;
            } else {
              const float v1 = val(ti, ml + half);
              out0 = v0 * cs_u[u].x - v1 * cs_u[u].y;
              out1 = v1 * cs_u[u].x + v0 * cs_u[u].y;
            }
            put(r, sec, m, g, i, pos, dep_u[u], out0, out1);
          }
        }
      }
    } break;
    case EPI_QKV_FX: {
      // RoPE is a rotation and the row scale a constant, so each split-K partial can be
      // rotated, scaled and added on its own: the fixed-point sums are exact and the same
      // for any order of arrival.  One output feature per thread, its rotation partner
      // (i +- hd/2, same head, same tile) read from the tile: every thread adds one value
      // per row.  The positions of sixteen rows are fetched together, then their RoPE
      // factors together, so a batch of rows waits for two dependent loads.
      const int hd = a.hd, half = hd >> 1;
      const int qend = a.nq * hd, kend = (a.nq + a.nkv) * hd, kvw = a.nkv * hd;
      constexpr int U = 16;
      for (int ml = tid; ml < mcount; ml += nthr) {
        const int m = m0 + ml;
        const int i = m % hd;
        const int sec = (m < qend) ? 0 : (m < kend ? 1 : 2);
        const bool first = i < half;  // i < hd/2: out = x_i c - x_{i+h} s, else x_i c + x_{i-h} s
        const int ip = first ? i : i - half;
        const int mlp = first ? ml + half : ml - half;
        fx_t* dst = sec == 0 ? a.q_fx + m
                    : sec == 1 ? a.kv_fx + (m - qend)
                               : a.kv_fx + kvw + (m - kend);
        const size_t ld = sec == 0 ? (size_t)qend : (size_t)2 * kvw;
        for (int t0 = 0; t0 < rcount; t0 += U) {
          int pos[U];
          float2 cs[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int ti = t0 + u;
            pos[u] = -1;
            if (sec != 2 && ti < rcount) pos[u] = rpos ? rpos[ti] : __ldg(a.row_pos + r0 + ti);
          }
#pragma unroll
          for (int u = 0; u < U; ++u)
            cs[u] = (pos[u] >= 0 && pos[u] < a.max_pos) ? __ldg(a.rope + (size_t)pos[u] * half + ip)
                                                        : make_float2(1.f, 0.f);
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int ti = t0 + u;
            if (ti >= rcount) break;
            const int r = r0 + ti;
            const float sc = rsc(ti);
            const float x = val(ti, ml) * sc;
            float out = x;
            if (sec != 2) {
              const float xp = val(ti, mlp) * sc;
              out = first ? x * cs[u].x - xp * cs[u].y : x * cs[u].x + xp * cs[u].y;
            }
            red_add_fx(dst + (size_t)r * ld, to_fx(out));
          }
        }
      }
    } break;
    case EPI_LMHEAD: {
      if (a.logits) {
        for (int idx = tid; idx < rcount * 128; idx += nthr) {
          int i = idx >> 7, ml = idx & 127;
          if (ml < mcount)
            a.logits[(size_t)(r0 + i) * a.Nout + m0 + ml] = val(i, ml) * rsc(i);
        }
      }
      // per row: best (value, index) over the tile -> one atomicMax per warp and row
      const int lane = tid & 31;
      const int nw = nthr >> 5;
      for (int i = tid >> 5; i < rcount; i += nw) {
        unsigned long long best = 0ull;
        const float sc = rsc(i);
        for (int ml = lane; ml < mcount; ml += 32) {
          unsigned long long k = argmax_key(val(i, ml) * sc, m0 + ml);
          best = k > best ? k : best;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
          best = other > best ? other : best;
        }
        if (lane == 0) atomicMax(a.keys + r0 + i, best);
      }
    } break;
  }
}

}  // namespace peagle
