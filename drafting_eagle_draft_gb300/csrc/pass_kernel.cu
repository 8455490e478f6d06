// Persistent kernel of the bf16 P-EAGLE draft pass on sm_103a.
//
// The draft pass is a chain of ~40 dependent steps (fc, input rows, per layer QKV /
// attention / merge / o-proj / norm / gate-up / down / norm, LM head, argmax) whose cost
// is streaming ~1 GB of weights.  As separate kernels every boundary drains the GPU: the
// tail of one projection, the launch and the ramp of the next leave HBM idle for several
// microseconds, ~40 times per pass.  Here one CTA per SM runs the whole chain:
//
//   warp 0 (TMA producer)  walks the weight tiles of every projection of the pass in
//       order and keeps the shared-memory ring full.  Weights do not depend on anything,
//       so while the CTAs finish one step (or run attention) the ring already fills with
//       the next projection's weights; the activation half of a ring stage is loaded once
//       the step it depends on has completed on every CTA.
//   warp 1 (MMA issuer)    tcgen05.mma on each full stage into one of two TMEM
//       accumulators, across projection boundaries.
//   warps 2-5 (workers)    drain the accumulators through the fused epilogues (stream-K
//       fix-up by the last contributor, as in the standalone GEMM) and run the steps that
//       are not projections: input rows, split-KV attention, merge, RMSNorm, argmax.
//
// Steps ("phases") complete when every CTA has signalled them (a release add on a
// per-phase counter after its own work, acquired by the consumers).  Each CTA signals
// phases in order, so a count of G on phase j implies every earlier phase is complete.
// All CTAs are co-resident (cooperative launch), every wait is bounded (2 s, then the
// device error word gets TIMEOUT and a global abort flag stops the other CTAs).
#include <cuda.h>
#include <stdio.h>

#include "attn_decode.cuh"
#include "pass_kernel.h"
#include "tc_ptx.cuh"

namespace peagle {

namespace {

constexpr int PK_THREADS = 224;
constexpr int PK_BWARP = 6;  // activation producer (warps 2-5 are the workers)
constexpr int PK_A_BYTES = 128 * 128 * PASS_KU;  // PASS_KU 128 x 64 bf16 weight tiles

__device__ __forceinline__ void wk_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Polling uses relaxed loads and one acquire fence once the value is seen: an acquiring
// load per spin would also invalidate the SM's L1 every time, and the other warps' local
// (spilled) variables with it.
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acquire_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ long long rbeg(long long c, long long total, int G) {
  return c * total / G;
}
__device__ __forceinline__ int owner(long long it, long long total, int G) {
  long long c = it * G / total;
  while (c + 1 < G && rbeg(c + 1, total, G) <= it) ++c;
  while (c > 0 && rbeg(c, total, G) > it) --c;
  return (int)c;
}

// Cursor over this CTA's (projection, iteration) sequence.  Everything the producers need
// per iteration is held in registers: reading the parameter block with a run-time index
// costs a memory round trip, far too slow for a loop that must issue a stage every few
// hundred nanoseconds.
struct Cur {
  int g;        // projection (n_gemm once exhausted)
  int left;     // iterations left in this projection's range
  int tile, kb; // 128-feature weight tile and 64-wide k-block of the current iteration
  int KB, BN, dep;
  const CUtensorMap* tw;
  const CUtensorMap* tx;
};
__device__ __forceinline__ void cur_seek(const PassParams& P, int c, Cur& k) {
  while (k.g < P.n_gemm) {
    const PassGemm& m = P.gemm[k.g];
    if (c < m.Gm) {
      const long long b = rbeg(c, m.total, m.Gm), e = rbeg(c + 1, m.total, m.Gm);
      if (b < e) {
        k.left = (int)(e - b);
        k.KB = m.KB;
        k.tile = (int)(b / m.KB);
        k.kb = (int)(b - (long long)k.tile * m.KB);
        k.BN = m.BN;
        k.dep = m.dep;
        k.tw = &P.tm[2 * k.g];
        k.tx = &P.tm[2 * k.g + 1];
        // bring the projection's tensor maps into the TMA descriptor cache (and the next
        // projection's weight map, which the weight producer reaches soon after)
        tc::tma_prefetch_desc(k.tw);
        tc::tma_prefetch_desc(k.tx);
        if (k.g + 1 < P.n_gemm) tc::tma_prefetch_desc(&P.tm[2 * k.g + 2]);
        return;
      }
    }
    ++k.g;
  }
}
__device__ __forceinline__ void cur_next(const PassParams& P, int c, Cur& k) {
  if (--k.left == 0) {
    ++k.g;
    cur_seek(P, c, k);
  } else if (++k.kb == k.KB) {
    k.kb = 0;
    ++k.tile;
  }
}

__device__ __forceinline__ bool aborted(const PassParams& P, volatile int* s_abort) {
  return *s_abort || *(volatile unsigned*)(P.phase_cnt + P.n_phase) != 0u;
}
__device__ __forceinline__ void set_abort(const PassParams& P, volatile int* s_abort) {
  raise_error(P.err, PEAGLE_DEV_TIMEOUT);
  *s_abort = 1;
  atomicExch(P.phase_cnt + P.n_phase, 1u);
}

// Worker thread 0 waits for phase `ph` to be complete on every CTA; the result is
// broadcast to the 128 workers.  Returns false on abort or timeout.
__device__ bool wk_wait_phase(const PassParams& P, int ph, int et, volatile int* s_abort,
                              volatile int* s_flag) {
  if (et == 0) {
    int ok = 1;
    const unsigned need = gridDim.x + (ph == P.stall_phase ? 1u : 0u);
    if (ph >= 0 && ld_relaxed(P.phase_cnt + ph) < need) {
      const uint64_t t0 = tc::globaltimer();
      unsigned spins = 0;
      while (ld_relaxed(P.phase_cnt + ph) < need) {
        if ((++spins & 63u) != 0) continue;
        if (aborted(P, s_abort)) {
          ok = 0;
          break;
        }
        if (tc::globaltimer() - t0 > P.wait_ns) {
          set_abort(P, s_abort);
          ok = 0;
          break;
        }
      }
    }
    fence_acquire_gpu();
    fence_proxy_async_global();
    *s_flag = ok;
  }
  wk_bar();
  const bool ok = *s_flag != 0;
  wk_bar();
  return ok;
}

// Worker thread 0 waits until *ctr >= need (bounded); the result is broadcast to the 128
// workers.  False on abort or timeout.
__device__ bool wk_wait_count(const PassParams& P, const unsigned* ctr, unsigned need, int et,
                              volatile int* s_abort, volatile int* s_flag) {
  if (et == 0) {
    int ok = 1;
    if (ld_relaxed(ctr) < need) {
      const uint64_t t0 = tc::globaltimer();
      unsigned spins = 0;
      while (ld_relaxed(ctr) < need) {
        if ((++spins & 63u) != 0) continue;
        if (aborted(P, s_abort)) {
          ok = 0;
          break;
        }
        if (tc::globaltimer() - t0 > P.wait_ns) {
          set_abort(P, s_abort);
          ok = 0;
          break;
        }
      }
    }
    fence_acquire_gpu();
    *s_flag = ok;
  }
  wk_bar();
  const bool ok = *s_flag != 0;
  wk_bar();
  return ok;
}

// Timing: event k of (phase, this CTA) -- projections: 0 activations ready (seen by the
// activation producer), 1 first MMA issued, 2 last accumulator committed; other steps: 0
// the previous step seen complete; attention: 1 the item's partials written, 2 every
// item of its (request, kv head) in; 3: done.
__device__ __forceinline__ void trace_ev(const PassParams& P, int ph, int k) {
  if (P.trace_cta)
    P.trace_cta[((size_t)ph * gridDim.x + blockIdx.x) * 4 + k] = tc::globaltimer();
}

// Every worker has finished its part of phase `ph`: publish it.  The CTA barrier orders
// the workers' writes before thread 0's release add, whose release semantics (cumulative
// at GPU scope) make them visible to every CTA that acquires the count.
__device__ __forceinline__ void wk_signal(const PassParams& P, int ph, int et) {
  wk_bar();
  if (et == 0) {
    fence_proxy_async_global();
    red_release_add(P.phase_cnt + ph, 1u);
    // timing: the phase completes when its last CTA signals
    if (P.trace) {
      const unsigned long long t = tc::globaltimer();
      atomicMax(P.trace + ph + 1, t);
      if (P.trace_cta) P.trace_cta[((size_t)ph * gridDim.x + blockIdx.x) * 4 + 3] = t;
    }
  }
}


// ---- steps spread over all CTAs -------------------------------------------------------
// CTA c owns the feature columns [c * cpc, (c+1) * cpc) of every row; per-row sums of
// squares are reduced in shared memory (fixed point) and added once per CTA and row.

__device__ __forceinline__ void col_range(const PassParams& P, int c, int G, int& c0, int& c1) {
  const int cpc = (P.H + G - 1) / G;
  c0 = min(P.H, c * cpc);
  c1 = min(P.H, c0 + cpc);
}

__device__ __forceinline__ void ss_flush(const PassParams& P, fx_t* dst, unsigned long long* s_rs,
                                         int et) {
  wk_bar();
  for (int r = et; r < P.R; r += 128) {
    const fx_t v = (fx_t)s_rs[r];
    if (v) red_add_fx(dst + r, v);
    s_rs[r] = 0ull;
  }
}

// NTP / MTP input rows: X0[:, :H] = e * g_in, X0[:, H:] = f * g_hid (hi / lo), residual = f,
// sums of squares of e and f (slots 0 and 1).  Row r = b*K + j: j = 0 takes
// embed[new_token[b]] and the fc row of request b, j >= 1 emb(mask) and fc(h_shared).
// The element loop issues the loads of four (row, column) pairs before using them.
__device__ void step_input(const PassParams& P, int c, int G, int et, unsigned long long* s_rs,
                           int* s_tok) {
  const int H = P.H, K = P.K, R = P.R;
  int c0, c1;
  col_range(P, c, G, c0, c1);
  const int nc = c1 - c0;
  const int n_tok = P.all_ntp ? R : P.B;  // catch-up: a token per row
  for (int b = et; b < n_tok; b += 128) {
    int tok = P.new_token[b];
    if (tok < 0 || tok >= P.Vt) {
      if (c == 0) raise_error(P.err, PEAGLE_DEV_BAD_TOKEN);
      tok = 0;
    }
    s_tok[b] = tok;
  }
  wk_bar();
  const bf16* gi = (const bf16*)P.input_norm;
  const bf16* gh = (const bf16*)P.hidden_norm;
  bf16* X0 = (bf16*)P.X0;
  constexpr int U = 4;
  for (int base = et; base < R * nc; base += 128 * U) {
    float ev[U], g1[U], g2[U];
    fx_t fq[U];
    int rr[U], cc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * 128;
      const bool ok = idx < R * nc;
      const int r = ok ? idx / nc : 0, col = ok ? c0 + idx - (idx / nc) * nc : c0;
      const int b = r / K, j = r - b * K;
      const bool ntp = P.all_ntp || j == 0;
      const int src = P.all_ntp ? r : b;  // token / fc row of an NTP row
      rr[u] = ok ? r : -1;
      cc[u] = col;
      const bf16* e = ntp ? (const bf16*)P.embed + (size_t)s_tok[src] * H : (const bf16*)P.emb_mask;
      ev[u] = ok ? ld(e + col) : 0.f;
      fq[u] = ok ? (ntp ? P.F[(size_t)src * H + col] : P.f_shared[col]) : 0;
      g1[u] = ok ? ld(gi + col) : 0.f;
      g2[u] = ok ? ld(gh + col) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = rr[u];
      if (r < 0) continue;
      const int col = cc[u];
      const float fv = from_fx(fq[u]);
      store_act<bf16>(X0, 2 * H, r, R, P.split, col, ev[u] * g1[u]);
      store_act<bf16>(X0, 2 * H, r, R, P.split, H + col, fv * g2[u]);
      P.res[(size_t)r * H + col] = fq[u];
      // the fc rows are read only here: clear them for the next pass
      if (P.all_ntp) P.F[(size_t)r * H + col] = 0;
      else if (r % K == 0) P.F[(size_t)(r / K) * H + col] = 0;
      atomicAdd(&s_rs[r], (unsigned long long)to_fx(ev[u] * ev[u]));
      atomicAdd(&s_rs[PASS_MAX_ROWS + r], (unsigned long long)to_fx(fv * fv));
    }
  }
  ss_flush(P, P.ss, s_rs, et);
  for (int r = et; r < R; r += 128) {
    const fx_t v = (fx_t)s_rs[PASS_MAX_ROWS + r];
    if (v) red_add_fx(P.ss + R + r, v);
    s_rs[PASS_MAX_ROWS + r] = 0ull;
  }
  if (c == 0) {
    for (int r = et; r < R; r += 128) {
      P.keys[r] = 0ull;
      P.row_pos[r] = P.seq_lens[r / K] + r % K;
    }
  }
}

// RMSNorm operand: Xn = x * gamma (hi / lo) and the rows' sums of squares into `slot`.
__device__ void step_norm(const PassParams& P, int c, int G, int slot, const bf16* gamma, int et,
                          unsigned long long* s_rs) {
  const int H = P.H, R = P.R;
  int c0, c1;
  col_range(P, c, G, c0, c1);
  const int nc = c1 - c0;
  bf16* out = (bf16*)P.Xn;
  constexpr int U = 4;
  for (int base = et; base < R * nc; base += 128 * U) {
    fx_t q[U];
    float g[U];
    int rr[U], cc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * 128;
      const bool ok = idx < R * nc;
      const int r = ok ? idx / nc : 0, col = ok ? c0 + idx - (idx / nc) * nc : c0;
      rr[u] = ok ? r : -1;
      cc[u] = col;
      q[u] = ok ? P.res[(size_t)r * H + col] : 0;
      g[u] = ok ? ld(gamma + col) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (rr[u] < 0) continue;
      const float v = from_fx(q[u]);
      store_act<bf16>(out, H, rr[u], R, P.split, cc[u], v * g[u]);
      atomicAdd(&s_rs[rr[u]], (unsigned long long)to_fx(v * v));
    }
  }
  ss_flush(P, P.ss + (size_t)slot * R, s_rs, et);
}

// The cache rows that this CTA's attention items of `layer` read and that exist before the
// pass (positions below seq_lens[b]) are fetched into L2 while the QKV projection runs, so
// that the items' tile loads do not wait on HBM.
template <int HD>
__device__ void prefetch_attn_rows(const PassParams& P, int layer, int c, int G) {
  const AttnArgs& a = P.att;
  const char* kc = (const char*)a.kc + (size_t)layer * P.layer_stride;
  const char* vc = (const char*)a.vc + (size_t)layer * P.layer_stride;
  const int n_items = a.nchunk * a.nkv * a.B;
  for (int i = c; i < n_items; i += G) {
    const int cc = i % a.nchunk;
    const int g = (i / a.nchunk) % a.nkv;
    const int b = i / (a.nchunk * a.nkv);
    const int L = a.seq_lens[b];
    if (L <= 0) continue;
    int first, total;
    attn_span(a, L, &first, &total);
    const int kbeg = first + cc * a.chunk;
    const int kend = min(min(total, kbeg + a.chunk), L);
    if (kend <= kbeg) continue;
    const size_t off = (((size_t)b * a.nkv + g) * a.cap + kbeg) * HD * sizeof(bf16);
    const uint32_t bytes = (uint32_t)(kend - kbeg) * HD * (uint32_t)sizeof(bf16);
    tc::bulk_prefetch_l2(kc + off, bytes);
    tc::bulk_prefetch_l2(vc + off, bytes);
  }
}

template <int HD>
__global__ void __launch_bounds__(PK_THREADS, 1)
    pass_kernel(const __grid_constant__ PassParams P) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) EpiArgs s_epi_buf;
  __shared__ unsigned long long s_rs[2 * PASS_MAX_ROWS];  // per-row sums (fixed point)
  __shared__ float s_rscale[32];  // epilogue chunk: row norm scales
  __shared__ int s_rpos[32];      // epilogue chunk: RoPE positions
  __shared__ int s_tok[PASS_MAX_ROWS];  // input step: validated new tokens
  EpiArgs* s_epi = &s_epi_buf;
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int S = P.stages;
  const int BS = P.b_stage_bytes;
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)S * PK_A_BYTES;
  uint8_t* uni = sB + (size_t)S * BS;  // epilogue staging / attention tiles
  float* stg = (float*)uni;
  uint64_t* full = (uint64_t*)(uni + P.uni_bytes);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;  // the MMA issuer's last MMAs after an abort
  uint32_t* s_tmem = (uint32_t*)(drain + 1);
  volatile int* s_flag = (volatile int*)(s_tmem + 1);
  volatile int* s_abort = s_flag + 1;
  volatile int* s_adone = s_flag + 2;
  volatile int* s_fin = s_flag + 3;  // a tile's last contributor (read between two barriers)
  volatile long long* s_nA = (volatile long long*)(s_tmem + 8);
  volatile long long* s_nB = s_nA + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int G = gridDim.x;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&accf[i], 1);
      tc::mbar_init(&acce[i], 128);
    }
    tc::mbar_init(drain, 1);
    *s_abort = 0;
    *s_adone = 0;
    for (int i = 0; i < 2 * PASS_MAX_ROWS; ++i) s_rs[i] = 0ull;
    *s_nA = 0;
    *s_nB = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(s_tmem, (uint32_t)P.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  const uint64_t wns = P.wait_ns;
  if (P.trace && c == 0 && threadIdx.x == 0) P.trace[0] = tc::globaltimer();

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    // Weight halves of the ring stages, in pass order, as fast as stages free up.
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_first();
      // loop-invariant parameters in registers (a parameter read inside the loop is a
      // memory access the asm statements' clobbers force the compiler to repeat)
      const int n_gemm = P.n_gemm;
      Cur ca{};
      ca.g = 0;
      cur_seek(P, c, ca);
      long long nA = 0;
      int st = 0;
      uint32_t par = 0;  // parity of the empty-barrier phase the next reuse waits for
      while (ca.g < n_gemm) {
        if (nA >= S && !tc::mbar_wait(&empty[st], par, s_abort, wns)) {
          if (!*s_abort) set_abort(P, s_abort);
          break;
        }
        tc::mbar_expect_tx(&full[st], (uint32_t)(PK_A_BYTES + ca.BN * 128 * PASS_KU));
        tc::tma_load_3d(sA + (size_t)st * PK_A_BYTES, ca.tw, 0, ca.tile * 128, ca.kb * PASS_KU,
                        &full[st], pol_w);
        cur_next(P, c, ca);
        ++nA;
        if (++st == S) {
          st = 0;
          if (nA > S) par ^= 1u;
        }
        __threadfence_block();
        *s_nA = nA;  // the stage's transaction count is armed: its activations may follow
      }
      *s_adone = 1;
      if (*s_abort) {
        // wait until the activation producer has completed every issued stage, then for
        // the loads to land, before the CTA can exit (bounded)
        const uint64_t t0 = tc::globaltimer();
        while (*s_nB < nA && tc::globaltimer() - t0 < 20000000ull) {
        }
        int never = 0;
        for (long long n = (nA > S ? nA - S : 0); n < nA; ++n)
          tc::mbar_wait(&full[n % S], (uint32_t)((n / S) & 1), &never, 10000000ull);
      }
    }
  } else if (warp == PK_BWARP) {
    // ------------------------------------------------------------ activation producer
    // Activation halves, each once its stage's weight half is armed and the step that
    // writes the activations is complete on every CTA.
    if (lane == 0) {
      const uint64_t pol_x = tc::policy_evict_last();
      const int n_gemm = P.n_gemm;
      const unsigned* phase_cnt = P.phase_cnt;
      const bool tracing = P.trace_cta != nullptr;
      Cur cb{};
      cb.g = 0;
      cur_seek(P, c, cb);
      long long nB = 0;
      int st = 0;
      int ready = -1;  // every phase <= ready is complete on all CTAs
      int last_traced = -1;
      bool ok = true;
      while (cb.g < n_gemm) {
        const int dep = cb.dep;
        if (ok && *s_nA <= nB) {
          // spin on shared memory for the weight producer (bounded)
          const uint64_t t0 = tc::globaltimer();
          unsigned spins = 0;
          while (*s_nA <= nB) {
            if (*s_adone && *s_nA <= nB) {
              ok = false;  // the weight producer stopped (abort)
              break;
            }
            if ((++spins & 255u) == 0 && tc::globaltimer() - t0 > wns) {
              if (!*s_abort) set_abort(P, s_abort);
              ok = false;
              break;
            }
          }
        }
        if (!ok && *s_nA <= nB) break;
        if (ok && dep > ready) {
          const uint64_t t0 = tc::globaltimer();
          unsigned spins = 0;
          const unsigned need = (unsigned)G + (dep == P.stall_phase ? 1u : 0u);
          while (ld_relaxed(phase_cnt + dep) < need) {
            if ((++spins & 63u) == 0) {
              if (aborted(P, s_abort)) {
                ok = false;
                break;
              }
              if (tc::globaltimer() - t0 > wns) {
                set_abort(P, s_abort);
                ok = false;
                break;
              }
            }
          }
          if (ok) {
            ready = dep;
            fence_acquire_gpu();
            fence_proxy_async_global();
          }
        }
        // after an abort the remaining armed stages are completed with whatever the
        // activation buffers hold, so that no load is left in flight
        if (tracing && cb.g != last_traced) {
          trace_ev(P, P.gemm[cb.g].phase, 0);
          last_traced = cb.g;
        }
        tc::tma_load_3d(sB + (size_t)st * BS, cb.tx, 0, 0, cb.kb * PASS_KU, &full[st], pol_x);
        cur_next(P, c, cb);
        ++nB;
        if (++st == S) st = 0;
        *s_nB = nB;
        if (!ok) {
          // drain: wait (bounded) for the weight producer to stop, then arm nothing new
          const uint64_t t0 = tc::globaltimer();
          while (!*s_adone && tc::globaltimer() - t0 < 20000000ull) {
          }
        }
      }
      *s_nB = 0x7fffffffffffffffll;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int seg = 0;
      bool ok = true;
      const int n_gemm = P.n_gemm;
      const int acc_stride = P.acc_stride;
      for (int g = 0; g < n_gemm && ok; ++g) {
        // the projection's parameters in registers (see Cur)
        const int Gm = P.gemm[g].Gm, KB = P.gemm[g].KB;
        const int kstep = P.gemm[g].BN * 128;  // bytes between a stage's activation k-blocks
        const long long total = P.gemm[g].total;
        const uint32_t idesc = P.gemm[g].idesc;
        if (c >= Gm) continue;
        const long long beg = rbeg(c, total, Gm), end = rbeg(c + 1, total, Gm);
        const int gph = P.gemm[g].phase;
        for (long long it = beg; it < end && ok;) {
          const int tile = (int)(it / KB);
          long long seg_end = (long long)(tile + 1) * KB;
          if (seg_end > end) seg_end = end;
          const int buf = seg & 1;
          const uint32_t use = (uint32_t)(seg >> 1);
          if (!tc::mbar_wait(&acce[buf], (use & 1u) ^ 1u, s_abort, wns)) {
            if (!*s_abort) set_abort(P, s_abort);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + (uint32_t)(buf * acc_stride);
          const long long seg_beg = it;
          for (; it < seg_end; ++it) {
            if (!tc::mbar_wait(&full[st], ph, s_abort, wns)) {
              if (!*s_abort) set_abort(P, s_abort);
              ok = false;
              break;
            }
            tc::fence_after_sync();
            if (it == beg) trace_ev(P, gph, 1);
            // the stage's PASS_KU k-blocks: weight tiles 16 KB apart, activation tiles
            // BN x 128 bytes apart (the projection's own box height)
#pragma unroll
            for (int j = 0; j < PASS_KU; ++j) {
              const uint64_t ad = tc::smem_desc_sw128(
                  tc::smem_u32(sA + (size_t)st * PK_A_BYTES + (size_t)j * (PK_A_BYTES / PASS_KU)));
              const uint64_t bd = tc::smem_desc_sw128(
                  tc::smem_u32(sB + (size_t)st * BS + (size_t)j * kstep));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc::mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc,
                             (it != seg_beg || j > 0 || k > 0) ? 1u : 0u);
            }
            tc::mma_commit(&empty[st]);
            if (++st == S) {
              st = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          tc::mma_commit(&accf[buf]);
          if (it >= end) trace_ev(P, gph, 2);
          ++seg;
        }
      }
      if (!ok) {
        // aborted: the MMAs already issued still write tensor memory, which is freed when
        // the CTA leaves; wait (bounded) until they have completed
        int never = 0;
        tc::mma_commit(drain);
        tc::mbar_wait(drain, 0u, &never, 10000000ull);
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ workers
    const int et = threadIdx.x - 64;     // 0 .. 127
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int ml = quarter * 32 + lane;  // tile feature = TMEM lane
    const int wid = et >> 5;
    const int acc_stride = P.acc_stride, n_phase = P.n_phase;
    float* const ws = P.ws;
    unsigned* const tile_cnt = P.tile_cnt;
    int seg = 0;
    bool alive = true;
    // sums-of-squares slots start at zero: cleared before this CTA signals the first step,
    // so before any CTA's input step accumulates into them
    if (c == 0)
      for (int i = et; i < PASS_SS_SLOTS * P.R; i += 128) P.ss[i] = 0;
    for (int j = 0; j < n_phase && alive; ++j) {
      const PassPhase& ph = P.ph[j];
      if (ph.kind == PP_GEMM) {
        // the projection's parameters in registers and its epilogue arguments in shared
        // memory (see Cur)
        const PassGemm& m = P.gemm[ph.gemm];
        if (et == 0 && j + 1 < n_phase && P.ph[j + 1].kind == PP_ATTN)
          prefetch_attn_rows<HD>(P, P.ph[j + 1].layer, c, G);
        const int Gm = m.Gm, KB = m.KB, BN = m.BN, mR = m.R, split = m.split;
        const int lo_col = m.lo_col, additive = m.additive;
        const long long total = m.total;
        {
          const int* src = (const int*)&m.epi;
          int* dst = (int*)s_epi;
          for (int q = et; q < (int)(sizeof(EpiArgs) / 4); q += 128) dst[q] = src[q];
        }
        wk_bar();
        const EpiArgs& epi = *s_epi;
        // the first row chunk's norm scales and RoPE positions, read while the tensor
        // cores work (the norm step this projection depends on must be complete)
        const int step = split ? 16 : 32;
        if (c < Gm) {
          if (!wk_wait_phase(P, m.dep, et, s_abort, s_flag)) {
            alive = false;
            break;
          }
          if (et < min(step, mR)) {
            s_rscale[et] = epi_row_scale(epi, et);
            s_rpos[et] = epi.row_pos ? epi.row_pos[et] : 0;
          }
        }
        if (c < Gm) {
          const long long beg = rbeg(c, total, Gm), end = rbeg(c + 1, total, Gm);
          for (long long it = beg; it < end;) {
            const int tile = (int)(it / KB);
            long long seg_end = (long long)(tile + 1) * KB;
            if (seg_end > end) seg_end = end;
            it = seg_end;
            const int buf = seg & 1;
            const uint32_t use = (uint32_t)(seg >> 1);
            ++seg;
            if (et == 0) {
              *s_flag = tc::mbar_wait(&accf[buf], use & 1u, s_abort, wns) ? 1 : 0;
              if (!*s_flag && !*s_abort) set_abort(P, s_abort);
            }
            wk_bar();
            if (!*s_flag) {
              alive = false;
              break;
            }
            tc::fence_after_sync();
            const int m0 = tile * 128;  // one activation tile: rows 0 .. R-1
            const int row0 = 0;
            const int lrows = mR;
            const long long t_beg = (long long)tile * KB;
            const int cf = owner(t_beg, total, Gm), cl = owner(t_beg + KB - 1, total, Gm);
            const uint32_t tb = tmem + (uint32_t)(buf * acc_stride) + ((uint32_t)(quarter * 32) << 16);
            const int nch = (lrows + step - 1) / step;
            if (cf == cl || additive) {
              for (int ch = 0; ch < nch; ++ch) {
                const int i0 = ch * step;
                float v[16], w[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) w[q] = 0.f;
                tc::tmem_ld16(tb + i0, v);
                if (split) {
                  tc::tmem_ld16(tb + lo_col + i0, w);
                } else if (i0 + 16 < BN) {
                  tc::tmem_ld16(tb + i0 + 16, w);
                }
                tc::tmem_ld_wait();
                if (epi.kind == EPI_RESID || epi.kind == EPI_STORE) {
                  // elementwise fixed-point adds: straight from the registers, no staging
                  if (ch == nch - 1) {
                    tc::fence_before_sync();
                    tc::mbar_arrive(&acce[buf]);
                  }
                  const int rc = min(step, lrows - i0);
                  fx_t* dst = epi.kind == EPI_STORE ? epi.out_fx : epi.resid;
                  const int ldd = epi.kind == EPI_STORE ? epi.out_ld : epi.ld_res;
                  if (m0 + ml < epi.Nout) {
                    fx_t* col = dst + (size_t)(row0 + i0) * ldd + m0 + ml;
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                      if (split) {
                        if (q < rc) red_add_fx(col + (size_t)q * ldd, to_fx(v[q] + w[q]));
                      } else {
                        if (q < rc) red_add_fx(col + (size_t)q * ldd, to_fx(v[q]));
                        if (16 + q < rc) red_add_fx(col + (size_t)(16 + q) * ldd, to_fx(w[q]));
                      }
                    }
                  }
                  continue;
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                  stg[q * 128 + ml] = v[q];
                  stg[(16 + q) * 128 + ml] = w[q];
                }
                if (ch == nch - 1) {
                  tc::fence_before_sync();
                  tc::mbar_arrive(&acce[buf]);
                }
                if (nch > 1 && et < min(step, lrows - i0)) {
                  s_rscale[et] = epi_row_scale(epi, row0 + i0 + et);
                  s_rpos[et] = epi.row_pos ? epi.row_pos[row0 + i0 + et] : 0;
                }
                wk_bar();
                epilogue_tile<bf16>(epi, stg, 128, split ? 16 : -1, m0, row0 + i0,
                                    min(step, lrows - i0), et, 128, s_rscale, s_rpos);
                wk_bar();
              }
            } else {
              const int slot = (rbeg(c, total, Gm) >= t_beg) ? 2 * c : 2 * c + 1;
              float* wsl = ws + (size_t)slot * BN * 128;
              for (int c0 = 0; c0 < BN; c0 += 16) {
                float v[16];
                tc::tmem_ld16(tb + c0, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q) wsl[(size_t)(c0 + q) * 128 + ml] = v[q];
              }
              tc::fence_before_sync();
              tc::mbar_arrive(&acce[buf]);
              wk_bar();
              if (et == 0) {
                const unsigned prev = atom_add_acq_rel(tile_cnt + tile, 1u);
                *s_fin = (prev == (unsigned)(cl - cf)) ? 1 : 0;
              }
              wk_bar();
              if (*s_fin) {
                const int slot_f = (rbeg(cf, total, Gm) == t_beg) ? 2 * cf : 2 * cf + 1;
                for (int ch = 0; ch < nch; ++ch) {
                  const int i0 = ch * step;
                  int col[32];
                  float acc[32];
#pragma unroll
                  for (int q = 0; q < 32; ++q) {
                    if (split) {
                      const int ii = i0 + (q & 15);
                      col[q] = min((q < 16) ? ii : lo_col + ii, BN - 1);
                    } else {
                      col[q] = min(i0 + q, BN - 1);
                    }
                    acc[q] = 0.f;
                  }
                  for (int cc = cf; cc <= cl; ++cc) {
                    const float* src =
                        ws + (size_t)(cc == cf ? slot_f : 2 * cc) * BN * 128 + ml;
#pragma unroll
                    for (int q = 0; q < 32; ++q) acc[q] += __ldcg(src + (size_t)col[q] * 128);
                  }
#pragma unroll
                  for (int q = 0; q < 32; ++q) stg[q * 128 + ml] = acc[q];
                  if (nch > 1 && et < min(step, lrows - i0)) {
                    s_rscale[et] = epi_row_scale(epi, row0 + i0 + et);
                    s_rpos[et] = epi.row_pos ? epi.row_pos[row0 + i0 + et] : 0;
                  }
                  wk_bar();
                  epilogue_tile<bf16>(epi, stg, 128, split ? 16 : -1, m0, row0 + i0,
                                      min(step, lrows - i0), et, 128, s_rscale, s_rpos);
                  wk_bar();
                }
                if (et == 0) tile_cnt[tile] = 0u;
              }
            }
          }
          if (!alive) break;
        }
      } else {
        if (!wk_wait_phase(P, j - 1, et, s_abort, s_flag)) {
          alive = false;
          break;
        }
        if (et == 0) trace_ev(P, j, 0);
        if (ph.kind == PP_INPUT) {
          step_input(P, c, G, et, s_rs, s_tok);
        } else if (ph.kind == PP_NORM) {
          step_norm(P, c, G, ph.slot, (const bf16*)ph.gamma, et, s_rs);
        } else if (ph.kind == PP_ATTN) {
          // One split-KV item (request b, kv head g, key chunk cc) per CTA.  The item reads
          // its queries straight from the QKV projection's fixed-point sums and first moves
          // the draft block's keys / values in its key range from the sums into their cache
          // slots.  Once every item of (b, g) has written its partials (a count per layer,
          // request and kv head), item cc merges the query rows
          // [cc * rows / nv, (cc + 1) * rows / nv) and clears their q / k / v sums for the
          // next layer; for a request without keys item 0 writes zero rows.
          AttnArgs a = P.att;
          const int layer = ph.layer;
          a.kc = (const char*)a.kc + (size_t)layer * P.layer_stride;
          a.vc = (const char*)a.vc + (size_t)layer * P.layer_stride;
          a.q = P.q_fx;
          const int Gq = a.nq / a.nkv;
          const int rows = a.K * Gq;
          const int hd = a.hd, kvw = a.nkv * hd;
          fx_t* const qx = P.q_fx;
          fx_t* const kvx = P.kv_fx;
          const int n_items = a.nchunk * a.nkv * a.B;
          for (int i = c; i < n_items; i += G) {
            const int cc = i % a.nchunk;
            const int g = (i / a.nchunk) % a.nkv;
            const int b = i / (a.nchunk * a.nkv);
            const int L = a.seq_lens[b];
            int first = 0, total = 0;
            attn_span(a, L, &first, &total);
            const int nv = L < 0 ? 0 : attn_nvalid(a, first, total);
            if (cc < nv) {
              const int kbeg = first + cc * a.chunk, kend = min(total, kbeg + a.chunk);
              const int p0 = max(kbeg, L), p1 = min(kend, L + a.K);
              bf16* kc = (bf16*)a.kc + ((size_t)b * a.nkv + g) * a.cap * hd;
              bf16* vc = (bf16*)a.vc + ((size_t)b * a.nkv + g) * a.cap * hd;
              const int nd = p1 > p0 ? (p1 - p0) * hd : 0;
              // every load of a batch is issued before the first store
              constexpr int UM = 4;
              for (int e0 = et; e0 < nd; e0 += 128 * UM) {
                fx_t kq[UM], vq[UM];
#pragma unroll
                for (int u = 0; u < UM; ++u) {
                  const int e = e0 + u * 128;
                  kq[u] = vq[u] = 0;
                  if (e < nd) {
                    const int p = p0 + e / hd, d = e % hd;
                    const fx_t* src = kvx + ((size_t)b * a.K + (p - L)) * 2 * kvw + g * hd + d;
                    kq[u] = __ldcg(src);
                    vq[u] = __ldcg(src + kvw);
                  }
                }
#pragma unroll
                for (int u = 0; u < UM; ++u) {
                  const int e = e0 + u * 128;
                  if (e < nd) {
                    const int p = p0 + e / hd, d = e % hd;
                    kc[(size_t)p * hd + d] = __float2bfloat16_rn(from_fx(kq[u]));
                    vc[(size_t)p * hd + d] = __float2bfloat16_rn(from_fx(vq[u]));
                  }
                }
              }
              if (et == 0 && g == 0 && cc == nv - 1 && L + a.K > a.cap)
                raise_error(P.err, PEAGLE_DEV_KV_OVERFLOW);
              wk_bar();
              auto bar = []() { wk_bar(); };
              attn_mma_item<HD, pass_att_nbuf(HD), decltype(bar), true>(a, b, g, cc, et, 128, uni,
                                                                         bar);
              if (et == 0) trace_ev(P, j, 1);
            }
            const int share = nv > 0 ? nv : 1;
            if (cc >= share) continue;
            unsigned* acnt = P.phase_cnt + P.n_phase + 1 + ((size_t)layer * a.B + b) * a.nkv + g;
            wk_bar();
            if (et == 0) red_release_add(acnt, 1u);
            if (!wk_wait_count(P, acnt, (unsigned)share, et, s_abort, s_flag)) {
              alive = false;
              break;
            }
            if (et == 0) trace_ev(P, j, 2);
            const int r0 = cc * rows / share, r1 = (cc + 1) * rows / share;
            if (nv > 0) {
              for (int rr = r0 + wid; rr < r1; rr += 4)
                attn_merge_rows<bf16, HD>(a, b, g, rows, nv, rr, rr + 1, lane);
            } else {
              for (int e = et; e < (r1 - r0) * hd; e += 128) {
                const int rr = r0 + e / hd, d = e % hd;
                const int jr = rr / Gq, h = g * Gq + (rr - jr * Gq);
                store_act<bf16>((bf16*)a.o, (size_t)a.nq * hd, b * a.K + jr, a.B * a.K, a.split,
                                h * hd + d, 0.f);
              }
            }
            for (int e = et; e < (r1 - r0) * hd; e += 128) {
              const int rr = r0 + e / hd, d = e % hd;
              const int jr = rr / Gq, h = g * Gq + (rr - jr * Gq);
              const size_t r = (size_t)b * a.K + jr;
              qx[r * a.nq * hd + h * hd + d] = 0;
              if (rr - jr * Gq == 0) {  // one merged row per draft row clears its k / v
                kvx[r * 2 * kvw + g * hd + d] = 0;
                kvx[r * 2 * kvw + kvw + g * hd + d] = 0;
              }
            }
          }
          if (!alive) break;
        } else if (ph.kind == PP_ARGMAX) {
          if (P.out_tokens)
            for (int r = c * 128 + et; r < P.R; r += G * 128) {
              const int idx = argmax_key_index(P.keys[r]);
              P.out_tokens[r] = P.d2t ? idx + P.d2t[idx] : idx;
            }
        }
      }
      wk_signal(P, j, et);
    }
    if (!alive && et == 0) *s_abort = 1;
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, (uint32_t)P.tmem_cols);
  }
}

}  // namespace

size_t pass_smem_bytes(int stages, int b_stage_bytes, int uni_bytes) {
  return 1024 /*align slack*/ + (size_t)stages * (PK_A_BYTES + b_stage_bytes) + uni_bytes +
         (size_t)(2 * stages + 5) * 8 + 64 + 16;
}

int pass_launch(const PassParams& P, int head_dim, int grid, cudaStream_t s) {
  const size_t smem = pass_smem_bytes(P.stages, P.b_stage_bytes, P.uni_bytes);
  void (*kern)(const PassParams) = head_dim == 64 ? pass_kernel<64> : pass_kernel<128>;
  cudaError_t ae = smem_optin((const void*)kern, smem);
  if (ae != cudaSuccess) {
    fprintf(stderr, "peagle: pass kernel shared memory (%zu bytes): %s\n", smem,
            cudaGetErrorString(ae));
    return PEAGLE_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PK_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, P);
  if (e != cudaSuccess) {
    fprintf(stderr, "peagle: pass kernel launch failed: %s\n", cudaGetErrorString(e));
    return PEAGLE_ERR_CUDA;
  }
  return PEAGLE_OK;
}

}  // namespace peagle
