// stream.cu -- the drafter's layer projections between two attention
// launches as one persistent kernel, for small batches (at most 32 rows, one
// token tile): the batch-1 drafting step of the P-EAGLE pages (paper
// summary "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training",
// section 2: embedding + projected hidden state, N LLaMA layers; the vLLM
// blog's results at concurrency 1) is bound by streaming the drafter's
// weights, and one launch per projection leaves the memory system idle at
// every launch's ramp and tail.
//
// A segment is a short program of phases run by one CTA per SM:
//   first:   fc -> layer-0 input (row phase) -> QKV_0
//   middle:  O_l -> gate/up_l -> down_l -> QKV_{l+1}
//   last:    O_l -> gate/up_l -> down_l -> final norm of the sampled rows
// with the paged attention of each layer launched between segments.
//
// Roles (224 threads): warp 4 streams weight tiles (128 features x 64 k,
// 16 KB) through a ring of shared-memory stages, phase after phase, waiting
// only for free stages -- weights do not depend on activations, so the
// stream runs across phase boundaries and across the wait for the previous
// kernel.  Warp 5 issues the tcgen05 MMAs (M = 128 features, N = the token
// tile, fp32 accumulators in TMEM, two buffers).  Warps 0-3 load the
// activation panel of each phase (the k-blocks of this CTA's units, by TMA,
// once the phase it depends on is complete everywhere), drain the
// accumulators, and reduce and finish tiles.
//
// Work split: the (feature tile, k-block) units of a phase are dealt out in
// equal contiguous ranges (stream-K).  A tile covered by several CTAs is
// summed by its last-arriving contributor from fp32 partials in CTA order
// (deterministic).  The finisher applies the epilogue and then publishes
// the tile (a release add on the phase's done count); a phase that needs
// the previous phase's output waits (acquire, bounded) until the count
// covers every tile.
//
// Fusions: RMSNorm before a projection is a per-row scale r = rsqrt(mean
// x^2 + eps): the residual-add finisher writes bf16(x * g) (the gain of the
// next norm) and per-tile sums of x^2; the consuming projection multiplies
// its accumulator rows by r (y = W(x r g) = r W(x g)).  The QKV finisher
// applies rotate-half RoPE and writes q and the paged K/V (slot -1: no
// write, the blog's KV-cache rule for rejected rows).
//
// Every wait is bounded; a wait that gives up records PE_DEV_TIMEOUT, sets
// an abort word that the other CTAs' waits watch, and the kernel unwinds
// after its own copies and MMAs have drained.
#include "fp8_common.cuh"
#include "gemm_tc.cuh"

namespace pe {

template <int BN>
struct SCfg {
  static constexpr int STAGE = 128 * 64 * 2;            // one weight tile
  static constexpr int PANEL_KB = BN == 16 ? 32 : 20;   // k-blocks of activations per phase
  static constexpr int PANEL_SLOT = BN * 128;           // one k-block of BN token rows
  static constexpr int PANEL = PANEL_KB * PANEL_SLOT;
  static constexpr int XCHG = 128 * BN * 4;             // [128 features][BN] fp32
  static constexpr int TRIG = 2 * BN * 64 * 4;          // cos, sin [BN][64]
  static constexpr int MISC = 1024;
  static constexpr int BUDGET = 227 * 1024;
  static constexpr int NST = (BUDGET - 1024 - PANEL - XCHG - TRIG - MISC) / STAGE;
  static constexpr int SMEM = 1024 + NST * STAGE + PANEL + XCHG + TRIG + MISC;
  static constexpr int ACC_STRIDE = 2 * BN;             // room for the gate/up pair
  static constexpr int TMEM_COLS = 4 * BN;              // two accumulator buffers
  static constexpr uint32_t IDESC = idesc_bf16_f32(128, BN);
  static_assert(NST >= 6 && SMEM <= BUDGET, "shared memory");
  // barriers, the TMEM address and the broadcast words below offset 512 of MISC
  static_assert((2 * NST + 6) * 8 + 4 + (2 + kStreamMaxPhases) * 4 <= 512, "misc layout");
  static_assert(TMEM_COLS == 64 || TMEM_COLS == 128, "tensor memory");
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Fetch-and-add with acquire and release at GPU scope: publishes what this
// CTA wrote before its barrier, and sees what earlier arrivals published.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void give_up(int* abort_word, int* err) {
  record_error(err, PE_DEV_TIMEOUT);
  atomicExch(abort_word, 1);
}
// mbarrier wait that also gives up when another CTA has aborted.
__device__ __forceinline__ bool mbar_wait_ab(uint64_t* bar, uint32_t parity, int* abort_word,
                                             int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (ld_relaxed_gpu(abort_word)) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      give_up(abort_word, err);
      return false;
    }
  }
}
// *flag >= target (acquire), bounded, abandoned on abort.
__device__ __forceinline__ bool flag_wait_ab(const int* flag, int target, int* abort_word,
                                             int* err) {
  if (ld_acquire_gpu(flag) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (ld_acquire_gpu(flag) >= target) return true;
    if (ld_relaxed_gpu(abort_word)) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      give_up(abort_word, err);
      return false;
    }
  }
}

// 16 bytes global -> shared without the TMA unit (src_bytes 0: zeros)
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// diagnostic timeline stamp (no-op unless a buffer was given)
__device__ __forceinline__ void stamp(const StreamParams& p, int slot) {
  if (p.timeline)
    p.timeline[static_cast<size_t>(blockIdx.x) * kStreamTimelineSlots + slot] = global_timer_ns();
}

__device__ __forceinline__ float bf(const void* p, size_t i) {
  return __bfloat162float(static_cast<const bf16*>(p)[i]);
}

// CTAs that take part in phase P: all G, or one per unit when the phase
// has fewer units than that -- every participant then holds at least one
// unit, so every CTA between a tile's first and last contributor arrives
// at the tile's counter.
__device__ __forceinline__ int phase_ctas(const StreamPhase& P, int G) {
  const long long U = static_cast<long long>(P.tiles) * P.kb;
  return U < G ? static_cast<int>(U) : G;
}
// The units [lo, hi) of phase P that CTA `cta` takes (empty past the
// participants).
__device__ __forceinline__ void phase_range(const StreamPhase& P, int cta, int G, long long& lo,
                                            long long& hi) {
  const long long U = static_cast<long long>(P.tiles) * P.kb;
  const int Gp = phase_ctas(P, G);
  lo = cta < Gp ? unit_lo(cta, U, Gp) : U;
  hi = cta < Gp ? unit_lo(cta + 1, U, Gp) : U;
}

// This CTA's weight tiles in stream order: phase, unit, and for the gate/up
// pair which of the two matrices.
struct WeightCursor {
  int ph, a;
  long long u, hi;
};
__device__ __forceinline__ bool wc_next_phase(const StreamParams& p, int cta, int G,
                                              WeightCursor& c) {
  for (++c.ph; c.ph < p.nphases; ++c.ph) {
    const StreamPhase& P = p.ph[c.ph];
    if (P.kind != SK_GEMM) continue;
    long long lo, hi;
    phase_range(P, cta, G, lo, hi);
    if (lo < hi) {
      c.u = lo;
      c.hi = hi;
      c.a = 0;
      return true;
    }
  }
  return false;
}
__device__ __forceinline__ bool wc_advance(const StreamParams& p, int cta, int G,
                                           WeightCursor& c) {
  if (c.a < p.ph[c.ph].dual) {
    ++c.a;
    return true;
  }
  c.a = 0;
  if (++c.u < c.hi) return true;
  return wc_next_phase(p, cta, G, c);
}

__device__ __forceinline__ int phase_target(const StreamParams& p, int i) {
  const StreamPhase& P = p.ph[i];
  return P.kind == SK_GEMM ? P.tiles : P.kind == SK_EMBED ? p.rows : p.final_rows;
}

// 16 consecutive accumulator columns of this thread's lane, with the
// registers fenced behind the wait.
template <int BN>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float (&v)[BN / 16][16]) {
#pragma unroll
  for (int c = 0; c < BN / 16; ++c) tmem_ld16(taddr + 16 * c, v[c]);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < BN / 16; ++c) reg_fence16(v[c]);
}

// Sum of a[j] over the 128 epilogue threads for every token j < BN, in a
// fixed order (butterfly within the warp, then warps 0..3); thread j < BN
// returns the sum for token j.  Uses red[4][BN] of shared memory.
template <int BN>
__device__ __forceinline__ float sum_over_features(float (&a)[BN], float* red, int warp,
                                                   int lane) {
#pragma unroll
  for (int j = 0; j < BN; ++j) {
    float x = a[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    a[j] = x;
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < BN; ++j) red[warp * BN + j] = a[j];
  }
  named_bar_sync(1, 128);
  const int t = threadIdx.x;
  float s = 0.f;
  if (t < BN) s = ((red[t] + red[BN + t]) + red[2 * BN + t]) + red[3 * BN + t];
  named_bar_sync(1, 128);
  return s;
}

// ---------------------------------------------------------------------------
// tile epilogues (all 128 epilogue threads together; thread = feature row)
// ---------------------------------------------------------------------------
// The residual of this thread's feature for the BN tokens (0 past the batch
// or the features): loaded by the finisher before it sums the partials, so
// that the two sets of loads are in flight together.
template <int BN>
__device__ __forceinline__ void load_resid(const StreamParams& p, const StreamPhase& P, int tile,
                                           float (&old)[BN]) {
  const int o = tile * 128 + threadIdx.x;
  const bool valid = o < P.N;
#pragma unroll
  for (int j = 0; j < BN; ++j)
    old[j] = (j < p.rows && valid) ? __ldcg(p.resid + static_cast<size_t>(j) * p.d + o) : 0.f;
}

template <int BN>
__device__ void finish_tile(const StreamParams& p, const StreamPhase& P, int tile,
                            float (&v)[BN], float (&v2)[BN], const float (&old)[BN],
                            const float* rms, float* xchg, const float* cosT, const float* sinT,
                            const int* slot_s, int warp, int lane) {
  const int row = threadIdx.x;
  const int o = tile * 128 + row;
  const bool valid = o < P.N;
  const int rows = p.rows;
  if (P.norm_src >= 0) {
#pragma unroll
    for (int j = 0; j < BN; ++j) {
      v[j] *= rms[j];
      v2[j] *= rms[j];
    }
  }
  switch (P.epi) {
    case SE_STORE: {
#pragma unroll
      for (int j = 0; j < BN; ++j)
        if (j < rows && valid) p.resid[static_cast<size_t>(j) * p.d + o] = v[j];
      break;
    }
    case SE_ADD: {
      float* r = p.resid + o;
      const float gn = (valid && P.g_next) ? bf(P.g_next, o) : 0.f;
      float sq[BN];
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        const float nv = old[j] + v[j];
        sq[j] = 0.f;
        if (j < rows && valid) {
          r[static_cast<size_t>(j) * p.d] = nv;
          if (P.xg)
            static_cast<bf16*>(P.xg)[static_cast<size_t>(j) * P.N + o] = __float2bfloat16_rn(nv * gn);
          sq[j] = nv * nv;
        }
      }
      if (P.ssq) {
        const float s = sum_over_features<BN>(sq, xchg, warp, lane);
        if (row < BN) P.ssq[tile * 32 + row] = s;
      }
      break;
    }
    case SE_SILU_MUL: {
      bf16* out = static_cast<bf16*>(P.out);
#pragma unroll
      for (int j = 0; j < BN; ++j)
        if (j < rows && valid)
          out[static_cast<size_t>(j) * P.ldo + o] = __float2bfloat16_rn(silu_f(v[j]) * v2[j]);
      break;
    }
    case SE_ROPE_KV: {
      // features [0, Hq dh) are q, then Hkv dh of k, then Hkv dh of v; heads
      // never straddle a 128-feature tile (checked on the host)
      const int qd = p.Hq * p.dh, kd = p.Hkv * p.dh;
      const int jd = o % p.dh, half = p.dh / 2;
      const bool is_v = o >= qd + kd;
      if (!is_v) {
#pragma unroll
        for (int j = 0; j < BN; ++j) xchg[row * BN + j] = v[j];
        named_bar_sync(1, 128);
        const int prow = jd < half ? row + half : row - half;
        const int i = jd % half;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const float other = xchg[prow * BN + j];
          const float c = cosT[j * 64 + i], s = sinT[j * 64 + i];
          v2[j] = jd < half ? v[j] * c - other * s : v[j] * c + other * s;
        }
        named_bar_sync(1, 128);
      } else {
        // v rows take no rotation; keep the barrier count of the warps equal
        named_bar_sync(1, 128);
        named_bar_sync(1, 128);
#pragma unroll
        for (int j = 0; j < BN; ++j) v2[j] = v[j];
      }
      if (!valid) break;
      if (o < qd) {
        bf16* q = static_cast<bf16*>(p.q_out);
#pragma unroll
        for (int j = 0; j < BN; ++j)
          if (j < rows) q[static_cast<size_t>(j) * qd + o] = __float2bfloat16_rn(v2[j]);
      } else {
        const bool is_k = o < qd + kd;
        const int g = (o - (is_k ? qd : qd + kd)) / p.dh;
        void* cache = is_k ? p.k_cache : p.v_cache;
        const float inv = is_k ? p.k_inv_scale : p.v_inv_scale;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const int sl = slot_s[j];
          if (j < rows && sl >= 0) {
            const int blk = sl / 16, off = sl % 16;
            if (blk >= p.num_blocks) {
              if (jd == 0) record_error(p.err, PE_DEV_BAD_BLOCK);
            } else {
              const size_t at = ((static_cast<size_t>(blk) * p.Hkv + g) * 16 + off) * p.dh + jd;
              if (p.kv_fp8)
                static_cast<uint8_t*>(cache)[at] =
                    static_cast<uint8_t>(f32x2_to_e4m3x2(v2[j] * inv, 0.f) & 0xffu);
              else
                static_cast<bf16*>(cache)[at] = __float2bfloat16_rn(v2[j]);
            }
          }
        }
      }
      break;
    }
  }
}

// layer-0 input row r: [RMSNorm_e(emb[id]) ; RMSNorm_h(resid[r])], 2d wide
__device__ void embed_row(const StreamParams& p, int r, float* red) {
  const int t = threadIdx.x, d = p.d;
  int id = p.ids[r];
  if (id < 0 || id >= p.vocab) {
    if (t == 0) record_error(p.err, PE_DEV_BAD_TOKEN);
    id = 0;
  }
  const bf16* e = static_cast<const bf16*>(p.emb) + static_cast<size_t>(id) * d;
  const float* h = p.resid + static_cast<size_t>(r) * d;
  float se = 0.f, sh = 0.f;
  for (int k = t; k < d; k += 128) {
    const float ev = __bfloat162float(e[k]), hv = h[k];
    se += ev * ev;
    sh += hv * hv;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    se += __shfl_xor_sync(0xffffffffu, se, o);
    sh += __shfl_xor_sync(0xffffffffu, sh, o);
  }
  if ((t & 31) == 0) {
    red[t >> 5] = se;
    red[4 + (t >> 5)] = sh;
  }
  named_bar_sync(1, 128);
  se = ((red[0] + red[1]) + red[2]) + red[3];
  sh = ((red[4] + red[5]) + red[6]) + red[7];
  named_bar_sync(1, 128);
  const float re = rsqrtf(se / d + p.eps), rh = rsqrtf(sh / d + p.eps);
  bf16* x = static_cast<bf16*>(p.x_in) + static_cast<size_t>(r) * 2 * d;
  for (int k = t; k < d; k += 128) {
    x[k] = __float2bfloat16_rn(__bfloat162float(e[k]) * re * bf(p.g_e, k));
    x[d + k] = __float2bfloat16_rn(h[k] * rh * bf(p.g_h, k));
  }
}

// final norm of sampled row i (gathered through new_idx)
__device__ void final_row(const StreamParams& p, int i, float* red) {
  const int t = threadIdx.x, d = p.d;
  int src = p.new_idx[i];
  const bool bad = src < 0 || src >= p.rows;
  if (bad) {
    if (t == 0) record_error(p.err, PE_DEV_BAD_ROW);
    src = 0;
  }
  const float* x = p.resid + static_cast<size_t>(src) * d;
  float ss = 0.f;
  for (int k = t; k < d; k += 128) ss += x[k] * x[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((t & 31) == 0) red[t >> 5] = ss;
  named_bar_sync(1, 128);
  ss = ((red[0] + red[1]) + red[2]) + red[3];
  named_bar_sync(1, 128);
  const float r = rsqrtf(ss / d + p.eps);
  bf16* y = static_cast<bf16*>(p.out_hidden) + static_cast<size_t>(i) * d;
  for (int k = t; k < d; k += 128)
    y[k] = __float2bfloat16_rn(bad ? 0.f : x[k] * r * bf(p.g_final, k));
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int BN>
__global__ void __launch_bounds__(224, 1)
    stream_kernel(const __grid_constant__ StreamMaps maps, const __grid_constant__ StreamParams p) {
  using C = SCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint8_t* panel = ring + C::NST * C::STAGE;
  float* xchg = reinterpret_cast<float*>(panel + C::PANEL);
  float* cosT = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xchg) + C::XCHG);
  float* sinT = cosT + BN * 64;
  uint8_t* misc = reinterpret_cast<uint8_t*>(cosT) + C::TRIG;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);  // [NST]
  uint64_t* empty = full + C::NST;                      // [NST]
  uint64_t* acc_full = empty + C::NST;                  // [2]
  uint64_t* acc_empty = acc_full + 2;                   // [2]
  uint64_t* b_full = acc_empty + 2;                     // activation panel landed
  uint64_t* drain = b_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  // broadcast words of the epilogue warps: [0] accumulator wait, [1]
  // finisher election, [2 + phase] dependency wait (one per phase, so a
  // thread that runs ahead never overwrites a word others still read)
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [2 + kStreamMaxPhases]
  float* rms = reinterpret_cast<float*>(misc + 512);                     // [32]
  int* slot_s = reinterpret_cast<int*>(misc + 640);                      // [32]
  float* red = reinterpret_cast<float*>(misc + 768);                     // [8]
  volatile int* loaded = reinterpret_cast<volatile int*>(misc + 800);     // weight tiles issued
  volatile int* open_ph = reinterpret_cast<volatile int*>(misc + 804);    // phases whose inputs are ready

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  int* const abort_word = p.sync + kStreamSyncAbort;

  if (threadIdx.x == 0) {
    stamp(p, 0);
    *loaded = 0;
    *open_ph = 0;
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    mbar_init(b_full, 1);
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 4) {
    // ---- weight stream ----------------------------------------------------
    if (lane == 0) {
      for (int i = 0; i < kStreamMaxMaps; ++i) tma_prefetch_desc(&maps.m[i]);
      const uint64_t pol = l2_policy_evict_first();
      WeightCursor ld{-1, 0, 0, 0};
      bool has_ld = wc_next_phase(p, cta, G, ld);
      stamp(p, 2);
      long long ring_i = 0;
      int cur_ph = -1, in_ph = 0;   // phase of the last load, loads issued into it
      while (has_ld) {
        const StreamPhase& P = p.ph[ld.ph];
        if (ld.ph != cur_ph) {
          cur_ph = ld.ph;
          in_ph = 0;
        }
        // At most boundary_tiles loads into a phase whose inputs are not
        // ready yet: the refill burst at a phase boundary would otherwise
        // delay the finishers' and the next panel's memory accesses.
        if (p.boundary_tiles >= 0 && in_ph >= p.boundary_tiles && *open_ph < ld.ph) {
          const unsigned long long t0 = global_timer_ns();
          while (*open_ph < ld.ph && global_timer_ns() - t0 < kWaitTimeoutNs) __nanosleep(64);
        }
        ++in_ph;
        const int st = static_cast<int>(ring_i % C::NST);
        const long long rnd = ring_i / C::NST;
        if (rnd > 0 && !mbar_wait_ab(&empty[st], static_cast<uint32_t>(rnd - 1) & 1, abort_word,
                                     p.err))
          break;
        mbar_arrive_expect_tx(&full[st], C::STAGE);
        tma_load_2d(ring + st * C::STAGE, &maps.m[ld.a ? P.map_a2 : P.map_a], &full[st],
                    static_cast<int>(ld.u % P.kb) * 64, static_cast<int>(ld.u / P.kb) * 128, pol);
        ++ring_i;
        *loaded = static_cast<int>(ring_i);
        has_ld = wc_advance(p, cta, G, ld);
      }
      *loaded = 0x7fffffff;   // done (or gave up): the prefetcher stops
      // every copy this thread issued has landed before the CTA exits
      for (long long i = ring_i - 1; i >= 0 && i >= ring_i - C::NST; --i)
        mbar_wait(&full[i % C::NST], static_cast<uint32_t>(i / C::NST) & 1, p.err);
    }
  } else if (warp == 6) {
    // ---- L2 prefetch --------------------------------------------------------
    // Up to prefetch_tiles weight tiles ahead of the ring, one 128-byte line
    // per weight row and k-block, with prefetch.global.L2 (the load/store
    // path, not the TMA unit, whose queue carries the ring's copies): HBM
    // keeps streaming while the ring is full and the MMAs wait for a phase's
    // activations, and the ring refills from L2 afterwards.
    if (p.prefetch_tiles > 0) {
      WeightCursor pf{-1, 0, 0, 0};
      bool has = wc_next_phase(p, cta, G, pf);
      long long issued = 0;
      const unsigned long long t0 = global_timer_ns();
      while (has) {
        // lane 0 reads the producer's progress and the clock for the warp,
        // so all lanes take the same path
        const int done = __shfl_sync(0xffffffffu, *loaded, 0);
        if (done == 0x7fffffff) break;
        if (issued >= done + p.prefetch_tiles) {
          const int late = __shfl_sync(0xffffffffu, global_timer_ns() - t0 > kWaitTimeoutNs, 0);
          if (late) break;
          __nanosleep(256);
          continue;
        }
        const StreamPhase& P = p.ph[pf.ph];
        const int tile = static_cast<int>(pf.u / P.kb), kk = static_cast<int>(pf.u % P.kb);
        const char* w = static_cast<const char*>(pf.a ? P.w2 : P.w);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = tile * 128 + q * 32 + lane;
          if (r < P.N) {
            const char* line = w + (static_cast<size_t>(r) * P.K + kk * 64) * 2;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
          }
        }
        ++issued;
        has = wc_advance(p, cta, G, pf);
      }
    }
  } else if (warp == 5) {
    // ---- MMA issuer -------------------------------------------------------
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
    named_bar_sync(2, 160);
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (lane == 0) {
      long long ring_i = 0;
      int seg = 0, bph = 0;
      bool ok = true;
      for (int ph = 0; ph < p.nphases && ok; ++ph) {
        const StreamPhase& P = p.ph[ph];
        if (P.kind != SK_GEMM) continue;
        long long lo, hi;
        phase_range(P, cta, G, lo, hi);
        if (lo >= hi) continue;
        if (!mbar_wait_ab(b_full, bph & 1, abort_word, p.err)) break;
        stamp(p, 4 + 4 * ph + 1);
        ++bph;
        for (long long u = lo; u < hi && ok;) {
          const int tile = static_cast<int>(u / P.kb);
          const int k_lo = static_cast<int>(u - static_cast<long long>(tile) * P.kb);
          const int k_hi = static_cast<int>(P.kb < k_lo + (hi - u) ? P.kb : k_lo + (hi - u));
          const int acc = seg & 1;
          if (seg >= 2 && !mbar_wait_ab(&acc_empty[acc], ((seg >> 1) - 1) & 1, abort_word, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * C::ACC_STRIDE;
          for (int kk = k_lo; kk < k_hi; ++kk) {
            const int pi = static_cast<int>(u - lo) + (kk - k_lo);  // panel slot of this unit
            const int st_a = static_cast<int>(ring_i % C::NST);
            const int st_b = static_cast<int>((ring_i + 1) % C::NST);
            if (!mbar_wait_ab(&full[st_a], static_cast<uint32_t>(ring_i / C::NST) & 1, abort_word,
                              p.err) ||
                (P.dual && !mbar_wait_ab(&full[st_b],
                                         static_cast<uint32_t>((ring_i + 1) / C::NST) & 1,
                                         abort_word, p.err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(ring + st_a * C::STAGE);
            const uint32_t a2_addr = smem_u32(ring + st_b * C::STAGE);
            const uint32_t b_addr = smem_u32(panel + pi * C::PANEL_SLOT);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const uint64_t bdesc = sw128_kmajor_desc(b_addr + k4 * 32);
              const uint32_t accum = (kk > k_lo || k4 > 0) ? 1u : 0u;
              umma_bf16(d, sw128_kmajor_desc(a_addr + k4 * 32), bdesc, C::IDESC, accum);
              if (P.dual)
                umma_bf16(d + BN, sw128_kmajor_desc(a2_addr + k4 * 32), bdesc, C::IDESC, accum);
            }
            umma_commit(&empty[st_a]);
            if (P.dual) umma_commit(&empty[st_b]);
            ring_i += P.dual ? 2 : 1;
          }
          if (!ok) break;
          umma_commit(&acc_full[acc]);
          ++seg;
          u += k_hi - k_lo;
        }
        stamp(p, 4 + 4 * ph + 2);
      }
      // all MMAs of this thread complete before the tensor memory is freed
      umma_commit(drain);
      mbar_wait(drain, 0, p.err);
    }
    tc_fence_before();
  } else {
    // ---- warps 0-3: activation panels, accumulators, tile finishers --------
    named_bar_sync(2, 160);
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) stamp(p, 1);
    grid_dep_wait();
    // dependents may start once this CTA has waited for its inputs and holds
    // its tensor memory
    if (threadIdx.x == 0) grid_dep_launch();
    const int row = threadIdx.x;
    int seg = 0, bph = 0;
    bool dead = false;
    for (int ph = 0; ph < p.nphases && !dead; ++ph) {
      const StreamPhase& P = p.ph[ph];
      // wait until the previous phase is complete on every CTA
      if (ph > 0) {
        if (threadIdx.x == 0)
          bcast[2 + ph] = flag_wait_ab(p.sync + ph - 1, phase_target(p, ph - 1), abort_word, p.err);
        named_bar_sync(1, 128);
        if (!bcast[2 + ph]) {
          dead = true;
          break;
        }
        if (threadIdx.x == 0) {
          stamp(p, 4 + 4 * ph);
          *open_ph = ph;
        }
      }
      if (P.kind == SK_EMBED || P.kind == SK_FINAL) {
        const int n = P.kind == SK_EMBED ? p.rows : p.final_rows;
        if (cta < n) {
          if (P.kind == SK_EMBED) embed_row(p, cta, red);
          else final_row(p, cta, red);
          named_bar_sync(1, 128);
          if (threadIdx.x == 0) red_release_add(p.sync + ph, 1);
        }
        continue;
      }
      // ---- GEMM phase ----
      if (P.norm_src >= 0) {
        // r = rsqrt(mean x^2 + eps) of each row from the producing phase's
        // per-tile sums: all of them loaded at once (one round trip) into
        // the exchange buffer, then summed in tile order (deterministic)
        const StreamPhase& S = p.ph[P.norm_src];
        for (int idx = row; idx < S.tiles * BN; idx += 128)
          xchg[idx] = __ldcg(S.ssq + (idx / BN) * 32 + idx % BN);
        named_bar_sync(1, 128);
        if (row < BN) {
          float s = 0.f;
          for (int t = 0; t < S.tiles; ++t) s += xchg[t * BN + row];
          rms[row] = rsqrtf(s / P.norm_d + p.eps);
        }
      }
      if (P.epi == SE_ROPE_KV) {
        const int half = p.dh / 2;
        for (int idx = row; idx < BN * half; idx += 128) {
          const int j = idx / half, i = idx % half;
          float c = 1.f, s = 0.f;
          if (j < p.rows) {
            // angle in fp64, reduced to [-pi, pi] before the fp32 sine/cosine
            const double two_pi = 6.283185307179586476925286766559;
            const double ang = static_cast<double>(p.pos[j]) * p.inv_freq64[i];
            const double red_ang = ang - rint(ang * (1.0 / two_pi)) * two_pi;
            sincosf(static_cast<float>(red_ang), &s, &c);
          }
          cosT[j * 64 + i] = c;
          sinT[j * 64 + i] = s;
        }
        if (row < BN) slot_s[row] = row < p.rows ? p.slot[row] : -1;
      }
      named_bar_sync(1, 128);
      long long lo, hi;
      phase_range(P, cta, G, lo, hi);
      if (lo >= hi) continue;
      {
        // This CTA's activation k-blocks, one panel slot per unit, in the
        // 128-byte-swizzled K-major layout the MMA reads (16-byte chunk j of
        // row r at r * 128 + ((j ^ (r & 7)) * 16)); rows past the batch and
        // k past K are zero.  Copied with cp.async by the 128 threads, not
        // by TMA: the TMA unit of this SM is busy streaming weights, and a
        // panel queued behind that stream would wait for it.
        // thread t copies chunk t % 8 of rows t / 8 (+ 16 for 32-row tiles)
        // of every slot
        const bf16* x = static_cast<const bf16*>(P.x);
        const int j = row & 7, r0 = row >> 3;
        const int n = static_cast<int>(hi - lo);
        int kk = static_cast<int>(lo % P.kb);
        for (int sl = 0; sl < n; ++sl) {
          const int k = kk * 64 + j * 8;
#pragma unroll
          for (int r = r0; r < BN; r += 16) {
            const bool in = r < p.rows && k < P.K;
            const bf16* src = x + (in ? static_cast<size_t>(r) * P.ldx + k : 0);
            cp_async_16(panel + sl * C::PANEL_SLOT + r * 128 + ((j ^ (r & 7)) * 16), src,
                        in ? 16 : 0);
          }
          if (++kk == P.kb) kk = 0;
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (threadIdx.x == 0) mbar_arrive(b_full);
      }
      ++bph;
      const long long U = static_cast<long long>(P.tiles) * P.kb;
      const int Gp = phase_ctas(P, G);
      int fin[2], nfin = 0;   // at most the first and the last segment are partial
      for (long long u = lo; u < hi;) {
        const int tile = static_cast<int>(u / P.kb);
        const int k_lo = static_cast<int>(u - static_cast<long long>(tile) * P.kb);
        const int k_hi = static_cast<int>(P.kb < k_lo + (hi - u) ? P.kb : k_lo + (hi - u));
        const int acc = seg & 1;
        if (threadIdx.x == 0) bcast[0] = mbar_wait_ab(&acc_full[acc], (seg >> 1) & 1, abort_word, p.err);
        named_bar_sync(1, 128);
        if (!bcast[0]) {
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * C::ACC_STRIDE;
        float va[BN / 16][16], vb[BN / 16][16];
        tmem_row<BN>(taddr, va);
        if (P.dual) tmem_row<BN>(taddr + BN, vb);
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
        float v[BN], v2[BN];
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          v[j] = va[j / 16][j % 16];
          v2[j] = P.dual ? vb[j / 16][j % 16] : 0.f;
        }
        const int c_first = cta_of_unit(static_cast<long long>(tile) * P.kb, U, Gp);
        const int c_last = cta_of_unit(static_cast<long long>(tile + 1) * P.kb - 1, U, Gp);
        if (c_first == c_last) {
          // the whole tile is this CTA's: finish and publish it now
          float old[BN];
          if (P.epi == SE_ADD) load_resid<BN>(p, P, tile, old);
          finish_tile<BN>(p, P, tile, v, v2, old, rms, xchg, cosT, sinT, slot_s, warp, lane);
          named_bar_sync(1, 128);
          if (threadIdx.x == 0) red_release_add(p.sync + ph, 1);
        } else {
          // partial tile: to this CTA's slot, published by thread 0's release
          // after the barrier; the last arrival (acquire) finishes the tile,
          // but only after this CTA's other partials are out too
          const int slot = (u == lo) ? 0 : 1;
          float* wsp = p.ws + (static_cast<size_t>(cta) * 2 + slot) * (128 * 64);
#pragma unroll
          for (int j = 0; j < BN; ++j) {
            wsp[j * 128 + row] = v[j];
            if (P.dual) wsp[(BN + j) * 128 + row] = v2[j];
          }
          named_bar_sync(1, 128);
          if (threadIdx.x == 0) {
            if (ph < 4) stamp(p, 24 + 4 * ph + (u == lo ? 0 : 2));
            const int old = atom_add_acq_rel(P.counters + tile, 1);
            bcast[1] = (old == c_last - c_first) ? 1 : 0;
            if (ph < 4) stamp(p, 24 + 4 * ph + (u == lo ? 1 : 3));
          }
          named_bar_sync(1, 128);
          if (bcast[1]) fin[nfin++] = tile;
        }
        ++seg;
        u += k_hi - k_lo;
      }
      // Tiles this CTA arrived last at: sum every contributor's partial in
      // CTA order (deterministic), finish and publish.  Deferred so that a
      // finisher never holds back its own next partial, which another
      // tile's finisher may be waiting for.
      for (int f = 0; f < nfin && !dead; ++f) {
        const int tile = fin[f];
        const int c_first = cta_of_unit(static_cast<long long>(tile) * P.kb, U, Gp);
        const int c_last = cta_of_unit(static_cast<long long>(tile + 1) * P.kb - 1, U, Gp);
        if (threadIdx.x == 0) {
          P.counters[tile] = 0;   // every contributor has arrived
          if (ph < 4) stamp(p, 40 + 4 * ph);
        }
        float v[BN], v2[BN], old[BN];
        if (P.epi == SE_ADD) load_resid<BN>(p, P, tile, old);
#pragma unroll
        for (int j = 0; j < BN; ++j) v[j] = v2[j] = 0.f;
        // contributors in CTA order, UNR partials' loads in flight
        constexpr int UNR = BN == 16 ? 4 : 2;
        for (int c = c_first; c <= c_last; c += UNR) {
          float t[UNR][BN], t2[UNR][BN];
#pragma unroll
          for (int q = 0; q < UNR; ++q) {
            if (c + q > c_last) break;
            const int cq = c + q;
            const int cs = unit_lo(cq, U, Gp) >= static_cast<long long>(tile) * P.kb ? 0 : 1;
            const float* src = p.ws + (static_cast<size_t>(cq) * 2 + cs) * (128 * 64) + row;
#pragma unroll
            for (int j = 0; j < BN; ++j) {
              t[q][j] = __ldcg(src + j * 128);
              t2[q][j] = P.dual ? __ldcg(src + (BN + j) * 128) : 0.f;
            }
          }
#pragma unroll
          for (int q = 0; q < UNR; ++q) {
            if (c + q > c_last) break;
#pragma unroll
            for (int j = 0; j < BN; ++j) {
              v[j] += t[q][j];
              v2[j] += t2[q][j];
            }
          }
        }
        if (threadIdx.x == 0 && ph < 4) stamp(p, 40 + 4 * ph + 1);
        finish_tile<BN>(p, P, tile, v, v2, old, rms, xchg, cosT, sinT, slot_s, warp, lane);
        if (threadIdx.x == 0 && ph < 4) stamp(p, 40 + 4 * ph + 2);
        named_bar_sync(1, 128);
        if (threadIdx.x == 0) {
          red_release_add(p.sync + ph, 1);
          if (ph < 4) stamp(p, 40 + 4 * ph + 3);
        }
      }
      if (threadIdx.x == 0) stamp(p, 4 + 4 * ph + 3);
    }
    tc_fence_before();
  }

  __syncthreads();
  if (threadIdx.x == 0) stamp(p, 60);
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, C::TMEM_COLS);
  }
  // The last CTA out leaves the synchronisation words zero for the next
  // launch (the tile counters too, which finishers reset themselves unless
  // a wait gave up).
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(p.sync + kStreamSyncExit, 1);
    bcast[0] = old == G - 1 ? 1 + ld_relaxed_gpu(abort_word) : 0;
  }
  __syncthreads();
  if (bcast[0]) {
    __threadfence();
    if (bcast[0] > 1)
      for (int i = threadIdx.x; i < p.n_counters; i += blockDim.x) p.counters[i] = 0;
    if (threadIdx.x < kStreamMaxPhases) p.sync[threadIdx.x] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
      p.sync[kStreamSyncAbort] = 0;
      __threadfence();
      p.sync[kStreamSyncExit] = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int BN>
static cudaError_t stream_attr() {
  return cudaFuncSetAttribute(stream_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SCfg<BN>::SMEM);
}

cudaError_t init_stream() {
  cudaError_t e = stream_attr<16>();
  if (e == cudaSuccess) e = stream_attr<32>();
  return e;
}

int stream_panel_kb(int rows) { return rows <= 16 ? SCfg<16>::PANEL_KB : SCfg<32>::PANEL_KB; }

size_t stream_ws_floats(int grid) { return static_cast<size_t>(grid) * 2 * 128 * 64; }

cudaError_t launch_stream(const StreamMaps& maps, const StreamParams& p, int grid,
                          cudaStream_t s) {
  if (p.rows < 1 || p.rows > 32 || grid < 1) return cudaErrorInvalidValue;
  if (p.rows <= 16)
    return launch_pdl(stream_kernel<16>, dim3(grid), dim3(224), SCfg<16>::SMEM, s, maps, p);
  return launch_pdl(stream_kernel<32>, dim3(grid), dim3(224), SCfg<32>::SMEM, s, maps, p);
}

}  // namespace pe
