// gemm_tc.cuh -- pieces of the tensor-core projection kernel (gemm_tc.cu:
// stream-K / cluster split-K, one CTA per tile): the tile configuration,
// the kernel parameters and the epilogue.
#pragma once

#include "fp8_common.cuh"
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

template <int BN, bool DUAL>
struct TcCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int NA = DUAL ? 2 : 1;
  static constexpr int STAGE_BYTES = A_BYTES * NA + B_BYTES;
  static constexpr int ACC_COLS = BN * NA;
  static constexpr int NUM_ACC = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_RAW = ACC_COLS * NUM_ACC;
  static constexpr int TMEM_COLS = TMEM_RAW <= 32    ? 32
                                   : TMEM_RAW <= 64  ? 64
                                   : TMEM_RAW <= 128 ? 128
                                   : TMEM_RAW <= 256 ? 256
                                                     : 512;
  // Narrow token tiles (a few rows, weight streaming) keep the CTA near
  // 100 KB of shared memory so that the next projection's CTA fits on the
  // same SM and prefetches its weights while this one drains.
  static constexpr int SMEM_BUDGET = BN <= 32 ? 104 * 1024 : 200 * 1024;
  // a cluster split's partial in shared memory: row-major, rows padded to
  // PS floats (16-byte aligned rows, few bank conflicts) for vector reads
  static constexpr int PS = ACC_COLS + 4;
  static constexpr int STAGES_RAW = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  // barriers and flags, then (RS_OFF) the row scales of a folded RMSNorm:
  // float partial[4][32], float r[32], int slot[32]; then (TAB_OFF, token
  // tiles of at most 32) the rotary table of the tile's tokens for the
  // fused RoPE epilogue, [BN][64] floats (cos / sin of the dh / 2 angles)
  static constexpr int RS_OFF = 256;
  static constexpr int TAB_OFF = RS_OFF + 6 * 32 * 4;
  static constexpr int TAB_FLOATS = BN <= 32 ? BN * 64 : 0;
  static constexpr int BAR_BYTES = TAB_OFF + TAB_FLOATS * 4;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert((2 * STAGES + 6) * 8 + 12 <= RS_OFF, "barrier space");
  // Pushed cluster reduction: items are (32-row group, 16-column chunk)
  // pairs, four row groups a chunk; item i belongs to cluster rank i % S,
  // which receives every rank's 32 x PW floats of it (PW: the chunk's
  // columns, both halves of a dual pair) into the operand stages, slot
  // [i / S][rank].  Rows are 16-byte chunks XOR-swizzled by the row so a
  // quarter-warp's vector accesses of one chunk fall in distinct banks.
  static constexpr int ITEMS = 4 * (BN / 16);
  static constexpr int PW = 16 * NA;
  static __host__ __device__ constexpr int push_bytes(int S) {
    return ((ITEMS + S - 1) / S) * S * 32 * PW * 4;
  }
};

struct TcParams {
  int M, N, K, kb, tiles_m;
  long long units;
  EpiArgs epi;
  float* ws;
  int* counters;
  int* done;
  int* err;
  int tiles_n;  // weight tiles (128 output features each)
  // Tile t's weight tile and token tile: t / tiles_m and t % tiles_m, or
  // with m_major (stream-K over several token tiles) t % tiles_n and
  // t / tiles_n, the grid cut to a multiple of the live token tiles
  int m_major;
  int split_s;  // 0: stream-K over all units; >= 1: S CTAs (one cluster) per tile
  int a_heads;  // 0: weights by a 2-D map; else a 4-D interleaved QKV map, heads per tile
  int push;     // cluster split: 1 pushes each item's partials to its owner (st.async), 0 pulls them
  int pre_stages;  // weight stages loaded before the wait for the previous kernel (-1: all)
  int max_split;   // host side: the largest cluster split (2..8)
  // diagnostic timeline, or null: [cta][16] %globaltimer stamps (ns): [0]
  // start, [1] the producer's wait for the previous kernel returned, [2]
  // the first stage landed (MMA issuer), [3] the last MMA issued, [4] the
  // epilogue's main loop done, [5] every partial of the cluster ready, [8]
  // the partials of the first item summed, [7] this CTA's share of the
  // cluster reduction applied, [6] exit; pushed reduction: [5] every stage
  // of the cluster free, [8] this CTA's items received, [9] the first
  // item summed, [10] its epilogue done; stream-K: [13] the last partial
  // store began, [11] its contributor count taken, [12] the last fix-up
  // done, [14] the last whole tile's epilogue done
  unsigned long long* tl;
};
__device__ __forceinline__ void tc_stamp(const TcParams& p, int slot) {
  if (p.tl) p.tl[static_cast<size_t>(blockIdx.x) * 16 + slot] = global_timer_ns();
}

__device__ __forceinline__ long long unit_lo(int c, long long U, int G) {
  return static_cast<long long>(c) * U / G;
}
// The CTA whose unit range contains unit u.
__device__ __forceinline__ int cta_of_unit(long long u, long long U, int G) {
  int c = static_cast<int>((u * G) / U);
  if (c > G - 1) c = G - 1;
  while (c > 0 && unit_lo(c, U, G) > u) --c;
  while (c + 1 < G && unit_lo(c + 1, U, G) <= u) ++c;
  return c;
}

// Per-tile values the epilogue warps stage in shared memory while the
// mainloop runs (single token tile of at most 32 tokens; token t at [t]):
// the row scales of a folded RMSNorm, and for the fused RoPE epilogue the
// slots and rotary table (token t: cos at tab[t * dh + i], sin at
// tab[t * dh + dh / 2 + i]).  Null where unused.
struct EpiStaged {
  const float* rs;
  const float* tab;
  const int* slot;
};

// Apply the epilogue to 16 token columns [t0, t0 + 16) of output feature o.
// Called by all 32 lanes of a warp together (the argmax reduces across them).
// old_pre (ADD): the residual of these 16 tokens already loaded, then the
// next norm's gain of feature o (old_pre[16]), or null.
template <bool DUAL>
__device__ __forceinline__ void epi_chunk(const EpiArgs& e, int o, int t0, const float* v_in,
                                          const float* v2_in, int lane, const EpiStaged& sm,
                                          const float* old_pre = nullptr) {
  const float* rs = sm.rs;
  const bool of = o < e.N;
  float vs[16], vs2[16];
  const float* v = v_in;
  const float* v2 = v2_in;
  if (rs) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float r = t0 + j < 32 ? rs[t0 + j] : 1.f;
      vs[j] = v_in[j] * r;
      if (DUAL) vs2[j] = v2_in[j] * r;
    }
    v = vs;
    v2 = vs2;
  }
  switch (e.kind) {
    case EPI_STORE:
      if (e.row_map) {
        // rows through the map (fp32 output; the map is read-only while this
        // kernel runs, and all 16 entries are read before any store, so no
        // load waits behind a store it cannot be told apart from)
        float* out = static_cast<float*>(e.out);
        int tr[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) tr[j] = (of && t0 + j < e.M) ? __ldg(e.row_map + t0 + j) : -1;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (tr[j] >= 0) out[static_cast<size_t>(tr[j]) * e.ldo + o] = v[j];
      } else if (e.out_f32) {
        float* out = static_cast<float*>(e.out);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (of && t0 + j < e.M) out[static_cast<size_t>(t0 + j) * e.ldo + o] = v[j];
      } else {
        bf16* out = static_cast<bf16*>(e.out);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (of && t0 + j < e.M)
            out[static_cast<size_t>(t0 + j) * e.ldo + o] = __float2bfloat16_rn(v[j]);
      }
      break;
    case EPI_ADD: {
      // all 16 reads are issued before any write: written as `+=` in one
      // loop, each read would wait for the previous write (the compiler
      // cannot tell that the rows differ), one memory round trip per token
      float* r = e.resid + static_cast<size_t>(t0) * e.ldr + o;
      float old[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        old[j] = old_pre ? old_pre[j]
                         : (of && t0 + j < e.M) ? r[static_cast<size_t>(j) * e.ldr] : 0.f;
      const float gn = old_pre ? old_pre[16]
                       : (e.xg && of) ? __bfloat162float(static_cast<const bf16*>(e.g_next)[o])
                                      : 0.f;
      float sq[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float nv = old[j] + v[j];
        sq[j] = (of && t0 + j < e.M) ? nv * nv : 0.f;
        if (of && t0 + j < e.M) {
          r[static_cast<size_t>(j) * e.ldr] = nv;
          if (e.xg)
            static_cast<bf16*>(e.xg)[static_cast<size_t>(t0 + j) * e.ldxg + o] =
                __float2bfloat16_rn(nv * gn);
        }
      }
      if (e.ssq) {
        // sum of squares over the warp's 32 features for each of the 16
        // tokens: butterfly reduce-scatter (lane l ends with token
        // (l >> 1) & 15 over the lanes that differ in bits 1-4), then the
        // last pair; a fixed order, so deterministic
#pragma unroll
        for (int s = 16, L = 16; s >= 2; s >>= 1, L >>= 1) {
          const bool up = (lane & s) != 0;
#pragma unroll
          for (int i = 0; i < L / 2; ++i) {
            const float send = up ? sq[i] : sq[i + L / 2];
            const float keep = up ? sq[i + L / 2] : sq[i];
            sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
          }
        }
        const float tot = sq[0] + __shfl_xor_sync(0xffffffffu, sq[0], 1);
        const int t = t0 + ((lane >> 1) & 15);
        if ((lane & 1) == 0 && t < e.M) e.ssq[static_cast<size_t>(o >> 5) * e.ssq_ld + t] = tot;
      }
      break;
    }
    case EPI_SILU_MUL: {
      bf16* out = static_cast<bf16*>(e.out);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (of && t0 + j < e.M)
          out[static_cast<size_t>(t0 + j) * e.ldo + o] =
              __float2bfloat16_rn(silu_f(v[j]) * (DUAL ? v2[j] : 1.f));
      break;
    }
    case EPI_ROPE_KV: {
      // o is an interleaved row: row 2i + b of a head holds feature
      // i + b dh/2, so lanes 2i and 2i+1 hold a rotate-half pair
      const int half = e.dh >> 1, rel = o % e.dh, i = rel >> 1, b = rel & 1;
      const int f = (o - rel) + i + b * half;        // the feature in the standard layout
      const int qd = e.Hq * e.dh, kd = e.Hkv * e.dh;
      const int mlim = e.m_live ? min(e.M, __ldg(e.m_live)) : e.M;
      const bool rot = f < qd + kd;                  // q and k rotate, v does not (warp-uniform)
      // the projection's output is a bf16 activation: rounded before the
      // rotation (as when it goes through memory), then rotated in fp32
      float y[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float x = __bfloat162float(__float2bfloat16_rn(v[j]));
        const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
        y[j] = x;
        if (rot) {
          const int t = t0 + j < mlim ? t0 + j : 0;   // rows past the batch are not stored
          const float c = sm.tab[t * e.dh + i];
          const float s = sm.tab[t * e.dh + half + i];
          y[j] = b == 0 ? x * c - partner * s : x * c + partner * s;
        }
      }
      if (!of) break;
      if (f < qd) {
        bf16* q = static_cast<bf16*>(e.q_out);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (t0 + j < mlim) q[static_cast<size_t>(t0 + j) * qd + f] = __float2bfloat16_rn(y[j]);
      } else {
        const bool is_k = f < qd + kd;
        const int g = (f - (is_k ? qd : qd + kd)) / e.dh, jd = f % e.dh;
        void* cache = is_k ? e.k_cache : e.v_cache;
        const float inv = is_k ? e.k_inv_scale : e.v_inv_scale;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (t0 + j >= mlim) continue;
          const int sl = sm.slot[t0 + j];
          if (sl < 0) continue;                      // rejected row: no KV write
          const int blk = sl / 16, off = sl % 16;
          if (blk >= e.num_blocks) {
            if (jd == 0) record_error(e.err, PE_DEV_BAD_BLOCK);
            continue;
          }
          const size_t at = ((static_cast<size_t>(blk) * e.Hkv + g) * 16 + off) * e.dh + jd;
          if (e.kv_fp8)
            static_cast<uint8_t*>(cache)[at] =
                static_cast<uint8_t>(f32x2_to_e4m3x2(y[j] * inv, 0.f) & 0xffu);
          else
            static_cast<bf16*>(cache)[at] = __float2bfloat16_rn(y[j]);
        }
      }
      break;
    }
    case EPI_ARGMAX: {
      if (e.logits) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (of && t0 + j < e.M) e.logits[static_cast<size_t>(t0 + j) * e.ldl + o] = v[j];
      }
      // (value, feature) keys of this lane's feature for the 16 tokens
      unsigned long long k[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) k[j] = (of && t0 + j < e.M) ? argmax_key(v[j], o) : 0ull;
      // Butterfly reduce-scatter over the warp: with lane mask s = 16, 8,
      // 4, 2 a lane keeps half of its tokens (the upper half if its bit s
      // is set), trades the other half with lane ^ s and keeps the larger
      // keys.  Lane l then holds token (l >> 1) & 15, reduced over the 16
      // lanes that differ from it in bits 1-4; mask 1 finishes the warp.
      // 16 exchanges of 64-bit keys per 16 tokens instead of 5 per token.
#pragma unroll
      for (int s = 16, L = 16; s >= 2; s >>= 1, L >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < L / 2; ++i) {
          const unsigned long long send = up ? k[i] : k[i + L / 2];
          const unsigned long long keep = up ? k[i + L / 2] : k[i];
          const unsigned long long got = __shfl_xor_sync(0xffffffffu, send, s);
          k[i] = got > keep ? got : keep;
        }
      }
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, k[0], 1);
      const unsigned long long key = other > k[0] ? other : k[0];
      const int t = t0 + ((lane >> 1) & 15);
      if ((lane & 1) == 0 && t < e.M && key != 0ull) atomicMax(e.keys + t, key);
      break;
    }
  }
}

// Walk the BN accumulator columns of a TMEM lane quarter in 16-column
// chunks with the load of the next chunk in flight while fn(c0, v, v2)
// consumes the current one (the load latency is paid once, not per chunk).
template <int BN, bool DUAL, typename F>
__device__ __forceinline__ void tmem_walk(uint32_t taddr, F&& fn) {
  float a[16], a2[16], b[16], b2[16];
  tmem_ld16(taddr, a);
  if (DUAL) tmem_ld16(taddr + BN, a2);
  tmem_ld_wait();
  reg_fence16(a);
  if (DUAL) reg_fence16(a2);
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    const bool nb = c0 + 16 < BN;
    if (nb) {
      tmem_ld16(taddr + c0 + 16, b);
      if (DUAL) tmem_ld16(taddr + BN + c0 + 16, b2);
    }
    fn(c0, a, a2);
    if (nb) {
      tmem_ld_wait();
      reg_fence16(b);
      if (DUAL) reg_fence16(b2);
      const bool na = c0 + 32 < BN;
      if (na) {
        tmem_ld16(taddr + c0 + 32, a);
        if (DUAL) tmem_ld16(taddr + BN + c0 + 32, a2);
      }
      fn(c0 + 16, b, b2);
      if (na) {
        tmem_ld_wait();
        reg_fence16(a);
        if (DUAL) reg_fence16(a2);
      }
    }
  }
}

}  // namespace pe
