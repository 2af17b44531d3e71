// gemm_tc.cuh -- pieces of the tensor-core projection kernel (gemm_tc.cu:
// stream-K / cluster split-K, one CTA per tile): the tile configuration,
// the kernel parameters and the epilogue.
#pragma once

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
  static constexpr int STAGES_RAW = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(2 * STAGES + 5 <= BAR_BYTES / 8, "barrier space");
};

struct TcParams {
  int M, N, K, kb, tiles_m;
  long long units;
  EpiArgs epi;
  float* ws;
  int* counters;
  int* done;
  int* err;
  int split_s;  // 0: stream-K over all units; >= 1: S CTAs (one cluster) per tile
};

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

// Apply the epilogue to 16 token columns [t0, t0 + 16) of output feature o.
// Called by all 32 lanes of a warp together (the argmax reduces across them).
template <bool DUAL>
__device__ __forceinline__ void epi_chunk(const EpiArgs& e, int o, int t0, const float* v,
                                          const float* v2, int lane) {
  const bool of = o < e.N;
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
        old[j] = (of && t0 + j < e.M) ? r[static_cast<size_t>(j) * e.ldr] : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (of && t0 + j < e.M) r[static_cast<size_t>(j) * e.ldr] = old[j] + v[j];
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
