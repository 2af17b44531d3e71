// gemm_tc.cu -- the drafter's dense projections on 5th-generation tensor
// cores: y[t, o] = sum_k x[t, k] w[o, k] with bf16 operands and fp32
// accumulators in tensor memory (fc, QKV, O, gate/up, down, LM head; paper
// summary "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training",
// section 2: embedding + projected hidden state, N LLaMA layers, LM head).
//
// Layout: the weight rows are the MMA's M side (128 output features per
// tile) and the tokens its N side (16..256 per tile), so a batch of a few
// rows still fills the 128-lane accumulator.  Both operands are K-major and
// arrive by TMA in 128-byte-swizzled 64-wide k-blocks.
//
// Work split: persistent, one CTA per SM.  The (feature tile, token tile,
// k-block) units are dealt out in equal contiguous ranges ("stream-K"), so
// a 5120 x 2880 projection at batch 1 keeps all SMs streaming weights.  A
// tile split between CTAs is summed by its last-arriving CTA from fp32
// partials in a fixed order (deterministic, no float atomics, no waiting).
//
// Warp roles: warps 0-3 epilogue (TMEM lanes 0-127), warp 4 TMA producer,
// warp 5 MMA issuer and TMEM owner.  The producer loads the first weight
// tiles before waiting on the previous kernel (programmatic dependent
// launch), so weight streaming overlaps the previous kernel's tail.
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemm_tc.cuh"

namespace pe {

// Narrow token tiles: two CTAs per SM (at most 170 registers a thread), so
// the next kernel's CTA can start on an SM while this one drains.  From 64
// tokens on the stages fill the shared memory and one CTA runs per SM.
template <int BN, bool DUAL>
__global__ void __launch_bounds__(192, BN <= 32 ? 2 : 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p) {
  using C = TcCfg<BN, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain = acc_empty + 2;         // [1]
  uint64_t* recv_bar = drain + 1;          // [1] pushed cluster reduction: items received
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recv_bar + 1);
  volatile int* flag = reinterpret_cast<volatile int*>(tmem_slot + 1);     // reducer election
  volatile int* epi_ok = reinterpret_cast<volatile int*>(tmem_slot + 2);   // epilogue wait result
  float* rs_part = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES + C::RS_OFF);
  float* rs_smem = rs_part + 128;
  int* slot_smem = reinterpret_cast<int*>(rs_smem + 32);
  float* tab_smem = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES + C::TAB_OFF);
  EpiStaged staged;
  staged.rs = p.epi.rs_ssq ? rs_smem : nullptr;      // row scales of a folded RMSNorm
  staged.tab = tab_smem;                             // fused RoPE: rotary table, slots
  staged.slot = slot_smem;

  // Live token count of a compacted batch.  It was written two or more
  // launches back, so it is read before the wait, and its latency hides
  // behind the setup below.
  const int m_live = p.epi.m_live ? __ldcg(p.epi.m_live) : 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc_stamp(p, 0);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    mbar_init(drain, 1);
    mbar_init(recv_bar, 1);
    mbar_fence_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (DUAL) tma_prefetch_desc(&tmA2);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Dead token tiles (past the live count) are skipped: a cluster split
  // drops the clusters of dead tiles, stream-K deals the live units out
  // again.  With fewer live tiles than CTAs, every live tile gets the same
  // number of CTAs (an equal k-split, so each tile has a fixed number of
  // contributors) and the rest stay idle.  A dead CTA exits without waiting
  // on the previous kernel; token tile 0 is always live (every request
  // keeps its next-token row), so some CTA still waits before the grid lets
  // its dependents start.
  int tiles_m = p.tiles_m;
  const int tiles_n = p.tiles_n;
  const bool m_major = p.m_major != 0;
  // weight tile and token tile of tile t
  auto tile_f = [&](int t) { return m_major ? t % tiles_n : t / tiles_m; };
  auto tile_m = [&](int t) { return m_major ? t / tiles_n : t % tiles_m; };
  long long U = p.units;
  int G = gridDim.x;
  const int cta = blockIdx.x, kb = p.kb;
  bool dead = false;
  if (p.epi.m_live) {
    const int tm = (max(0, min(p.M, m_live)) + BN - 1) / BN;
    if (p.split_s >= 1) {
      dead = (cta / p.split_s) % p.tiles_m >= tm;  // the same for the whole cluster
    } else {
      tiles_m = tm;
      U = p.units / p.tiles_m * tm;
      const long long live_tiles = U / kb;
      if (live_tiles < G)
        G = live_tiles > 0 ? static_cast<int>(live_tiles * std::min<long long>(G / live_tiles, kb))
                           : 0;
      dead = cta >= G;
    }
  }
  if (m_major) {
    // Token-tile-major stream-K: the same number of CTAs for every live
    // token tile, so that CTA j of each token tile's group covers the same
    // k-blocks of the same weight tiles in the same order, all at once:
    // one read of a weight k-block from memory, the others from L2.
    const int g = G / tiles_m;
    G = g * tiles_m;
    dead = dead || cta >= G;
  }
  if (dead) {
    if (warp == 5) {
      tc_fence_after();
      tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    return;
  }

  long long lo, hi;
  if (p.split_s >= 1) {
    // cluster split: CTA s of the tile's cluster takes k-blocks
    // [s kb / S, (s + 1) kb / S) of that one tile
    const int S = p.split_s, tile = cta / S, sr = cta % S;
    lo = static_cast<long long>(tile) * kb + (static_cast<long long>(sr) * kb) / S;
    hi = static_cast<long long>(tile) * kb + (static_cast<long long>(sr + 1) * kb) / S;
  } else {
    lo = unit_lo(cta, U, G);
    hi = unit_lo(cta + 1, U, G);
  }

  if (warp == 4) {
    if (lane == 0) {
      const uint64_t pol_a = tiles_m == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_last();
      const long long n = hi - lo;
      // weight stages issued before the wait for the previous kernel
      const int pre_cap = p.pre_stages < 0 || p.pre_stages > C::STAGES ? C::STAGES : p.pre_stages;
      const int npre = static_cast<int>(n < pre_cap ? n : pre_cap);
      // weight tile f at k-block kk: a 2-D box, or the interleaved QKV box
      auto load_a = [&](uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int kk, int f) {
        if (p.a_heads) tma_load_4d(dst, m, bar, kk * 64, 0, 0, f * p.a_heads, pol_a);
        else tma_load_2d(dst, m, bar, kk * 64, f * 128, pol_a);
      };
      // weight tiles of the first stages do not depend on earlier kernels
      for (int i = 0; i < npre; ++i) {
        const long long u = lo + i;
        const int tile = static_cast<int>(u / kb), kk = static_cast<int>(u % kb);
        const int f = tile_f(tile);
        uint8_t* st = smem + i * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
        load_a(st, &tmA, &full[i], kk, f);
        if (DUAL) load_a(st + C::A_BYTES, &tmA2, &full[i], kk, f);
      }
      grid_dep_wait();
      tc_stamp(p, 1);
      // Dependents may launch once this CTA has waited for its own inputs;
      // TMEM is already held, so their allocation can only wait for this
      // grid to finish, never the other way round.
      grid_dep_launch();
      for (int i = 0; i < npre; ++i) {
        const long long u = lo + i;
        const int tile = static_cast<int>(u / kb), kk = static_cast<int>(u % kb);
        const int m = tile_m(tile);
        tma_load_2d(smem + i * C::STAGE_BYTES + C::NA * C::A_BYTES, &tmB, &full[i], kk * 64,
                    m * BN, pol_b);
      }
      long long issued = npre;
      for (long long i = npre; i < n; ++i) {
        const int stage = static_cast<int>(i % C::STAGES);
        const uint32_t round = static_cast<uint32_t>(i / C::STAGES);
        if (!mbar_wait(&empty[stage], (round - 1) & 1, p.err)) break;
        const long long u = lo + i;
        const int tile = static_cast<int>(u / kb), kk = static_cast<int>(u % kb);
        const int f = tile_f(tile), m = tile_m(tile);
        uint8_t* st = smem + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        load_a(st, &tmA, &full[stage], kk, f);
        if (DUAL) load_a(st + C::A_BYTES, &tmA2, &full[stage], kk, f);
        tma_load_2d(st + C::NA * C::A_BYTES, &tmB, &full[stage], kk * 64, m * BN, pol_b);
        issued = i + 1;
      }
      // drain: every copy this thread issued has landed before the CTA exits
      for (long long i = issued - 1; i >= 0 && i >= issued - C::STAGES; --i) {
        const int stage = static_cast<int>(i % C::STAGES);
        mbar_wait(&full[stage], static_cast<uint32_t>(i / C::STAGES) & 1, p.err);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      long long i = 0;
      int seg = 0;
      bool ok = true;
      for (long long u = lo; u < hi && ok;) {
        const int tile = static_cast<int>(u / kb);
        const int k_lo = static_cast<int>(u - static_cast<long long>(tile) * kb);
        const int k_hi = static_cast<int>(std::min<long long>(kb, k_lo + (hi - u)));
        const int acc = seg % C::NUM_ACC;
        const uint32_t around = static_cast<uint32_t>(seg / C::NUM_ACC);
        if (around > 0 && !mbar_wait(&acc_empty[acc], (around - 1) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * C::ACC_COLS;
        for (int kk = k_lo; kk < k_hi; ++kk, ++i) {
          const int stage = static_cast<int>(i % C::STAGES);
          if (!mbar_wait(&full[stage], static_cast<uint32_t>(i / C::STAGES) & 1, p.err)) {
            ok = false;
            break;
          }
          if (i == 0) tc_stamp(p, 2);
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::NA * C::A_BYTES;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint64_t bdesc = sw128_kmajor_desc(b_addr + k4 * 32);
            const uint32_t accum = (kk > k_lo || k4 > 0) ? 1u : 0u;
            umma_bf16(d, sw128_kmajor_desc(a_addr + k4 * 32), bdesc, C::IDESC, accum);
            if (DUAL)
              umma_bf16(d + BN, sw128_kmajor_desc(a_addr + C::A_BYTES + k4 * 32), bdesc,
                        C::IDESC, accum);
          }
          umma_commit(&empty[stage]);
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
        u += k_hi - k_lo;
        ++seg;
      }
      tc_stamp(p, 3);
      // drain: all MMAs of this thread are complete before TMEM is freed
      umma_commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else {
    grid_dep_wait();
    if (p.epi.rs_ssq) {
      // the folded RMSNorm's row scales of the (single) token tile, while
      // the mainloop runs: four slices of the 32-feature groups, summed in
      // a fixed order
      float* part = rs_part;
      const int t = threadIdx.x & 31, sl = threadIdx.x >> 5;
      float s = 0.f;
      if (t < p.M)
        for (int gr = sl; gr < p.epi.rs_groups; gr += 4)
          s += __ldcg(p.epi.rs_ssq + static_cast<size_t>(gr) * p.epi.rs_ld + t);
      part[sl * 32 + t] = s;
      named_bar_sync(1, 128);
      if (threadIdx.x < 32)
        rs_smem[t] = rsqrtf((((part[t] + part[32 + t]) + part[64 + t]) + part[96 + t]) /
                                p.epi.rs_d + p.epi.rs_eps);
      named_bar_sync(1, 128);
    }
    if (p.epi.kind == EPI_ROPE_KV) {
      // the tile's rotary table and slots (tokens of a live count past it
      // are never stored)
      const int mt = min(p.M, BN);
      for (int idx = threadIdx.x; idx < mt * p.epi.dh; idx += 128)
        tab_smem[idx] = __ldg(p.epi.rope_tab + idx);
      if (threadIdx.x < mt) slot_smem[threadIdx.x] = __ldg(p.epi.slot + threadIdx.x);
      named_bar_sync(1, 128);
    }
    int seg = 0;
    const int row = warp * 32 + lane;
    bool arrived = false;  // pushed cluster reduction: this thread's cluster-barrier arrival
    // Pushed cluster reduction with a residual-add epilogue: the residual
    // and gain of this warp's first item, when the item is this CTA's
    // (warp = rank mod S), loaded while the mainloop runs; at the end of
    // the kernel the memory system is busy with the next kernel's weights.
    float old_pre[17];
    bool pre = false;
    if (BN <= 32 && p.split_s >= 2 && p.push && p.epi.kind == EPI_ADD) {
      pre = warp % p.split_s == static_cast<int>(cluster_ctarank());
      if (pre) {
        const int tile = static_cast<int>(lo / kb);
        const int o = tile_f(tile) * 128 + row, t0 = tile_m(tile) * BN;
        const float* r = p.epi.resid + static_cast<size_t>(t0) * p.epi.ldr + o;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          old_pre[j] = (o < p.epi.N && t0 + j < p.epi.M) ? r[static_cast<size_t>(j) * p.epi.ldr] : 0.f;
        old_pre[16] = (p.epi.xg && o < p.epi.N)
                          ? __bfloat162float(static_cast<const bf16*>(p.epi.g_next)[o])
                          : 0.f;
      }
    }
    for (long long u = lo; u < hi;) {
      const int tile = static_cast<int>(u / kb);
      const int k_lo = static_cast<int>(u - static_cast<long long>(tile) * kb);
      const int k_hi = static_cast<int>(std::min<long long>(kb, k_lo + (hi - u)));
      const int acc = seg % C::NUM_ACC;
      const uint32_t around = static_cast<uint32_t>(seg / C::NUM_ACC);
      // one thread waits (bounded) and the outcome is shared, so the four
      // epilogue warps always take the same path through the barriers below
      if (threadIdx.x == 0) *epi_ok = mbar_wait(&acc_full[acc], around & 1, p.err) ? 1 : 0;
      named_bar_sync(1, 128);
      if (!*epi_ok) break;
      tc_fence_after();
      const int f = tile_f(tile), m = tile_m(tile);
      const int o = f * 128 + row;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * C::ACC_COLS;
      if (k_lo == 0 && k_hi == kb) {
        tmem_walk<BN, DUAL>(taddr, [&](int c0, const float* v, const float* v2) {
          epi_chunk<DUAL>(p.epi, o, m * BN + c0, v, v2, lane, staged);
        });
        if (threadIdx.x == 0) tc_stamp(p, 14);
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
      } else if (BN <= 32 && p.split_s >= 2 && p.push) {
        // Pushed cluster reduction.  This CTA's MMAs are complete, so its
        // operand stages are free: it arrives on the cluster barrier, and
        // once every CTA of the cluster has, it sends each item's partial
        // (read from TMEM) straight into the owner's stages with st.async,
        // counted on the owner's recv_bar.  The owner sums its items in
        // rank order (the same order as the pulled reduction).
        const int S = p.split_s;
        const int rk = static_cast<int>(cluster_ctarank());
        fence_proxy_async_smem();
        cluster_arrive_release();
        arrived = true;
        cluster_wait_acquire();
        if (threadIdx.x == 0) tc_stamp(p, 5);
        constexpr int NQ = C::PW / 4;   // 16-byte chunks of a row
        auto swz = [&](int q) { return NQ == 4 ? (q ^ ((lane >> 1) & 3)) : (q ^ (lane & 7)); };
        float* recv = reinterpret_cast<float*>(smem);
        const uint32_t bar_local = smem_u32(recv_bar);
        tmem_walk<BN, DUAL>(taddr, [&](int c0, const float* v, const float* v2) {
          const int item = (c0 / 16) * 4 + warp, owner = item % S;
          const int off = (((item / S) * S + rk) * 32 + lane) * C::PW;   // floats
          if (owner == rk) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              const float* s4 = q < 4 ? v + 4 * q : v2 + 4 * (q - 4);
              *reinterpret_cast<float4*>(recv + off + swz(q) * 4) = make_float4(s4[0], s4[1], s4[2], s4[3]);
            }
          } else {
            const uint32_t dst = cluster_map_shared(smem_u32(recv + off), owner);
            const uint32_t mb = cluster_map_shared(bar_local, owner);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              const float* s4 = q < 4 ? v + 4 * q : v2 + 4 * (q - 4);
              st_async_v4(dst + swz(q) * 16, s4[0], s4[1], s4[2], s4[3], mb);
            }
          }
        });
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
        int mine = 0;   // items of this CTA
        for (int i = rk; i < C::ITEMS; i += S) ++mine;
        if (threadIdx.x == 0 && mine > 0)
          mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(mine * (S - 1) * 32 * C::PW * 4));
        {
          bool any = false;
          for (int c0 = 0; c0 < BN; c0 += 16) any |= ((c0 / 16) * 4 + warp) % S == rk;
          // warp-uniform outcome: the epilogue below shuffles across lanes
          const bool got = __all_sync(0xffffffffu, any && mbar_wait(recv_bar, 0, p.err));
          if (got) {
            if (lane == 0 && warp == rk % 4) tc_stamp(p, 8);
            const bool stamp = lane == 0 && warp == rk % 4;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
              const int item = (c0 / 16) * 4 + warp;
              if (item % S != rk) continue;
              float v[16], v2[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = v2[j] = 0.f;
              const float* base = recv + ((item / S) * S * 32 + lane) * C::PW;
              // ranks in order; two ranks' loads in flight together (one
              // for a dual pair: registers)
              constexpr int RB = DUAL ? 1 : 2;
              for (int q = 0; q < S; q += RB) {
                float4 t[RB][NQ];
#pragma unroll
                for (int h = 0; h < RB; ++h)
#pragma unroll
                  for (int c = 0; c < NQ; ++c)
                    t[h][c] = q + h < S ? *reinterpret_cast<const float4*>(
                                              base + (q + h) * 32 * C::PW + swz(c) * 4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int h = 0; h < RB; ++h) {
                  if (q + h >= S) break;
#pragma unroll
                  for (int c = 0; c < NQ; ++c) {
                    float* d = c < 4 ? v + 4 * c : v2 + 4 * (c - 4);
                    d[0] += t[h][c].x;
                    d[1] += t[h][c].y;
                    d[2] += t[h][c].z;
                    d[3] += t[h][c].w;
                  }
                }
              }
              if (stamp && c0 == 0) tc_stamp(p, 9);
              epi_chunk<DUAL>(p.epi, o, m * BN + c0, v, v2, lane, staged,
                              pre && c0 == 0 ? old_pre : nullptr);
              if (stamp && c0 == 0) tc_stamp(p, 10);
            }
          }
        }
        if (threadIdx.x == 0) tc_stamp(p, 7);
      } else if (p.split_s >= 2) {
        // cluster split: the partial goes to this CTA's own shared memory
        // (the operand stages are all consumed); rank 0 sums the cluster's
        // partials after the cluster barrier below
        float* part = reinterpret_cast<float*>(smem) + row * C::PS;
        tmem_walk<BN, DUAL>(taddr, [&](int c0, const float* v, const float* v2) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            *reinterpret_cast<float4*>(part + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            if (DUAL)
              *reinterpret_cast<float4*>(part + BN + c0 + j) =
                  make_float4(v2[j], v2[j + 1], v2[j + 2], v2[j + 3]);
          }
        });
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
      } else {
        const int slot = (u == lo) ? 0 : 1;
        if (threadIdx.x == 0) tc_stamp(p, 13);
        float* wsp = p.ws + (static_cast<size_t>(cta) * 2 + slot) * (128 * C::ACC_COLS);
        tmem_walk<BN, DUAL>(taddr, [&](int c0, const float* v, const float* v2) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            wsp[(c0 + j) * 128 + row] = v[j];
            if (DUAL) wsp[(BN + c0 + j) * 128 + row] = v2[j];
          }
        });
        tc_fence_before();
        mbar_arrive(&acc_empty[acc]);
        __threadfence();
        named_bar_sync(1, 128);
        const int c_first = cta_of_unit(static_cast<long long>(tile) * kb, U, G);
        const int c_last = cta_of_unit(static_cast<long long>(tile + 1) * kb - 1, U, G);
        if (threadIdx.x == 0) {
          const int old = atomicAdd(p.counters + tile, 1);
          *flag = (old == c_last - c_first) ? 1 : 0;
          tc_stamp(p, 11);
        }
        named_bar_sync(1, 128);
        // Two contributors and this CTA's last segment (its stages are free,
        // its accumulator stays in TMEM): the other contributor's partial
        // comes into the stages in bulk copies, one round trip, and is added
        // to the accumulator read from TMEM, in contributor order.
        const bool last_seg = u + (k_hi - k_lo) >= hi;
        const size_t part_bytes = static_cast<size_t>(128) * C::ACC_COLS * 4;
        if (*flag && c_last - c_first == 1 && last_seg &&
            part_bytes <= static_cast<size_t>(C::STAGES) * C::STAGE_BYTES) {
          const int other = cta == c_first ? c_last : c_first;
          const int cs = unit_lo(other, U, G) >= static_cast<long long>(tile) * kb ? 0 : 1;
          const float* osrc = p.ws + (static_cast<size_t>(other) * 2 + cs) * (128 * C::ACC_COLS);
          float* ostage = reinterpret_cast<float*>(smem);
          if (threadIdx.x == 0) {
            __threadfence();
            fence_proxy_async_global();
            mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(part_bytes));
            for (size_t off = 0; off < part_bytes; off += 16384)
              bulk_copy_g2s(reinterpret_cast<uint8_t*>(ostage) + off,
                            reinterpret_cast<const uint8_t*>(osrc) + off,
                            static_cast<uint32_t>(part_bytes - off < 16384 ? part_bytes - off : 16384),
                            recv_bar);
          }
          // warp-uniform outcome (the epilogue below shuffles across lanes)
          const bool got = __all_sync(0xffffffffu, mbar_wait(recv_bar, 0, p.err));
          if (got) {
            const bool own_first = cta == c_first;
            tc_fence_after();
            tmem_walk<BN, DUAL>(taddr, [&](int c0, const float* v, const float* v2) {
              float w[16], w2[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float ot = ostage[(c0 + j) * 128 + row];
                w[j] = own_first ? (0.f + v[j]) + ot : (0.f + ot) + v[j];
                if (DUAL) {
                  const float ot2 = ostage[(BN + c0 + j) * 128 + row];
                  w2[j] = own_first ? (0.f + v2[j]) + ot2 : (0.f + ot2) + v2[j];
                } else {
                  w2[j] = 0.f;
                }
              }
              epi_chunk<DUAL>(p.epi, o, m * BN + c0, w, w2, lane, staged);
            });
          }
          if (threadIdx.x == 0) {
            p.counters[tile] = 0;
            tc_stamp(p, 12);
          }
          u += k_hi - k_lo;
          ++seg;
          continue;
        }
        // contributors the pipelined path holds in registers: a tile spans at
        // most three CTAs at the wide-tile shapes of the drafter (k-blocks
        // per tile below twice the k-blocks per CTA), two at the others;
        // none for the gate/up pair, whose two accumulators' partials would
        // spill registers across the whole kernel (its usual fix-up, a
        // finisher at the end of its range, takes the bulk-copy path)
        constexpr int NCM = DUAL ? 0 : (BN <= 64) ? 2 : 3;
        if (NCM > 0 && *flag && c_last - c_first < NCM) {
          // up to NCM contributors (the usual split): the loads of the next
          // chunk's partials are in flight while this chunk is summed (in
          // contributor order) and stored
          __threadfence();
          const int nc = c_last - c_first + 1;
          constexpr int NCA = NCM > 0 ? NCM : 1;
          const float* src[NCA];
#pragma unroll
          for (int q = 0; q < NCA; ++q) {
            const int cq = min(c_first + q, c_last);
            const int cs = unit_lo(cq, U, G) >= static_cast<long long>(tile) * kb ? 0 : 1;
            src[q] = p.ws + (static_cast<size_t>(cq) * 2 + cs) * (128 * C::ACC_COLS) + row;
          }
          constexpr int W = DUAL ? 32 : 16;  // values per contributor and chunk
          float xa[NCA][W], xb[NCA][W];
          auto load = [&](int c0, float (&x)[NCA][W]) {
#pragma unroll
            for (int q = 0; q < NCA; ++q)
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                x[q][j] = q < nc ? __ldcg(src[q] + (c0 + j) * 128) : 0.f;
                if (DUAL) x[q][16 + j] = q < nc ? __ldcg(src[q] + (BN + c0 + j) * 128) : 0.f;
              }
          };
          auto finish = [&](int c0, const float (&x)[NCA][W]) {
            float v[16], v2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = v2[j] = 0.f;
#pragma unroll
            for (int q = 0; q < NCA; ++q)
              if (q < nc)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  v[j] += x[q][j];
                  if (DUAL) v2[j] += x[q][16 + j];
                }
            epi_chunk<DUAL>(p.epi, o, m * BN + c0, v, v2, lane, staged);
          };
          load(0, xa);
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 32) {
            if (c0 + 16 < BN) load(c0 + 16, xb);
            finish(c0, xa);
            if (c0 + 16 < BN) {
              if (c0 + 32 < BN) load(c0 + 32, xa);
              finish(c0 + 16, xb);
            }
          }
          if (threadIdx.x == 0) {
            p.counters[tile] = 0;
            tc_stamp(p, 12);
          }
        } else if (*flag) {
          __threadfence();
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16], v2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = v2[j] = 0.f;
            // contributors in order; four at a time so their loads overlap
            constexpr int UNR = DUAL ? 2 : 4;
            for (int c = c_first; c <= c_last; c += UNR) {
              float t[UNR][16], t2[UNR][DUAL ? 16 : 1];
#pragma unroll
              for (int q = 0; q < UNR; ++q) {
                if (c + q > c_last) break;
                const int cq = c + q;
                const int cs = unit_lo(cq, U, G) >= static_cast<long long>(tile) * kb ? 0 : 1;
                const float* src = p.ws + (static_cast<size_t>(cq) * 2 + cs) * (128 * C::ACC_COLS);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  t[q][j] = __ldcg(src + (c0 + j) * 128 + row);
                  if (DUAL) t2[q][j] = __ldcg(src + (BN + c0 + j) * 128 + row);
                }
              }
#pragma unroll
              for (int q = 0; q < UNR; ++q) {
                if (c + q > c_last) break;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  v[j] += t[q][j];
                  if (DUAL) v2[j] += t2[q][j];
                }
              }
            }
            epi_chunk<DUAL>(p.epi, o, m * BN + c0, v, v2, lane, staged);
          }
          if (threadIdx.x == 0) {
            p.counters[tile] = 0;
            tc_stamp(p, 12);
          }
        }
      }
      u += k_hi - k_lo;
      ++seg;
    }
    // every thread of the cluster arrives once, also after an abort
    if (p.split_s >= 2 && p.push && !arrived) cluster_arrive_relaxed();
  }
  // the producer and MMA warps arrive for their CTA (they never wait)
  if (p.split_s >= 2 && p.push && warp >= 4) cluster_arrive_relaxed();

  if (threadIdx.x == 0) tc_stamp(p, 4);
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (p.split_s >= 2 && !p.push) {
    // Every CTA of the cluster has its partial in shared memory.  The sum
    // is scattered over the cluster: the tile's (32-row group, 16-column
    // chunk) items go round-robin to the S CTAs, and the warp of that row
    // group reads its item from all S partials with the loads of 8 columns
    // in flight together (two 16-byte DSMEM loads per partial, one round
    // trip per 8 columns), adds them in rank order (deterministic) and
    // applies the epilogue.  A residual-add epilogue's residual (untouched
    // by this kernel) is loaded before the cluster barrier, for one chunk.
    const int S = p.split_s, tile = cta / S;
    const int rk = static_cast<int>(cluster_ctarank());
    const int f = tile_f(tile), m = tile_m(tile);
    const int row = warp * 32 + lane;
    float old_pre[17];
    const bool pre = p.epi.kind == EPI_ADD && BN == 16 && warp < 4 && warp % S == rk;
    if (pre) {
      const int o = f * 128 + row, t0 = m * BN;
      const float* r = p.epi.resid + static_cast<size_t>(t0) * p.epi.ldr + o;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        old_pre[j] = (o < p.epi.N && t0 + j < p.epi.M) ? r[static_cast<size_t>(j) * p.epi.ldr] : 0.f;
      old_pre[16] = (p.epi.xg && o < p.epi.N)
                        ? __bfloat162float(static_cast<const bf16*>(p.epi.g_next)[o])
                        : 0.f;
    }
    cluster_sync_all();
    if (threadIdx.x == 0) tc_stamp(p, 5);
    if (warp < 4) {
      const uint32_t base = smem_u32(smem) + row * C::PS * 4;
      constexpr int kMaxS = 8;  // cluster split sizes are at most 8
      for (int c0 = 0; c0 < BN; c0 += 16) {
        if (((c0 / 16) * 4 + warp) % S != rk) continue;
        float v[16], v2[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = v2[j] = 0.f;
#pragma unroll
        for (int part = 0; part < (DUAL ? 4 : 2); ++part) {
          const int col = (part & 2 ? BN : 0) + c0 + (part & 1) * 8;
          float4 t[kMaxS][2];
#pragma unroll
          for (int q = 0; q < kMaxS; ++q) {
            if (q < S) {
              const uint32_t rb = cluster_map_shared(base, q) + col * 4;
              t[q][0] = ld_shared_cluster_v4(rb);
              t[q][1] = ld_shared_cluster_v4(rb + 16);
            }
          }
          float* dst = (part & 2 ? v2 : v) + (part & 1) * 8;
#pragma unroll
          for (int q = 0; q < kMaxS; ++q)
            if (q < S) {
              dst[0] += t[q][0].x;
              dst[1] += t[q][0].y;
              dst[2] += t[q][0].z;
              dst[3] += t[q][0].w;
              dst[4] += t[q][1].x;
              dst[5] += t[q][1].y;
              dst[6] += t[q][1].z;
              dst[7] += t[q][1].w;
            }
        }
        if (threadIdx.x == 0 && c0 == 0) tc_stamp(p, 8);
        epi_chunk<DUAL>(p.epi, f * 128 + row, m * BN + c0, v, v2, lane, staged,
                        pre && c0 == 0 ? old_pre : nullptr);
      }
    }
    if (threadIdx.x == 0) tc_stamp(p, 7);
    // every CTA keeps its shared memory until all of the cluster has read it
    cluster_sync_relaxed();
  }
  if (p.epi.kind == EPI_ARGMAX) {
    // the last CTA turns the packed (value, index) keys into token ids
    if (threadIdx.x == 0) {
      __threadfence();
      const int old = atomicAdd(p.done, 1);
      *flag = (old == G - 1) ? 1 : 0;
    }
    __syncthreads();
    if (*flag) {
      __threadfence();
      for (int t = threadIdx.x; t < p.epi.M; t += blockDim.x) {
        const unsigned long long k = atomicExch(p.epi.keys + t, 0ull);
        p.epi.tokens[t] = k ? argmax_key_index(k) : -1;
      }
      if (threadIdx.x == 0) *p.done = 0;
    }
  }
  if (threadIdx.x == 0) tc_stamp(p, 6);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

bool tensor_map_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                        uint64_t ld_elems, uint32_t box_cols, uint32_t box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || (ld_elems * 2) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tensor_map_qkv_interleaved(CUtensorMap* m, const void* ptr, int heads, int dh, uint64_t K) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || (K * 2) % 16 != 0 || dh <= 0 ||
      128 % dh != 0 || dh % 2 != 0)
    return false;
  const uint64_t half = static_cast<uint64_t>(dh / 2);
  // dims (innermost first): k, half index b, row within the half i, head
  cuuint64_t dims[4] = {K, 2, half, static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[3] = {half * K * 2, K * 2, static_cast<cuuint64_t>(dh) * K * 2};
  cuuint32_t box[4] = {64, 2, static_cast<cuuint32_t>(half), static_cast<cuuint32_t>(128 / dh)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of S CTAs (2..8) that can be resident at once, per
// instantiation and device, queried at init (0 when unknown).
constexpr int kMaxDev = 64;
template <int BN, bool DUAL>
int g_tc_clusters[kMaxDev][9];

template <int BN, bool DUAL>
int tc_max_clusters(int S) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  return g_tc_clusters<BN, DUAL>[dev][S];
}

template <int BN, bool DUAL>
static cudaError_t set_smem_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, DUAL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<BN, DUAL>::SMEM);
  int dev = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  for (int S = 2; S <= 8 && e == cudaSuccess; ++S) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 32);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = TcCfg<BN, DUAL>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, DUAL>, &cfg);
    g_tc_clusters<BN, DUAL>[dev][S] = n;
  }
  return e;
}

// Opt every instantiation into its dynamic shared memory (once per process
// and device, before any launch or stream capture).
cudaError_t init_gemm_tc() {
  cudaError_t e = cudaSuccess;
#define PE_TC_ATTR(BNV)                                            \
  if (e == cudaSuccess) e = set_smem_attr<BNV, false>();           \
  if (e == cudaSuccess) e = set_smem_attr<BNV, true>();
  PE_TC_ATTR(16)
  PE_TC_ATTR(32)
  PE_TC_ATTR(64)
  PE_TC_ATTR(128)
  PE_TC_ATTR(224)
  PE_TC_ATTR(256)
#undef PE_TC_ATTR
  return e;
}

size_t tc_partial_floats(int grid, int bn, bool dual);

template <int BN, bool DUAL>
static cudaError_t run_tc(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                          TcParams p, int tiles, long long units, int sm_count,
                          size_t partial_floats, cudaStream_t s) {
  using C = TcCfg<BN, DUAL>;
  // Fewer tiles than SMs: split k across a cluster of S CTAs per tile and
  // reduce through distributed shared memory.  Otherwise stream-K.
  const bool fits = static_cast<size_t>(C::PS) * 128 * 4 <=
                    static_cast<size_t>(C::STAGES) * C::STAGE_BYTES;
  // S CTAs a tile, about one CTA per SM in all (measured best in the
  // drafting step: with two CTAs an SM resident, the next kernel's CTAs
  // start beside these), at most 8 a tile and one k-block each; the whole
  // grid fits one wave (two CTAs an SM when the stages fit in about half
  // of the shared memory, otherwise one).
  const int per_sm = C::SMEM <= 113 * 1024 ? 2 : 1;
  int S = per_sm == 2 ? (sm_count + tiles / 2) / std::max(1, tiles) : sm_count / std::max(1, tiles);
  if (per_sm == 2) {
    // the next power of two, if the grid still fits two CTAs an SM
    int S2 = 1;
    while (S2 < S) S2 *= 2;
    if (tiles * S2 <= per_sm * sm_count) S = S2;
  }
  S = std::min(S, std::min(std::max(1, std::min(8, p.max_split)), p.kb));
  // One CTA an SM: clusters are placed whole within a GPC, so no more than
  // the resident-cluster count the runtime reports (a cluster left for a
  // second wave doubles the time; measured on 256-row projections).  With
  // two an SM that count measured too low, and the one-per-SM total fits.
  if (per_sm == 1)
    while (S >= 2 && tiles > tc_max_clusters<BN, DUAL>(S)) --S;
  if (tiles < sm_count && fits && (S >= 2 || per_sm == 2) && S >= 1 &&
      tiles * S <= per_sm * sm_count) {
    p.split_s = S;
    p.m_major = 0;   // one tile a cluster
    // the pushed reduction receives its items in the operand stages
    // (token tiles of at most 32; wider tiles pull)
    if (BN > 32 || C::push_bytes(S) > C::STAGES * C::STAGE_BYTES) p.push = 0;
    if (S == 1)
      return launch_pdl(gemm_tc_kernel<BN, DUAL>, dim3(tiles), dim3(192), C::SMEM, s, a, a2, b, p);
    return launch_pdl_cluster(gemm_tc_kernel<BN, DUAL>, dim3(tiles * S), dim3(192), C::SMEM, s, S,
                              a, a2, b, p);
  }
  p.split_s = 0;
  // as many CTAs as the SMs hold (two an SM for narrow token tiles: twice
  // the weight bytes in flight), within the caller's partial workspace
  const long long ws_ctas = static_cast<long long>(partial_floats / tc_partial_floats(1, BN, DUAL));
  const int grid = static_cast<int>(
      std::min<long long>(std::min<long long>(per_sm * sm_count, units), ws_ctas));
  if (grid < 1) return cudaErrorInvalidValue;
  return launch_pdl(gemm_tc_kernel<BN, DUAL>, dim3(grid), dim3(192), C::SMEM, s, a, a2, b, p);
}

// Token-tile width for M rows.  The gate/up pair (dual) stays at 128 from
// there on: at 256 its two accumulators fill the tensor memory (no overlap
// of the epilogue with the next tile) and its 64 KB stages leave room for
// three (measured 136 us against about 90 us at 128 on 896 x 15360 x 2880).
// Above 128 rows the others take ceil(M / 256) tiles of 224 tokens when
// they cover M (448 and 896 rows: no padded columns) and of 256 otherwise.
//
// (A 448-token tile -- two 224-token MMAs into one 448-column accumulator,
// so that the LM head at 448 rows streams each weight tile once -- measured
// slower: 495 us against about 445 us on 448 x 201088 x 2880.  One
// accumulator leaves the tensor cores idle during the argmax epilogue of
// every tile, and that kernel is bound by the tensor pipe, not by memory.)
int tc_pick_bn(int M, bool dual) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128 || dual) return 128;
  const int tm = (M + 255) / 256;
  return (M + tm - 1) / tm <= 224 ? 224 : 256;
}

// Rows of the token box in the x tensor map that launch_gemm_tc_maps
// expects for an M x N projection: the token tile.
int tc_b_box_rows(int M, int N, int sm_count, bool dual, bool live_rows) {
  (void)N;
  (void)sm_count;
  (void)live_rows;
  return tc_pick_bn(M, dual);
}

size_t tc_partial_floats(int grid, int bn, bool dual) {
  return static_cast<size_t>(grid) * 2 * 128 * bn * (dual ? 2 : 1);
}

cudaError_t launch_gemm_tc_maps(const CUtensorMap& wa, const CUtensorMap& wa2,
                                const CUtensorMap& xb, bool dual, int M, int N, int K,
                                const EpiArgs& epi, const TcGemmWorkspace& ws, int* err,
                                cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if ((epi.m_live && epi.kind == EPI_ARGMAX) || (epi.row_map && !epi.out_f32))
    return cudaErrorInvalidValue;
  const int bn = tc_pick_bn(M, dual);
  TcParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.kb = (K + 63) / 64;
  p.tiles_m = (M + bn - 1) / bn;
  const int tiles_n = (N + 127) / 128;
  p.units = static_cast<long long>(tiles_n) * p.tiles_m * p.kb;
  p.epi = epi;
  p.ws = ws.partials;
  p.counters = ws.tile_counters;
  p.done = ws.done_counter;
  p.err = err;
  const int tiles = tiles_n * p.tiles_m;
  p.tiles_n = tiles_n;
  // Token-tile-major where the weights cannot stay in L2 from one token
  // tile of a weight tile to the next (the LM head at a few hundred rows):
  // measured faster there, and slower for the layer projections, whose
  // weights (24-90 MB) L2 partly keeps between token tiles.  Stream-K only
  // (run_tc).
  // (At most one token tile an SM: the grid, at least the SM count here,
  // then holds one CTA a token tile or more.)
  p.m_major = ws.tile_order == 1 && p.tiles_m > 1 && p.tiles_m <= ws.sm_count &&
                      ws.l2_bytes > 0 && static_cast<long long>(N) * K * 2 > ws.l2_bytes
                  ? 1
                  : 0;
  p.split_s = 0;
  p.a_heads = 0;
  p.tl = ws.timeline;
  p.push = ws.cluster_push;
  p.pre_stages = ws.pre_stages;
  p.max_split = ws.max_split > 0 ? ws.max_split : 8;
  if (epi.kind == EPI_ROPE_KV) {
    // one token tile whose rotary table fits the staged [BN][64] floats
    if (dual || epi.dh <= 0 || 128 % epi.dh != 0 || N % 128 != 0 || M > bn || bn > 32 ||
        static_cast<long long>(M) * epi.dh > bn * 64 || epi.m_live)
      return cudaErrorInvalidValue;
    // the weight rows interleaved by a 4-D tensor map, unless the caller
    // gives an already interleaved copy (epi.rope_rows_interleaved)
    p.a_heads = epi.rope_rows_interleaved ? 0 : 128 / epi.dh;
  }
  // a folded RMSNorm: one token tile of at most 32 rows
  if ((epi.rs_ssq || epi.ssq) && (M > 32 || bn > 32 || epi.m_live)) return cudaErrorInvalidValue;
  if (tiles > ws.max_tiles) return cudaErrorInvalidValue;
#define PE_TC_CASE(BNV)                                                                       \
  case BNV:                                                                                   \
    return dual ? run_tc<BNV, true>(wa, wa2, xb, p, tiles, p.units, ws.sm_count,              \
                                    ws.partial_floats, s)                                     \
                : run_tc<BNV, false>(wa, wa2, xb, p, tiles, p.units, ws.sm_count,             \
                                     ws.partial_floats, s);
  switch (bn) {
    PE_TC_CASE(16)
    PE_TC_CASE(32)
    PE_TC_CASE(64)
    PE_TC_CASE(128)
    PE_TC_CASE(224)
    PE_TC_CASE(256)
  }
#undef PE_TC_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(const void* x, int ldx, const void* w, const void* w2, int M, int N,
                           int K, const EpiArgs& epi, const TcGemmWorkspace& ws, int* err,
                           cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  CUtensorMap wa, wa2, xb;
  if (!tensor_map_2d_bf16(&wa, w, N, K, K, 64, 128)) return cudaErrorInvalidValue;
  wa2 = wa;
  if (w2 && !tensor_map_2d_bf16(&wa2, w2, N, K, K, 64, 128)) return cudaErrorInvalidValue;
  if (!tensor_map_2d_bf16(&xb, x, M, K, ldx, 64, tc_b_box_rows(M, N, ws.sm_count, w2 != nullptr, epi.m_live != nullptr)))
    return cudaErrorInvalidValue;
  return launch_gemm_tc_maps(wa, wa2, xb, w2 != nullptr, M, N, K, epi, ws, err, s);
}

}  // namespace pe
