// gemm_mc.cu -- the tensor-core projection for many token tiles' worth of
// output (the LM head over a large batch): y[t, o] = sum_k x[t, k] w[o, k],
// bf16 operands, fp32 accumulators in tensor memory, the same epilogues as
// gemm_tc.cu.
//
// What it changes: a 128-feature x 256-token tile consumes 48 KB of
// operands per 64-wide k-block, 32 KB of them the token tile that every
// feature tile of the same tokens reads again.  Here CS CTAs of a
// thread-block cluster take CS neighbouring feature tiles of one token
// tile; each loads its own weight tile and 1/CS of the token tile, and the
// token slice goes by one TMA multicast into the same stage of every CTA of
// the cluster, so L2 delivers 16 KB of weights plus 32/CS KB of tokens per
// k-block and CTA.  On the LM head at 448-896 tokens, pairs are about 5%
// faster than one CTA per tile (gemm_tc.cu).  Token tiles of 224 or 256.
//
// Pipeline per CTA (warp roles as in gemm_tc.cu: warps 0-3 epilogue, warp 4
// TMA producer, warp 5 MMA issuer and TMEM owner):
//   full[s]  -- one arrival (this CTA's producer, expecting the weight tile
//               and the whole token tile) plus the bytes of all CS slices;
//   empty[s] -- CS arrivals, one multicast commit from the MMA issuer of
//               every CTA: a producer refills stage s of all CTAs, so it
//               waits until every one of them has consumed it.
// The CTAs of a cluster walk the same list of (feature group, token tile)
// pairs, so their k-block sequences stay in step.  Before exit the producer
// waits for the last release of every stage (no arrive from a peer is still
// on its way) and the cluster meets at a barrier.
#include "gemm_tc.cuh"

namespace pe {

template <int BN, bool DUAL, int CS>
__global__ void __launch_bounds__(192, 1)
    gemm_mc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p) {
  using C = TcCfg<BN, DUAL>;
  constexpr int SLICE_ROWS = BN / CS;
  constexpr int SLICE_BYTES = SLICE_ROWS * 128;  // 64 bf16 of k per token row
  static_assert(SLICE_ROWS % 8 == 0, "a slice is whole 8-row swizzle atoms");
  constexpr uint16_t ALL = static_cast<uint16_t>((1u << CS) - 1);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain = acc_empty + 2;         // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* flag = reinterpret_cast<volatile int*>(tmem_slot + 1);    // argmax finaliser
  volatile int* epi_ok = reinterpret_cast<volatile int*>(tmem_slot + 2);  // epilogue wait result

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    mbar_init(drain, 1);
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
  // peers multicast into this CTA's stages and arrive on its barriers: all
  // barriers of the cluster exist before anyone starts
  cluster_sync_all();

  // (feature group, token tile) pairs of this cluster: a contiguous range
  const int tiles_f = (p.N + 127) / 128;
  const long long groups = static_cast<long long>((tiles_f + CS - 1) / CS) * p.tiles_m;
  const int ncl = static_cast<int>(gridDim.x) / CS, cl = static_cast<int>(blockIdx.x) / CS;
  const long long g_lo = groups * cl / ncl, g_hi = groups * (cl + 1) / ncl;
  const int kb = p.kb;
  const long long n = (g_hi - g_lo) * kb;  // k-blocks of every CTA of the cluster

  if (warp == 4) {
    if (lane == 0) {
      const uint64_t pol_a = p.tiles_m == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_last();
      const int npre = static_cast<int>(n < C::STAGES ? n : C::STAGES);
      // weight tiles of the first stages do not depend on earlier kernels
      for (int i = 0; i < npre; ++i) {
        const long long g = g_lo + i / kb;
        const int kk = i % kb, f = static_cast<int>(g / p.tiles_m) * CS + rank;
        uint8_t* st = smem + i * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
        tma_load_2d(st, &tmA, &full[i], kk * 64, f * 128, pol_a);
        if (DUAL) tma_load_2d(st + C::A_BYTES, &tmA2, &full[i], kk * 64, f * 128, pol_a);
      }
      grid_dep_wait();
      grid_dep_launch();
      for (int i = 0; i < npre; ++i) {
        const long long g = g_lo + i / kb;
        const int kk = i % kb, m = static_cast<int>(g % p.tiles_m);
        tma_load_2d_mcast(smem + i * C::STAGE_BYTES + C::NA * C::A_BYTES + rank * SLICE_BYTES,
                          &tmB, &full[i], kk * 64, m * BN + rank * SLICE_ROWS, ALL, pol_b);
      }
      bool ok = true;
      for (long long i = npre; i < n; ++i) {
        const int stage = static_cast<int>(i % C::STAGES);
        const uint32_t round = static_cast<uint32_t>(i / C::STAGES);
        if (!mbar_wait(&empty[stage], (round - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        const long long g = g_lo + i / kb;
        const int kk = static_cast<int>(i % kb);
        const int f = static_cast<int>(g / p.tiles_m) * CS + rank, m = static_cast<int>(g % p.tiles_m);
        uint8_t* st = smem + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        tma_load_2d(st, &tmA, &full[stage], kk * 64, f * 128, pol_a);
        if (DUAL) tma_load_2d(st + C::A_BYTES, &tmA2, &full[stage], kk * 64, f * 128, pol_a);
        tma_load_2d_mcast(st + C::NA * C::A_BYTES + rank * SLICE_BYTES, &tmB, &full[stage],
                          kk * 64, m * BN + rank * SLICE_ROWS, ALL, pol_b);
      }
      // tail: the last use of every stage has been released by every CTA,
      // so no copy into this CTA and no arrive on its barriers is pending
      if (ok)
        for (long long i = n > C::STAGES ? n - C::STAGES : 0; i < n; ++i)
          if (!mbar_wait(&empty[i % C::STAGES], static_cast<uint32_t>(i / C::STAGES) & 1, p.err))
            break;
    }
  } else if (warp == 5) {
    if (lane == 0) {
      long long i = 0;
      int seg = 0;
      bool ok = true;
      for (long long g = g_lo; g < g_hi && ok; ++g, ++seg) {
        const int acc = seg % C::NUM_ACC;
        const uint32_t around = static_cast<uint32_t>(seg / C::NUM_ACC);
        if (around > 0 && !mbar_wait(&acc_empty[acc], (around - 1) & 1, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * C::ACC_COLS;
        for (int kk = 0; kk < kb; ++kk, ++i) {
          const int stage = static_cast<int>(i % C::STAGES);
          if (!mbar_wait(&full[stage], static_cast<uint32_t>(i / C::STAGES) & 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::NA * C::A_BYTES;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint64_t bdesc = sw128_kmajor_desc(b_addr + k4 * 32);
            const uint32_t accum = (kk > 0 || k4 > 0) ? 1u : 0u;
            umma_bf16(d, sw128_kmajor_desc(a_addr + k4 * 32), bdesc, C::IDESC, accum);
            if (DUAL)
              umma_bf16(d + BN, sw128_kmajor_desc(a_addr + C::A_BYTES + k4 * 32), bdesc,
                        C::IDESC, accum);
          }
          // stage consumed here: tell every CTA of the cluster
          umma_commit_mcast(&empty[stage], ALL);
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
      }
      // drain: all MMAs of this thread are complete before TMEM is freed
      umma_commit(drain);
      mbar_wait(drain, 0, p.err);
    }
  } else {
    grid_dep_wait();
    int seg = 0;
    const int row = warp * 32 + lane;
    for (long long g = g_lo; g < g_hi; ++g, ++seg) {
      const int acc = seg % C::NUM_ACC;
      const uint32_t around = static_cast<uint32_t>(seg / C::NUM_ACC);
      if (threadIdx.x == 0) *epi_ok = mbar_wait(&acc_full[acc], around & 1, p.err) ? 1 : 0;
      named_bar_sync(1, 128);
      if (!*epi_ok) break;
      tc_fence_after();
      const int f = static_cast<int>(g / p.tiles_m) * CS + rank, m = static_cast<int>(g % p.tiles_m);
      const int o = f * 128 + row;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * C::ACC_COLS;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16], v2[16];
        tmem_ld16(taddr + c0, v);
        if (DUAL) tmem_ld16(taddr + BN + c0, v2);
        tmem_ld_wait();
        reg_fence16(v);
        if (DUAL) reg_fence16(v2);
        epi_chunk<DUAL>(p.epi, o, m * BN + c0, v, v2, lane);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  cluster_sync_all();
  if (p.epi.kind == EPI_ARGMAX) {
    // the last CTA turns the packed (value, index) keys into token ids
    if (threadIdx.x == 0) {
      __threadfence();
      const int old = atomicAdd(p.done, 1);
      *flag = (old == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
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
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

constexpr int kMaxDev = 64;
// clusters of each instantiation that can be resident at once, per device
int g_max_clusters[kMaxDev][2];  // [device][token tile 224 / 256]
int bn_slot(int bn) { return bn == 224 ? 0 : 1; }

template <int BN, bool DUAL, int CS>
cudaError_t init_one(int dev) {
  using C = TcCfg<BN, DUAL>;
  cudaError_t e = cudaFuncSetAttribute(gemm_mc_kernel<BN, DUAL, CS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS * 64);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, gemm_mc_kernel<BN, DUAL, CS>, &cfg);
  if (e != cudaSuccess) return e;
  g_max_clusters[dev][bn_slot(BN)] = n;
  return cudaSuccess;
}

template <int BN, bool DUAL, int CS>
cudaError_t run_mc(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                   const TcParams& p, int dev, cudaStream_t s) {
  using C = TcCfg<BN, DUAL>;
  const int tiles_f = (p.N + 127) / 128;
  const long long groups = static_cast<long long>((tiles_f + CS - 1) / CS) * p.tiles_m;
  const int most = g_max_clusters[dev][bn_slot(BN)];
  const int ncl = static_cast<int>(std::min<long long>(groups, most));
  if (ncl < 1) return cudaErrorInvalidValue;
  return launch_pdl_cluster(gemm_mc_kernel<BN, DUAL, CS>, dim3(ncl * CS), dim3(192), C::SMEM, s,
                            CS, a, a2, b, p);
}

}  // namespace

cudaError_t init_gemm_mc() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
#define PE_MC_INIT(BNV, DV, CSV) \
  if (e == cudaSuccess) e = init_one<BNV, DV, CSV>(dev);
  PE_MC_INIT(224, false, 2)
  PE_MC_INIT(256, false, 2)
#undef PE_MC_INIT
  return e;
}

// Measured on the LM head (d 2880, vocab 201088): pairs sharing 256-token
// tiles gain about 5% at 448 and 896 tokens over one CTA per tile; clusters
// of 4 leave 8 SMs idle (36 resident clusters) and lose; for 128-token
// tiles the one-CTA kernel is faster.  So: pairs, for 224- and 256-token
// tiles, with at least four tiles per SM; the gate/up pair (dual) keeps
// gemm_tc.cu.
int gemm_mc_cluster(int bn, bool dual, long long tiles, int sm_count) {
  if ((bn != 224 && bn != 256) || dual) return 1;
  return tiles >= 4LL * sm_count ? 2 : 1;
}

cudaError_t launch_gemm_mc(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                           bool dual, int bn, int cs, const TcParams& p, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  if (dual) return cudaErrorInvalidValue;
#define PE_MC_CASE(BNV, CSV) \
  if (bn == BNV && cs == CSV) return run_mc<BNV, false, CSV>(a, a2, b, p, dev, s);
  PE_MC_CASE(224, 2)
  PE_MC_CASE(256, 2)
#undef PE_MC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pe
