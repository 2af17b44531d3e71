// attention_tc.cu -- paged causal attention of the drafting rows on 5th-gen
// tensor cores (bf16 operands, fp32 scores and accumulators in TMEM).
//
// Semantics (what the oracle states): each non-rejected row at position P
// attends key positions 0..P of its request through the block table; query
// head h reads kv head h / (Hq / Hkv); softmax of q.k / sqrt(dh); rejected
// rows (vLLM blog summary "P-EAGLE: Faster LLM Inference with Parallel
// Speculative Decoding in vLLM", KV-cache bullet) produce zeros.  The rows of
// one request are [accepted window rows, next-token row, MASK rows] (after
// the live-row compaction there are no rejected rows and is_rejected is
// null), so a shorter request's mask is the top-left block of a longer
// one's (paper summary "P-EAGLE: Parallel-Drafting EAGLE with Scalable
// Training", Fig. 3).
//
// Work unit (one CTA): request r, kv head g, a tile of up to 128 query rows
// (the request's rows x the g-th group of q heads -- GQA packs the group
// into the MMA's M side), and one split of the key range.  Per 128-key chunk:
//   S = Q K^T      (tcgen05, M=128 queries, N=128 keys, K=dh)
//   P = softmax    (8 warps: each query row is served by two threads, one per
//                   64-key half of the chunk; each half keeps its own running
//                   max (rescaling its O in TMEM only when the max grows past
//                   2^8), its own sum and its own O, combined once at the end)
//   O_h += P_h V_h (tcgen05, M=128, N=64 per half of dh, K=64 keys)
// S and P are double-buffered (S in TMEM, P in shared memory): S of the next
// chunk is computed while this chunk's softmax runs, and it needs only that
// every softmax warp has read the S two chunks back, so a slow warp never
// waits for the scores of its next chunk.  K and V pages come by TMA (16 keys x 64 dims per copy,
// 128-byte swizzle) into a 3-stage ring (2 for dh=128).  Splits of one
// (r, g, tile) are merged by the CTA that finishes last, in split order
// (deterministic).
#include <cudaTypedefs.h>

#include "fp8_common.cuh"
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

struct AttnTcParams {
  AttnArgs a;
  const int32_t* seq_lens;
  int G;             // q heads per kv head
  int rows_per_qt;   // request rows per query tile (128 / G)
  int qtiles;        // query tiles per request
  int split_keys;    // keys per split (multiple of 128)
  int max_splits;
  float* part;       // [B, Hkv, qtiles, max_splits, 128, dh + 2]
  int* counters;     // [2][B, Hkv, qtiles]: splits written, splits merged
  // 1: every split CTA merges its own slice of the unit's rows once all the
  // unit's splits are written (the grid is one wave, so they are all
  // resident); 0: the last split to finish merges the whole unit
  int parallel_merge;
  // K/V chunks brought into L2 ahead of the shared-memory ring: the first
  // l2_ahead before the wait for the previous kernel (the context pages do
  // not depend on it; L2 is where its new rows land, so nothing stale is
  // read), then chunk c + l2_ahead when chunk c is loaded; 0: none
  int l2_ahead;
  // longest work first, or null: the grid is (kv heads x query tiles,
  // B x max_splits) and CTA row y takes work item order[y] = request << 8 |
  // split (-1: none), the items sorted by their chunk count, most first
  const int32_t* order;
  // diagnostic timeline, or null: [cta][16] %globaltimer stamps (ns): [0]
  // start, [1] set up (barriers, tensor memory, block ids), [2] the wait
  // for the previous kernel returned, [3] Q in shared memory, [4] the first
  // scores ready, [5] the last P.V done, [6] the partial written, [7] every
  // split of the unit written, [10] the slice's partials in shared memory,
  // [11] the slice merged, [8] merged (after the barrier), [9] exit
  unsigned long long* tl;
};

__device__ __forceinline__ void attn_stamp(const AttnTcParams& p, int slot) {
  const unsigned cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  if (p.tl && cta < 448) p.tl[static_cast<size_t>(cta) * 16 + slot] = global_timer_ns();
}
// Per-chunk stamps of the CTAs of split 0, kv head 0, query tile 0 of the
// first two requests, chunks 0..31, after the 448 CTAs' stamps: [0] the
// chunk's K/V copies issued, [1] landed (MMA issuer), [2] S issued, [3] S
// seen by the softmax, [4] S in registers, [5] P stored, [6] P seen by the
// MMA issuer, [7] P.V issued; then, for the first request's CTA, every
// softmax warp's (S seen, P stored) per chunk.
__device__ __forceinline__ void attn_chunk_stamp(const AttnTcParams& p, int c, int slot) {
  if (p.tl && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z < 2 && c < 32)
    p.tl[448 * 16 + (blockIdx.z * 32 + c) * 8 + slot] = global_timer_ns();
}
__device__ __forceinline__ void attn_warp_stamp(const AttnTcParams& p, int c, int w, int slot) {
  if (p.tl && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && c < 32)
    p.tl[448 * 16 + 512 + c * 16 + w * 2 + slot] = global_timer_ns();
}

// FP8: the pools hold e4m3 codes.  Their pages come by TMA into a two-stage
// staging ring, the producer warp widens them to f16 in the K/V stages
// (every e4m3 value is an f16), and the MMAs run on f16 Q, K, V and P.
template <int DH, bool FP8 = false>
struct AttnCfg {
  static constexpr int NH = DH / 64;            // 64-wide halves of the head dim
  static constexpr int KEYS = 128;              // keys per chunk (two 64-key halves)
  static constexpr int TILE = 128 * 128;        // 128 rows x 128 B
  // K/V rings.  P lives in tensor memory (over the S columns it was
  // computed from), so shared memory holds Q and the rings only.  At dh
  // 128 K and V are separate rings: a K stage is free once S of its chunk
  // is computed, a V stage only once P.V has read it, so V is the deeper
  // ring (two K, four V stages).  At dh 64 one ring carries K and V of a
  // chunk together (six stages, four with the fp8 staging ring; split
  // rings measured 6 % slower there).
  static constexpr bool SPLIT = DH != 64;
  static constexpr int K_STAGES = DH == 64 ? (FP8 ? 4 : 6) : 2;
  static constexpr int V_STAGES = DH == 64 ? K_STAGES : 4;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NH * TILE;                 // [stage][NH]
  static constexpr int V_OFF = K_OFF + K_STAGES * NH * TILE;      // [stage][NH]
  static constexpr int RING_END = V_OFF + V_STAGES * NH * TILE;
  // Key slices of a chunk: each query row is served by NQ softmax threads,
  // one per KPW-key slice, each with its own running max, sum and O.  Two
  // slices (8 softmax warps); four (16 warps) measured no faster at dh 64.
  static constexpr int NQ = 2;
  static constexpr int KPW = KEYS / NQ;
  static constexpr int SOFT = 128 * NQ;          // softmax threads
  // float[2 NQ][128] for combining the slices; used only after the last
  // P.V has finished (every S, and so every read of Q, is done), so it
  // shares Q's space
  static constexpr int RED_OFF = Q_OFF;
  static constexpr int BAR_OFF = RING_END;
  // block ids of the CTA's pages, read once: a split covers at most
  // BT_ENTRIES pages of 16 keys (64 chunks at dh 64, 32 at dh 128, where
  // shared memory is full)
  static constexpr int BT_ENTRIES = DH == 64 ? 512 : 256;
  static constexpr int BT_OFF = BAR_OFF + 256;
  // fp8 staging: [stage][K pages 8 x 1 KB | V pages 8 x 1 KB]
  static constexpr int F8_STAGES = 2;
  static constexpr int F8_STAGE = 2 * 8 * 16 * DH;
  static constexpr int F8_OFF = (BT_OFF + BT_ENTRIES * 4 + 1023) / 1024 * 1024;
  static constexpr int SMEM = 1024 + (FP8 ? F8_OFF + F8_STAGES * F8_STAGE : BT_OFF + BT_ENTRIES * 4);
  // TMEM: two S buffers at columns 0..255 (S of chunk c in buffer c % 2);
  // O of key slice h at 256 + h * DH
  static constexpr int O_COL = 256;
  static constexpr int TMEM_COLS = 512;
  // fp8 pools: four warps widen the staged codes (one per scheduler)
  static constexpr int WIDEN_WARPS = FP8 ? 4 : 0;
  static constexpr int THREADS = 64 + SOFT + 32 * WIDEN_WARPS;  // producer, MMA, softmax, widening
  static constexpr uint32_t IDESC_S = FP8 ? idesc_f16_f32(128, 128) : idesc_bf16_f32(128, 128);
  static constexpr uint32_t IDESC_PV =
      FP8 ? idesc_f16_f32_bmn(128, 64) : idesc_bf16_f32_bmn(128, 64);
  static_assert(SMEM <= 232448, "shared memory");
  static_assert((2 * K_STAGES + (SPLIT ? 2 * V_STAGES : 0) + 18) * 8 <= 256, "barrier space");
  static_assert(SPLIT || K_STAGES == V_STAGES, "one ring");
  static_assert(!FP8 || DH == 64, "the fp8 pools are read at dh 64");
  static_assert(O_COL + NQ * DH <= TMEM_COLS && KPW % 16 == 0, "slices");
};

template <int DH, bool FP8 = false>
__global__ void __launch_bounds__(AttnCfg<DH, FP8>::THREADS, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnTcParams p) {
  using C = AttnCfg<DH, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // one ring (dh 64): the V barriers are the K barriers
  uint64_t* k_full = bars;                                              // [K_STAGES]
  uint64_t* k_empty = k_full + C::K_STAGES;                             // [K_STAGES]
  uint64_t* v_full = C::SPLIT ? k_empty + C::K_STAGES : k_full;         // [V_STAGES]
  uint64_t* v_empty = C::SPLIT ? v_full + C::V_STAGES : k_empty;        // [V_STAGES]
  uint64_t* q_ready = bars + 2 * C::K_STAGES + (C::SPLIT ? 2 * C::V_STAGES : 0);
  // [2] each: one per S buffer.  S(c + 2) reuses the buffer of S(c), so it
  // waits only until every softmax warp has read S(c): the next chunk's
  // scores are ready when the slowest warp gets to them.
  uint64_t* s_full = q_ready + 8;
  uint64_t* s_free = q_ready + 10;
  // [2]: one per P buffer.  The softmax warps are only loosely coupled: a
  // warp may finish chunk c + 1 while another still computes chunk c, so
  // the arrivals of consecutive chunks must land on different barriers (on
  // one shared barrier they would complete chunk c's phase early).  A warp
  // reaches chunk c + 2 only after every warp has read S(c + 1), so two
  // barriers suffice.
  uint64_t* p_full = q_ready + 3;
  uint64_t* pv_done = q_ready + 5;                // [2]: one per P buffer
  uint64_t* drain = q_ready + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_ready + 12);
  uint64_t* kv8_full = q_ready + 14;               // [2]: fp8 staging stages landed
  uint64_t* kv8_empty = q_ready + 16;              // [2]: fp8 staging stages widened
  volatile int* flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* red = reinterpret_cast<float*>(smem + C::RED_OFF);

  const AttnArgs& a = p.a;
  int split, g, qt, r;
  if (p.order) {
    g = blockIdx.x % a.Hkv;
    qt = blockIdx.x / a.Hkv;
    const int item = __ldg(p.order + blockIdx.y);   // written two or more launches back
    r = item >= 0 ? (item >> 8) : 0;
    split = item >= 0 ? (item & 255) : p.max_splits;  // past every sequence: no work
  } else {
    split = blockIdx.x;
    g = blockIdx.y % a.Hkv;
    qt = blockIdx.y / a.Hkv;
    r = blockIdx.z;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which rows and keys this CTA covers (uniform across the CTA) ------
  // The request offsets, sequence lengths, positions and block ids come
  // from the expansion (several launches back) or the caller, so they are
  // read, and the barriers and tensor memory set up, before the wait for
  // the previous kernel (which writes q and this step's K/V): that wait
  // sits right before the Q and K/V loads.
  if (threadIdx.x == 0) attn_stamp(p, 0);
  const int row0 = a.cu_out[r];
  const int nrows = a.cu_out[r + 1] - row0;
  const int tile_row0 = qt * p.rows_per_qt;
  const int tile_rows = min(p.rows_per_qt, nrows - tile_row0);
  if (qt == p.qtiles - 1 && split == 0 && g == 0 && threadIdx.x == 0 &&
      nrows > p.qtiles * p.rows_per_qt)
    record_error(a.err, PE_DEV_BAD_ROW);
  const int seq = p.seq_lens[r];
  const int key0 = split * p.split_keys;
  const int nsplits = (seq + p.split_keys - 1) / p.split_keys;
  if (tile_rows <= 0 || key0 >= seq || seq > a.bt_stride * 16) {
    if (threadIdx.x == 0 && seq > a.bt_stride * 16 && split == 0 && g == 0 && qt == 0)
      record_error(a.err, PE_DEV_BAD_POSITION);
    grid_dep_wait();
    grid_dep_launch();
    return;
  }
  const int key1 = min(seq, key0 + p.split_keys);
  const int nchunks = (key1 - key0 + C::KEYS - 1) / C::KEYS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::K_STAGES; ++i) {
      mbar_init(&k_full[i], FP8 ? C::WIDEN_WARPS : 1);   // fp8: one arrival a widening warp
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < (C::SPLIT ? C::V_STAGES : 0); ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(q_ready, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&s_free[0], C::SOFT);
    mbar_init(&s_free[1], C::SOFT);
    mbar_init(&p_full[0], C::SOFT);
    mbar_init(&p_full[1], C::SOFT);
    mbar_init(&pv_done[0], 1);
    mbar_init(&pv_done[1], 1);
    mbar_init(drain, 1);
    if (FP8) {
      mbar_init(&kv8_full[0], 1);
      mbar_init(&kv8_full[1], 1);
      mbar_init(&kv8_empty[0], C::WIDEN_WARPS);
      mbar_init(&kv8_empty[1], C::WIDEN_WARPS);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The block ids of all pages of [key0, key1), read by the whole warp in
    // one round trip (not one per chunk on the loads' critical path) and
    // checked here; -1 marks a bad id (recorded, its page not loaded).
    int* bt_s = reinterpret_cast<int*>(smem + C::BT_OFF);
    {
      const int32_t* bt = a.block_table + static_cast<size_t>(r) * a.bt_stride + (key0 >> 4);
      const int npages = (key1 - key0 + 15) >> 4;  // <= BT_ENTRIES (split size on the host)
      int v[C::BT_ENTRIES / 32];
#pragma unroll
      for (int k = 0; k < C::BT_ENTRIES / 32; ++k) {
        const int i = lane + 32 * k;
        v[k] = i < npages ? bt[i] : 0;
      }
#pragma unroll
      for (int k = 0; k < C::BT_ENTRIES / 32; ++k) {
        const int i = lane + 32 * k;
        if (i < npages) {
          int b = v[k];
          if (b < 0 || b >= a.num_blocks) {
            record_error(a.err, PE_DEV_BAD_BLOCK);
            b = -1;
          }
          bt_s[i] = b;
        }
      }
      __syncwarp();
    }
    if (lane == 0) attn_stamp(p, 1);
    // the pages of chunk c into L2 (valid block ids only)
    auto prefetch_chunk = [&](int c) {
      const int t0 = key0 + c * C::KEYS;
#pragma unroll
      for (int pg = 0; pg < 8; ++pg) {
        const int b = t0 + pg * 16 < key1 ? bt_s[c * 8 + pg] : -1;
        if (b < 0) continue;
        const int row = (b * a.Hkv + g) * 16;
#pragma unroll
        for (int h = 0; h < (FP8 ? 1 : C::NH); ++h) {
          tma_prefetch_l2_2d(&tmK, h * 64, row);
          tma_prefetch_l2_2d(&tmV, h * 64, row);
        }
      }
    };
    const int ahead = min(p.l2_ahead, nchunks);
    if (lane == 0)
      for (int c = 0; c < ahead; ++c) prefetch_chunk(c);
    grid_dep_wait();   // the previous kernel wrote this step's K/V
    if (lane == 0) attn_stamp(p, 2);
    if constexpr (!FP8) {
      // The page copies of a chunk go out from eight lanes at once (lane pg
      // takes page pg): one copy instruction for the warp instead of eight
      // issued one after another by one thread.  Lane 0 waits for the
      // stage and posts the byte count first.
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      const uint64_t pol = l2_policy_evict_first();
      int k_issued = 0, v_issued = 0;   // chunks whose copies went out
      for (int c = 0; c < nchunks; ++c) {
        const int ks = c % C::K_STAGES, kround = c / C::K_STAGES;
        const int vs = c % C::V_STAGES, vround = c / C::V_STAGES;
        const int t0 = key0 + c * C::KEYS;
        const int blk = (lane < 8 && t0 + lane * 16 < key1) ? bt_s[c * 8 + lane] : -1;
        const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, blk >= 0)) * C::NH * 2048u;
        const int row = (blk * a.Hkv + g) * 16;
        // K of the chunk once S of the chunk K_STAGES back is computed (one
        // ring: K and V once P.V of that chunk has read the stage)
        int ok0 = 1;
        if (lane == 0) {
          if (kround > 0 && !mbar_wait(&k_empty[ks], (kround - 1) & 1, a.err)) {
            ok0 = 0;
          } else {
            mbar_arrive_expect_tx(&k_full[ks], C::SPLIT ? bytes : 2 * bytes);
            attn_chunk_stamp(p, c, 0);
            if (ahead > 0 && c + ahead < nchunks) prefetch_chunk(c + ahead);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok0, 0)) break;
        k_issued = c + 1;
        if (!C::SPLIT) v_issued = c + 1;
        if (blk >= 0) {
#pragma unroll
          for (int h = 0; h < C::NH; ++h) {
            tma_load_2d(smem + C::K_OFF + (ks * C::NH + h) * C::TILE + lane * 2048, &tmK,
                        &k_full[ks], h * 64, row, pol);
            if (!C::SPLIT)
              tma_load_2d(smem + C::V_OFF + (ks * C::NH + h) * C::TILE + lane * 2048, &tmV,
                          &k_full[ks], h * 64, row, pol);
          }
        }
        if (C::SPLIT) {
          // V of the chunk once P.V of the chunk V_STAGES back has read it
          if (lane == 0) {
            if (vround > 0 && !mbar_wait(&v_empty[vs], (vround - 1) & 1, a.err)) ok0 = 0;
            else mbar_arrive_expect_tx(&v_full[vs], bytes);
          }
          if (!__shfl_sync(0xffffffffu, ok0, 0)) break;
          v_issued = c + 1;
          if (blk >= 0) {
#pragma unroll
            for (int h = 0; h < C::NH; ++h)
              tma_load_2d(smem + C::V_OFF + (vs * C::NH + h) * C::TILE + lane * 2048, &tmV,
                          &v_full[vs], h * 64, row, pol);
          }
        }
      }
      // drain: the copies of the last stages have landed before exit
      if (lane == 0) {
        for (int c = max(0, k_issued - C::K_STAGES); c < k_issued; ++c)
          mbar_wait(&k_full[c % C::K_STAGES], (c / C::K_STAGES) & 1, a.err);
        if (C::SPLIT)
          for (int c = max(0, v_issued - C::V_STAGES); c < v_issued; ++c)
            mbar_wait(&v_full[c % C::V_STAGES], (c / C::V_STAGES) & 1, a.err);
      }
    } else {
      // fp8 pages by TMA into a two-stage staging ring (eight lanes at once);
      // the widening warps turn each staged chunk into f16 rows of its K/V
      // stage (per chunk 2 x 8 pages x 16 keys x 4 groups of 16 codes) and
      // release the staging stage.
      uint8_t* f8 = smem + C::F8_OFF;
      const uint64_t pol = l2_policy_evict_first();
      // (the whole warp: lane pg < 8 copies page pg; lane 0 posts the bytes)
      auto issue8 = [&](int c) {
        const int s8 = c & 1;
        const int t0 = key0 + c * C::KEYS;
        const int blk = (lane < 8 && t0 + lane * 16 < key1) ? bt_s[c * 8 + lane] : -1;
        const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, blk >= 0)) * 2u * 16u * DH;
        if (lane == 0) mbar_arrive_expect_tx(&kv8_full[s8], bytes);
        __syncwarp();
        if (blk >= 0) {
          const int row = (blk * a.Hkv + g) * 16;
          uint8_t* base = f8 + s8 * C::F8_STAGE + lane * 16 * DH;
          tma_load_2d(base, &tmK, &kv8_full[s8], 0, row, pol);
          tma_load_2d(base + 8 * 16 * DH, &tmV, &kv8_full[s8], 0, row, pol);
        }
      };
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      int issued = 0;
      for (int c = 0; c < nchunks; ++c) {
        if (c >= C::F8_STAGES) {
          // the staging stage is free once every widening warp has read it
          int ok0 = 1;
          if (lane == 0 &&
              !mbar_wait(&kv8_empty[c & 1], ((c - C::F8_STAGES) >> 1) & 1, a.err))
            ok0 = 0;
          if (!__shfl_sync(0xffffffffu, ok0, 0)) break;
        }
        issue8(c);
        issued = c + 1;
        if (lane == 0 && ahead > 0 && c + ahead < nchunks) prefetch_chunk(c + ahead);
      }
      // drain: the last staging copies have landed before the CTA exits
      if (lane == 0)
        for (int c = max(0, issued - C::F8_STAGES); c < issued; ++c)
          mbar_wait(&kv8_full[c & 1], (c >> 1) & 1, a.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(smem + C::Q_OFF);
      // S(c) = Q K(c)^T into TMEM columns (c & 1) * 128 .. + 127
      auto issue_s = [&](int c) {
        const int ks = c % C::K_STAGES;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + C::K_OFF + ks * C::NH * C::TILE);
#pragma unroll
        for (int h = 0; h < C::NH; ++h)
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            umma_bf16(tmem + (c & 1) * 128, sw128_kmajor_desc(q_addr + h * C::TILE + k4 * 32),
                      sw128_kmajor_desc(k_addr + h * C::TILE + k4 * 32), C::IDESC_S,
                      (h | k4) != 0);
        umma_commit(&s_full[c & 1]);
        if (C::SPLIT) umma_commit(&k_empty[ks]);  // K(c) is read once S(c) is done
        attn_chunk_stamp(p, c, 2);
      };
      // O_h += P(keys of slice h) V(keys of slice h), per 64-wide part of
      // dh; P comes from tensor memory: slice h's probabilities, packed two
      // to a column, over the first half of its own S columns (the A
      // operand of a 16-key step is 8 columns)
      auto issue_pv = [&](int c) {
        tc_fence_after();
        const int vs = c % C::V_STAGES;
        const uint32_t v_addr = smem_u32(smem + C::V_OFF + vs * C::NH * C::TILE);
#pragma unroll
        for (int sl = 0; sl < C::NQ; ++sl)
#pragma unroll
          for (int k = 0; k < C::KPW / 16; ++k) {
            const int kk = sl * C::KPW + k * 16;     // first key of this step
            const uint32_t a_tmem = tmem + (c & 1) * 128 + sl * C::KPW + k * 8;
#pragma unroll
            for (int j = 0; j < C::NH; ++j)
              umma_f16_ts(tmem + C::O_COL + sl * DH + j * 64, a_tmem,
                          sw128_mnmajor_desc(v_addr + j * C::TILE + kk * 128), C::IDESC_PV,
                          (c > 0 || k > 0) ? 1u : 0u);
          }
        umma_commit(&v_empty[vs]);
        umma_commit(&pv_done[c & 1]);
        attn_chunk_stamp(p, c, 7);
      };
      // S(c) needs chunk c's K and, from c = 2 on, the softmax's read of
      // S(c - 2) (its buffer); P.V(c) needs P(c) and chunk c's V.  One
      // thread polls both and
      // issues whichever is ready -- S first, and S at most one chunk ahead
      // of P.V (P.V is on the softmax's critical path) -- so that P.V(c)
      // never waits for chunk c + 1's copy.  A bounded poll: no progress
      // for kWaitTimeoutNs records PE_DEV_TIMEOUT and stops.
      bool ok = mbar_wait(q_ready, 0, a.err);
      int cs = 0, cp = 0;            // next S, next P.V
      unsigned long long idle_since = 0;
      while (ok && cp < nchunks) {
        bool did = false;
        if (cs < nchunks && cs <= cp + 1 &&
            mbar_test_wait(&k_full[cs % C::K_STAGES], (cs / C::K_STAGES) & 1) &&
            (cs < 2 || mbar_test_wait(&s_free[cs & 1], ((cs - 2) >> 1) & 1))) {
          attn_chunk_stamp(p, cs, 1);
          issue_s(cs);
          ++cs;
          did = true;
        }
        if (cp < cs && mbar_test_wait(&p_full[cp & 1], (cp >> 1) & 1) &&
            mbar_test_wait(&v_full[cp % C::V_STAGES], (cp / C::V_STAGES) & 1)) {
          attn_chunk_stamp(p, cp, 6);
          issue_pv(cp);
          ++cp;
          did = true;
        }
        if (did) {
          idle_since = 0;
        } else {
          // idle: yield the scheduler to the softmax warps that share it
          __nanosleep(64);
          if (idle_since == 0) {
            idle_since = global_timer_ns();
          } else if (global_timer_ns() - idle_since > kWaitTimeoutNs) {
            record_error(a.err, PE_DEV_TIMEOUT);
            ok = false;
          }
        }
      }
      umma_commit(drain);
      mbar_wait(drain, 0, a.err);
    }
  } else if (warp >= 2 + C::SOFT / 32) {
    // ------------------------------------------------------------ widening
    // (fp8 pools) The staged e4m3 codes of a chunk become f16 rows of its
    // K/V stage, a quarter of the 16-byte groups a warp (warps 0-1 of the
    // four: K, 2-3: V); each warp releases the staging stage and arrives on
    // the chunk's K/V barrier (one arrival a warp).  Keys past the split
    // (and pages whose block id was bad) become zeros, so no stale value
    // reaches S or O.
    if constexpr (FP8) {
      const int wi = warp - (2 + C::SOFT / 32);
      uint8_t* f8 = smem + C::F8_OFF;
      // the split's block ids (written by the producer warp before its
      // first copy; the staging barrier's phase orders them before here)
      const int* bt_s = reinterpret_cast<const int*>(smem + C::BT_OFF);
      for (int c = 0; c < nchunks; ++c) {
        const int s8 = c & 1;
        const int ks = c % C::K_STAGES, kround = c / C::K_STAGES;
        const int vs = ks;   // one ring at dh 64
        // every lane waits (each needs the barrier's acquire); the outcome is
        // made warp-uniform so the lanes leave together
        if (!__all_sync(0xffffffffu, mbar_wait(&kv8_full[s8], (c >> 1) & 1, a.err))) break;
        if (kround > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&k_empty[ks], (kround - 1) & 1, a.err)))
          break;
        const int t0 = key0 + c * C::KEYS;
        const uint8_t* src = f8 + s8 * C::F8_STAGE;
#pragma unroll 4
        for (int k = wi * 8; k < wi * 8 + 8; ++k) {
          const int item = lane + 32 * k;
          const int which = item >> 9, pg = (item >> 6) & 7, kr = (item >> 2) & 15, q4 = item & 3;
          const int kk = pg * 16 + kr;                 // key within the chunk
          uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
          if (t0 + kk < key1 && bt_s[c * 8 + pg] >= 0) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + which * 8 * 16 * DH +
                                                            pg * 16 * DH + kr * DH + q4 * 16);
            lo = make_uint4(e4m3x2_to_f16x2(x.x), e4m3x2_to_f16x2(x.x >> 16),
                            e4m3x2_to_f16x2(x.y), e4m3x2_to_f16x2(x.y >> 16));
            hi = make_uint4(e4m3x2_to_f16x2(x.z), e4m3x2_to_f16x2(x.z >> 16),
                            e4m3x2_to_f16x2(x.w), e4m3x2_to_f16x2(x.w >> 16));
          }
          // row kk of the 128-byte-swizzled stage: dims q4*16 .. +15 are its
          // 16-byte chunks 2 q4 and 2 q4 + 1
          uint8_t* dst = smem + (which ? C::V_OFF + vs * C::TILE : C::K_OFF + ks * C::TILE) + kk * 128;
          *reinterpret_cast<uint4*>(dst + (((2 * q4) ^ (kk & 7)) * 16)) = lo;
          *reinterpret_cast<uint4*>(dst + (((2 * q4 + 1) ^ (kk & 7)) * 16)) = hi;
        }
        fence_proxy_async_smem();   // the stage's f16 rows, for the MMA's reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&kv8_empty[s8]);
          mbar_arrive(&k_full[ks]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // NQ warps per TMEM lane quarter: slice h takes keys h*KPW..h*KPW+KPW-1
    // of every chunk and runs its own online softmax into its own O
    const int qrow = 32 * (warp & 3) + lane;
    const int h = (warp - 2) >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int lr = qrow / p.G, hl = qrow % p.G;
    const bool in_tile = lr < tile_rows;
    const int row = row0 + tile_row0 + lr;          // expanded row
    const int head = g * p.G + hl;
    int P = -1;                                     // last key this row reads
    if (in_tile && (a.is_rejected == nullptr || a.is_rejected[row] == 0)) P = a.pos[row];
    grid_dep_wait();   // the previous kernel wrote q
    // Q -> shared memory (128-byte swizzle; zero for padding / rejected rows)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const bf16*>(a.q) + (static_cast<size_t>(row) * a.Hq + head) * DH);
#pragma unroll
      for (int i = 0; i < 8 * C::NH / C::NQ; ++i) {
        const int ch = h * (8 * C::NH / C::NQ) + i;
        const int tl = ch >> 3, cc = ch & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (P >= 0) v = src[ch];
        if (FP8)  // the MMAs run on f16 operands
          v = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                         bf16x2_to_f16x2(v.w));
        *reinterpret_cast<uint4*>(smem + C::Q_OFF + tl * C::TILE + qrow * 128 +
                                  ((cc ^ (qrow & 7)) * 16)) = v;
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, C::SOFT);
    if (threadIdx.x == 64) {
      mbar_arrive(q_ready);
      attn_stamp(p, 3);
    }

    // log2(e) / sqrt(dh), times the K scale of an fp8 pool (S holds
    // q . code; the score is q . code * k_scale)
    const float sc = a.scale * 1.4426950408889634f * (FP8 ? a.k_scale : 1.f);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    const uint32_t o_col = C::O_COL + h * DH;
    // rows that read no key of this split (padding, rejected, or a position
    // before the split): P rows of zeros, l = 0
    const bool dead = P < key0;
    const bool warp_dead = __all_sync(0xffffffffu, dead);
    for (int c = 0; c < nchunks; ++c) {
      if (!mbar_wait(&s_full[c & 1], (c >> 1) & 1, a.err)) { ok = false; break; }
      if (c == 0 && threadIdx.x == 64) attn_stamp(p, 4);
      if (threadIdx.x == 64) attn_chunk_stamp(p, c, 3);
      if (lane == 0) attn_warp_stamp(p, c, warp - 2, 0);
      tc_fence_after();
      constexpr int KPW = C::KPW;
      uint32_t pk[KPW / 2];
      float factor = 1.f;
      if (warp_dead) {
        // no row of this warp reads a key of this split: its P rows are
        // zeros, nothing else to compute
        tc_fence_before();
        mbar_arrive(&s_free[c & 1]);
#pragma unroll
        for (int j = 0; j < KPW / 2; ++j) pk[j] = 0u;
      } else {
        float sv[KPW / 16][16];
#pragma unroll
        for (int q = 0; q < KPW / 16; ++q)
          tmem_ld16(tmem + lane_off + (c & 1) * 128 + h * KPW + q * 16, sv[q]);
        tmem_ld_wait();
        if (threadIdx.x == 64) attn_chunk_stamp(p, c, 4);
#pragma unroll
        for (int q = 0; q < KPW / 16; ++q) reg_fence16(sv[q]);
        const float* s = &sv[0][0];
        tc_fence_before();
        mbar_arrive(&s_free[c & 1]);                  // this S buffer may be reused
        const int tb = key0 + c * C::KEYS + h * KPW;  // first key of this slice
        // no masking inside the slice for any row of the warp (one path for
        // the warp: a row with no key of the split counts as unmasked, its
        // probabilities are replaced by zeros below)
        const bool whole = __all_sync(0xffffffffu, dead || tb + KPW - 1 <= P);
        // masked maximum (four independent chains)
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (whole) {
          // two scores per instruction in each of the four chains
#pragma unroll
          for (int j = 0; j < KPW; j += 8) {
            m4[0] = fmax3(m4[0], s[j], s[j + 1]);
            m4[1] = fmax3(m4[1], s[j + 2], s[j + 3]);
            m4[2] = fmax3(m4[2], s[j + 4], s[j + 5]);
            m4[3] = fmax3(m4[3], s[j + 6], s[j + 7]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < KPW; ++j)
            if (tb + j <= P) m4[j & 3] = fmaxf(m4[j & 3], s[j]);
        }
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sc;  // sc > 0
        // lazy rescale: keep the old reference unless the max grew past 2^8
        float m_new = m_used;
        if (mx > -INFINITY && !dead) {
          if (m_used == -INFINITY) m_new = mx;
          else if (mx > m_used + 8.f) {
            m_new = mx;
            factor = fast_exp2(m_used - mx);
          }
        }
        // probabilities: one FFMA and one MUFU.EX2 a score; the row sum is
        // kept in fp32 (two chains), P goes to the MMA as bf16 pairs (f16
        // with fp8 pools)
        float ps0 = 0.f, ps1 = 0.f;
        const float nm = -m_new;
        if (whole) {
#pragma unroll
          for (int j = 0; j < KPW; j += 2) {
            const float p0 = fast_exp2(fmaf(s[j], sc, nm));
            const float p1 = fast_exp2(fmaf(s[j + 1], sc, nm));
            ps0 += p0;
            ps1 += p1;
            pk[j / 2] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
          if (dead) {
#pragma unroll
            for (int j = 0; j < KPW / 2; ++j) pk[j] = 0u;
            ps0 = ps1 = 0.f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < KPW; j += 2) {
            const float e0 = fast_exp2(fmaf(s[j], sc, nm));
            const float e1 = fast_exp2(fmaf(s[j + 1], sc, nm));
            const float p0 = (tb + j <= P) ? e0 : 0.f;
            const float p1 = (tb + j + 1 <= P) ? e1 : 0.f;
            ps0 += p0;
            ps1 += p1;
            pk[j / 2] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
        }
        const float psum = ps0 + ps1;
        l = l * factor + psum;
        m_used = m_new;
      }
      // O must hold every earlier chunk before it is rescaled
      if (c >= 1 && __any_sync(0xffffffffu, factor != 1.f)) {
        if (!mbar_wait(&pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1, a.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 16) {
          float o[16];
          tmem_ld16(tmem + lane_off + o_col + c0, o);
          tmem_ld_wait();
          reg_fence16(o);
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] *= factor;
          tmem_st16(tmem + lane_off + o_col + c0, o);
        }
        tmem_st_wait();
      }
      // P row of this slice -> tensor memory, over the first half of the
      // slice's own S columns (this thread has read them; the next S into
      // this buffer, of chunk c + 2, is issued after P.V of chunk c, and
      // the tensor pipe runs them in order)
      {
        const uint32_t pcol = tmem + lane_off + (c & 1) * 128 + h * KPW;
#pragma unroll
        for (int q = 0; q < KPW / 32; ++q) tmem_st16u(pcol + q * 16, pk + q * 16);
        tmem_st_wait();
      }
      // keys past the sequence end: zero their V rows so 0 * garbage cannot
      // reach O (the pool may hold anything there)
      const int t0 = key0 + c * C::KEYS;
      if (h == 0 && t0 + C::KEYS > key1 && t0 + qrow >= key1) {
        // (after the chunk's V copies have landed, so none lands on top)
        const int vs = c % C::V_STAGES;
        if (!mbar_wait(&v_full[vs], (c / C::V_STAGES) & 1, a.err)) ok = false;
#pragma unroll
        for (int j = 0; j < C::NH; ++j) {
          uint4* vr = reinterpret_cast<uint4*>(smem + C::V_OFF + (vs * C::NH + j) * C::TILE +
                                               qrow * 128);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) vr[cc] = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[c & 1]);
      if (threadIdx.x == 64) attn_chunk_stamp(p, c, 5);
      if (lane == 0) attn_warp_stamp(p, c, warp - 2, 1);
    }
    if (ok && !mbar_wait(&pv_done[(nchunks - 1) & 1], ((nchunks - 1) >> 1) & 1, a.err)) ok = false;
    if (threadIdx.x == 64) attn_stamp(p, 5);
    if (!ok) *abort_flag = 1;
    // combine the slices: (m, l) through shared memory
    red[h * 128 + qrow] = m_used;
    red[(C::NQ + h) * 128 + qrow] = l;
    named_bar_sync(1, C::SOFT);
    if (!*abort_flag) {
      tc_fence_after();
      float mi[C::NQ], wi[C::NQ];
      float M = -INFINITY;
#pragma unroll
      for (int i = 0; i < C::NQ; ++i) {
        mi[i] = red[i * 128 + qrow];
        M = fmaxf(M, mi[i]);
      }
      float L = 0.f;
#pragma unroll
      for (int i = 0; i < C::NQ; ++i) {
        wi[i] = mi[i] > -INFINITY ? exp2f(mi[i] - M) : 0.f;
        L += red[(C::NQ + i) * 128 + qrow] * wi[i];
      }
      // this thread finishes columns h*HC .. h*HC + HC - 1 of its row
      constexpr int HC = DH / C::NQ;
      float o[HC];
#pragma unroll
      for (int c0 = 0; c0 < HC; c0 += 16) {
        float x[C::NQ][16];
#pragma unroll
        for (int i = 0; i < C::NQ; ++i)
          tmem_ld16(tmem + lane_off + C::O_COL + i * DH + h * HC + c0, x[i]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < C::NQ; ++i) reg_fence16(x[i]);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < C::NQ; ++i) acc += x[i][j] * wi[i];
          o[c0 + j] = FP8 ? acc * a.v_scale : acc;   // O holds P . code for fp8 pools
        }
      }
      bf16* out = static_cast<bf16*>(a.out) + (static_cast<size_t>(row) * a.Hq + head) * DH + h * HC;
      if (nsplits == 1) {
        if (in_tile) {
          const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
          for (int j = 0; j < HC; j += 2)
            *reinterpret_cast<__nv_bfloat162*>(out + j) =
                __floats2bfloat162_rn(o[j] * inv, o[j + 1] * inv);
        }
      } else {
        // partial [split][column][query row]: a warp's accesses of one column
        // are contiguous
        const size_t unit = (static_cast<size_t>(r) * a.Hkv + g) * p.qtiles + qt;
        const size_t stride = static_cast<size_t>(128) * (DH + 2);
        // (rows of the tile only: the merge reads no other)
        float* mine = p.part + (unit * p.max_splits + split) * stride + qrow;
        if (in_tile) {
#pragma unroll
          for (int j = 0; j < HC; ++j) mine[(h * HC + j) * 128] = o[j];
          if (h == 0) {
            mine[DH * 128] = M;
            mine[(DH + 1) * 128] = L;
          }
        }
        __threadfence();
        named_bar_sync(1, C::SOFT);
        if (p.parallel_merge) {
          // Wait (bounded) until the unit's splits have all written their
          // partials, then merge rows [q0, q1) of the unit's 128: the
          // slice's (m, l) and columns of every split come into shared
          // memory (the K/V stages, idle now) in one round of cp.async,
          // and each thread combines one row's group of columns in split
          // order (deterministic).
          int* arrived = p.counters + unit;
          int* merged = arrived + static_cast<size_t>(a.B) * a.Hkv * p.qtiles;
          if (threadIdx.x == 64) {
            attn_stamp(p, 6);
            atomicAdd(arrived, 1);
            *flag = flag_wait_geq(arrived, nsplits, a.err) ? 1 : 0;
            attn_stamp(p, 7);
          }
          named_bar_sync(1, C::SOFT);
          // the tile's rows are query slots [0, tile_rows G)
          const int live = tile_rows * p.G;
          const int per = ((live + nsplits - 1) / nsplits + 3) & ~3;   // rows, a multiple of 4
          const int q0 = split * per, q1 = min(live, q0 + per);
          if (*flag && q0 < q1) {
            const float* base = p.part + unit * p.max_splits * stride;
            float* stage = reinterpret_cast<float*>(smem + C::K_OFF);   // [split][col][per]
            const int t = threadIdx.x - 64;
            const int quads = per / 4;                                   // 16-byte row groups
            const int items = nsplits * (DH + 2) * quads;
            for (int it = t; it < items; it += C::SOFT) {
              const int qd = it % quads, col = (it / quads) % (DH + 2), sp = it / (quads * (DH + 2));
              const int q = q0 + qd * 4;
              const float* src = base + sp * stride + col * 128 + q;
              const uint32_t dst = smem_u32(stage + (sp * (DH + 2) + col) * per + qd * 4);
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                           "r"(q < q1 ? 16 : 0)
                           : "memory");
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            named_bar_sync(1, C::SOFT);
            if (threadIdx.x == 64) attn_stamp(p, 10);
            // Combine in parallel passes (row maxima; the weight of every
            // (row, split); row sums; the columns).  Every sum runs over the
            // splits in order, with the same operations as one thread per
            // row would use.
            const int nr = q1 - q0;                               // rows of the slice
            float* mx = stage + nsplits * (DH + 2) * per;          // [per]
            float* inv = mx + per;                                 // [per]
            float* wgt = inv + per;                                // [per][nsplits]
            auto st_m = [&](int sp, int rr) { return stage[(sp * (DH + 2) + DH) * per + rr]; };
            auto st_l = [&](int sp, int rr) { return stage[(sp * (DH + 2) + DH + 1) * per + rr]; };
            // (loops over the splits without branches, unrolled: their
            // shared-memory loads are issued together, not one round trip
            // per split)
            for (int rr = t; rr < nr; rr += C::SOFT) {
              float Mx = -INFINITY;
#pragma unroll 8
              for (int sp = 0; sp < nsplits; ++sp) {
                const float l = st_l(sp, rr), m = st_m(sp, rr);
                Mx = l > 0.f ? fmaxf(Mx, m) : Mx;
              }
              mx[rr] = Mx;
            }
            named_bar_sync(1, C::SOFT);
            for (int it = t; it < nr * nsplits; it += C::SOFT) {
              const int rr = it / nsplits, sp = it % nsplits;
              wgt[it] = st_l(sp, rr) > 0.f ? exp2f(st_m(sp, rr) - mx[rr]) : 0.f;
            }
            named_bar_sync(1, C::SOFT);
            for (int rr = t; rr < nr; rr += C::SOFT) {
              float Ls = 0.f;
#pragma unroll 8
              for (int sp = 0; sp < nsplits; ++sp) {
                const float ls = st_l(sp, rr), w = wgt[rr * nsplits + sp];
                Ls = ls > 0.f ? Ls + w * ls : Ls;
              }
              inv[rr] = Ls > 0.f ? 1.f / Ls : 0.f;
            }
            named_bar_sync(1, C::SOFT);
            // thread -> (row, column pair), rows fastest
            for (int it = t; it < nr * (DH / 2); it += C::SOFT) {
              const int rr = it % nr, c = (it / nr) * 2;
              const int q = q0 + rr, mlr = q / p.G, mhl = q % p.G;
              float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
              for (int sp = 0; sp < nsplits; ++sp) {
                const bool in = st_l(sp, rr) > 0.f;
                const float w = wgt[rr * nsplits + sp];
                const float x0 = stage[(sp * (DH + 2) + c) * per + rr];
                const float x1 = stage[(sp * (DH + 2) + c + 1) * per + rr];
                a0 = in ? a0 + w * x0 : a0;
                a1 = in ? a1 + w * x1 : a1;
              }
              if (mlr < tile_rows) {
                bf16* o2 = static_cast<bf16*>(a.out) +
                           (static_cast<size_t>(row0 + tile_row0 + mlr) * a.Hq + g * p.G + mhl) * DH + c;
                *reinterpret_cast<__nv_bfloat162*>(o2) =
                    __floats2bfloat162_rn(a0 * inv[rr], a1 * inv[rr]);
              }
            }
          }
          // the last split to finish its slice leaves both counts zero
          if (threadIdx.x == 64) attn_stamp(p, 11);
          named_bar_sync(1, C::SOFT);
          if (threadIdx.x == 64) attn_stamp(p, 8);
          if (threadIdx.x == 64 && *flag) {
            const int old = atomicAdd(merged, 1);
            if (old == nsplits - 1) {
              *arrived = 0;
              *merged = 0;
            }
          }
        } else {
        if (threadIdx.x == 64) {
          const int old = atomicAdd(p.counters + unit, 1);
          *flag = (old == nsplits - 1) ? 1 : 0;
        }
        named_bar_sync(1, C::SOFT);
        if (*flag) {
          __threadfence();
          const float* base = p.part + unit * p.max_splits * stride + qrow;
          float Mx = -INFINITY;
          for (int s0 = 0; s0 < nsplits; s0 += 8) {
            float ms[8], ls[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const bool in = s0 + q < nsplits;
              ms[q] = in ? __ldcg(base + (s0 + q) * stride + DH * 128) : -INFINITY;
              ls[q] = in ? __ldcg(base + (s0 + q) * stride + (DH + 1) * 128) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (ls[q] > 0.f) Mx = fmaxf(Mx, ms[q]);
          }
          float acc[HC];
#pragma unroll
          for (int j = 0; j < HC; ++j) acc[j] = 0.f;
          float Ls = 0.f;
          // QN splits at a time: their weights and columns are all loaded
          // before any of them is added (in split order)
          constexpr int QN = DH == 64 ? 2 : 1;   // splits loaded together
          for (int s2 = 0; s2 < nsplits; s2 += QN) {
            float wq[QN], lq[QN], col[QN][HC];
#pragma unroll
            for (int q = 0; q < QN; ++q) {
              const bool in = s2 + q < nsplits;
              const float* src = base + (s2 + q) * stride;
              lq[q] = in ? __ldcg(src + (DH + 1) * 128) : 0.f;
              wq[q] = in ? __ldcg(src + DH * 128) : -INFINITY;
#pragma unroll
              for (int j = 0; j < HC; ++j) col[q][j] = in ? __ldcg(src + (h * HC + j) * 128) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < QN; ++q) {
              if (!(lq[q] > 0.f)) continue;
              const float w = exp2f(wq[q] - Mx);
              Ls += w * lq[q];
#pragma unroll
              for (int j = 0; j < HC; ++j) acc[j] += w * col[q][j];
            }
          }
          if (in_tile) {
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
            for (int j = 0; j < HC; j += 2)
              *reinterpret_cast<__nv_bfloat162*>(out + j) =
                  __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
          }
          if (threadIdx.x == 64) p.counters[unit] = 0;
        }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) attn_stamp(p, 9);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

struct AttnPlan {
  int G, rows_per_qt, qtiles, split_keys, max_splits;
};

// min_cps: the fewest chunks a split takes (2 by default; the workspace is
// sized for that, so a larger value only needs less of it)
static AttnPlan plan_attention(const AttnArgs& a, int max_rows_per_req, int sm_count,
                               int min_cps = 2, int max_cps = 32) {
  AttnPlan pl;
  pl.G = a.Hq / a.Hkv;
  pl.rows_per_qt = 128 / pl.G;
  pl.qtiles = (max_rows_per_req + pl.rows_per_qt - 1) / pl.rows_per_qt;
  const int max_seq = a.bt_stride * 16;
  const int chunks_max = (max_seq + 127) / 128;
  const long long pairs = static_cast<long long>(a.B) * a.Hkv * pl.qtiles;
  const int want = static_cast<int>(std::max<long long>(1, (sm_count + pairs - 1) / pairs));
  // A split is at most 64 chunks at dh 64 and 32 at dh 128 (its block ids
  // fit the CTA's table).
  // Fewer units than SMs: about 8 splits per unit, 16 where 8 would leave
  // more than half of the SMs idle (batch 1: 1.5 % faster step; at 16
  // requests 16 splits lost 5 %); otherwise enough splits to give every SM
  // a unit, 2 to 32 chunks each (32 measured best at batch 64).  The splits of a unit are merged through global memory by
  // the last one to finish: at batch 16 that beat merging the splits of a
  // thread-block cluster through distributed shared memory by a sixth of
  // the step (8-CTA clusters of one-CTA-per-SM kernels leave SMs idle), and
  // tied with it at batch 1.
  // A few units (batch 1): as many splits as keep the grid one wave, two
  // chunks or more each; their merge is then parallel (every split merges
  // a slice of the rows, parallel_merge below).
  const int kMaxCps = std::max(2, std::min(a.dh == 64 ? 64 : 32, max_cps));
  int cps = pairs * 16 <= sm_count ? (chunks_max * static_cast<int>(pairs) + sm_count - 1) / sm_count
            : pairs < sm_count     ? (chunks_max + 7) / 8
                                   : (chunks_max + want - 1) / want;
  cps = std::max(std::max(2, min_cps), std::min(kMaxCps, cps));
  pl.split_keys = cps * 128;
  pl.max_splits = (max_seq + pl.split_keys - 1) / pl.split_keys;
  return pl;
}

size_t attention_tc_partial_floats(const AttnArgs& a, int max_rows_per_req, int sm_count,
                                   int min_cps, int max_cps) {
  const AttnPlan pl = plan_attention(a, max_rows_per_req, sm_count, min_cps, max_cps);
  return static_cast<size_t>(a.B) * a.Hkv * pl.qtiles * pl.max_splits * 128 * (a.dh + 2);
}

size_t attention_tc_counters(const AttnArgs& a, int max_rows_per_req, int sm_count,
                             int min_cps, int max_cps) {
  const AttnPlan pl = plan_attention(a, max_rows_per_req, sm_count, min_cps, max_cps);
  return 2 * static_cast<size_t>(a.B) * a.Hkv * pl.qtiles;   // splits written, merged
}

// Tensor map of an fp8 pool viewed as [rows, cols] bytes (rows = blocks x
// kv heads x 16 keys, cols = dh), boxes of box_rows keys x cols bytes,
// unswizzled (the pages are widened by threads, not read by the MMA).
bool tensor_map_2d_u8(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
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
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || cols % 16 != 0 || cols > 256) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t init_attention_tc() {
  cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       AttnCfg<64>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attention_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttnCfg<128>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attention_tc_kernel<64, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<64, true>::SMEM);
  return e;
}

// Work items of an attention launch, longest first: item (request r, split
// s) has min(split chunks, chunks left in r's sequence past s's first key)
// chunks; a counting sort by that count, most first, items without keys
// last as -1.  One CTA; the order among items of equal length is whatever
// the atomics give (each item's result does not depend on it).
__global__ void attention_order_kernel(const int32_t* seq_lens, int B, int split_keys,
                                       int max_splits, int32_t* order) {
  constexpr int kBuckets = 65;              // 0..64 chunks
  __shared__ int count[kBuckets], start[kBuckets];
  const int n = B * max_splits;
  const int cps = split_keys / 128;
  for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) count[i] = 0;
  __syncthreads();
  auto chunks_of = [&](int it) {
    const int r = it / max_splits, s = it % max_splits;
    const int left = seq_lens[r] - s * split_keys;
    return left <= 0 ? 0 : min(cps, (left + 127) / 128);
  };
  for (int it = threadIdx.x; it < n; it += blockDim.x) atomicAdd(&count[chunks_of(it)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int c = kBuckets - 1; c >= 0; --c) {   // most chunks first, empty items last
      start[c] = acc;
      acc += count[c];
    }
  }
  __syncthreads();
  for (int it = threadIdx.x; it < n; it += blockDim.x) {
    const int c = chunks_of(it);
    const int at = atomicAdd(&start[c], 1);
    order[at] = c > 0 ? ((it / max_splits) << 8) | (it % max_splits) : -1;
  }
}

// Whether a launch of this shape takes its work in a sorted order (many CTAs:
// more than one wave), and then the order buffer entries it needs.
int attention_tc_order_entries(const AttnArgs& a, int max_rows_per_req, int sm_count, int min_cps,
                               int max_cps) {
  const AttnPlan pl = plan_attention(a, max_rows_per_req, sm_count, min_cps, max_cps);
  const long long ctas = static_cast<long long>(pl.max_splits) * a.Hkv * pl.qtiles * a.B;
  if (ctas <= sm_count || pl.max_splits > 255 || a.B >= (1 << 22)) return 0;
  return a.B * pl.max_splits;
}

cudaError_t launch_attention_order(const AttnArgs& a, const int32_t* seq_lens,
                                   int max_rows_per_req, int sm_count, int min_cps, int max_cps,
                                   int32_t* order, cudaStream_t s) {
  const AttnPlan pl = plan_attention(a, max_rows_per_req, sm_count, min_cps, max_cps);
  if (pl.split_keys / 128 > 64) return cudaErrorInvalidValue;
  attention_order_kernel<<<1, 1024, 0, s>>>(seq_lens, a.B, pl.split_keys, pl.max_splits, order);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const int32_t* seq_lens, int max_rows_per_req, int sm_count,
                                float* part, size_t part_floats, int* counters,
                                size_t n_counters, unsigned long long* timeline, int l2_ahead,
                                int min_cps, int max_cps, const int32_t* order,
                                cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  const AttnPlan pl = plan_attention(a, max_rows_per_req, sm_count, min_cps, max_cps);
  AttnTcParams p;
  p.a = a;
  p.seq_lens = seq_lens;
  p.G = pl.G;
  p.rows_per_qt = pl.rows_per_qt;
  p.qtiles = pl.qtiles;
  p.split_keys = pl.split_keys;
  p.max_splits = pl.max_splits;
  p.part = part;
  p.counters = counters;
  p.tl = timeline;
  p.l2_ahead = l2_ahead < 0 ? 0 : l2_ahead;
  p.order = nullptr;
  // every split CTA resident at once (one wave of one CTA per SM), at most
  // 32 splits: the splits merge their unit in parallel
  const long long ctas = static_cast<long long>(pl.max_splits) * a.Hkv * pl.qtiles * a.B;
  p.parallel_merge = (ctas <= sm_count && pl.max_splits <= 32) ? 1 : 0;
  if (pl.split_keys / 16 > (a.dh == 64 ? AttnCfg<64>::BT_ENTRIES : AttnCfg<128>::BT_ENTRIES))
    return cudaErrorInvalidValue;
  const size_t need = static_cast<size_t>(a.B) * a.Hkv * pl.qtiles * pl.max_splits * 128 * (a.dh + 2);
  if (need > part_floats || 2 * static_cast<size_t>(a.B) * a.Hkv * pl.qtiles > n_counters)
    return cudaErrorInvalidValue;
  dim3 grid(pl.max_splits, a.Hkv * pl.qtiles, a.B);
  if (order && !p.parallel_merge) {
    p.order = order;
    grid = dim3(a.Hkv * pl.qtiles, a.B * pl.max_splits, 1);
  }
  if (a.kv_fp8) {
    if (a.dh != 64 || !(a.k_scale > 0.f) || !(a.v_scale > 0.f)) return cudaErrorInvalidValue;
    return launch_pdl(attention_tc_kernel<64, true>, grid, dim3(AttnCfg<64, true>::THREADS),
                      AttnCfg<64, true>::SMEM, s, tmK, tmV, p);
  }
  if (a.dh == 64)
    return launch_pdl(attention_tc_kernel<64>, grid, dim3(AttnCfg<64>::THREADS),
                      AttnCfg<64>::SMEM, s, tmK, tmV, p);
  return launch_pdl(attention_tc_kernel<128>, grid, dim3(AttnCfg<128>::THREADS),
                    AttnCfg<128>::SMEM, s, tmK, tmV, p);
}

}  // namespace pe
