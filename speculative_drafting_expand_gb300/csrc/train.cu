// train.cu -- index work of P-EAGLE's long-context training layout (paper
// summary "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training",
// section 3): the amortized attention mask over (position, depth) rows
// (3.1), conditional drop-token (COD) sampling of the depth rows, and the
// sequence partitioning that keeps every cross-depth dependency inside one
// segment (3.2).
//
// Rows: (p, d) is depth d at position p, laid out position-major (index
// p K + d); depth d >= 1 is the d-th MASK row of the draft whose
// next-token row is (p - d, 0).  Row (p, d) attends the depth-0 rows
// q <= p - d and its draft's MASK rows (p - d + e, e), 1 <= e <= d: the
// rule depends on p - q only, so the mask of an n-token sample is the
// top-left n K x n K block of the mask built once for the longest one
// (ScienceStack page, Figure 3).
//
// Partitioning: the pages assign depths 0 and 1 by index and then each
// deeper row to its dependency's segment, depth by depth.  Unrolled, the
// chain of (p, d) ends at (p - d + 1, 1), so its segment is the one whose
// index range holds p - d + 1: every row is assigned independently here.
#include <algorithm>

#include "../../include/peagle_train.h"
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

// ------------------------------------------------------------------ mask

// A CTA writes whole mask rows, its threads 16-byte chunks of a row.  Row
// (p, d) has three column ranges: positions q <= p - d (context: only the
// depth-0 column of each position may be attended, a pattern that repeats
// every K columns, so its chunks come from a per-phase table), the draft's
// positions p - d < q <= p (the rule, element by element: a few chunks a
// row) and later positions (nothing may be attended).  A thread's column
// phase (j mod K) advances by a fixed step, so no chunk divides by K.
template <bool ADDITIVE>
__global__ void __launch_bounds__(256) train_mask_kernel(uint8_t* out, int n_max, int K,
                                                         long long ld, int chunks_per_row) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int EPC = ADDITIVE ? 8 : 16;  // elements per 16-byte chunk
  constexpr int EB = ADDITIVE ? 2 : 1;
  constexpr uint32_t kAllow = ADDITIVE ? 0x0000u : 1u, kBlock = ADDITIVE ? 0xff80u : 0u;
  constexpr uint32_t kBlockWord = ADDITIVE ? (kBlock | (kBlock << 16)) : 0u;
  extern __shared__ uint4 phase_tab[];  // [K]: context chunk starting at depth phase e0
  auto pack = [](uint32_t (&w)[4], int k, bool ok) {
    const uint32_t v = ok ? kAllow : kBlock;
    if (ADDITIVE) w[k >> 1] |= v << ((k & 1) * 16);
    else w[k >> 2] |= v << ((k & 3) * 8);
  };
  for (int e0 = threadIdx.x; e0 < K; e0 += blockDim.x) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    int e = e0;
#pragma unroll
    for (int k = 0; k < EPC; ++k) {
      pack(w, k, e == 0);
      if (++e == K) e = 0;
    }
    phase_tab[e0] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  const long long N = static_cast<long long>(n_max) * K;
  const int step = static_cast<int>((static_cast<long long>(blockDim.x) * EPC) % K);
  const int phase0 = static_cast<int>((static_cast<long long>(threadIdx.x) * EPC) % K);
  const uint4 blocked = make_uint4(kBlockWord, kBlockWord, kBlockWord, kBlockWord);
  for (long long i = blockIdx.x; i < N; i += gridDim.x) {
    const int p = static_cast<int>(i / K), d = static_cast<int>(i - static_cast<long long>(p) * K);
    uint4* row = reinterpret_cast<uint4*>(out + i * ld * EB);
    const long long a_end = static_cast<long long>(p - d + 1) * K;  // context columns
    const long long b_end = static_cast<long long>(p + 1) * K;      // + the draft's columns
    int phase = phase0;
    for (int c = threadIdx.x; c < chunks_per_row; c += blockDim.x) {
      const long long j0 = static_cast<long long>(c) * EPC;
      uint4 v;
      if (p < d || j0 >= b_end) {
        v = blocked;
      } else if (j0 + EPC <= a_end) {
        v = phase_tab[phase];
      } else {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        int e = phase;
        int q = static_cast<int>((j0 - phase) / K);
#pragma unroll
        for (int k = 0; k < EPC; ++k) {
          pack(w, k, j0 + k < N && q >= e && (e == 0 ? q <= p - d : (e <= d && q - e == p - d)));
          if (++e == K) {
            e = 0;
            ++q;
          }
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      __stcs(row + c, v);
      phase += step;
      if (phase >= K) phase -= K;
    }
  }
}

// ------------------------------------------------------------ partition

constexpr int kMaxSegments = 64;

struct PartitionArgs {
  int n, K, S;
  float r;
  const float* u;       // [n, K] draws (depth 0 unused)
  uint8_t* keep;        // [n, K]
  int32_t* seg;         // [n, K], -1 for dropped rows
  int32_t* counts;      // [S] owned rows per segment (zero on entry)
  int32_t* offsets;     // [S + 1]
  int32_t* rows;        // layout indices, segment by segment
  uint8_t* owned;       // 1 = owned by the segment, 0 = context
  int bounds[kMaxSegments + 1];
};

__device__ __forceinline__ int segment_of(int x, const PartitionArgs& a) {
  int lo = 0, hi = a.S - 1;  // largest s with bounds[s] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.bounds[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// COD keep flag and owning segment of every row, one thread per row.
__global__ void __launch_bounds__(256) cod_assign_kernel(const PartitionArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int hist[kMaxSegments];
  for (int s = threadIdx.x; s < a.S; s += blockDim.x) hist[s] = 0;
  __syncthreads();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < a.n * a.K) {
    const int p = idx / a.K, d = idx - p * a.K;
    // kept when every link of its chain back to depth 0 drew below r
    bool kept = p >= d;
    for (int j = 0; j < d && kept; ++j) kept = a.u[(p - j) * a.K + (d - j)] < a.r;
    int s = -1;
    if (kept) {
      s = segment_of(d <= 1 ? p : p - d + 1, a);
      atomicAdd(&hist[s], 1);
    }
    a.keep[idx] = kept ? 1 : 0;
    a.seg[idx] = s;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < a.S; s += blockDim.x)
    if (hist[s]) atomicAdd(a.counts + s, hist[s]);
}

// Rows of segment blockIdx.x in layout order: the depth-0 rows before its
// first index (context, owned elsewhere), then its own rows, which all sit
// at positions [bounds[s], bounds[s + 1] + K - 2).
__global__ void __launch_bounds__(1024) segment_rows_kernel(const PartitionArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int warp_excl[32];
  __shared__ int s_base;
  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long off = 0;
  for (int t = 0; t < s; ++t) off += a.bounds[t] + __ldcg(a.counts + t);
  const int b0 = a.bounds[s];
  if (tid == 0) {
    a.offsets[s] = static_cast<int32_t>(off);
    if (s == a.S - 1) a.offsets[a.S] = static_cast<int32_t>(off + b0 + __ldcg(a.counts + s));
    s_base = 0;
  }
  for (int q = tid; q < b0; q += 1024) {
    a.rows[off + q] = q * a.K;
    a.owned[off + q] = 0;
  }
  const long long own0 = off + b0;
  const int i_lo = b0 * a.K;
  const int i_hi = min(a.n, a.bounds[s + 1] + max(a.K - 2, 0)) * a.K;
  __syncthreads();
  for (int i0 = i_lo; i0 < i_hi; i0 += 1024) {
    const int i = i0 + tid;
    const int mine = (i < i_hi && __ldcg(a.seg + i) == s) ? 1 : 0;
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_excl[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int w = warp_excl[lane];
      int z = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      warp_excl[lane] = z - w;
    }
    __syncthreads();
    const int rank = s_base + warp_excl[warp] + x - mine;
    if (mine) {
      a.rows[own0 + rank] = i;
      a.owned[own0 + rank] = 1;
    }
    __syncthreads();
    if (tid == 1023) s_base = rank + mine;
    __syncthreads();
  }
}

// --------------------------------------------------------------- launchers

cudaError_t launch_train_mask(int n_max, int K, bool additive, void* out, long long ld,
                              int sm_count, cudaStream_t s) {
  const long long eb = additive ? 2 : 1;
  const long long chunks_per_row = ld * eb / 16;
  const long long N = static_cast<long long>(n_max) * K;
  if (N <= 0 || chunks_per_row <= 0) return cudaSuccess;
  if (chunks_per_row > (1LL << 31) - 1 || static_cast<size_t>(K) * 16 > 48 * 1024)
    return cudaErrorInvalidValue;
  const int grid = static_cast<int>(std::min<long long>(N, 8LL * sm_count));
  const size_t smem = static_cast<size_t>(K) * 16;
  if (additive)
    return launch_pdl(train_mask_kernel<true>, dim3(grid), dim3(256), smem, s,
                      static_cast<uint8_t*>(out), n_max, K, ld, static_cast<int>(chunks_per_row));
  return launch_pdl(train_mask_kernel<false>, dim3(grid), dim3(256), smem, s,
                    static_cast<uint8_t*>(out), n_max, K, ld, static_cast<int>(chunks_per_row));
}

cudaError_t launch_train_partition(int n, int K, float r, const float* u, int S,
                                   const int32_t* bounds, uint8_t* keep, int32_t* seg,
                                   int32_t* counts, int32_t* offsets, int32_t* rows,
                                   uint8_t* owned, cudaStream_t s) {
  if (S < 1 || S > kMaxSegments) return cudaErrorInvalidValue;
  PartitionArgs a;
  a.n = n;
  a.K = K;
  a.S = S;
  a.r = r;
  a.u = u;
  a.keep = keep;
  a.seg = seg;
  a.counts = counts;
  a.offsets = offsets;
  a.rows = rows;
  a.owned = owned;
  for (int t = 0; t <= kMaxSegments; ++t) a.bounds[t] = t <= S ? bounds[t] : n;
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * S, s);
  if (e == cudaSuccess)
    e = launch_pdl(cod_assign_kernel, dim3((n * K + 255) / 256), dim3(256), 0, s, a);
  if (e == cudaSuccess) e = launch_pdl(segment_rows_kernel, dim3(S), dim3(1024), 0, s, a);
  return e;
}

}  // namespace pe

extern "C" {

pe_status pe_train_build_mask(int32_t n_max, int32_t K, int32_t mask_type, void* out,
                              int64_t ld, void* stream) {
  if (n_max < 1 || K < 1 || K > 1024 || !out ||
      (mask_type != PE_MASK_BOOL_U8 && mask_type != PE_MASK_ADDITIVE_BF16))
    return PE_ERR_INVALID_ARGUMENT;
  const long long N = static_cast<long long>(n_max) * K;
  const long long eb = mask_type == PE_MASK_ADDITIVE_BF16 ? 2 : 1;
  if (N > (1LL << 31) - 1 || ld < N || (ld * eb) % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(out) & 15) != 0)
    return PE_ERR_INVALID_ARGUMENT;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PE_ERR_CUDA;
  const cudaError_t e = pe::launch_train_mask(n_max, K, mask_type == PE_MASK_ADDITIVE_BF16, out,
                                              ld, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

pe_status pe_train_mask_view(const void* mask, int64_t ld, int32_t n_max, int32_t K, int32_t n,
                             const void** view, int64_t* view_rows, int64_t* view_ld) {
  if (!mask || !view || !view_rows || !view_ld || K < 1 || n < 1 || n > n_max ||
      ld < static_cast<int64_t>(n_max) * K)
    return PE_ERR_INVALID_ARGUMENT;
  *view = mask;
  *view_rows = static_cast<int64_t>(n) * K;
  *view_ld = ld;
  return PE_OK;
}

pe_status pe_train_partition(int32_t n, int32_t K, float r, const float* u, int32_t S,
                             const int32_t* bounds, uint8_t* keep, int32_t* seg,
                             int32_t* counts, int32_t* offsets, int32_t* rows,
                             uint8_t* owned, int64_t capacity, void* stream) {
  if (n < 1 || K < 1 || S < 1 || S > pe::kMaxSegments || !u || !bounds || !keep || !seg ||
      !counts || !offsets || !rows || !owned)
    return PE_ERR_INVALID_ARGUMENT;
  if (static_cast<long long>(n) * K > (1LL << 30)) return PE_ERR_INVALID_ARGUMENT;
  if (bounds[0] != 0 || bounds[S] != n) return PE_ERR_INVALID_ARGUMENT;
  long long need = static_cast<long long>(n) * K;
  for (int s = 0; s < S; ++s) {
    if (bounds[s + 1] <= bounds[s]) return PE_ERR_INVALID_ARGUMENT;
    need += bounds[s];
  }
  if (capacity < need || need > (1LL << 31) - 1) return PE_ERR_INVALID_ARGUMENT;
  const cudaError_t e = pe::launch_train_partition(n, K, r, u, S, bounds, keep, seg, counts,
                                                   offsets, rows, owned,
                                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

}  // extern "C"
