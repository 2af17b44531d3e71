// compact.cu -- live-row compaction of the expanded batch.
//
// The expanded layout keeps every window row of a request, including the
// ones after its accepted count (vLLM blog summary "P-EAGLE: Faster LLM
// Inference with Parallel Speculative Decoding in vLLM", KV-cache bullet:
// rejected tokens get slot -1 and never write the cache).  Nothing reads
// what such a row computes: no sampled row is rejected, and attention reads
// other positions only through the cache.  So after the fc projection the
// drafter layers run on the live rows alone.  Each request's live rows stay
// together and in order (window rows 0..a, then the MASK rows), so their
// positions are still consecutive and the request offsets carry over.
//
// One CTA: a block-wide prefix count over the rejected flags, 1024 rows at
// a time (the step has a few thousand rows at most).
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

constexpr int kCompactThreads = 1024;

__global__ void __launch_bounds__(kCompactThreads) compact_rows_kernel(const CompactArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int warp_excl[32];
  __shared__ int s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (int p0 = 0; p0 < a.T_out; p0 += kCompactThreads) {
    const int p = p0 + tid;
    const int live = (p < a.T_out && a.is_rejected[p] == 0) ? 1 : 0;
    int x = live;  // inclusive count within the warp
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
    const int c = s_base + warp_excl[warp] + x - live;  // live rows before p
    if (p < a.T_out) {
      a.live_before[p] = c;
      a.row_map[p] = live ? c : -1;
      if (live) {
        a.live_row[c] = p;
        a.ids_c[c] = a.ids[p];
        a.pos_c[c] = a.pos[p];
        a.slot_c[c] = a.slot[p];
        if (a.masked_c) a.masked_c[c] = a.is_masked[p];
      }
    }
    __syncthreads();  // every thread has read s_base and warp_excl
    if (tid == kCompactThreads - 1) s_base = c + live;
    __syncthreads();
  }
  const int n = s_base;
  if (tid == 0) {
    a.live_before[a.T_out] = n;
    *a.n_live = n;
  }
  __syncthreads();  // the block's global writes above are visible to it
  for (int r = tid; r <= a.B; r += kCompactThreads) {
    int q = r < a.B ? a.cu_out[r] : a.T_out;
    q = min(max(q, 0), a.T_out);
    a.cu_live[r] = a.live_before[q];
  }
  for (int i = tid; i < a.B * a.K; i += kCompactThreads) {
    const int q = a.new_idx[i];
    a.new_c[i] = (q >= 0 && q < a.T_out) ? a.row_map[q] : -1;
  }
  if (a.fc_map)
    for (int t = tid; t < a.T; t += kCompactThreads) {
      const int q = a.hidden_map[t];
      a.fc_map[t] = (q >= 0 && q < a.T_out) ? a.row_map[q] : -1;
    }
}

__global__ void __launch_bounds__(128) scatter_rows_kernel(uint8_t* dst, const uint8_t* src,
                                                           const int32_t* live_row,
                                                           const int32_t* n_live, int row_bytes) {
  grid_dep_wait();
  grid_dep_launch();
  const int c = blockIdx.x;
  if (c >= __ldcg(n_live)) return;
  const int p = __ldcg(live_row + c);
  const uint4* from = reinterpret_cast<const uint4*>(src + static_cast<size_t>(c) * row_bytes);
  uint4* to = reinterpret_cast<uint4*>(dst + static_cast<size_t>(p) * row_bytes);
  for (int v = threadIdx.x; v < row_bytes / 16; v += 128) to[v] = from[v];
}

cudaError_t launch_compact_rows(const CompactArgs& a, cudaStream_t s) {
  if (a.T_out <= 0 || a.B <= 0) return cudaErrorInvalidValue;
  return launch_pdl(compact_rows_kernel, dim3(1), dim3(kCompactThreads), 0, s, a);
}

cudaError_t launch_scatter_rows(void* dst, const void* src, const int32_t* live_row,
                                const int32_t* n_live, int rows_max, int row_bytes,
                                cudaStream_t s) {
  if (rows_max <= 0) return cudaSuccess;
  if (row_bytes % 16 || (reinterpret_cast<uintptr_t>(dst) & 15) ||
      (reinterpret_cast<uintptr_t>(src) & 15))
    return cudaErrorInvalidValue;
  return launch_pdl(scatter_rows_kernel, dim3(rows_max), dim3(128), 0, s,
                    static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), live_row, n_live,
                    row_bytes);
}

}  // namespace pe
