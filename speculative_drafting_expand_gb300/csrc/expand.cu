// expand.cu -- batch expansion for parallel drafting, fused with the hidden
// state scatter and the h_shared broadcast (one launch, one CTA per
// expanded row).
//
// What it computes follows the vLLM blog summary "P-EAGLE: Faster LLM
// Inference with Parallel Speculative Decoding in vLLM":
//   * fused-kernel bullet: copy the previous token ids and positions into
//     the new slots, insert each request's sampled token, fill the extra
//     parallel-drafting slots with the MASK id, and produce the rejected
//     mask, MASK mask, new-token indices and hidden-state map;
//   * hidden-state bullet: target hidden rows go to their mapped rows, MASK
//     rows receive the learned shared hidden state;
//   * KV-cache bullet: slot mapping from the new positions, -1 for rejected
//     tokens so that they never write the cache;
//   * prompt-position handling: the row at position i carries the hidden
//     state of position i-1 (so window row j sits at q_j + 1).
// The pages run the metadata and the hidden copy as two kernels; here one
// CTA per output row does both, since each row's metadata is a handful of
// integers and its hidden row is one contiguous 16-byte-vector copy.
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

// Warp 0 finds the row's request (32 candidates a round: two rounds up to
// 1024 requests) and publishes its source hidden row; warps 1-3 then copy
// the row (all their 16-byte loads in flight before the stores) while warp 0
// gathers the rest of the metadata, one independent load per lane.
__global__ void __launch_bounds__(128) expand_kernel(const ExpandArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;  // expanded row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int s_src;      // source hidden row (-1: h_shared)

  int r = 0, in0 = 0, n = 0, acc = 0, s = 0, out0 = 0, j = 0;
  if (warp == 0) {
    // request of this row: the largest r with cu_in[r] + r (K - 1) <= i
    // (non-decreasing in r, so the lanes that pass form a prefix)
    int lo = 0, cnt = a.B;
    while (cnt > 1) {
      const int step = (cnt + 31) / 32;
      const int cand = lo + lane * step;
      const bool ok = lane * step < cnt && a.cu_in[cand] + cand * (a.K - 1) <= i;
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      const int last = m ? 31 - __clz(static_cast<int>(m)) : 0;
      lo += last * step;
      cnt = min(step, cnt - last * step);
    }
    r = lo;
    const int v = lane == 0 ? a.cu_in[r]
                : lane == 1 ? a.cu_in[r + 1]
                : lane == 2 ? a.num_accepted[r]
                : lane == 3 ? a.sampled_ids[r]
                            : 0;
    in0 = __shfl_sync(0xffffffffu, v, 0);
    n = __shfl_sync(0xffffffffu, v, 1) - in0;
    acc = __shfl_sync(0xffffffffu, v, 2);
    s = __shfl_sync(0xffffffffu, v, 3);
    out0 = in0 + r * (a.K - 1);
    j = i - out0;
    if (acc < 0 || acc > n - 1) {
      // (an empty window, n = 0, is reported the same way)
      if (lane == 0) record_error(a.err, PE_DEV_BAD_ACCEPTED);
      acc = acc < 0 || n < 1 ? 0 : n - 1;
    }
    if (lane == 0) s_src = j < n ? in0 + j : -1;
  }
  __syncthreads();

  if (warp == 0) {
    // the rest of the row's metadata, independent loads on separate lanes
    const int v = (lane == 0 && n > 0) ? a.target_pos[in0 + acc]
                : (lane == 1 && j < n) ? a.target_pos[in0 + j]
                : (lane == 2 && j + 1 < n) ? a.target_ids[in0 + j + 1]
                                           : 0;
    const int q_a = __shfl_sync(0xffffffffu, v, 0);
    const int q_j = __shfl_sync(0xffffffffu, v, 1);
    const int next_id = __shfl_sync(0xffffffffu, v, 2);
    if (lane == 0) {
      int id, p, rejected = 0, masked = 0;
      if (j < n) {
        // window row j: hidden of target row j, one position later, carrying
        // the token at that position (the next window token, or s at row a)
        id = (j + 1 < n) ? next_id : s;
        if (j == acc) id = s;
        p = q_j + 1;
        rejected = (j > acc) ? 1 : 0;
        a.hidden_map[in0 + j] = i;
        if (j == acc) a.new_idx[r * a.K] = i;
      } else {
        const int k = j - n + 1;  // MASK rows k = 1..K-1
        id = a.mask_token_id;
        p = q_a + 1 + k;
        masked = 1;
        a.new_idx[r * a.K + k] = i;
      }
      int sl = -1;
      if (!rejected) {
        const int page = p / a.page_size;
        if (p < 0 || page >= a.bt_stride) {
          record_error(a.err, PE_DEV_BAD_POSITION);
        } else {
          const int blk = a.block_table[static_cast<long long>(r) * a.bt_stride + page];
          if (blk < 0 || blk >= a.num_blocks) record_error(a.err, PE_DEV_BAD_BLOCK);
          else sl = blk * a.page_size + p % a.page_size;
        }
      }
      a.ids[i] = id;
      a.pos[i] = p;
      a.slot[i] = sl;
      a.is_rejected[i] = static_cast<uint8_t>(rejected);
      a.is_masked[i] = static_cast<uint8_t>(masked);
      if (j == 0) {
        a.cu_out[r] = out0;
        a.seq_lens[r] = q_a + a.K + 1;
        if (r == a.B - 1) a.cu_out[a.B] = a.T_out;
      }
    }
  } else {
    // hidden row: target row (scatter through the map) or h_shared (broadcast)
    const int src = s_src;
    const uint4* from = reinterpret_cast<const uint4*>(
        src >= 0 ? static_cast<const uint8_t*>(a.target_hidden) +
                       static_cast<size_t>(src) * a.row_bytes
                 : static_cast<const uint8_t*>(a.h_shared));
    uint4* to = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.hidden) +
                                         static_cast<size_t>(i) * a.row_bytes);
    const int nvec = a.row_bytes / 16;
    constexpr int kCopiers = 96, kInFlight = 12;
    for (int v0 = threadIdx.x - 32; v0 < nvec; v0 += kCopiers * kInFlight) {
      uint4 x[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k)
        if (v0 + k * kCopiers < nvec) x[k] = from[v0 + k * kCopiers];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k)
        if (v0 + k * kCopiers < nvec) to[v0 + k * kCopiers] = x[k];
    }
  }
}

cudaError_t launch_expand(const ExpandArgs& a, cudaStream_t s) {
  if (a.T_out <= 0) return cudaSuccess;
  return launch_pdl(expand_kernel, dim3(a.T_out), dim3(128), 0, s, a);
}

}  // namespace pe
