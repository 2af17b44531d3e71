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

__global__ void __launch_bounds__(128) expand_kernel(const ExpandArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;  // expanded row
  __shared__ int s_src;      // source hidden row (-1: h_shared)

  if (threadIdx.x == 0) {
    // request of this row: largest r with cu_in[r] + r (K - 1) <= i
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu_in[mid] + mid * (a.K - 1) <= i) lo = mid;
      else hi = mid - 1;
    }
    const int r = lo;
    const int in0 = a.cu_in[r];
    const int n = a.cu_in[r + 1] - in0;
    const int out0 = in0 + r * (a.K - 1);
    const int j = i - out0;
    int acc = a.num_accepted[r];
    if (acc < 0 || acc > n - 1) {
      record_error(a.err, PE_DEV_BAD_ACCEPTED);
      acc = acc < 0 ? 0 : n - 1;
    }
    const int q_a = a.target_pos[in0 + acc];
    const int s = a.sampled_ids[r];

    int id, p, rejected = 0, masked = 0, src = -1;
    if (j < n) {
      // window row j: hidden of target row j, one position later, carrying
      // the token at that position (the next window token, or s at row a)
      id = (j + 1 < n) ? a.target_ids[in0 + j + 1] : s;
      if (j == acc) id = s;
      p = a.target_pos[in0 + j] + 1;
      rejected = (j > acc) ? 1 : 0;
      src = in0 + j;
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
    s_src = src;
  }
  __syncthreads();

  // hidden row: target row (scatter through the map) or h_shared (broadcast)
  const int src = s_src;
  const uint4* from = reinterpret_cast<const uint4*>(
      src >= 0 ? static_cast<const uint8_t*>(a.target_hidden) + static_cast<size_t>(src) * a.row_bytes
               : static_cast<const uint8_t*>(a.h_shared));
  uint4* to = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.hidden) +
                                       static_cast<size_t>(i) * a.row_bytes);
  const int nvec = a.row_bytes / 16;
  int v = threadIdx.x;
  // four 16-byte loads in flight per thread before the stores
  for (; v + 3 * 128 < nvec; v += 4 * 128) {
    const uint4 x0 = from[v], x1 = from[v + 128], x2 = from[v + 256], x3 = from[v + 384];
    to[v] = x0;
    to[v + 128] = x1;
    to[v + 256] = x2;
    to[v + 384] = x3;
  }
  for (; v < nvec; v += 128) to[v] = from[v];
}

cudaError_t launch_expand(const ExpandArgs& a, cudaStream_t s) {
  if (a.T_out <= 0) return cudaSuccess;
  return launch_pdl(expand_kernel, dim3(a.T_out), dim3(128), 0, s, a);
}

}  // namespace pe
