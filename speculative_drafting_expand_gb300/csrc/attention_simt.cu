// attention_simt.cu -- paged causal attention with FFMA (the fp32 path).
//
// Each non-rejected row at position P attends positions 0..P of its request
// through the block table; query head h reads kv head h / (Hq / Hkv); scores
// are scaled by 1/sqrt(dh) and normalised with an online softmax.  Rejected
// rows (vLLM blog summary, KV-cache bullet) produce zeros.  One warp per
// (row, query head); lanes split the head dimension.
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

template <typename T, int DH>
__global__ void __launch_bounds__(128) attention_simt_kernel(const AttnArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int E = DH / 32;  // elements per lane
  const int i = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= a.Hq) return;
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
  T* out = static_cast<T*>(a.out) + static_cast<size_t>(i) * a.Hq * DH + h * DH;
  if (a.is_rejected && a.is_rejected[i]) {
#pragma unroll
    for (int e = 0; e < E; ++e) out[lane + 32 * e] = from_f<T>(0.f);
    return;
  }
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.cu_out[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo;
  const int P = a.pos[i];
  const int g = h / (a.Hq / a.Hkv);
  const T* qp = static_cast<const T*>(a.q) + static_cast<size_t>(i) * a.Hq * DH + h * DH;
  float q[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = to_f(qp[lane + 32 * e]) * a.scale;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const T* kc = static_cast<const T*>(a.k_cache);
  const T* vc = static_cast<const T*>(a.v_cache);
  const int32_t* bt = a.block_table + static_cast<size_t>(r) * a.bt_stride;
  for (int t = 0; t <= P; ++t) {
    const int page = t / 16;
    int blk = page < a.bt_stride ? bt[page] : -1;
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) record_error(a.err, PE_DEV_BAD_BLOCK);
      break;
    }
    const size_t base = ((static_cast<size_t>(blk) * a.Hkv + g) * 16 + (t % 16)) * DH;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) s += q[e] * to_f(kc[base + lane + 32 * e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float m_new = fmaxf(m, s);
    const float corr = expf(m - m_new);
    const float pw = expf(s - m_new);
    l = l * corr + pw;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = acc[e] * corr + pw * to_f(vc[base + lane + 32 * e]);
    m = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) out[lane + 32 * e] = from_f<T>(acc[e] * inv);
}

cudaError_t launch_attention_simt(int dtype, const AttnArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  dim3 grid(a.rows, (a.Hq + 3) / 4);
  if (dtype == PE_DTYPE_BF16) {
    if (a.dh == 64) return launch_pdl(attention_simt_kernel<bf16, 64>, grid, dim3(128), 0, s, a);
    return launch_pdl(attention_simt_kernel<bf16, 128>, grid, dim3(128), 0, s, a);
  }
  if (a.dh == 64) return launch_pdl(attention_simt_kernel<float, 64>, grid, dim3(128), 0, s, a);
  return launch_pdl(attention_simt_kernel<float, 128>, grid, dim3(128), 0, s, a);
}

}  // namespace pe
