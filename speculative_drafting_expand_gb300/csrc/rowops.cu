// rowops.cu -- per-row kernels of the drafter layer (LLaMA 3 pieces named in
// the paper summary "P-EAGLE: Parallel-Drafting EAGLE with Scalable
// Training", section 2 and Figure 2):
//   * layer-0 input: token embedding and projected target hidden state, each
//     RMS-normalised, concatenated (2d wide);
//   * RMSNorm of the fp32 residual stream (optionally gathering rows, for
//     the final norm of the sampled rows);
//   * rotate-half RoPE of q and k at the row's position, with k and v written
//     into the paged KV cache at the row's slot (slot -1: no write, as the
//     vLLM blog summary's KV-cache bullet requires for rejected tokens).
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

constexpr int kRowThreads = 256;

// Block-wide sum; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  const int nw = blockDim.x >> 5;
  for (int k = 0; k < nw; ++k) t += red[k];
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) embed_concat_kernel(const EmbedConcatArgs a) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;
  int id = a.ids[i];
  if (id < 0 || id >= a.vocab) {
    if (threadIdx.x == 0) record_error(a.err, PE_DEV_BAD_TOKEN);
    id = 0;
  }
  const T* e = static_cast<const T*>(a.emb) + static_cast<size_t>(id) * a.d;
  const float* h = a.h + static_cast<size_t>(i) * a.d;
  float se = 0.f, sh = 0.f;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
    const float ev = to_f(e[c]);
    const float hv = h[c];
    se += ev * ev;
    sh += hv * hv;
  }
  se = block_sum(se, red);
  sh = block_sum(sh, red);
  const float re = rsqrtf(se / a.d + a.eps);
  const float rh = rsqrtf(sh / a.d + a.eps);
  const T* ge = static_cast<const T*>(a.g_e);
  const T* gh = static_cast<const T*>(a.g_h);
  T* x = static_cast<T*>(a.x) + static_cast<size_t>(i) * 2 * a.d;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) {
    x[c] = from_f<T>(to_f(e[c]) * re * to_f(ge[c]));
    x[a.d + c] = from_f<T>(h[c] * rh * to_f(gh[c]));
  }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const RmsNormArgs a) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;
  int src = a.row_index ? a.row_index[i] : i;
  T* y = static_cast<T*>(a.y) + static_cast<size_t>(i) * a.d;
  if (src < 0 || src >= a.rows_in) {
    if (threadIdx.x == 0) record_error(a.err, PE_DEV_BAD_ROW);
    for (int c = threadIdx.x; c < a.d; c += blockDim.x) y[c] = from_f<T>(0.f);
    return;
  }
  const float* x = a.x + static_cast<size_t>(src) * a.d;
  float ss = 0.f;
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) ss += x[c] * x[c];
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / a.d + a.eps);
  const T* g = static_cast<const T*>(a.g);
  for (int c = threadIdx.x; c < a.d; c += blockDim.x) y[c] = from_f<T>(x[c] * r * to_f(g[c]));
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) rope_kv_kernel(const RopeKvArgs a) {
  __shared__ float cs[64], sn[64];
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;
  const int half = a.dh / 2;
  const int p = a.pos[i];
  if (threadIdx.x < half) {
    // angle in fp64, reduced to [0, 2 pi) before the fp32 sine/cosine
    const double two_pi = 6.283185307179586476925286766559;
    double ang = static_cast<double>(p) * a.inv_freq64[threadIdx.x];
    ang -= floor(ang / two_pi) * two_pi;
    float s, c;
    sincosf(static_cast<float>(ang), &s, &c);
    cs[threadIdx.x] = c;
    sn[threadIdx.x] = s;
  }
  __syncthreads();
  const int width = (a.Hq + 2 * a.Hkv) * a.dh;
  const T* qkv = static_cast<const T*>(a.qkv) + static_cast<size_t>(i) * width;
  T* qo = static_cast<T*>(a.q_out) + static_cast<size_t>(i) * a.Hq * a.dh;
  const int sl = a.slot[i];
  int blk = -1, off = 0;
  if (sl >= 0) {
    blk = sl / 16;
    off = sl % 16;
    if (blk >= a.num_blocks) {
      if (threadIdx.x == 0) record_error(a.err, PE_DEV_BAD_BLOCK);
      blk = -1;
    }
  }
  T* kc = static_cast<T*>(a.k_cache);
  T* vc = static_cast<T*>(a.v_cache);
  const int pairs = (a.Hq + a.Hkv) * half;
  for (int w = threadIdx.x; w < pairs; w += blockDim.x) {
    const int h = w / half, t = w % half;
    const float x1 = to_f(qkv[h * a.dh + t]);
    const float x2 = to_f(qkv[h * a.dh + t + half]);
    const float y1 = x1 * cs[t] - x2 * sn[t];
    const float y2 = x2 * cs[t] + x1 * sn[t];
    if (h < a.Hq) {
      qo[h * a.dh + t] = from_f<T>(y1);
      qo[h * a.dh + t + half] = from_f<T>(y2);
    } else if (blk >= 0) {
      const int g = h - a.Hq;
      T* dst = kc + ((static_cast<size_t>(blk) * a.Hkv + g) * 16 + off) * a.dh;
      dst[t] = from_f<T>(y1);
      dst[t + half] = from_f<T>(y2);
    }
  }
  if (blk >= 0) {
    const T* v = qkv + (a.Hq + a.Hkv) * a.dh;
    for (int w = threadIdx.x; w < a.Hkv * a.dh; w += blockDim.x) {
      const int g = w / a.dh, t = w % a.dh;
      vc[((static_cast<size_t>(blk) * a.Hkv + g) * 16 + off) * a.dh + t] = v[w];
    }
  }
}

cudaError_t launch_embed_concat(int dtype, const EmbedConcatArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dtype == PE_DTYPE_BF16)
    return launch_pdl(embed_concat_kernel<bf16>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
  return launch_pdl(embed_concat_kernel<float>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}

cudaError_t launch_rmsnorm(int dtype, const RmsNormArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dtype == PE_DTYPE_BF16)
    return launch_pdl(rmsnorm_kernel<bf16>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
  return launch_pdl(rmsnorm_kernel<float>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}

cudaError_t launch_rope_kv(int dtype, const RopeKvArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dtype == PE_DTYPE_BF16)
    return launch_pdl(rope_kv_kernel<bf16>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
  return launch_pdl(rope_kv_kernel<float>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}

}  // namespace pe
