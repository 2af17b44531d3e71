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
#include "fp8_common.cuh"
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

constexpr int kRowThreads = 256;

// cos and sin of the rotary angles of one row (threads k < dh / 2; the
// angle in fp64, reduced to [-pi, pi] before the fp32 sine and cosine, as
// in the RoPE kernel below)
__device__ __forceinline__ void rope_table_row(const EmbedConcatArgs& a, int i) {
  if (!a.rope_tab) return;
  const int half = a.dh / 2;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const double two_pi = 6.283185307179586476925286766559;
    const double ang = static_cast<double>(a.pos[i]) * a.inv_freq64[k];
    const double red_ang = ang - rint(ang * (1.0 / two_pi)) * two_pi;
    float sv, cv;
    sincosf(static_cast<float>(red_ang), &sv, &cv);
    a.rope_tab[static_cast<size_t>(i) * a.dh + k] = cv;
    a.rope_tab[static_cast<size_t>(i) * a.dh + half + k] = sv;
  }
}

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
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
  int id = a.ids[i];
  if (id < 0 || id >= a.vocab) {
    if (threadIdx.x == 0) record_error(a.err, PE_DEV_BAD_TOKEN);
    id = 0;
  }
  const T* e = static_cast<const T*>(a.emb) + static_cast<size_t>(id) * a.d;
  // a MASK row's projected hidden state is the fc of h_shared
  const bool mrow = a.masked && a.masked[i];
  const float* h = mrow ? a.fc_hs : a.h + static_cast<size_t>(i) * a.d;
  if (mrow)
    for (int c = threadIdx.x; c < a.d; c += blockDim.x)
      a.h_w[static_cast<size_t>(i) * a.d + c] = h[c];
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
  rope_table_row(a, i);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const RmsNormArgs a) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
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
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
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

// ---------------------------------------------------------------------------
// Vectorised variants.  These kernels move little data and sit between
// projections on the critical path, so their cost is the latency of their
// dependent memory round trips: every operand of the row is loaded into
// registers with 16-byte (fp32 residual) or 8-byte (4 x bf16) accesses
// before any arithmetic, the norm gains are fetched before the wait on
// earlier kernels (they are weights), and the reduction runs once.  The
// scalar kernels above stay for widths or pointers these cannot take.

__device__ __forceinline__ void ld4(const float* p, float v[4]) {
  const float4 r = *reinterpret_cast<const float4*>(p);
  v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
}
__device__ __forceinline__ void ld4(const bf16* p, float v[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void st4(float* p, const float v[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st4(bf16* p, const float v[4]) {
  uint2 r;
  r.x = pack_bf16x2(v[0], v[1]);
  r.y = pack_bf16x2(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = r;
}

// NV groups of 4 columns per thread: d <= 4 * NV * kRowThreads.
template <typename T, int NV>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_vec_kernel(const RmsNormArgs a) {
  __shared__ float red[32];
  const int n4 = a.d >> 2;
  const T* __restrict__ gp = static_cast<const T*>(a.g);
  float g[NV][4];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c4 = threadIdx.x + j * kRowThreads;
    if (c4 < n4) ld4(gp + 4 * c4, g[j]);
  }
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
  const int src = a.row_index ? a.row_index[i] : i;
  T* __restrict__ y = static_cast<T*>(a.y) + static_cast<size_t>(i) * a.d;
  const bool bad = src < 0 || src >= a.rows_in;
  if (bad && threadIdx.x == 0) record_error(a.err, PE_DEV_BAD_ROW);
  const float* __restrict__ x = a.x + static_cast<size_t>(bad ? 0 : src) * a.d;
  float v[NV][4];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c4 = threadIdx.x + j * kRowThreads;
    if (c4 < n4) {
      ld4(x + 4 * c4, v[j]);
      if (bad) v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.f;
    } else {
      v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.f;
    }
  }
  if (a.add && !bad) {
    // the deferred residual add: x + add, written back (all loads first)
    const float* __restrict__ ad = a.add + static_cast<size_t>(src) * a.d;
    float t[NV][4];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c4 = threadIdx.x + j * kRowThreads;
      if (c4 < n4) ld4(ad + 4 * c4, t[j]);
    }
    float* __restrict__ xw = a.x_w + static_cast<size_t>(src) * a.d;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int c4 = threadIdx.x + j * kRowThreads;
      if (c4 < n4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[j][q] = v[j][q] + t[j][q];
        *reinterpret_cast<float4*>(xw + 4 * c4) = make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NV; ++j)
    ss += v[j][0] * v[j][0] + v[j][1] * v[j][1] + v[j][2] * v[j][2] + v[j][3] * v[j][3];
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / a.d + a.eps);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c4 = threadIdx.x + j * kRowThreads;
    if (c4 < n4) {
      float o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = v[j][q] * r * g[j][q];
      st4(y + 4 * c4, o);
    }
  }
}

template <typename T, int NV>
__global__ void __launch_bounds__(kRowThreads) embed_concat_vec_kernel(const EmbedConcatArgs a) {
  __shared__ float red[32];
  const int n4 = a.d >> 2;
  const T* __restrict__ gep = static_cast<const T*>(a.g_e);
  const T* __restrict__ ghp = static_cast<const T*>(a.g_h);
  float ge[NV][4], gh[NV][4];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c4 = threadIdx.x + j * kRowThreads;
    if (c4 < n4) {
      ld4(gep + 4 * c4, ge[j]);
      ld4(ghp + 4 * c4, gh[j]);
    }
  }
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x;
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
  int id = a.ids[i];
  if (id < 0 || id >= a.vocab) {
    if (threadIdx.x == 0) record_error(a.err, PE_DEV_BAD_TOKEN);
    id = 0;
  }
  const T* __restrict__ e = static_cast<const T*>(a.emb) + static_cast<size_t>(id) * a.d;
  // a MASK row's projected hidden state is the fc of h_shared
  const bool mrow = a.masked && a.masked[i];
  const float* __restrict__ h = mrow ? a.fc_hs : a.h + static_cast<size_t>(i) * a.d;
  float ev[NV][4], hv[NV][4];
  float se = 0.f, sh = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c4 = threadIdx.x + j * kRowThreads;
    if (c4 < n4) {
      ld4(e + 4 * c4, ev[j]);
      ld4(h + 4 * c4, hv[j]);
      if (mrow) st4(a.h_w + static_cast<size_t>(i) * a.d + 4 * c4, hv[j]);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) ev[j][q] = hv[j][q] = 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < NV; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      se += ev[j][q] * ev[j][q];
      sh += hv[j][q] * hv[j][q];
    }
  // both sums in one pass through shared memory
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    se += __shfl_xor_sync(0xffffffffu, se, o);
    sh += __shfl_xor_sync(0xffffffffu, sh, o);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[w] = se;
    red[16 + w] = sh;
  }
  __syncthreads();
  se = 0.f;
  sh = 0.f;
#pragma unroll
  for (int k = 0; k < kRowThreads / 32; ++k) {
    se += red[k];
    sh += red[16 + k];
  }
  const float re = rsqrtf(se / a.d + a.eps);
  const float rh = rsqrtf(sh / a.d + a.eps);
  T* __restrict__ x = static_cast<T*>(a.x) + static_cast<size_t>(i) * 2 * a.d;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c4 = threadIdx.x + j * kRowThreads;
    if (c4 < n4) {
      float oe[4], oh[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        oe[q] = ev[j][q] * re * ge[j][q];
        oh[q] = hv[j][q] * rh * gh[j][q];
      }
      st4(x + 4 * c4, oe);
      st4(x + a.d + 4 * c4, oh);
    }
  }
  rope_table_row(a, i);
}

// 16-byte vectors of the head dimension: EPV elements each.  A rope item is
// EPV columns of the first half of one q or k head and the matching EPV
// columns of its second half; a v item is EPV columns of one v head.
template <typename T>
struct RopeVec {
  static constexpr int EPV = 16 / static_cast<int>(sizeof(T));
  static constexpr int PER_THREAD = 2;  // items a thread takes, loads hoisted
};

__device__ __forceinline__ void ldv(const bf16* p, float v[8]) {
  const uint4 r = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    v[2 * k] = f.x;
    v[2 * k + 1] = f.y;
  }
}
__device__ __forceinline__ void ldv(const float* p, float v[4]) { ld4(p, v); }
__device__ __forceinline__ void stv(bf16* p, const float v[8]) {
  uint4 r;
  r.x = pack_bf16x2(v[0], v[1]);
  r.y = pack_bf16x2(v[2], v[3]);
  r.z = pack_bf16x2(v[4], v[5]);
  r.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void stv(float* p, const float v[4]) { st4(p, v); }
// eight values -> eight e4m3 codes of v * inv (an fp8 pool row, 8 bytes)
__device__ __forceinline__ void stv_e4m3(uint8_t* p, const float v[8], float inv) {
  uint2 r;
  r.x = static_cast<uint32_t>(f32x2_to_e4m3x2(v[0] * inv, v[1] * inv)) |
        (static_cast<uint32_t>(f32x2_to_e4m3x2(v[2] * inv, v[3] * inv)) << 16);
  r.y = static_cast<uint32_t>(f32x2_to_e4m3x2(v[4] * inv, v[5] * inv)) |
        (static_cast<uint32_t>(f32x2_to_e4m3x2(v[6] * inv, v[7] * inv)) << 16);
  *reinterpret_cast<uint2*>(p) = r;
}

// FP8: the K and V rows go to e4m3 pools (bf16 activations only).
template <typename T, bool FP8 = false>
__global__ void __launch_bounds__(kRowThreads) rope_kv_vec_kernel(const RopeKvArgs a) {
  using R = RopeVec<T>;
  constexpr int E = R::EPV;
  __shared__ float cs[64], sn[64];
  // The positions, slots and live count come from the expansion and the
  // compaction, several launches back (each kernel waits for its
  // predecessor before its dependents may start), so the rotary angles and
  // the cache slot are worked out before the wait for the QKV projection,
  // the one input that kernel writes.  Row 0 is always live: its CTA waits,
  // so this grid never completes before the projection does.
  const int i = blockIdx.x;
  if (a.live && i >= __ldcg(a.live)) return;  // past the live rows
  const int half = a.dh / 2;
  if (threadIdx.x < half) {
    // angle in fp64, reduced to [-pi, pi] before the fp32 sine/cosine
    const double two_pi = 6.283185307179586476925286766559;
    const double ang = static_cast<double>(a.pos[i]) * a.inv_freq64[threadIdx.x];
    const double red_ang = ang - rint(ang * (1.0 / two_pi)) * two_pi;
    float sv, cv;
    sincosf(static_cast<float>(red_ang), &sv, &cv);
    cs[threadIdx.x] = cv;
    sn[threadIdx.x] = sv;
  }
  const int width = (a.Hq + 2 * a.Hkv) * a.dh;
  const T* __restrict__ qkv = static_cast<const T*>(a.qkv) + static_cast<size_t>(i) * width;
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
  grid_dep_wait();
  grid_dep_launch();
  const int gpr = half / E;                        // vectors per half head
  const int n_rope = (a.Hq + a.Hkv) * gpr;
  const int n_v = blk >= 0 ? a.Hkv * a.dh / E : 0;
  // all loads first
  float x1[R::PER_THREAD][E], x2[R::PER_THREAD][E];
  int item[R::PER_THREAD];
#pragma unroll
  for (int k = 0; k < R::PER_THREAD; ++k) {
    const int it = threadIdx.x + k * kRowThreads;
    item[k] = it;
    if (it < n_rope) {
      const int h = it / gpr, t = (it % gpr) * E;
      ldv(qkv + h * a.dh + t, x1[k]);
      ldv(qkv + h * a.dh + half + t, x2[k]);
    } else if (it < n_rope + n_v) {
      ldv(qkv + (a.Hq + a.Hkv) * a.dh + (it - n_rope) * E, x1[k]);
    }
  }
  __syncthreads();                                  // cs / sn ready
  T* __restrict__ qo = static_cast<T*>(a.q_out) + static_cast<size_t>(i) * a.Hq * a.dh;
  T* __restrict__ kc = static_cast<T*>(a.k_cache);
  T* __restrict__ vc = static_cast<T*>(a.v_cache);
#pragma unroll
  for (int k = 0; k < R::PER_THREAD; ++k) {
    const int it = item[k];
    if (it < n_rope) {
      const int h = it / gpr, t = (it % gpr) * E;
      float y1[E], y2[E];
#pragma unroll
      for (int q = 0; q < E; ++q) {
        y1[q] = x1[k][q] * cs[t + q] - x2[k][q] * sn[t + q];
        y2[q] = x2[k][q] * cs[t + q] + x1[k][q] * sn[t + q];
      }
      if (h < a.Hq) {
        stv(qo + h * a.dh + t, y1);
        stv(qo + h * a.dh + half + t, y2);
      } else if (blk >= 0) {
        const size_t row = ((static_cast<size_t>(blk) * a.Hkv + (h - a.Hq)) * 16 + off) * a.dh;
        if constexpr (FP8) {
          uint8_t* dst = static_cast<uint8_t*>(a.k_cache) + row;
          stv_e4m3(dst + t, y1, a.k_inv_scale);
          stv_e4m3(dst + half + t, y2, a.k_inv_scale);
        } else {
          stv(kc + row + t, y1);
          stv(kc + row + half + t, y2);
        }
      }
    } else if (it < n_rope + n_v) {
      const int w = (it - n_rope) * E;
      const int g = w / a.dh, t = w % a.dh;
      const size_t row = ((static_cast<size_t>(blk) * a.Hkv + g) * 16 + off) * a.dh;
      if constexpr (FP8) stv_e4m3(static_cast<uint8_t*>(a.v_cache) + row + t, x1[k], a.v_inv_scale);
      else stv(vc + row + t, x1[k]);
    }
  }
}

namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// groups of 4 columns a thread takes in the vector kernels; 0: scalar kernel
int row_nv(int d) {
  if (d % 4) return 0;
  const int nv = (d / 4 + kRowThreads - 1) / kRowThreads;
  return nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 8 ? 8 : 0;
}
template <typename T, int NV>
cudaError_t rms_vec(const RmsNormArgs& a, cudaStream_t s) {
  return launch_pdl(rmsnorm_vec_kernel<T, NV>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}
template <typename T>
cudaError_t rms_launch(const RmsNormArgs& a, cudaStream_t s) {
  const int nv = al16(a.x) && al16(a.y) && al16(a.g) ? row_nv(a.d) : 0;
  // the deferred residual add runs in the vector kernel only
  if (a.add && (nv == 0 || a.row_index || !al16(a.add) || a.x_w != a.x))
    return cudaErrorInvalidValue;
  switch (nv) {
    case 1: return rms_vec<T, 1>(a, s);
    case 2: return rms_vec<T, 2>(a, s);
    case 4: return rms_vec<T, 4>(a, s);
    case 8: return rms_vec<T, 8>(a, s);
    default: return launch_pdl(rmsnorm_kernel<T>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
  }
}
template <typename T, int NV>
cudaError_t emb_vec(const EmbedConcatArgs& a, cudaStream_t s) {
  return launch_pdl(embed_concat_vec_kernel<T, NV>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}
template <typename T>
cudaError_t emb_launch(const EmbedConcatArgs& a, cudaStream_t s) {
  // every row of emb and x starts 16-byte aligned when the bases do and a
  // row of d elements is a whole number of 16-byte vectors
  const bool ok = al16(a.emb) && al16(a.h) && al16(a.g_e) && al16(a.g_h) && al16(a.x) &&
                  (a.d * static_cast<int>(sizeof(T))) % 16 == 0;
  const int nv = ok ? row_nv(a.d) : 0;
  switch (nv) {
    case 1: return emb_vec<T, 1>(a, s);
    case 2: return emb_vec<T, 2>(a, s);
    case 4: return emb_vec<T, 4>(a, s);
    case 8: return emb_vec<T, 8>(a, s);
    default: return launch_pdl(embed_concat_kernel<T>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
  }
}
template <typename T>
cudaError_t rope_launch(const RopeKvArgs& a, cudaStream_t s) {
  constexpr int E = RopeVec<T>::EPV;
  const int half = a.dh / 2;
  const bool ok = al16(a.qkv) && al16(a.q_out) && al16(a.k_cache) && al16(a.v_cache) &&
                  half % E == 0 &&
                  (a.Hq + a.Hkv) * (half / E) + a.Hkv * a.dh / E <=
                      RopeVec<T>::PER_THREAD * kRowThreads;
  if (a.kv_fp8) {
    if constexpr (sizeof(T) == 2) {
      if (ok) return launch_pdl(rope_kv_vec_kernel<T, true>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
    }
    return cudaErrorInvalidValue;
  }
  if (ok) return launch_pdl(rope_kv_vec_kernel<T>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
  return launch_pdl(rope_kv_kernel<T>, dim3(a.rows), dim3(kRowThreads), 0, s, a);
}
}  // namespace

cudaError_t launch_embed_concat(int dtype, const EmbedConcatArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  return dtype == PE_DTYPE_BF16 ? emb_launch<bf16>(a, s) : emb_launch<float>(a, s);
}

cudaError_t launch_rmsnorm(int dtype, const RmsNormArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  return dtype == PE_DTYPE_BF16 ? rms_launch<bf16>(a, s) : rms_launch<float>(a, s);
}

cudaError_t launch_rope_kv(int dtype, const RopeKvArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  return dtype == PE_DTYPE_BF16 ? rope_launch<bf16>(a, s) : rope_launch<float>(a, s);
}

}  // namespace pe
