// gemm_simt.cu -- y = x . w^T with FFMA for the fp32 path (tcgen05 has no
// fp32 operand type), with the projection epilogues of the drafter layer:
// store, residual add, SiLU(gate) * up, and the LM-head argmax.
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

constexpr int SBF = 64, SBT = 16, SBK = 32;  // features x tokens x k per tile

template <bool DUAL>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* __restrict__ x, int ldx,
                                                        const float* __restrict__ w,
                                                        const float* __restrict__ w2, int M,
                                                        int N, int K, const EpiArgs epi) {
  __shared__ float sw[SBF][SBK + 1];
  __shared__ float sw2[DUAL ? SBF : 1][SBK + 1];
  __shared__ float sx[SBT][SBK + 1];
  grid_dep_wait();
  grid_dep_launch();
  const int f0 = blockIdx.x * SBF, t0 = blockIdx.y * SBT;
  if (epi.m_live) {
    // compacted batch: tokens at or past the live count are skipped
    M = min(M, __ldcg(epi.m_live));
    if (t0 >= M) return;
  }
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < K; k0 += SBK) {
    for (int e = threadIdx.x; e < SBF * SBK; e += 256) {
      const int r = e / SBK, c = e % SBK, f = f0 + r, k = k0 + c;
      const bool ok = f < N && k < K;
      sw[r][c] = ok ? w[static_cast<size_t>(f) * K + k] : 0.f;
      if (DUAL) sw2[r][c] = ok ? w2[static_cast<size_t>(f) * K + k] : 0.f;
    }
    for (int e = threadIdx.x; e < SBT * SBK; e += 256) {
      const int r = e / SBK, c = e % SBK, t = t0 + r, k = k0 + c;
      sx[r][c] = (t < M && k < K) ? x[static_cast<size_t>(t) * ldx + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < SBK; ++c) {
      const float xv = sx[ty][c];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[q] = fmaf(sw[tx + 16 * q][c], xv, acc[q]);
        if (DUAL) acc2[q] = fmaf(sw2[tx + 16 * q][c], xv, acc2[q]);
      }
    }
    __syncthreads();
  }
  const int t = t0 + ty;
  if (t >= M) return;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int f = f0 + tx + 16 * q;
    if (f >= N) continue;
    const float v = acc[q];
    switch (epi.kind) {
      case EPI_STORE: {
        const int tr = epi.row_map ? __ldcg(epi.row_map + t) : t;
        if (tr >= 0) static_cast<float*>(epi.out)[static_cast<size_t>(tr) * epi.ldo + f] = v;
        break;
      }
      case EPI_ADD:
        epi.resid[static_cast<size_t>(t) * epi.ldr + f] += v;
        break;
      case EPI_SILU_MUL:
        static_cast<float*>(epi.out)[static_cast<size_t>(t) * epi.ldo + f] = silu_f(v) * acc2[q];
        break;
      case EPI_ARGMAX:
        if (epi.logits) epi.logits[static_cast<size_t>(t) * epi.ldl + f] = v;
        atomicMax(epi.keys + t, argmax_key(v, f));
        break;
    }
  }
}

__global__ void argmax_finalize_kernel(int M, unsigned long long* keys, int32_t* tokens) {
  grid_dep_wait();
  grid_dep_launch();
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < M; t += gridDim.x * blockDim.x) {
    const unsigned long long k = keys[t];
    tokens[t] = k ? argmax_key_index(k) : -1;
    keys[t] = 0ull;
  }
}

cudaError_t launch_gemm_simt(const float* x, int ldx, const float* w, const float* w2, int M,
                             int N, int K, const EpiArgs& epi, int* err, cudaStream_t s) {
  (void)err;
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + SBF - 1) / SBF, (M + SBT - 1) / SBT);
  if (w2) return launch_pdl(gemm_simt_kernel<true>, grid, dim3(256), 0, s, x, ldx, w, w2, M, N, K, epi);
  return launch_pdl(gemm_simt_kernel<false>, grid, dim3(256), 0, s, x, ldx, w, w, M, N, K, epi);
}

cudaError_t launch_argmax_finalize(int M, unsigned long long* keys, int32_t* tokens,
                                   cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_pdl(argmax_finalize_kernel, dim3((M + 255) / 256), dim3(256), 0, s, M, keys, tokens);
}

}  // namespace pe
