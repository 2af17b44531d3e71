// noalloc.cu -- pe_linear_static: the bf16 tensor-core projection
// y = x . w^T for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a
// custom allocator or memory-pool callback, in a process whose device memory
// is carved up and owned by a framework that forbids side allocations, or
// in a latency-critical path that must never hit the driver's allocator.
// pe_create allocates its workspace, so such callers cannot use pe_linear.
//
// The split-K partial tiles and per-tile counters of the GEMM live instead
// in one file-scope device array (kScratchBytes, below).  Every GPU that
// loads this library reserves that array until the process exits.  Host
// code cannot use the array's name as a device address, so the first call
// on each device looks the address up (cudaGetSymbolAddress) with that
// device current and caches it; make that first call before any stream
// capture.  All calls share the one array: calls that overlap on the GPU
// (different streams, or different host threads on one device) race on it.
//
// A bounded wait inside the GEMM that gives up records PE_DEV_TIMEOUT in an
// error word that also lives in the array; it stays set across calls until
// pe_linear_static_error reads and clears it.
#include <mutex>

#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {
cudaError_t init_gemm_tc();
cudaError_t launch_gemm_tc_maps(const CUtensorMap& wa, const CUtensorMap& wa2,
                                const CUtensorMap& xb, bool dual, int M, int N, int K,
                                const EpiArgs& epi, const TcGemmWorkspace& ws, int* err,
                                cudaStream_t s);
int tc_b_box_rows(int M, int N, int sm_count, bool dual, bool live_rows);
}  // namespace pe

namespace {

// Limits of the static workspace: at most 32 tokens (one 32-wide token
// tile), at most kMaxTiles output tiles of 128 features, and split-K
// partials for one CTA per SM on GPUs of up to kMaxSms SMs (two CTAs per SM
// at 16 tokens or fewer); a GPU with more SMs runs on kMaxSms of them.
constexpr int kMaxTokens = 32;
constexpr int kMaxSms = 160;
constexpr int kMaxTiles = 4096;
constexpr size_t kPartialFloats = static_cast<size_t>(kMaxSms) * 2 * 128 * kMaxTokens;
constexpr size_t kScratchBytes =
    kPartialFloats * sizeof(float) + (kMaxTiles + 64) * sizeof(int);  // ~5.3 MB

// [partials: kPartialFloats floats][tile counters: kMaxTiles ints][error word]
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceSlot {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_scratch
  int sm_count = 0;
};
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceSlot g_slots[kMaxDevices];

// Once per device, with that device current: find the array's device
// address, opt the GEMM kernels into their shared memory, read the SM count.
cudaError_t device_setup(DeviceSlot** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    e = pe::init_gemm_tc();
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<unsigned char*>(p);
    s.sm_count = sms;
    s.ready = true;
  }
  *out = &s;
  return cudaSuccess;
}

}  // namespace

extern "C" pe_status pe_linear_static(const void* x, const void* w, float* y, int32_t M,
                                      int32_t N, int32_t K, void* stream) {
  using namespace pe;
  if (!x || !w || !y || M < 1 || N < 1 || K < 8 || K % 8 != 0) return PE_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(w) & 15))
    return PE_ERR_INVALID_ARGUMENT;
  // sizes beyond the static workspace are refused before anything launches
  if (M > kMaxTokens || (N + 127) / 128 > kMaxTiles) return PE_ERR_UNSUPPORTED;
  DeviceSlot* slot = nullptr;
  if (device_setup(&slot) != cudaSuccess) return PE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* partials = reinterpret_cast<float*>(slot->scratch);
  int* counters = reinterpret_cast<int*>(slot->scratch + kPartialFloats * sizeof(float));
  int* err = counters + kMaxTiles;
  // the tile counters must start at zero; the error word is left for
  // pe_linear_static_error
  if (cudaMemsetAsync(counters, 0, kMaxTiles * sizeof(int), s) != cudaSuccess)
    return PE_ERR_CUDA;
  const int sms = slot->sm_count < kMaxSms ? slot->sm_count : kMaxSms;
  CUtensorMap wa, xb;
  if (!tensor_map_2d_bf16(&wa, w, N, K, K, 64, 128) ||
      !tensor_map_2d_bf16(&xb, x, M, K, K, 64, tc_b_box_rows(M, N, sms, false, false)))
    return PE_ERR_INVALID_ARGUMENT;
  TcGemmWorkspace ws = {};
  ws.partials = partials;
  ws.partial_floats = kPartialFloats;
  ws.tile_counters = counters;
  ws.max_tiles = kMaxTiles;
  ws.done_counter = nullptr;  // only the argmax epilogue uses it
  ws.timeline = nullptr;
  ws.cluster_push = 1;
  ws.pre_stages = -1;
  ws.max_split = 8;
  ws.tile_order = 0;   // one weight-tile-major order for these launches
  ws.l2_bytes = 0;
  ws.sm_count = sms;
  EpiArgs ep = {};
  ep.kind = EPI_STORE;
  ep.M = M;
  ep.N = N;
  ep.out = y;
  ep.ldo = N;
  ep.out_f32 = 1;
  const cudaError_t e = launch_gemm_tc_maps(wa, wa, xb, false, M, N, K, ep, ws, err, s);
  if (e == cudaErrorInvalidValue) return PE_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

// Read and clear the error word of the static array (0: no violation
// recorded since the last read).  Copies on `stream` and waits for it, so
// it also orders after every pe_linear_static call issued there.
extern "C" pe_status pe_linear_static_error(int32_t* code, void* stream) {
  if (!code) return PE_ERR_INVALID_ARGUMENT;
  DeviceSlot* slot = nullptr;
  if (device_setup(&slot) != cudaSuccess) return PE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = reinterpret_cast<int*>(slot->scratch + kPartialFloats * sizeof(float)) + kMaxTiles;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *code = v;
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}
