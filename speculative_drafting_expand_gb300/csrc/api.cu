// api.cu -- the C ABI declared in include/peagle.h: handle and workspace,
// host-side validation, and the order of kernels in one drafting step.
#include <algorithm>
#include <cmath>
#include <map>
#include <new>
#include <tuple>
#include <vector>

#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {
cudaError_t launch_gemm_tc_maps(const CUtensorMap& wa, const CUtensorMap& wa2,
                                const CUtensorMap& xb, bool dual, int M, int N, int K,
                                const EpiArgs& epi, const TcGemmWorkspace& ws, int* err,
                                cudaStream_t s);
int tc_pick_bn(int M, bool dual);
int tc_b_box_rows(int M, int N, int sm_count, bool dual, bool live_rows);
cudaError_t init_gemm_tc();
size_t tc_partial_floats(int grid, int bn, bool dual);
cudaError_t init_attention_tc();
bool tensor_map_2d_u8(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);
size_t attention_tc_partial_floats(const AttnArgs& a, int max_rows_per_req, int sm_count,
                                   int min_cps, int max_cps);
size_t attention_tc_counters(const AttnArgs& a, int max_rows_per_req, int sm_count, int min_cps,
                             int max_cps);
cudaError_t launch_attention_tc(const AttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const int32_t* seq_lens, int max_rows_per_req, int sm_count,
                                float* part, size_t part_floats, int* counters,
                                size_t n_counters, unsigned long long* timeline, int l2_ahead,
                                int min_cps, int max_cps, const int32_t* order,
                                cudaStream_t s);
int attention_tc_order_entries(const AttnArgs& a, int max_rows_per_req, int sm_count, int min_cps,
                               int max_cps);
cudaError_t launch_attention_order(const AttnArgs& a, const int32_t* seq_lens,
                                   int max_rows_per_req, int sm_count, int min_cps, int max_cps,
                                   int32_t* order, cudaStream_t s);
cudaError_t launch_bounded_wait_check(int* flag, int32_t* out, int* err, cudaStream_t s);
}  // namespace pe

namespace {
// streaming-segment workspace: tile counters and sums of squares per phase
constexpr int kStreamCounterStride = 1024;  // tiles of one phase, at most
constexpr int kStreamSsqTiles = 256;        // residual tiles of 128 features, at most
}  // namespace

using namespace pe;

struct pe_handle {
  pe_model_desc desc;
  pe_weights w;
  std::vector<pe_layer_weights> layers;
  int device = 0;
  int sm_count = 0;
  int max_tokens = 0, max_reqs = 0;
  size_t esize = 2;  // bytes per element of the model dtype

  int* err = nullptr;
  int* diag_flag = nullptr;  // the flag the bounded-wait self-check waits on
  float* resid = nullptr;   // [max_tokens, d] fp32 residual stream
  float* o_delta = nullptr; // [max_tokens, d] fp32 O-projection output, added by the next norm
  void* x_in = nullptr;     // [max_tokens, 2d] QKV input
  void* qkv = nullptr;      // [max_tokens, (Hq + 2Hkv) dh]
  void* q = nullptr;        // [max_tokens, Hq dh] rotated queries
  void* attn = nullptr;     // [max_tokens, Hq dh]
  void* xn = nullptr;       // [max_tokens, d] MLP input
  void* act = nullptr;      // [max_tokens, F]
  unsigned long long* keys = nullptr;  // [max_tokens] argmax keys (kept zero)
  double* inv_freq64 = nullptr;        // [dh / 2]
  float* rope_tab = nullptr;           // [max_tokens, dh] cos / sin of each row's angles
  int fusions = PE_FUSE_NORM;          // epilogue fusions of the per-projection path
  int cluster_push = PE_REDUCE_PUSH;   // cluster split-K reduction: push (1) or pull (0)
  // projection weight stages loaded before the dependency wait: three
  // (measured on the GPT-OSS-20B-shaped batch-1 step: 498-505 us against
  // 505-513 us with all five; fewer weight loads compete with the previous
  // kernel's epilogue; no change at batch 64)
  int gemm_pre_stages = 3;
  // K/V chunks the attention brings into L2 ahead of its shared-memory ring:
  // none (measured slower with 2, 4 or 8 at batch 1, batch 64 and the Qwen
  // batch-16 step: 2900 -> 3230 us at batch 64)
  int attn_l2_ahead = 0;
  int gemm_max_split = 8;              // the largest cluster split-K of a projection
  // stream-K over several token tiles, weights larger than L2: token-tile-major
  int gemm_tile_order = 1;
  int l2_bytes = 0;                    // the device's L2 size
  int attn_min_chunks = 2;             // the fewest 128-key chunks an attention split takes
  // the most (a split's block ids: at most 64 chunks at dh 64, 32 at dh
  // 128); longer splits measured better at batch 64 (16: 2757, 32: 2576, 64:
  // 2544-2561 us a step), fewer CTAs each paying its setup and merge
  int attn_max_chunks = 64;
  float* fc_hs = nullptr;              // [d] fc(h_shared), the projected hidden of every MASK row
  int32_t* fc_map = nullptr;           // [max_tokens] target row -> compact row
  uint8_t* masked_c = nullptr;         // [max_tokens] MASK flag of every compact row
  float* ssq_post = nullptr;           // [ceil(d / 32), max_tokens] folded-norm sums
  float* ssq_in = nullptr;
  float* gemm_partials = nullptr;
  size_t gemm_partial_floats = 0;
  int* tile_counters = nullptr;
  int max_tiles = 0;
  int* done_counter = nullptr;
  float* attn_partials = nullptr;
  size_t attn_partial_floats = 0;
  int* attn_counters = nullptr;
  int32_t* attn_order = nullptr;       // attention work items, longest first
  size_t attn_order_cap = 0;
  size_t attn_n_counters = 0;
  // live-row compaction of the expanded batch (compact.cu)
  int32_t* row_map = nullptr;      // [max_tokens]
  int32_t* live_before = nullptr;  // [max_tokens + 1]
  int32_t* live_row = nullptr;     // [max_tokens]
  int32_t* ids_c = nullptr;        // [max_tokens]
  int32_t* pos_c = nullptr;
  int32_t* slot_c = nullptr;
  int32_t* cu_live = nullptr;      // [max_reqs + 1]
  int32_t* new_c = nullptr;        // [max_tokens]
  int32_t* n_live = nullptr;       // [1]
  // fp8 (e4m3) KV pools: one K and one V scale per layer
  bool kv_fp8 = false;
  std::vector<float> k_scales, v_scales;
  float* trace = nullptr;
  void* attn_trace = nullptr;
  std::vector<cudaEvent_t> phase_events;  // 2 + 2 L events, or none
  // small batches: projections between attention launches as one
  // persistent kernel per segment (stream.cu)
  bool stream_on = false;
  unsigned long long* stream_timeline = nullptr;  // diagnostic, caller-owned
  unsigned long long* gemm_timeline = nullptr;    // diagnostic, caller-owned
  int gemm_timeline_launches = 0;
  int gemm_ordinal = 0;                           // projection launches since the step began
  int stream_prefetch = 0;  // weight tiles prefetched into L2 ahead of the ring
  int stream_boundary = -1;  // loads into a phase before its inputs are ready (-1: any)
  float* stream_ws = nullptr;
  int* stream_sync = nullptr;
  int* stream_counters = nullptr;
  float* stream_ssq = nullptr;
  long long launches = 0;

  std::map<std::tuple<const void*, uint64_t, uint64_t, uint64_t, uint32_t>, CUtensorMap> maps;
  std::map<std::pair<const void*, uint64_t>, CUtensorMap> maps_u8;  // fp8 pools
  std::map<std::pair<const void*, uint64_t>, CUtensorMap> maps_qkv;  // interleaved QKV weights
  // the QKV weights with each head's halves interleaved (row 2i + b = row
  // i + b dh/2), one copy per layer, for the fused RoPE epilogue
  std::vector<void*> qkv_il;
  std::vector<void*> allocations;
};

namespace {

pe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PE_OK : PE_ERR_CUDA; }

// Count one kernel launch of the handle when it was issued successfully.
cudaError_t counted(pe_handle* h, cudaError_t e) {
  if (e == cudaSuccess) ++h->launches;
  return e;
}

template <typename T>
cudaError_t dev_alloc(pe_handle* h, T** p, size_t count) {
  void* raw = nullptr;
  cudaError_t e = cudaMalloc(&raw, std::max<size_t>(count, 1) * sizeof(T));
  if (e != cudaSuccess) return e;
  h->allocations.push_back(raw);
  *p = static_cast<T*>(raw);
  return cudaMemset(raw, 0, std::max<size_t>(count, 1) * sizeof(T));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

const CUtensorMap* get_map(pe_handle* h, const void* ptr, uint64_t rows, uint64_t cols,
                           uint64_t ld, uint32_t box_rows) {
  auto key = std::make_tuple(ptr, rows, cols, ld, box_rows);
  auto it = h->maps.find(key);
  if (it != h->maps.end()) return &it->second;
  CUtensorMap m;
  if (!tensor_map_2d_bf16(&m, ptr, rows, cols, ld, 64, box_rows)) return nullptr;
  return &h->maps.emplace(key, m).first->second;
}

const CUtensorMap* get_map_u8(pe_handle* h, const void* ptr, uint64_t rows) {
  auto key = std::make_pair(ptr, rows);
  auto it = h->maps_u8.find(key);
  if (it != h->maps_u8.end()) return &it->second;
  CUtensorMap m;
  if (!tensor_map_2d_u8(&m, ptr, rows, h->desc.head_dim, 16)) return nullptr;
  return &h->maps_u8.emplace(key, m).first->second;
}

const CUtensorMap* get_map_qkv(pe_handle* h, const void* ptr, uint64_t K) {
  auto key = std::make_pair(ptr, K);
  auto it = h->maps_qkv.find(key);
  if (it != h->maps_qkv.end()) return &it->second;
  CUtensorMap m;
  const pe_model_desc& d = h->desc;
  if (!tensor_map_qkv_interleaved(&m, ptr, d.n_heads + 2 * d.n_kv_heads, d.head_dim, K))
    return nullptr;
  return &h->maps_qkv.emplace(key, m).first->second;
}

// Copy every layer's QKV weight with each head's halves interleaved (one
// strided copy per head half; synchronous, at set-up).
cudaError_t make_interleaved_qkv(pe_handle* h) {
  const pe_model_desc& d = h->desc;
  const int heads = d.n_heads + 2 * d.n_kv_heads, half = d.head_dim / 2;
  for (int l = 0; l < d.n_layers; ++l) {
    const size_t K = l == 0 ? 2 * d.d : d.d, rb = K * 2;
    unsigned char* dst = nullptr;
    cudaError_t e = dev_alloc(h, &dst, static_cast<size_t>(heads) * d.head_dim * rb);
    if (e != cudaSuccess) return e;
    const unsigned char* src = static_cast<const unsigned char*>(h->layers[l].qkv);
    for (int hd = 0; hd < heads && e == cudaSuccess; ++hd)
      for (int b = 0; b < 2 && e == cudaSuccess; ++b)
        e = cudaMemcpy2D(dst + (static_cast<size_t>(hd) * d.head_dim + b) * rb, 2 * rb,
                         src + (static_cast<size_t>(hd) * d.head_dim + b * half) * rb, rb, rb, half,
                         cudaMemcpyDeviceToDevice);
    if (e != cudaSuccess) return e;
    h->qkv_il.push_back(dst);
  }
  return cudaDeviceSynchronize();
}

TcGemmWorkspace tc_ws(pe_handle* h) {
  TcGemmWorkspace ws = {};
  ws.timeline = nullptr;
  if (h->gemm_timeline && h->gemm_ordinal < h->gemm_timeline_launches)
    ws.timeline = h->gemm_timeline + static_cast<size_t>(h->gemm_ordinal) * 512 * 16;
  ++h->gemm_ordinal;
  ws.partials = h->gemm_partials;
  ws.partial_floats = h->gemm_partial_floats;
  ws.tile_counters = h->tile_counters;
  ws.max_tiles = h->max_tiles;
  ws.done_counter = h->done_counter;
  ws.sm_count = h->sm_count;
  ws.cluster_push = h->cluster_push;
  ws.pre_stages = h->gemm_pre_stages;
  ws.max_split = h->gemm_max_split;
  ws.tile_order = h->gemm_tile_order;
  ws.l2_bytes = h->l2_bytes;
  return ws;
}

// y = x . w^T (+ epilogue) with the GEMM of the model dtype.
cudaError_t linear(pe_handle* h, const void* x, int ldx, const void* w, const void* w2, int M,
                   int N, int K, const EpiArgs& epi, cudaStream_t s) {
  if (h->desc.dtype == PE_DTYPE_F32)
    return counted(h, launch_gemm_simt(static_cast<const float*>(x), ldx,
                                       static_cast<const float*>(w),
                                       static_cast<const float*>(w2), M, N, K, epi, h->err, s));
  const CUtensorMap* wa = get_map(h, w, N, K, K, 128);
  const CUtensorMap* wa2 = w2 ? get_map(h, w2, N, K, K, 128) : wa;
  const CUtensorMap* xb = get_map(h, x, M, K, ldx, tc_b_box_rows(M, N, h->sm_count, w2 != nullptr, epi.m_live != nullptr));
  if (!wa || !wa2 || !xb) return cudaErrorInvalidValue;
  return counted(h, launch_gemm_tc_maps(*wa, *wa2, *xb, w2 != nullptr, M, N, K, epi, tc_ws(h),
                                        h->err, s));
}

EpiArgs epi_none() {
  EpiArgs e = {};
  return e;
}

}  // namespace

extern "C" {

const char* pe_status_string(pe_status s) {
  switch (s) {
    case PE_OK: return "ok";
    case PE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PE_ERR_UNSUPPORTED: return "unsupported shape";
    case PE_ERR_CUDA: return "CUDA runtime error";
    case PE_ERR_OUT_OF_MEMORY: return "out of device memory";
    case PE_ERR_DEVICE: return "device-side violation recorded";
  }
  return "unknown status";
}

pe_status pe_destroy(pe_handle* h) {
  if (!h) return PE_ERR_INVALID_ARGUMENT;
  cudaDeviceSynchronize();
  for (void* p : h->allocations) cudaFree(p);
  delete h;
  return PE_OK;
}

pe_status pe_create(const pe_model_desc* desc, const pe_weights* weights, int32_t max_tokens,
                    int32_t max_reqs, pe_handle** out) {
  if (!desc || !weights || !out || max_tokens < 1 || max_reqs < 1) return PE_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  const pe_model_desc& d = *desc;
  if (d.d < 1 || d.n_layers < 1 || d.n_heads < 1 || d.n_kv_heads < 1 || d.ffn < 1 ||
      d.vocab < 2 || d.hidden3 < 1 || d.head_dim < 1 || d.n_heads % d.n_kv_heads != 0 ||
      d.mask_token_id < 0 || d.mask_token_id >= d.vocab || !(d.rms_eps >= 0.f) ||
      !(d.rope_theta > 0.f))
    return PE_ERR_INVALID_ARGUMENT;
  if (d.dtype != PE_DTYPE_BF16 && d.dtype != PE_DTYPE_F32) return PE_ERR_INVALID_ARGUMENT;
  if (d.page_size != 16 || (d.head_dim != 64 && d.head_dim != 128)) return PE_ERR_UNSUPPORTED;
  const size_t es = d.dtype == PE_DTYPE_BF16 ? 2 : 4;
  if ((d.hidden3 * es) % 16 != 0) return PE_ERR_UNSUPPORTED;
  if (d.dtype == PE_DTYPE_BF16 &&
      (d.d % 8 || d.ffn % 8 || d.hidden3 % 8 || (d.n_heads * d.head_dim) % 8))
    return PE_ERR_UNSUPPORTED;
  const pe_weights& w = *weights;
  if (!w.emb || !w.fc || !w.h_shared || !w.norm_final || !w.lm_head || !w.layers)
    return PE_ERR_INVALID_ARGUMENT;
  for (int l = 0; l < d.n_layers; ++l) {
    const pe_layer_weights& L = w.layers[l];
    if (!L.qkv || !L.o || !L.gate || !L.up || !L.down || !L.norm_post) return PE_ERR_INVALID_ARGUMENT;
    if (l == 0 ? (!L.norm_e || !L.norm_h) : !L.norm_in) return PE_ERR_INVALID_ARGUMENT;
    if (d.dtype == PE_DTYPE_BF16 &&
        !(aligned16(L.qkv) && aligned16(L.o) && aligned16(L.gate) && aligned16(L.up) &&
          aligned16(L.down)))
      return PE_ERR_INVALID_ARGUMENT;
  }
  if (d.dtype == PE_DTYPE_BF16 && !(aligned16(w.fc) && aligned16(w.lm_head)))
    return PE_ERR_INVALID_ARGUMENT;
  if (!aligned16(w.h_shared)) return PE_ERR_INVALID_ARGUMENT;

  pe_handle* h = new (std::nothrow) pe_handle();
  if (!h) return PE_ERR_OUT_OF_MEMORY;
  h->desc = d;
  h->w = w;
  h->layers.assign(w.layers, w.layers + d.n_layers);
  h->w.layers = h->layers.data();
  h->max_tokens = max_tokens;
  h->max_reqs = max_reqs;
  h->esize = es;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->l2_bytes, cudaDevAttrL2CacheSize, h->device);
  const size_t T = max_tokens;
  const int qkv_rows = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  const int qd = d.n_heads * d.head_dim;
  auto alloc_bytes = [&](void** p, size_t bytes) {
    unsigned char* q = nullptr;
    cudaError_t r = dev_alloc(h, &q, bytes);
    *p = q;
    return r;
  };
  if (e == cudaSuccess) e = dev_alloc(h, &h->err, 1);
  if (e == cudaSuccess) e = dev_alloc(h, &h->diag_flag, 1);
  if (e == cudaSuccess) e = dev_alloc(h, &h->resid, T * d.d);
  if (e == cudaSuccess) e = dev_alloc(h, &h->o_delta, T * d.d);
  if (e == cudaSuccess) e = alloc_bytes(&h->x_in, T * 2 * d.d * es);
  if (e == cudaSuccess) e = alloc_bytes(&h->qkv, T * qkv_rows * es);
  if (e == cudaSuccess) e = alloc_bytes(&h->q, T * qd * es);
  if (e == cudaSuccess) e = alloc_bytes(&h->attn, T * qd * es);
  if (e == cudaSuccess) e = alloc_bytes(&h->xn, T * d.d * es);
  if (e == cudaSuccess) e = alloc_bytes(&h->act, T * d.ffn * es);
  if (e == cudaSuccess) e = dev_alloc(h, &h->keys, T);
  for (int32_t** p : {&h->row_map, &h->live_row, &h->ids_c, &h->pos_c, &h->slot_c, &h->new_c})
    if (e == cudaSuccess) e = dev_alloc(h, p, T);
  if (e == cudaSuccess) e = dev_alloc(h, &h->live_before, T + 1);
  if (e == cudaSuccess) e = dev_alloc(h, &h->cu_live, static_cast<size_t>(max_reqs) + 1);
  if (e == cudaSuccess) e = dev_alloc(h, &h->n_live, 1);
  if (e == cudaSuccess) e = dev_alloc(h, &h->inv_freq64, d.head_dim / 2);
  if (e == cudaSuccess) e = dev_alloc(h, &h->rope_tab, T * d.head_dim);
  if (e == cudaSuccess) e = dev_alloc(h, &h->fc_hs, d.d);
  if (e == cudaSuccess) e = dev_alloc(h, &h->fc_map, T);
  if (e == cudaSuccess) e = dev_alloc(h, &h->masked_c, T);
  if (e == cudaSuccess) e = dev_alloc(h, &h->ssq_post, T * ((d.d + 31) / 32));
  if (e == cudaSuccess) e = dev_alloc(h, &h->ssq_in, T * ((d.d + 31) / 32));
  if (e == cudaSuccess) {
    std::vector<double> inv(d.head_dim / 2);
    for (int i = 0; i < d.head_dim / 2; ++i)
      inv[i] = std::pow(static_cast<double>(d.rope_theta), -2.0 * i / d.head_dim);
    e = cudaMemcpy(h->inv_freq64, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && d.dtype == PE_DTYPE_BF16) e = init_gemm_tc();
  if (e == cudaSuccess && d.dtype == PE_DTYPE_BF16) e = init_attention_tc();
  if (e == cudaSuccess && d.dtype == PE_DTYPE_BF16) e = init_stream();
  if (e == cudaSuccess && d.dtype == PE_DTYPE_BF16) {
    e = dev_alloc(h, &h->stream_ws, stream_ws_floats(h->sm_count));
    if (e == cudaSuccess) e = dev_alloc(h, &h->stream_sync, kStreamSyncInts);
    if (e == cudaSuccess)
      e = dev_alloc(h, &h->stream_counters, kStreamMaxPhases * kStreamCounterStride);
    if (e == cudaSuccess)
      e = dev_alloc(h, &h->stream_ssq, static_cast<size_t>(kStreamMaxPhases) * kStreamSsqTiles * 32);
  }
  if (e == cudaSuccess && d.dtype == PE_DTYPE_BF16) {
    // the widest token tile any row count up to max_tokens can take
    const int bn = max_tokens > 128 ? 256 : tc_pick_bn(max_tokens, false);
    // stream-K runs two CTAs an SM for token tiles up to 32 wide
    h->gemm_partial_floats = tc_partial_floats((bn <= 32 ? 2 : 1) * h->sm_count, bn, true);
    e = dev_alloc(h, &h->gemm_partials, h->gemm_partial_floats);
    const int widest = std::max({d.vocab, qkv_rows, d.ffn, d.d, qd});
    h->max_tiles = ((widest + 127) / 128) * ((max_tokens + 15) / 16);
    if (e == cudaSuccess) e = dev_alloc(h, &h->tile_counters, h->max_tiles);
    if (e == cudaSuccess) e = dev_alloc(h, &h->done_counter, 1);
  }
  if (e == cudaSuccess) {
    // fc(h_shared): every MASK row carries h_shared, so its projection is a
    // constant of the weights, computed once here
    EpiArgs ep = epi_none();
    ep.kind = EPI_STORE;
    ep.M = 1;
    ep.N = d.d;
    ep.out = h->fc_hs;
    ep.ldo = d.d;
    ep.out_f32 = 1;
    e = linear(h, w.h_shared, d.hidden3, w.fc, nullptr, 1, d.d, d.hidden3, ep, nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
  }
  if (e != cudaSuccess) {
    pe_destroy(h);
    return e == cudaErrorMemoryAllocation ? PE_ERR_OUT_OF_MEMORY : PE_ERR_CUDA;
  }
  *out = h;
  return PE_OK;
}

pe_status pe_get_launch_count(pe_handle* h, int64_t* count) {
  if (!h || !count) return PE_ERR_INVALID_ARGUMENT;
  *count = h->launches;
  return PE_OK;
}

pe_status pe_set_kv_cache_fp8(pe_handle* h, const float* k_scales, const float* v_scales) {
  if (!h || (!k_scales) != (!v_scales)) return PE_ERR_INVALID_ARGUMENT;
  if (!k_scales) {
    h->kv_fp8 = false;
    return PE_OK;
  }
  if (h->desc.dtype != PE_DTYPE_BF16 || h->desc.head_dim != 64) return PE_ERR_UNSUPPORTED;
  std::vector<float> ks(k_scales, k_scales + h->desc.n_layers);
  std::vector<float> vs(v_scales, v_scales + h->desc.n_layers);
  for (int l = 0; l < h->desc.n_layers; ++l)
    if (!(ks[l] > 0.f) || !(vs[l] > 0.f) || !std::isfinite(ks[l]) || !std::isfinite(vs[l]))
      return PE_ERR_INVALID_ARGUMENT;
  h->k_scales = ks;
  h->v_scales = vs;
  h->kv_fp8 = true;
  return PE_OK;
}

pe_status pe_set_tuning(pe_handle* h, int32_t key, int32_t value) {
  if (!h) return PE_ERR_INVALID_ARGUMENT;
  switch (key) {
    case PE_TUNE_GEMM_PRE_STAGES:
      if (value < -1) return PE_ERR_INVALID_ARGUMENT;
      h->gemm_pre_stages = value;
      return PE_OK;
    case PE_TUNE_GEMM_MAX_SPLIT:
      if (value < 1 || value > 8) return PE_ERR_INVALID_ARGUMENT;
      h->gemm_max_split = value;
      return PE_OK;
    case PE_TUNE_ATTN_MIN_CHUNKS:
      if (value < 2 || value > 32) return PE_ERR_INVALID_ARGUMENT;
      h->attn_min_chunks = value;
      return PE_OK;
    case PE_TUNE_ATTN_MAX_CHUNKS:
      if (value < 2 || value > 64) return PE_ERR_INVALID_ARGUMENT;
      h->attn_max_chunks = value;
      return PE_OK;
    case PE_TUNE_ATTN_L2_AHEAD:
      if (value < 0 || value > 64) return PE_ERR_INVALID_ARGUMENT;
      h->attn_l2_ahead = value;
      return PE_OK;
    case PE_TUNE_GEMM_TILE_ORDER:
      if (value < 0 || value > 1) return PE_ERR_INVALID_ARGUMENT;
      h->gemm_tile_order = value;
      return PE_OK;
    default:
      return PE_ERR_INVALID_ARGUMENT;
  }
}

pe_status pe_set_split_reduce(pe_handle* h, int32_t mode) {
  if (!h || (mode != PE_REDUCE_PULL && mode != PE_REDUCE_PUSH)) return PE_ERR_INVALID_ARGUMENT;
  h->cluster_push = mode;
  return PE_OK;
}

pe_status pe_set_fusions(pe_handle* h, int32_t mask) {
  if (!h || (mask & ~PE_FUSE_ALL)) return PE_ERR_INVALID_ARGUMENT;
  if ((mask & PE_FUSE_ROPE_KV) && h->desc.dtype == PE_DTYPE_BF16 && h->qkv_il.empty()) {
    const cudaError_t e = make_interleaved_qkv(h);
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? PE_ERR_OUT_OF_MEMORY : PE_ERR_CUDA;
  }
  h->fusions = mask;
  return PE_OK;
}

pe_status pe_set_small_batch_stream(pe_handle* h, int32_t enable) {
  if (!h) return PE_ERR_INVALID_ARGUMENT;
  h->stream_on = enable != 0;
  return PE_OK;
}

pe_status pe_set_stream_prefetch(pe_handle* h, int32_t tiles, int32_t boundary_tiles) {
  if (!h || tiles < 0 || tiles > 4096 || boundary_tiles < -1) return PE_ERR_INVALID_ARGUMENT;
  h->stream_prefetch = tiles;
  h->stream_boundary = boundary_tiles;
  return PE_OK;
}

pe_status pe_set_gemm_timeline(pe_handle* h, uint64_t* stamps, int32_t launches) {
  if (!h || launches < 0) return PE_ERR_INVALID_ARGUMENT;
  h->gemm_timeline = reinterpret_cast<unsigned long long*>(stamps);
  h->gemm_timeline_launches = stamps ? launches : 0;
  return PE_OK;
}

pe_status pe_set_stream_timeline(pe_handle* h, uint64_t* stamps) {
  if (!h) return PE_ERR_INVALID_ARGUMENT;
  h->stream_timeline = reinterpret_cast<unsigned long long*>(stamps);
  return PE_OK;
}

pe_status pe_set_phase_events(pe_handle* h, void* const* events, int32_t n) {
  if (!h || n < 0 || (n > 0 && !events)) return PE_ERR_INVALID_ARGUMENT;
  if (n != 0 && n != 2 + 2 * h->desc.n_layers) return PE_ERR_INVALID_ARGUMENT;
  h->phase_events.clear();
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return PE_ERR_INVALID_ARGUMENT;
    h->phase_events.push_back(static_cast<cudaEvent_t>(events[i]));
  }
  return PE_OK;
}

pe_status pe_set_trace(pe_handle* h, float* residual_trace, void* attn_trace) {
  if (!h) return PE_ERR_INVALID_ARGUMENT;
  h->trace = residual_trace;
  h->attn_trace = attn_trace;
  return PE_OK;
}

pe_status pe_get_device_error(pe_handle* h, int32_t* code, void* stream) {
  if (!h || !code) return PE_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, h->err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *code = v;
  return cuda_status(e);
}

pe_status pe_check_bounded_wait(pe_handle* h, int32_t* out, void* stream) {
  if (!h || !out) return PE_ERR_INVALID_ARGUMENT;
  return cuda_status(counted(
      h, launch_bounded_wait_check(h->diag_flag, out, h->err, static_cast<cudaStream_t>(stream))));
}

pe_status pe_expand_batch(pe_handle* h, int32_t B, int32_t K, int32_t T, const int32_t* target_ids,
                          const int32_t* target_pos, const int32_t* cu_in,
                          const int32_t* num_accepted, const int32_t* sampled_ids,
                          const int32_t* block_table, int32_t bt_stride, int32_t num_blocks,
                          const void* target_hidden, pe_expanded* out, void* stream) {
  if (!h || !out || B < 1 || B > h->max_reqs || K < 1 || K > 64 || T < B || bt_stride < 1 ||
      num_blocks < 1)
    return PE_ERR_INVALID_ARGUMENT;
  const long long T_out = static_cast<long long>(T) + static_cast<long long>(B) * (K - 1);
  if (T_out > h->max_tokens) return PE_ERR_INVALID_ARGUMENT;
  if (!target_ids || !target_pos || !cu_in || !num_accepted || !sampled_ids || !block_table ||
      !target_hidden || !out->ids || !out->pos || !out->slot || !out->is_rejected ||
      !out->is_masked || !out->new_idx || !out->hidden_map || !out->cu_out || !out->seq_lens ||
      !out->hidden)
    return PE_ERR_INVALID_ARGUMENT;
  if (!aligned16(target_hidden) || !aligned16(out->hidden)) return PE_ERR_INVALID_ARGUMENT;
  ExpandArgs a;
  a.B = B;
  a.K = K;
  a.T = T;
  a.T_out = static_cast<int>(T_out);
  a.target_ids = target_ids;
  a.target_pos = target_pos;
  a.cu_in = cu_in;
  a.num_accepted = num_accepted;
  a.sampled_ids = sampled_ids;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.num_blocks = num_blocks;
  a.page_size = h->desc.page_size;
  a.mask_token_id = h->desc.mask_token_id;
  a.target_hidden = target_hidden;
  a.h_shared = h->w.h_shared;
  a.row_bytes = static_cast<int>(h->desc.hidden3 * h->esize);
  a.ids = out->ids;
  a.pos = out->pos;
  a.slot = out->slot;
  a.is_rejected = out->is_rejected;
  a.is_masked = out->is_masked;
  a.new_idx = out->new_idx;
  a.hidden_map = out->hidden_map;
  a.cu_out = out->cu_out;
  a.seq_lens = out->seq_lens;
  a.hidden = out->hidden;
  a.err = h->err;
  cudaError_t e = counted(h, launch_expand(a, static_cast<cudaStream_t>(stream)));
  if (e != cudaSuccess) return PE_ERR_CUDA;
  out->B = B;
  out->K = K;
  out->T = T;
  out->T_out = a.T_out;
  out->target_hidden = target_hidden;
  return PE_OK;
}

pe_status pe_draft_forward(pe_handle* h, const pe_expanded* ex, int32_t B, int32_t K,
                           const int32_t* block_table, int32_t bt_stride, void* const* k_cache,
                           void* const* v_cache, int32_t num_blocks, void* out_hidden,
                           void* stream) {
  if (!h || !ex || !block_table || !k_cache || !v_cache || !out_hidden || bt_stride < 1 ||
      num_blocks < 1)
    return PE_ERR_INVALID_ARGUMENT;
  if (B < 1 || B > h->max_reqs || ex->B != B || ex->K != K || ex->T_out < 1 ||
      ex->T_out > h->max_tokens ||
      ex->T_out != ex->T + B * (K - 1))
    return PE_ERR_INVALID_ARGUMENT;
  const pe_model_desc& d = h->desc;
  for (int l = 0; l < d.n_layers; ++l)
    if (!k_cache[l] || !v_cache[l]) return PE_ERR_INVALID_ARGUMENT;
  if (static_cast<long long>(B) * K > h->max_tokens) return PE_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->gemm_ordinal = 0;
  const int rows = ex->T_out;
  const int dt = d.dtype;
  const int qkv_rows = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  const int qd = d.n_heads * d.head_dim;
  const uint64_t cache_rows = static_cast<uint64_t>(num_blocks) * d.n_kv_heads * 16;
  // rows of one request: its verify window (at most K + 1 rows, and at most
  // what the batch leaves it) plus the K - 1 MASK rows
  const int max_rows_per_req = std::min(ex->T - B + 1, K + 1) + K - 1;
  cudaError_t e;
  AttnArgs probe = {};                 // the attention's shape, for its plan
  probe.B = B;
  probe.Hq = d.n_heads;
  probe.Hkv = d.n_kv_heads;
  probe.dh = d.head_dim;
  probe.bt_stride = bt_stride;
  int order_entries = 0;               // > 0: the attention takes its work longest first
  if (dt == PE_DTYPE_BF16) {
    if (d.head_dim % 64 || (d.n_heads / d.n_kv_heads) > 128) return PE_ERR_UNSUPPORTED;
    for (int l = 0; l < d.n_layers; ++l)
      if (!aligned16(k_cache[l]) || !aligned16(v_cache[l])) return PE_ERR_INVALID_ARGUMENT;
    // the split-KV workspace depends on the batch and the block table; the
    // first call that needs more grows it (make that call before capturing
    // the step into a CUDA graph)
    const size_t need = attention_tc_partial_floats(probe, max_rows_per_req, h->sm_count,
                                                    h->attn_min_chunks, h->attn_max_chunks);
    const size_t need_c = attention_tc_counters(probe, max_rows_per_req, h->sm_count,
                                                h->attn_min_chunks, h->attn_max_chunks);
    if (need > h->attn_partial_floats) {
      if ((e = dev_alloc(h, &h->attn_partials, need))) return PE_ERR_OUT_OF_MEMORY;
      h->attn_partial_floats = need;
    }
    if (need_c > h->attn_n_counters) {
      if ((e = dev_alloc(h, &h->attn_counters, need_c))) return PE_ERR_OUT_OF_MEMORY;
      h->attn_n_counters = need_c;
    }
    order_entries = attention_tc_order_entries(probe, max_rows_per_req, h->sm_count,
                                               h->attn_min_chunks, h->attn_max_chunks);
    if (static_cast<size_t>(order_entries) > h->attn_order_cap) {
      if ((e = dev_alloc(h, &h->attn_order, static_cast<size_t>(order_entries))))
        return PE_ERR_OUT_OF_MEMORY;
      h->attn_order_cap = static_cast<size_t>(order_entries);
    }
  }

  // Rejected rows (window rows after the accepted count) write no KV and
  // feed no sampled row: after fc the layers run on the live rows only.
  // The compaction pays only if the live rows can need fewer token tiles
  // in some projection: a batch of one window row per request has no
  // rejected rows, and when even B*K live rows (every request accepting
  // nothing) fill as many tiles as the expanded batch, nothing shrinks.
  auto tiles_of = [&](int m, bool dual) {
    const int bn = d.dtype == PE_DTYPE_BF16 ? tc_pick_bn(rows, dual) : 16;
    return (m + bn - 1) / bn;
  };
  const bool compact = ex->T > B && (tiles_of(B * K, false) < tiles_of(rows, false) ||
                                     tiles_of(B * K, true) < tiles_of(rows, true));
  const int32_t* live = nullptr;
  const int32_t* ids_l = ex->ids;
  const int32_t* pos_l = ex->pos;
  const int32_t* slot_l = ex->slot;
  const int32_t* cu_l = ex->cu_out;
  const int32_t* new_l = ex->new_idx;
  const uint8_t* rej_l = ex->is_rejected;
  if (compact) {
    CompactArgs ca = {};
    ca.B = B;
    ca.K = K;
    ca.T_out = rows;
    ca.cu_out = ex->cu_out;
    ca.is_rejected = ex->is_rejected;
    ca.ids = ex->ids;
    ca.pos = ex->pos;
    ca.slot = ex->slot;
    ca.new_idx = ex->new_idx;
    ca.row_map = h->row_map;
    ca.live_before = h->live_before;
    ca.live_row = h->live_row;
    ca.ids_c = h->ids_c;
    ca.pos_c = h->pos_c;
    ca.slot_c = h->slot_c;
    ca.cu_live = h->cu_live;
    ca.new_c = h->new_c;
    ca.n_live = h->n_live;
    if (ex->target_hidden) {
      ca.T = ex->T;
      ca.hidden_map = ex->hidden_map;
      ca.is_masked = ex->is_masked;
      ca.fc_map = h->fc_map;
      ca.masked_c = h->masked_c;
    }
    if ((e = counted(h, launch_compact_rows(ca, s)))) return PE_ERR_CUDA;
    live = h->n_live;
    ids_l = h->ids_c;
    pos_l = h->pos_c;
    slot_l = h->slot_c;
    cu_l = h->cu_live;
    new_l = h->new_c;
    rej_l = nullptr;
  }
  // phase timing (diagnostic): event 0 here, 1 + 2 l before layer l's
  // attention, 2 + 2 l after it, 1 + 2 L at the end
  auto mark = [&](int i) -> cudaError_t {
    // inside a stream capture an external record becomes an event node that
    // every replay of the graph records; outside one, a plain record
    if (h->phase_events.empty()) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t q = cudaStreamIsCapturing(s, &cs);
    if (q != cudaSuccess) return q;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(h->phase_events[i], s, cudaEventRecordExternal)
               : cudaEventRecord(h->phase_events[i], s);
  };
  if ((e = mark(0))) return PE_ERR_CUDA;
  // debug copies of per-row activations, in the expanded row order (zero
  // for rejected rows)
  auto trace_rows = [&](void* dst, const void* src, size_t row_bytes) -> cudaError_t {
    if (!compact) return cudaMemcpyAsync(dst, src, rows * row_bytes, cudaMemcpyDeviceToDevice, s);
    cudaError_t r = cudaMemsetAsync(dst, 0, rows * row_bytes, s);
    if (r == cudaSuccess)
      r = counted(h, launch_scatter_rows(dst, src, h->live_row, h->n_live, rows,
                                         static_cast<int>(row_bytes), s));
    return r;
  };

  // paged causal attention of layer l (with the phase marks and the
  // attention trace around it)
  auto attention = [&](int l) -> pe_status {
    cudaError_t e;
    if ((e = mark(1 + 2 * l))) return PE_ERR_CUDA;
    AttnArgs at = {};
    at.rows = rows;
    at.B = B;
    at.Hq = d.n_heads;
    at.Hkv = d.n_kv_heads;
    at.dh = d.head_dim;
    at.bt_stride = bt_stride;
    at.num_blocks = num_blocks;
    at.max_seq = bt_stride * d.page_size;
    at.q = h->q;
    at.k_cache = k_cache[l];
    at.v_cache = v_cache[l];
    at.live = live;
    at.pos = pos_l;
    at.is_rejected = rej_l;
    at.cu_out = cu_l;
    at.block_table = block_table;
    at.out = h->attn;
    at.scale = 1.0f / std::sqrt(static_cast<float>(d.head_dim));
    at.err = h->err;
    if (dt == PE_DTYPE_F32) {
      if ((e = counted(h, launch_attention_simt(dt, at, s)))) return PE_ERR_CUDA;
    } else {
      if (h->kv_fp8) {
        at.kv_fp8 = 1;
        at.k_scale = h->k_scales[l];
        at.v_scale = h->v_scales[l];
      }
      const CUtensorMap* tk = h->kv_fp8 ? get_map_u8(h, k_cache[l], cache_rows)
                                        : get_map(h, k_cache[l], cache_rows, d.head_dim, d.head_dim, 16);
      const CUtensorMap* tv = h->kv_fp8 ? get_map_u8(h, v_cache[l], cache_rows)
                                        : get_map(h, v_cache[l], cache_rows, d.head_dim, d.head_dim, 16);
      if (!tk || !tv) return PE_ERR_INVALID_ARGUMENT;
      unsigned long long* tl = nullptr;
      if (h->gemm_timeline && h->gemm_ordinal < h->gemm_timeline_launches)
        tl = h->gemm_timeline + static_cast<size_t>(h->gemm_ordinal) * 512 * 16;
      ++h->gemm_ordinal;
      e = counted(h, launch_attention_tc(at, *tk, *tv, ex->seq_lens, max_rows_per_req,
                                         h->sm_count, h->attn_partials, h->attn_partial_floats,
                                         h->attn_counters, h->attn_n_counters, tl,
                                         h->attn_l2_ahead, h->attn_min_chunks,
                                         h->attn_max_chunks,
                                         order_entries > 0 ? h->attn_order : nullptr, s));
      if (e) return PE_ERR_CUDA;
    }
    if ((e = mark(2 + 2 * l))) return PE_ERR_CUDA;
    if (h->attn_trace) {
      const size_t per = static_cast<size_t>(qd) * h->esize;
      if ((e = trace_rows(static_cast<char*>(h->attn_trace) + l * h->max_tokens * per, h->attn,
                          per)))
        return PE_ERR_CUDA;
    }
    return PE_OK;
  };

  // ---- small batches: one persistent kernel per segment of projections ----
  // (stream.cu): fc -> layer-0 input -> QKV_0, then after each layer's
  // attention O -> gate/up -> down -> next QKV (or the final norm).  Used
  // when the rows fit one 16- or 32-token tile and every phase's share of
  // activations fits a CTA's panel.
  const int G = h->sm_count;
  auto units_per_cta = [&](int N, int K) {
    const long long U = static_cast<long long>((N + 127) / 128) * ((K + 63) / 64);
    return (U + G - 1) / G;
  };
  const int pkb = stream_panel_kb(std::min(rows, 32));
  const bool use_stream =
      dt == PE_DTYPE_BF16 && h->stream_on && rows <= 32 && !compact &&
      qd % 128 == 0 && (d.n_kv_heads * d.head_dim) % 128 == 0 && (d.head_dim == 64 || d.head_dim == 128) &&
      (d.d + 127) / 128 <= 128 &&  // a norm's per-tile sums fit the CTA's exchange buffer
      (std::max({d.d, d.ffn, qkv_rows}) + 127) / 128 <= kStreamCounterStride &&
      units_per_cta(d.d, d.hidden3) <= pkb && units_per_cta(qkv_rows, 2 * d.d) <= pkb &&
      units_per_cta(qkv_rows, d.d) <= pkb && units_per_cta(d.d, qd) <= pkb &&
      units_per_cta(d.ffn, d.d) <= pkb && units_per_cta(d.d, d.ffn) <= pkb;
  if (use_stream) {
    StreamMaps sm;
    StreamParams sp;
    int nmaps = 0;
    bool maps_ok = true;
    auto add_map = [&](const CUtensorMap* m) {
      if (!m || nmaps >= kStreamMaxMaps) {
        maps_ok = false;
        return 0;
      }
      sm.m[nmaps] = *m;
      return nmaps++;
    };
    auto begin = [&]() {
      sp = StreamParams{};
      nmaps = 0;
      sp.rows = rows;
      sp.d = d.d;
      sp.resid = h->resid;
      sp.eps = d.rms_eps;
      sp.ids = ex->ids;
      sp.emb = h->w.emb;
      sp.vocab = d.vocab;
      sp.g_e = h->layers[0].norm_e;
      sp.g_h = h->layers[0].norm_h;
      sp.x_in = h->x_in;
      sp.pos = ex->pos;
      sp.slot = ex->slot;
      sp.Hq = d.n_heads;
      sp.Hkv = d.n_kv_heads;
      sp.dh = d.head_dim;
      sp.num_blocks = num_blocks;
      sp.inv_freq64 = h->inv_freq64;
      sp.q_out = h->q;
      sp.new_idx = ex->new_idx;
      sp.final_rows = B * K;
      sp.g_final = h->w.norm_final;
      sp.out_hidden = out_hidden;
      sp.timeline = h->stream_timeline;
      sp.prefetch_tiles = h->stream_prefetch;
      sp.boundary_tiles = h->stream_boundary;
      sp.ws = h->stream_ws;
      sp.sync = h->stream_sync;
      sp.counters = h->stream_counters;
      sp.n_counters = kStreamMaxPhases * kStreamCounterStride;
      sp.err = h->err;
    };
    // a GEMM phase: y[rows, N] = x[rows, K] . w[N, K]^T (+ w2 for gate/up)
    auto gemm = [&](int epi, const void* w, const void* w2, int N, int Kd, const void* x,
                    int ldx) {
      StreamPhase& P = sp.ph[sp.nphases];
      P = StreamPhase{};
      P.kind = SK_GEMM;
      P.epi = epi;
      P.dual = w2 != nullptr;
      P.N = N;
      P.K = Kd;
      P.kb = (Kd + 63) / 64;
      P.tiles = (N + 127) / 128;
      P.map_a = add_map(get_map(h, w, N, Kd, Kd, 128));
      P.map_a2 = w2 ? add_map(get_map(h, w2, N, Kd, Kd, 128)) : P.map_a;
      P.w = w;
      P.w2 = w2 ? w2 : w;
      P.x = x;
      P.ldx = ldx;
      P.norm_src = -1;
      P.counters = h->stream_counters + sp.nphases * kStreamCounterStride;
      return sp.nphases++;
    };
    auto row_phase = [&](int kind) {
      StreamPhase& P = sp.ph[sp.nphases];
      P = StreamPhase{};
      P.kind = kind;
      P.norm_src = -1;
      return sp.nphases++;
    };
    auto ssq_of = [&](int ph) {
      return h->stream_ssq + static_cast<size_t>(ph) * kStreamSsqTiles * 32;
    };
    auto launch = [&]() -> cudaError_t {
      if (!maps_ok) return cudaErrorInvalidValue;
      return counted(h, launch_stream(sm, sp, G, s));
    };
    // segment 0: fc, the layer-0 input, QKV_0 (+ RoPE and the KV write)
    auto set_kv = [&](int l) {
      sp.k_cache = k_cache[l];
      sp.v_cache = v_cache[l];
      sp.kv_fp8 = h->kv_fp8 ? 1 : 0;
      if (h->kv_fp8) {
        sp.k_inv_scale = 1.f / h->k_scales[l];
        sp.v_inv_scale = 1.f / h->v_scales[l];
      }
    };
    begin();
    set_kv(0);
    gemm(SE_STORE, h->w.fc, nullptr, d.d, d.hidden3, ex->hidden, d.hidden3);
    row_phase(SK_EMBED);
    gemm(SE_ROPE_KV, h->layers[0].qkv, nullptr, qkv_rows, 2 * d.d, h->x_in, 2 * d.d);
    if ((e = launch())) return PE_ERR_CUDA;
    for (int l = 0; l < d.n_layers; ++l) {
      if (const pe_status st = attention(l); st != PE_OK) return st;
      const pe_layer_weights& L = h->layers[l];
      const bool last = l + 1 == d.n_layers;
      begin();
      if (!last) set_kv(l + 1);
      const int o_ph = gemm(SE_ADD, L.o, nullptr, d.d, qd, h->attn, qd);
      sp.ph[o_ph].g_next = L.norm_post;
      sp.ph[o_ph].xg = h->xn;
      sp.ph[o_ph].ssq = ssq_of(o_ph);
      const int gu_ph = gemm(SE_SILU_MUL, L.gate, L.up, d.ffn, d.d, h->xn, d.d);
      sp.ph[gu_ph].norm_src = o_ph;
      sp.ph[gu_ph].norm_d = d.d;
      sp.ph[gu_ph].out = h->act;
      sp.ph[gu_ph].ldo = d.ffn;
      const int dn_ph = gemm(SE_ADD, L.down, nullptr, d.d, d.ffn, h->act, d.ffn);
      if (!last) {
        sp.ph[dn_ph].g_next = h->layers[l + 1].norm_in;
        sp.ph[dn_ph].xg = h->x_in;
        sp.ph[dn_ph].ssq = ssq_of(dn_ph);
        const int q_ph = gemm(SE_ROPE_KV, h->layers[l + 1].qkv, nullptr, qkv_rows, d.d,
                              h->x_in, d.d);
        sp.ph[q_ph].norm_src = dn_ph;
        sp.ph[q_ph].norm_d = d.d;
      } else {
        row_phase(SK_FINAL);
      }
      if ((e = launch())) return PE_ERR_CUDA;
      if (h->trace) {
        if ((e = trace_rows(h->trace + static_cast<size_t>(l) * h->max_tokens * d.d, h->resid,
                            static_cast<size_t>(d.d) * sizeof(float))))
          return PE_ERR_CUDA;
      }
    }
    if ((e = mark(1 + 2 * d.n_layers))) return PE_ERR_CUDA;
    return PE_OK;
  }

  // fc: projected target hidden state -> residual stream (fp32), live rows
  // to their compact rows.  With the target rows recorded, fc runs on those
  // T rows only (through the hidden map) and the MASK rows take fc(h_shared)
  // in the layer-0 input kernel below.
  const bool fc_once = ex->target_hidden != nullptr;
  EpiArgs ep = epi_none();
  ep.kind = EPI_STORE;
  ep.N = d.d;
  ep.out = h->resid;
  ep.ldo = d.d;
  ep.out_f32 = 1;
  if (fc_once) {
    ep.M = ex->T;
    ep.row_map = compact ? h->fc_map : ex->hidden_map;
    if ((e = linear(h, ex->target_hidden, d.hidden3, h->w.fc, nullptr, ex->T, d.d, d.hidden3, ep,
                    s)))
      return PE_ERR_CUDA;
  } else {
    ep.M = rows;
    ep.row_map = compact ? h->row_map : nullptr;
    if ((e = linear(h, ex->hidden, d.hidden3, h->w.fc, nullptr, rows, d.d, d.hidden3, ep, s)))
      return PE_ERR_CUDA;
  }
  // layer-0 input: [RMSNorm_e(emb[id]) ; RMSNorm_h(fc h)]
  EmbedConcatArgs ec = {};
  ec.rows = rows;
  ec.d = d.d;
  ec.vocab = d.vocab;
  ec.ids = ids_l;
  ec.live = live;
  ec.emb = h->w.emb;
  ec.h = h->resid;
  ec.g_e = h->layers[0].norm_e;
  ec.g_h = h->layers[0].norm_h;
  ec.eps = d.rms_eps;
  ec.x = h->x_in;
  ec.err = h->err;
  if (fc_once) {
    ec.masked = compact ? h->masked_c : ex->is_masked;
    ec.fc_hs = h->fc_hs;
    ec.h_w = h->resid;
  }
  // RoPE and the KV write in the QKV projection's epilogue (bf16): the
  // rotary table of every row comes with the layer-0 input
  // (one token tile of at most 32 rows whose rotary table fits the tile's
  // staged [tile][64] floats; larger batches keep the separate kernel)
  const bool fuse_rope = dt == PE_DTYPE_BF16 && (h->fusions & PE_FUSE_ROPE_KV) &&
                         (qkv_rows % 128) == 0 && rows <= 32 && live == nullptr &&
                         rows * d.head_dim <= tc_pick_bn(rows, false) * 64;
  if (fuse_rope) {
    ec.pos = pos_l;
    ec.inv_freq64 = h->inv_freq64;
    ec.rope_tab = h->rope_tab;
    ec.dh = d.head_dim;
  }
  if ((e = counted(h, launch_embed_concat(dt, ec, s)))) return PE_ERR_CUDA;
  // More attention CTAs than one wave: the step's attention work items
  // sorted longest first, once for all layers (same sequences); written
  // well before the first attention reads it (two launches back at least)
  if (order_entries > 0 &&
      (e = counted(h, launch_attention_order(probe, ex->seq_lens, max_rows_per_req, h->sm_count,
                                             h->attn_min_chunks, h->attn_max_chunks,
                                             h->attn_order, s))))
    return PE_ERR_CUDA;
  // RMSNorm folded into the projections (bf16, one token tile of at most 32
  // rows): O and down write x g_next and per-group sums of squares, the
  // next projection scales its rows by r
  const bool fuse_norm = dt == PE_DTYPE_BF16 && (h->fusions & PE_FUSE_NORM) && rows <= 32 &&
                         live == nullptr;
  const int ssq_groups = (d.d + 31) / 32;
  auto fold_out = [&](EpiArgs& ep2, const void* g, void* xg, float* ssq) {
    ep2.g_next = g;
    ep2.xg = xg;
    ep2.ldxg = d.d;
    ep2.ssq = ssq;
    ep2.ssq_ld = h->max_tokens;
  };
  auto fold_in = [&](EpiArgs& ep2, const float* ssq) {
    ep2.rs_ssq = ssq;
    ep2.rs_groups = ssq_groups;
    ep2.rs_ld = h->max_tokens;
    ep2.rs_d = static_cast<float>(d.d);
    ep2.rs_eps = d.rms_eps;
  };

  bool down_deferred = false;   // the last down-projection left its residual add to the next norm
  for (int l = 0; l < d.n_layers; ++l) {
    const pe_layer_weights& L = h->layers[l];
    const int d_in = l == 0 ? 2 * d.d : d.d;
    if (l > 0 && !fuse_norm) {
      RmsNormArgs rn = {};
      rn.rows = rows;
      rn.d = d.d;
      rn.x = h->resid;
      rn.rows_in = rows;
      rn.g = L.norm_in;
      rn.eps = d.rms_eps;
      rn.y = h->x_in;
      rn.err = h->err;
      rn.live = live;
      if (down_deferred) {         // the previous layer's down-projection output
        rn.add = h->o_delta;
        rn.x_w = h->resid;
      }
      if ((e = counted(h, launch_rmsnorm(dt, rn, s)))) return PE_ERR_CUDA;
    }
    if (fuse_rope) {
      // QKV projection, rotate-half RoPE of q and k, q stored, k and v to
      // the paged cache (slot -1: nothing written), all in the epilogue
      ep = epi_none();
      ep.kind = EPI_ROPE_KV;
      ep.M = rows;
      ep.N = qkv_rows;
      ep.m_live = live;
      ep.q_out = h->q;
      ep.k_cache = k_cache[l];
      ep.v_cache = v_cache[l];
      ep.slot = slot_l;
      ep.rope_tab = h->rope_tab;
      ep.rope_rows_interleaved = h->qkv_il.empty() ? 0 : 1;
      ep.Hq = d.n_heads;
      ep.Hkv = d.n_kv_heads;
      ep.dh = d.head_dim;
      ep.num_blocks = num_blocks;
      ep.err = h->err;
      if (l > 0 && fuse_norm) fold_in(ep, h->ssq_in);
      if (h->kv_fp8) {
        ep.kv_fp8 = 1;
        ep.k_inv_scale = 1.f / h->k_scales[l];
        ep.v_inv_scale = 1.f / h->v_scales[l];
      }
      const CUtensorMap* wa = h->qkv_il.empty() ? get_map_qkv(h, L.qkv, d_in)
                                                : get_map(h, h->qkv_il[l], qkv_rows, d_in, d_in, 128);
      const CUtensorMap* xb =
          get_map(h, h->x_in, rows, d_in, d_in,
                  tc_b_box_rows(rows, qkv_rows, h->sm_count, false, live != nullptr));
      if (!wa || !xb) return PE_ERR_INVALID_ARGUMENT;
      if ((e = counted(h, launch_gemm_tc_maps(*wa, *wa, *xb, false, rows, qkv_rows, d_in, ep,
                                              tc_ws(h), h->err, s))))
        return PE_ERR_CUDA;
    } else {
      // QKV projection
      ep = epi_none();
      ep.kind = EPI_STORE;
      ep.M = rows;
      ep.N = qkv_rows;
      ep.out = h->qkv;
      ep.ldo = qkv_rows;
      ep.out_f32 = dt == PE_DTYPE_F32 ? 1 : 0;
      ep.m_live = live;
      if (l > 0 && fuse_norm) fold_in(ep, h->ssq_in);
      if ((e = linear(h, h->x_in, d_in, L.qkv, nullptr, rows, qkv_rows, d_in, ep, s)))
        return PE_ERR_CUDA;
      // RoPE + paged KV write (slot -1: nothing written)
      RopeKvArgs rk = {};
      rk.rows = rows;
      rk.Hq = d.n_heads;
      rk.Hkv = d.n_kv_heads;
      rk.dh = d.head_dim;
      rk.num_blocks = num_blocks;
      rk.qkv = h->qkv;
      rk.pos = pos_l;
      rk.slot = slot_l;
      rk.live = live;
      rk.inv_freq = nullptr;
      rk.inv_freq64 = h->inv_freq64;
      rk.q_out = h->q;
      rk.k_cache = k_cache[l];
      rk.v_cache = v_cache[l];
      rk.err = h->err;
      if (h->kv_fp8) {
        rk.kv_fp8 = 1;
        rk.k_inv_scale = 1.f / h->k_scales[l];
        rk.v_inv_scale = 1.f / h->v_scales[l];
      }
      if ((e = counted(h, launch_rope_kv(dt, rk, s)))) return PE_ERR_CUDA;
    }
    // paged causal attention
    if (const pe_status st = attention(l); st != PE_OK) return st;
    // O projection + residual.  Where the norm after it is a kernel of its
    // own (bf16, more than 32 rows), the projection stores its fp32 output
    // and that norm does the residual add (the same fp32 addition): the
    // projection's epilogue then has no residual reads, each a dependent
    // round trip per 16-token chunk of a wide tile.
    const bool defer_add = !fuse_norm && dt == PE_DTYPE_BF16 && d.d % 4 == 0;
    ep = epi_none();
    ep.kind = defer_add ? EPI_STORE : EPI_ADD;
    ep.M = rows;
    ep.N = d.d;
    if (defer_add) {
      ep.out = h->o_delta;
      ep.ldo = d.d;
      ep.out_f32 = 1;
    } else {
      ep.resid = h->resid;
      ep.ldr = d.d;
    }
    ep.m_live = live;
    if (fuse_norm) fold_out(ep, L.norm_post, h->xn, h->ssq_post);
    if ((e = linear(h, h->attn, qd, L.o, nullptr, rows, d.d, qd, ep, s))) return PE_ERR_CUDA;
    // MLP
    if (!fuse_norm) {
      RmsNormArgs rn = {};
      rn.rows = rows;
      rn.d = d.d;
      rn.x = h->resid;
      rn.rows_in = rows;
      rn.g = L.norm_post;
      rn.eps = d.rms_eps;
      rn.y = h->xn;
      rn.err = h->err;
      rn.live = live;
      if (defer_add) {
        rn.add = h->o_delta;
        rn.x_w = h->resid;
      }
      if ((e = counted(h, launch_rmsnorm(dt, rn, s)))) return PE_ERR_CUDA;
    }
    ep = epi_none();
    ep.kind = EPI_SILU_MUL;
    ep.M = rows;
    ep.N = d.ffn;
    ep.out = h->act;
    ep.ldo = d.ffn;
    ep.out_f32 = dt == PE_DTYPE_F32 ? 1 : 0;
    ep.m_live = live;
    if (fuse_norm) fold_in(ep, h->ssq_post);
    if ((e = linear(h, h->xn, d.d, L.gate, L.up, rows, d.ffn, d.d, ep, s))) return PE_ERR_CUDA;
    // down-projection + residual; deferred into the next layer's input norm
    // like the O projection's (not after the last layer, whose final norm
    // gathers rows, nor when the per-layer residual is traced)
    down_deferred = defer_add && l + 1 < d.n_layers && !h->trace;
    ep = epi_none();
    ep.kind = down_deferred ? EPI_STORE : EPI_ADD;
    ep.M = rows;
    ep.N = d.d;
    if (down_deferred) {
      ep.out = h->o_delta;
      ep.ldo = d.d;
      ep.out_f32 = 1;
    } else {
      ep.resid = h->resid;
      ep.ldr = d.d;
    }
    ep.m_live = live;
    if (fuse_norm && l + 1 < d.n_layers)
      fold_out(ep, h->layers[l + 1].norm_in, h->x_in, h->ssq_in);
    if ((e = linear(h, h->act, d.ffn, L.down, nullptr, rows, d.d, d.ffn, ep, s)))
      return PE_ERR_CUDA;
    if (h->trace) {
      if ((e = trace_rows(h->trace + static_cast<size_t>(l) * h->max_tokens * d.d, h->resid,
                          static_cast<size_t>(d.d) * sizeof(float))))
        return PE_ERR_CUDA;
    }
  }
  // final norm of the B*K sampled rows
  RmsNormArgs rn = {};
  rn.rows = B * K;
  rn.d = d.d;
  rn.x = h->resid;
  rn.row_index = new_l;
  rn.rows_in = rows;
  rn.g = h->w.norm_final;
  rn.eps = d.rms_eps;
  rn.y = out_hidden;
  rn.err = h->err;
  if ((e = counted(h, launch_rmsnorm(dt, rn, s)))) return PE_ERR_CUDA;
  if ((e = mark(1 + 2 * d.n_layers))) return PE_ERR_CUDA;
  return PE_OK;
}

pe_status pe_lmhead_argmax(pe_handle* h, const void* hidden, int32_t M, int32_t* out_tokens,
                           float* out_logits, void* stream) {
  if (!h || !hidden || !out_tokens || M < 1 || M > h->max_tokens) return PE_ERR_INVALID_ARGUMENT;
  const pe_model_desc& d = h->desc;
  if (d.dtype == PE_DTYPE_BF16 && !aligned16(hidden)) return PE_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EpiArgs ep = epi_none();
  ep.kind = EPI_ARGMAX;
  ep.M = M;
  ep.N = d.vocab;
  ep.logits = out_logits;
  ep.ldl = d.vocab;
  ep.keys = h->keys;
  ep.tokens = out_tokens;
  cudaError_t e = linear(h, hidden, d.d, h->w.lm_head, nullptr, M, d.vocab, d.d, ep, s);
  if (e == cudaSuccess && d.dtype == PE_DTYPE_F32)
    e = counted(h, launch_argmax_finalize(M, h->keys, out_tokens, s));
  return cuda_status(e);
}

pe_status pe_linear(pe_handle* h, const void* x, const void* w, float* y, int32_t M, int32_t N,
                    int32_t K, void* stream) {
  if (!h || !x || !w || !y || M < 1 || N < 1 || K < 1 || M > h->max_tokens)
    return PE_ERR_INVALID_ARGUMENT;
  if (h->desc.dtype == PE_DTYPE_BF16 && (K % 8 || !aligned16(x) || !aligned16(w)))
    return PE_ERR_INVALID_ARGUMENT;
  if (h->desc.dtype == PE_DTYPE_BF16) {
    const int bn = tc_pick_bn(M, false);
    const long long tiles = static_cast<long long>((N + 127) / 128) * ((M + bn - 1) / bn);
    if (tiles > h->max_tiles) return PE_ERR_INVALID_ARGUMENT;
  }
  EpiArgs ep = epi_none();
  ep.kind = EPI_STORE;
  ep.M = M;
  ep.N = N;
  ep.out = y;
  ep.ldo = N;
  ep.out_f32 = 1;
  return cuda_status(linear(h, x, K, w, nullptr, M, N, K, ep, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
