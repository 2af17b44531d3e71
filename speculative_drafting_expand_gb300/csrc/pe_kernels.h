// pe_kernels.h -- launchers of the sm_103a kernels (host side, internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pe {

// Launch with programmatic stream serialization so a kernel's prologue
// (barrier setup, TMEM allocation, weight prefetch) overlaps the tail of the
// kernel before it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a thread-block cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- expansion
struct ExpandArgs {
  int B, K, T, T_out;
  const int32_t* target_ids;
  const int32_t* target_pos;
  const int32_t* cu_in;
  const int32_t* num_accepted;
  const int32_t* sampled_ids;
  const int32_t* block_table;
  int bt_stride, num_blocks, page_size, mask_token_id;
  const void* target_hidden;
  const void* h_shared;
  int row_bytes;  // hidden3 * element size (multiple of 16)
  int32_t* ids;
  int32_t* pos;
  int32_t* slot;
  uint8_t* is_rejected;
  uint8_t* is_masked;
  int32_t* new_idx;
  int32_t* hidden_map;
  int32_t* cu_out;
  int32_t* seq_lens;
  void* hidden;
  int* err;
};
cudaError_t launch_expand(const ExpandArgs& a, cudaStream_t s);

// Live-row compaction of the expanded batch: the rejected rows of a request
// (window rows after its accepted count) never write the KV cache and feed
// no sampled row, so the drafter layers skip them.  One CTA scans the
// is_rejected flags and writes, for the n_live live rows in expanded order:
// ids/pos/slot copies, the compact index of every expanded row (-1 when
// rejected), the expanded row of every compact row, the compact request
// offsets and the compact index of every sampled row.
struct CompactArgs {
  int B, K, T_out;
  const int32_t* cu_out;        // [B + 1]
  const uint8_t* is_rejected;   // [T_out]
  const int32_t* ids;           // [T_out]
  const int32_t* pos;
  const int32_t* slot;
  const int32_t* new_idx;       // [B K]
  int32_t* row_map;             // [T_out] expanded -> compact, -1 rejected
  int32_t* live_before;         // [T_out + 1] live rows before each expanded row
  int32_t* live_row;            // [T_out] compact -> expanded
  int32_t* ids_c;               // [T_out] (first n_live used)
  int32_t* pos_c;
  int32_t* slot_c;
  int32_t* cu_live;             // [B + 1]
  int32_t* new_c;               // [B K]
  int32_t* n_live;              // [1]
  // optional (fc of the target rows only): the compact row of every target
  // row (-1 when rejected) and the MASK flag of every compact row
  int T;
  const int32_t* hidden_map;    // [T] target row -> expanded row
  const uint8_t* is_masked;     // [T_out]
  int32_t* fc_map;              // [T]
  uint8_t* masked_c;            // [T_out]
};
cudaError_t launch_compact_rows(const CompactArgs& a, cudaStream_t s);

// dst[live_row[c]] = src[c] for the first *n_live compact rows (row_bytes a
// multiple of 16); the other dst rows are left as they are.
cudaError_t launch_scatter_rows(void* dst, const void* src, const int32_t* live_row,
                                const int32_t* n_live, int rows_max, int row_bytes,
                                cudaStream_t s);

// ---------------------------------------------------------------- row ops
// dtype tag: 0 = bf16, 1 = f32 (activations, weights, caches share it)
// `live` (optional, device): rows at or past *live are skipped -- the
// compacted row count, written by a kernel earlier on the stream.
struct EmbedConcatArgs {
  int rows, d, vocab;
  const int32_t* live;
  const int32_t* ids;
  const void* emb;      // [V, d]
  const float* h;       // [rows, d] fp32 fc output (the residual)
  const void* g_e;      // [d]
  const void* g_h;      // [d]
  float eps;
  void* x;              // [rows, 2d] activations
  int* err;
  // optional (fc of the target rows only): MASK rows take the fc of
  // h_shared as their projected hidden state and write it to the residual
  const uint8_t* masked;  // [rows] MASK flags
  const float* fc_hs;     // [d]
  float* h_w;             // the residual (= h), written for MASK rows
  // optional: the rotary table of each row, rope_tab[row][k] = cos and
  // rope_tab[row][dh/2 + k] = sin of pos[row] * inv_freq64[k] (angle in fp64)
  const int32_t* pos;
  const double* inv_freq64;
  float* rope_tab;
  int dh;
};
cudaError_t launch_embed_concat(int dtype, const EmbedConcatArgs& a, cudaStream_t s);

struct RmsNormArgs {
  int rows, d;
  const int32_t* live;
  const float* x;       // [*, d] fp32 residual
  const int32_t* row_index;  // optional gather: out row i reads x[row_index[i]]
  int rows_in;          // bound for row_index values
  const void* g;        // [d]
  float eps;
  void* y;              // [rows, d] activations
  int* err;
  // optional: a projection's output [rows, d] fp32 added to x first (x <-
  // x + add, written back to x_w, the same storage as x), the residual add
  // of that projection done here instead of in its epilogue (no row_index)
  const float* add;
  float* x_w;
};
cudaError_t launch_rmsnorm(int dtype, const RmsNormArgs& a, cudaStream_t s);

struct RopeKvArgs {
  int rows, Hq, Hkv, dh, num_blocks;
  const int32_t* live;
  const void* qkv;          // [rows, (Hq + 2 Hkv) dh]
  const int32_t* pos;       // [rows]
  const int32_t* slot;      // [rows], -1 = no KV write
  const float* inv_freq;    // [dh / 2] (fp32 copy of fp64 table, unused)
  const double* inv_freq64; // [dh / 2]
  void* q_out;              // [rows, Hq dh]
  void* k_cache;            // [num_blocks, Hkv, 16, dh]
  void* v_cache;
  int* err;
  // fp8 (e4m3) pools: k / k_scale and v / v_scale are stored as codes
  int kv_fp8;
  float k_inv_scale, v_inv_scale;
};
cudaError_t launch_rope_kv(int dtype, const RopeKvArgs& a, cudaStream_t s);

struct AttnArgs {
  int rows, B, Hq, Hkv, dh, bt_stride, num_blocks, max_seq;
  int kv_fp8;                // pools hold e4m3 codes; values are code * scale
  float k_scale, v_scale;
  const int32_t* live;       // optional live-row count (per-row kernel only)
  const void* q;             // [rows, Hq dh] (roped)
  const void* k_cache;
  const void* v_cache;
  const int32_t* pos;        // [rows]
  const uint8_t* is_rejected;  // nullable: no rejected rows (compacted batch)
  const int32_t* cu_out;     // [B+1] first row of each request
  const int32_t* block_table;
  void* out;                 // [rows, Hq dh]
  float scale;
  int* err;
};
cudaError_t launch_attention_simt(int dtype, const AttnArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- GEMM
enum EpiKind { EPI_STORE = 0, EPI_ADD = 1, EPI_SILU_MUL = 2, EPI_ARGMAX = 3, EPI_ROPE_KV = 4 };

struct EpiArgs {
  int kind;
  int M, N;                 // valid tokens, valid output features
  void* out;                // STORE / SILU_MUL destination [M, ldo]
  int ldo;
  int out_f32;              // 1: fp32 output, 0: bf16 (or model dtype)
  float* resid;             // ADD: resid[M, ldr] += acc
  int ldr;
  float* logits;            // ARGMAX: optional fp32 [M, ldl]
  int ldl;
  unsigned long long* keys; // ARGMAX: [M] packed (value, index), zero on entry
  int32_t* tokens;          // ARGMAX: [M] result
  const int32_t* row_map;   // STORE (optional): token t goes to row row_map[t], skipped if < 0
  // ROPE_KV (the QKV projection): the weight rows arrive interleaved so
  // that features i and i + dh/2 of every head are neighbouring rows (the
  // A operand through a 4-D tensor map), lanes 2i and 2i+1 of a warp; the
  // epilogue rotates q and k (rotate-half RoPE, cos / sin of each token row
  // from rope_tab), stores q and writes k and v to the paged cache at the
  // row's slot (-1: no write).
  void* q_out;              // [M, Hq dh]
  void* k_cache;            // [num_blocks, Hkv, 16, dh]
  void* v_cache;
  const int32_t* slot;      // [M]
  const float* rope_tab;    // [M, dh]: cos of the dh/2 angles, then their sines
  int rope_rows_interleaved;  // 1: the weight itself is stored interleaved (2-D map)
  int Hq, Hkv, dh, num_blocks;
  int kv_fp8;
  float k_inv_scale, v_inv_scale;
  int* err;
  // RMSNorm folded across two projections (one token tile, M <= 32):
  // ADD also writes xg[t][o] = bf16(new residual * g_next[o]) and, per 32
  // features, ssq[(o / 32) * ssq_ld + t] = the sum of the new residual's
  // squares; a projection of xg with rs_ssq set scales its accumulator row
  // t by r[t] = rsqrt(sum of rs_ssq over the groups / rs_d + rs_eps), since
  // W (x r g) = r W (x g).
  const void* g_next;
  void* xg;
  int ldxg;
  float* ssq;
  int ssq_ld;
  const float* rs_ssq;
  int rs_groups, rs_ld;
  float rs_d, rs_eps;
  // Optional live token count (device): token tiles at or past *m_live are
  // skipped and the work of the live ones is dealt out again.  The
  // tensor-core kernel reads it before waiting on the previous kernel, so
  // it must be written at least two launches earlier on the stream (every
  // kernel here waits on its predecessor before it lets its dependents
  // start).  Not used with the ARGMAX epilogue.
  const int32_t* m_live;
};

// y = x . w^T (+ epilogue) with tcgen05 tensor cores (bf16 in, fp32 accumulate).
// x [M, K] row stride ldx, w [N, K] (w2 the second matrix for SILU_MUL).
struct TcGemmWorkspace {
  float* partials;          // split-K partial tiles
  size_t partial_floats;
  int* tile_counters;       // zero on entry, left zero on exit
  int max_tiles;
  int* done_counter;        // zero on entry, left zero on exit
  int sm_count;
  unsigned long long* timeline;  // diagnostic per-CTA stamps of this launch, or null
  int cluster_push;         // cluster split-K: 1 pushes partials to their owners, 0 pulls
  int pre_stages;           // weight stages loaded before the dependency wait (-1: all)
  int max_split;            // the largest cluster split-K (2..8; 0: 8)
  // stream-K over several token tiles with weights larger than L2
  // (l2_bytes, 0: unknown): 1 token-tile-major, 0 weight-tile-major
  int tile_order;
  long long l2_bytes;
};
cudaError_t launch_gemm_tc(const void* x, int ldx, const void* w, const void* w2, int M, int N,
                           int K, const EpiArgs& epi, const TcGemmWorkspace& ws, int* err,
                           cudaStream_t s);

// The same contraction with FFMA for the fp32 path.
cudaError_t launch_gemm_simt(const float* x, int ldx, const float* w, const float* w2, int M,
                             int N, int K, const EpiArgs& epi, int* err, cudaStream_t s);
cudaError_t launch_argmax_finalize(int M, unsigned long long* keys, int32_t* tokens,
                                   cudaStream_t s);

// ---------------------------------------------------------------- streaming segments
// The layer projections between two attention launches as one persistent
// kernel for small row counts (at most 32 rows: one token tile), stream.cu.
// A segment is a short program of phases: GEMM phases (fc, O, gate/up,
// down, QKV) and row phases (the layer-0 input, the final norm).
constexpr int kStreamMaxPhases = 5;
constexpr int kStreamMaxMaps = 12;
constexpr int kStreamSyncInts = 16;   // [0, kStreamMaxPhases): phase done counts
constexpr int kStreamSyncExit = 8;    // CTAs that finished the kernel
constexpr int kStreamSyncAbort = 9;   // set when a bounded wait gave up
// Diagnostic timeline of one segment launch (%globaltimer, ns), per CTA:
// [0] start, [1] tensor memory held, [2] weight stream issued its first
// load; then per phase ph at 4 + 4 ph: [+0] previous phase complete
// everywhere, [+1] activation panel landed (MMA issuer), [+2] the issuer
// committed its last MMA of the phase, [+3] this CTA's last tile of the
// phase done (partial stored, or finished and published); [60] end.
constexpr int kStreamTimelineSlots = 64;
enum StreamKind { SK_GEMM = 0, SK_EMBED = 1, SK_FINAL = 2 };
enum StreamEpi { SE_STORE = 0, SE_ADD = 1, SE_SILU_MUL = 2, SE_ROPE_KV = 3 };

struct StreamPhase {
  int kind, epi, dual;
  int N, K, kb, tiles;     // GEMM: y[rows, N] = x[rows, K] . w[N, K]^T
  int map_a, map_a2;       // weight tensor maps (indices into StreamMaps)
  const void* w;           // the same weights [N, K] bf16 (row stride K), for L2 prefetch
  const void* w2;
  const void* x;           // activations [rows, K] bf16, row stride ldx (16-byte aligned)
  int ldx;
  int norm_src;            // phase whose sums of squares scale this GEMM's rows (-1: none)
  int norm_d;              // width of that norm
  const void* g_next;      // ADD: gain of the next norm; xg = bf16(residual * g_next)
  void* xg;                // ADD: [rows, N] bf16 (nullable)
  float* ssq;              // ADD: [tiles][32] sums of squares of the new residual
  void* out;               // SILU_MUL: [rows, ldo] bf16
  int ldo;
  int* counters;           // [tiles] arrivals (zeroed at kernel exit)
};

struct StreamParams {
  int rows, nphases, final_rows, d;
  StreamPhase ph[kStreamMaxPhases];
  float* resid;            // [rows, d] fp32 residual stream
  float eps;
  // layer-0 input: x_in[r] = [RMSNorm_e(emb[ids[r]]) ; RMSNorm_h(resid[r])]
  const int32_t* ids;
  const void* emb;
  int vocab;
  const void* g_e;
  const void* g_h;
  void* x_in;              // [rows, 2d] bf16
  // QKV epilogue: rotate-half RoPE of q and k, k and v to the paged cache
  const int32_t* pos;
  const int32_t* slot;
  int Hq, Hkv, dh, num_blocks;
  const double* inv_freq64;
  void* q_out;             // [rows, Hq dh] bf16
  void* k_cache;           // [num_blocks, Hkv, 16, dh] bf16 (e4m3 codes when kv_fp8)
  void* v_cache;
  int kv_fp8;              // pools hold e4m3 codes of k / k_scale and v / v_scale
  float k_inv_scale, v_inv_scale;
  // final norm of the sampled rows
  const int32_t* new_idx;  // [final_rows]
  const void* g_final;
  void* out_hidden;        // [final_rows, d] bf16
  int prefetch_tiles;      // weight tiles brought into L2 ahead of the ring (0: none)
  int boundary_tiles;      // loads into a phase before its inputs are ready (-1: no limit)
  unsigned long long* timeline;  // diagnostic: [grid][kStreamTimelineSlots] ns stamps, or null
  float* ws;               // split-K partials [grid][2][128 * 32 * 2]
  int* sync;               // [kStreamSyncInts], zero on entry, left zero
  int* counters;           // every phase's tile counters, zero on entry, left zero
  int n_counters;
  int* err;
};

struct StreamMaps {
  CUtensorMap m[kStreamMaxMaps];
};

// Launch one segment (rows <= 32); grid = one CTA per SM.
cudaError_t launch_stream(const StreamMaps& maps, const StreamParams& p, int grid,
                          cudaStream_t s);
cudaError_t init_stream();
// Largest number of k-blocks one CTA may take in a GEMM phase (its
// activation panel), for rows token rows.
int stream_panel_kb(int rows);
size_t stream_ws_floats(int grid);

// tensor-map encoder (fetched once through cudart)
bool tensor_map_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                        uint64_t ld_elems, uint32_t box_cols, uint32_t box_rows);
// The QKV weight [(Hq + 2 Hkv) dh, K] as [heads][2][dh/2][K]: a box of
// 128 / dh heads x both halves x dh/2 rows x 64 k lands in shared memory as
// 128 rows with the halves interleaved (row 2i + b = feature i + b dh/2).
bool tensor_map_qkv_interleaved(CUtensorMap* m, const void* ptr, int heads, int dh, uint64_t K);

}  // namespace pe
