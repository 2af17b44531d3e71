/*
 * peagle.h -- C ABI of the P-EAGLE parallel drafting step on one GB300 (sm_103a).
 *
 * One drafting step turns the verified target batch into all K draft tokens
 * of every request in a single drafter pass:
 *
 *   pe_expand_batch   -> expanded rows [token, MASK, ..., MASK] + metadata
 *                        + expanded target hidden states (h_shared in MASK rows)
 *   pe_draft_forward  -> N LLaMA-style drafter layers over the expanded rows,
 *                        paged-KV causal attention, final RMSNorm of the
 *                        B*K rows that get sampled
 *   pe_lmhead_argmax  -> LM head and argmax: one draft token per sampled row
 *
 * Sources (web pages on P-EAGLE), cited by title and section:
 *   [paper] "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training",
 *           section 2 (architecture) and Figure 2.
 *   [blog]  "P-EAGLE: Faster LLM Inference with Parallel Speculative Decoding
 *           in vLLM": the input formula (Input_i = emb(new) (+) h_context for
 *           i = 1, emb(mask) (+) h_shared for 2 <= i <= K), prompt-position
 *           handling (position i carries the hidden state of i-1), and the
 *           engineering section (fused expansion kernel, hidden-state
 *           management, KV-cache slot mapping with -1 for rejected tokens).
 *
 * Conventions shared by every entry point
 *   - All tensors are caller-owned DEVICE memory on the current device unless
 *     a parameter says "host".  The library never frees caller memory.  The
 *     handle owns only its workspace, allocated in pe_create.
 *   - Every compute call is asynchronous on the given stream (cudaStream_t
 *     passed as void*; NULL = legacy default stream).  Calls on one handle
 *     must not overlap in time (they share the workspace).
 *   - Host-checkable errors are returned synchronously and launch nothing:
 *     PE_ERR_INVALID_ARGUMENT (bad size, null pointer, misaligned pointer),
 *     PE_ERR_UNSUPPORTED (a shape the kernels do not implement),
 *     PE_ERR_CUDA (a CUDA runtime call or launch failed).
 *   - Data-dependent violations found by the kernels (an accepted count
 *     outside the window, a block id outside [0, num_blocks), a position past
 *     the block table, a token id outside the vocabulary, a wait that timed
 *     out) never trap: the kernel records a code, skips the offending write,
 *     and pe_get_device_error reports it.
 *   - Matrices are row-major [out, in].  bf16 tensors are IEEE bfloat16.
 *   - No C++ exception crosses this ABI and the library keeps no global state
 *     besides the per-device tensor-map encoder entry point.
 */
#ifndef PEAGLE_H_
#define PEAGLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pe_status;
enum {
  PE_OK = 0,
  PE_ERR_INVALID_ARGUMENT = 1,
  PE_ERR_UNSUPPORTED = 2,
  PE_ERR_CUDA = 3,
  PE_ERR_OUT_OF_MEMORY = 4,
  PE_ERR_DEVICE = 5 /* a kernel recorded a data-dependent violation */
};

/* Device-side error codes reported by pe_get_device_error (first one wins). */
enum {
  PE_DEV_OK = 0,
  PE_DEV_BAD_ACCEPTED = 1,    /* num_accepted[r] outside [0, n_r - 1] */
  PE_DEV_BAD_BLOCK = 2,       /* block id outside [0, num_blocks) */
  PE_DEV_BAD_POSITION = 3,    /* position beyond bt_stride * page_size */
  PE_DEV_BAD_TOKEN = 4,       /* token id outside [0, vocab) */
  PE_DEV_TIMEOUT = 5,         /* a bounded wait inside a kernel gave up */
  PE_DEV_BAD_ROW = 6          /* a row index outside the expanded batch */
};

typedef enum { PE_DTYPE_BF16 = 0, PE_DTYPE_F32 = 1 } pe_dtype;

/* Drafter shape ([paper] section 2: N LLaMA 3 decoder layers with RoPE). */
typedef struct {
  int32_t d;             /* drafter hidden width */
  int32_t n_layers;      /* N */
  int32_t n_heads;       /* query heads Hq */
  int32_t n_kv_heads;    /* key/value heads Hkv (Hq % Hkv == 0) */
  int32_t head_dim;      /* dh: 64 or 128 */
  int32_t ffn;           /* SwiGLU inner width F */
  int32_t vocab;         /* V */
  int32_t hidden3;       /* width of the target hidden states = 3d ([paper] Fig. 2) */
  int32_t page_size;     /* KV page size: must be 16 */
  int32_t mask_token_id; /* the MASK token id ([blog] fused-kernel bullet) */
  float rope_theta;      /* rotate-half RoPE base */
  float rms_eps;         /* RMSNorm epsilon */
  int32_t dtype;         /* pe_dtype of weights, hidden states, KV cache */
} pe_model_desc;

/* One decoder layer's weights (borrowed device pointers, dtype of the model).
 * qkv [(Hq + 2 Hkv) dh, d_in] with rows ordered q heads, k heads, v heads;
 * d_in = 2d for layer 0 (input = [RMSNorm_e(emb) ; RMSNorm_h(fc h)]) and d
 * for later layers.  o [d, Hq dh]; gate, up [F, d]; down [d, F].
 * Norm gains are [d]: norm_e and norm_h for layer 0, norm_in for later
 * layers (NULL where not used), norm_post for every layer. */
typedef struct {
  const void* qkv;
  const void* o;
  const void* gate;
  const void* up;
  const void* down;
  const void* norm_e;
  const void* norm_h;
  const void* norm_in;
  const void* norm_post;
} pe_layer_weights;

/* Drafter weights (borrowed device pointers; must outlive the handle).
 * emb [V, d] (its MASK row is the learned emb(mask)); fc [d, hidden3];
 * h_shared [hidden3] ([blog] hidden-state management; [paper] section 2);
 * norm_final [d]; lm_head [V, d]; layers: HOST array of n_layers entries
 * (copied by pe_create). */
typedef struct {
  const void* emb;
  const void* fc;
  const void* h_shared;
  const void* norm_final;
  const void* lm_head;
  const pe_layer_weights* layers;
} pe_weights;

/* The expanded drafting batch.  Device pointers are caller-owned buffers
 * sized for T' = T + B (K - 1) rows; pe_expand_batch fills them and records
 * B, K, T and T_out (host fields) and the target_hidden pointer it was
 * given, for pe_draft_forward.  When target_hidden is recorded (not NULL),
 * pe_draft_forward projects the T target rows through fc and gives every
 * MASK row the fc of h_shared computed once at pe_create, instead of
 * projecting all T' rows of `hidden` (the same values: MASK rows carry
 * h_shared); that buffer must then still hold the same data when
 * pe_draft_forward runs.  Set it to NULL to make pe_draft_forward project
 * `hidden`.
 * Layout of request r: rows cu_out[r] .. cu_out[r] + n_r - 1 come from the
 * target window (row j carries the target hidden state of window row j and
 * sits one position after it), rows cu_out[r] + n_r .. + n_r + K - 2 are the
 * K - 1 MASK rows. */
typedef struct {
  int32_t* ids;          /* [T'] token ids */
  int32_t* pos;          /* [T'] positions */
  int32_t* slot;         /* [T'] KV slot = block * 16 + pos % 16; -1 if rejected */
  uint8_t* is_rejected;  /* [T'] 1 for window rows after the accepted prefix */
  uint8_t* is_masked;    /* [T'] 1 for MASK rows */
  int32_t* new_idx;      /* [B*K] rows that are sampled: next-token row, then MASK rows */
  int32_t* hidden_map;   /* [T] target row t -> expanded row */
  int32_t* cu_out;       /* [B+1] first expanded row of each request */
  int32_t* seq_lens;     /* [B] drafter sequence length after this step */
  void* hidden;          /* [T', hidden3] expanded target hidden states */
  int32_t B, K, T, T_out;  /* host fields written by pe_expand_batch */
  const void* target_hidden;  /* [T, hidden3] the target rows (see above), or NULL */
} pe_expanded;

typedef struct pe_handle pe_handle;

/* Create a handle: validates the shape, copies the layer-pointer array,
 * builds the TMA descriptors of the weights and allocates the workspace for
 * up to max_tokens expanded rows and max_reqs requests.  Weights are
 * borrowed; every weight buffer must hold its full shape.  fc and h_shared
 * are read here (fc of h_shared, on the default stream, synchronised before
 * returning).  Returns PE_ERR_UNSUPPORTED for shapes the kernels do not cover
 * (d, F, hidden3 and Hq*dh must be multiples of 64; dh in {64, 128};
 * page_size 16). */
pe_status pe_create(const pe_model_desc* desc, const pe_weights* weights,
                    int32_t max_tokens, int32_t max_reqs, pe_handle** out);

/* Free the handle's workspace (synchronises the device first). */
pe_status pe_destroy(pe_handle* h);

/* Batch expansion + hidden-state broadcast ([blog] engineering section:
 * fused expansion kernel and hidden-state management; KV-cache bullet).
 *
 * Inputs (device): target_ids/target_pos [T] int32, the verify window of
 * every request back to back; cu_in [B+1] int32 window offsets (n_r =
 * cu_in[r+1] - cu_in[r] >= 1); num_accepted [B] int32 (a_r in [0, n_r-1]);
 * sampled_ids [B] int32 (the target's sampled token per request);
 * block_table [B, bt_stride] int32 physical page ids; target_hidden
 * [T, hidden3] (model dtype).  B, K, T, bt_stride, num_blocks are host ints.
 * Rules per request r (a = a_r, s = sampled, q_j = target_pos of window
 * row j): row j < n_r gets position q_j + 1 and token target_ids[j+1] (s for
 * the last row), then row a gets s; rows j > a are rejected (slot -1);
 * MASK rows k = 1..K-1 get the MASK id at position q_a + 1 + k;
 * new_idx = [row a, MASK rows]; seq_lens = q_a + K + 1;
 * hidden[hidden_map[t]] = target_hidden[t], then MASK rows = h_shared.
 * Writes every field of *out (which the caller fills with buffer pointers).
 * Requires 1 <= K <= 16 and n_r + K - 1 <= 32. */
pe_status pe_expand_batch(pe_handle* h, int32_t B, int32_t K, int32_t T,
                          const int32_t* target_ids, const int32_t* target_pos,
                          const int32_t* cu_in, const int32_t* num_accepted,
                          const int32_t* sampled_ids, const int32_t* block_table,
                          int32_t bt_stride, int32_t num_blocks,
                          const void* target_hidden, pe_expanded* out,
                          void* stream);

/* The drafter pass over the expanded batch ([paper] section 2: all rows go
 * through the N layers at once; [blog] "parallel prediction").
 *
 * Per row: e = emb[id], h = fc x hidden; layer 0 input [RMSNorm_e(e) ;
 * RMSNorm_h(h)], residual h; each layer: QKV projection, rotate-half RoPE at
 * the row's position, K/V written to the paged cache at slot (rows with
 * slot -1 write nothing), causal attention of every non-rejected row over
 * positions 0..pos of its request (GQA), O projection + residual, RMSNorm,
 * SwiGLU MLP + residual.  Finally the rows new_idx are gathered and
 * RMSNorm'ed with norm_final into out_hidden [B*K, d] (model dtype).
 * Rejected rows write nothing and feed no sampled row, so after fc the
 * layers run on the live rows only (found on the device, so the call's
 * launches do not depend on the accepted counts and can be captured in a
 * CUDA graph); this changes no result.
 * k_cache/v_cache: HOST arrays of n_layers device pointers, each a pool
 * [num_blocks, Hkv, 16, dh] (model dtype, 16-byte aligned); block_table as
 * in pe_expand_batch.  B and K must match the values recorded in *ex, and
 * B <= max_reqs.
 * Each request's verify window is expected to hold at most K + 1 rows (the
 * previous step's drafts plus one); a request with more rows than that is
 * reported as PE_DEV_BAD_ROW.  The bf16 path keeps a split-KV workspace
 * sized by B and bt_stride: the first call with a larger batch or block
 * table grows it with cudaMalloc, so make that call before capturing the
 * step into a CUDA graph. */
pe_status pe_draft_forward(pe_handle* h, const pe_expanded* ex, int32_t B,
                           int32_t K, const int32_t* block_table,
                           int32_t bt_stride, void* const* k_cache,
                           void* const* v_cache, int32_t num_blocks,
                           void* out_hidden, void* stream);

/* LM head + argmax ([paper] section 2: LM head after the N layers).
 * hidden [M, d] (model dtype, already final-normed), M <= max_tokens.
 * out_tokens [M] int32: argmax over the vocabulary of hidden x lm_head^T,
 * lowest index on ties.  out_logits: NULL, or [M, V] fp32 logits. */
pe_status pe_lmhead_argmax(pe_handle* h, const void* hidden, int32_t M,
                           int32_t* out_tokens, float* out_logits,
                           void* stream);

/* Synchronise the stream, return the first device-side error code recorded
 * since the last call (PE_DEV_*), and clear it. */
pe_status pe_get_device_error(pe_handle* h, int32_t* code, void* stream);

/* Self-check of the bounded waits (no counterpart on the pages; the
 * failure handling of every kernel here rests on it).  Launches one kernel
 * that waits on an mbarrier nobody arrives on and then on a global flag
 * nobody sets; each wait gives up after the library's wait limit (2 s),
 * records PE_DEV_TIMEOUT in the handle's error word and the kernel returns.
 * out: caller-owned device int32[2], set to 1 for each wait that gave up
 * (0 if it was satisfied).  Asynchronous on `stream`; takes about 4 s of
 * GPU time; the context stays usable afterwards. */
pe_status pe_check_bounded_wait(pe_handle* h, int32_t* out, void* stream);

/* fp8 KV cache (the pages' deployment runs with --kv-cache-dtype fp8): after
 * this call the k_cache / v_cache pools that pe_draft_forward receives hold
 * OCP FP8 E4M3 codes, one byte per element in the same [num_blocks, Hkv, 16,
 * dh] layout; layer l stores k / k_scales[l] and v / v_scales[l], rounded to
 * the nearest e4m3 value (ties to even) and saturated to +-448, and its
 * attention reads code * scale.  k_scales, v_scales: HOST arrays of
 * n_layers positive finite floats, copied; both NULL return to pools of the
 * model dtype.  PE_ERR_UNSUPPORTED unless the model is bf16 with head_dim
 * 64; PE_ERR_INVALID_ARGUMENT for a non-positive or non-finite scale or only
 * one of the two arrays. */
pe_status pe_set_kv_cache_fp8(pe_handle* h, const float* k_scales, const float* v_scales);

/* Optional diagnostics: when residual_trace is non-NULL, every later
 * pe_draft_forward copies the fp32 residual stream [T', d] after each layer
 * (rows in expanded order; rows the layers skipped as rejected read zero)
 * into residual_trace + layer * max_tokens * d (caller-owned device buffer of
 * n_layers * max_tokens * d floats).  When attn_trace is non-NULL, it copies
 * each layer's attention output [T', Hq * dh] (model dtype, rejected rows
 * zero) into
 * attn_trace + layer * max_tokens * Hq * dh elements.  NULL turns a trace
 * off. */
pe_status pe_set_trace(pe_handle* h, float* residual_trace, void* attn_trace);

/* Phase timing (diagnostic; no counterpart on the pages).  events: n =
 * 2 + 2 * n_layers caller-created CUDA events (cudaEvent_t, passed as
 * void*), or n = 0 to turn it off.  While set, pe_draft_forward records
 * event 0 when it starts, event 1 + 2l just before layer l's attention,
 * event 2 + 2l just after it, and event 1 + 2 n_layers at its end, on its
 * stream, so that the caller can split the step's time into attention and
 * the rest.  Recording events between kernels breaks the overlap of
 * consecutive kernels, so a timed step runs a little slower with them.
 * The handle keeps the event handles, not the events: they must outlive
 * their use. */
pe_status pe_set_phase_events(pe_handle* h, void* const* events, int32_t n);

/* Small-batch streaming (off by default).  With enable = 1, when a step's
 * expanded rows fit one 16- or 32-row token tile, pe_draft_forward runs the
 * projections between two attention launches (fc, the layer-0 input and
 * QKV; then O, gate/up, down and the next QKV or the final norm) as one
 * persistent kernel per segment, with RMSNorm, RoPE and the KV write fused
 * into it, instead of one launch per projection.  The results agree with
 * the per-projection path up to fp32 summation order.  Measured slower on
 * the GPT-OSS-20B-shaped batch-1 step (about 655 against 515 us): every
 * phase boundary waits for the slowest tile's split-K finisher, a chain of
 * dependent L2 round trips of about 1 us each. */
pe_status pe_set_small_batch_stream(pe_handle* h, int32_t enable);

/* Epilogue fusions of the per-projection path (bf16), a bit mask; the
 * default is PE_FUSE_NORM:
 *   PE_FUSE_ROPE_KV  at most 32 expanded rows: rotate-half RoPE of q and k
 *                    and the paged K/V write in the QKV projection's
 *                    epilogue (no separate kernel and no round trip of the
 *                    qkv activations through memory);
 *   PE_FUSE_NORM     at most 32 expanded rows: the RMSNorms before gate/up
 *                    and before the next layer's QKV folded into the
 *                    projections (the residual add writes x * g and sums of
 *                    squares, the next projection scales its rows by
 *                    rsqrt(mean x^2 + eps)), instead of a norm kernel;
 * 0 selects the separate kernels.  Measured on the GPT-OSS-20B-shaped
 * batch-1 step (us per step): none 526, PE_FUSE_ROPE_KV 535,
 * PE_FUSE_NORM 516, both 521 -- the fused RoPE epilogue loses what the
 * removed kernel costs, hence the default. */
enum { PE_FUSE_ROPE_KV = 1, PE_FUSE_NORM = 2, PE_FUSE_ALL = 3 };
pe_status pe_set_fusions(pe_handle* h, int32_t mask);

/* How a projection split over the k dimension across a thread-block
 * cluster (few token rows: fewer weight tiles than SMs) sums its partial
 * tiles.  PE_REDUCE_PUSH (the default): every CTA, once the cluster's
 * operand stages are free, stores each (32-row, 16-column) item of its
 * fp32 partial into the shared memory of the CTA that owns the item
 * (st.async, counted on the owner's mbarrier), and the owner adds the
 * partials in rank order.  PE_REDUCE_PULL: every CTA keeps its partial,
 * a cluster barrier, and the owner reads the peers' partials with
 * distributed-shared-memory loads.  Both add in the same order: the
 * results are bit-identical.  Returns PE_ERR_INVALID_ARGUMENT for another
 * value. */
enum { PE_REDUCE_PULL = 0, PE_REDUCE_PUSH = 1 };
pe_status pe_set_split_reduce(pe_handle* h, int32_t mode);

/* Launch tuning of the projection kernels, one key at a time.
 *   PE_TUNE_GEMM_PRE_STAGES  how many of a CTA's weight stages it loads
 *                            before its wait for the previous kernel (the
 *                            weights do not depend on it); -1: all of its
 *                            shared-memory stages, 0: none; default 3
 *                            (measured on the GPT-OSS-20B-shaped batch-1
 *                            step: about 500 us against 509 us with all
 *                            five stages of the narrow token tile).
 *   PE_TUNE_ATTN_L2_AHEAD    how many 128-key chunks of K/V pages each
 *                            attention CTA brings into L2 ahead of its
 *                            shared-memory ring (cp.async.bulk.prefetch;
 *                            the first ones before its wait for the
 *                            previous kernel), 0..64; default 0 (2, 4
 *                            and 8 measured slower: 2900 against 3230 us
 *                            a GPT-OSS-shaped batch-64 step).
 *   PE_TUNE_GEMM_MAX_SPLIT   the largest number of CTAs (a thread-block
 *                            cluster) that split one projection tile's k
 *                            range when there are fewer tiles than SMs,
 *                            1..8; default 8 (4, 3 and 2 measured slower
 *                            at batch 1 and on the Qwen-shaped batch 16).
 *   PE_TUNE_ATTN_MIN_CHUNKS  the fewest 128-key chunks one attention CTA
 *                            (key split) takes, 2..32; default 2 (splits
 *                            are otherwise sized to fill the SMs).
 *   PE_TUNE_ATTN_MAX_CHUNKS  the most chunks one attention split takes,
 *                            2..64 (at most 32 at dh 128); default 64.
 *                            More splits need a larger
 *                            split workspace, which the next
 *                            pe_draft_forward outside a graph capture
 *                            allocates.
 *   PE_TUNE_GEMM_TILE_ORDER  a stream-K projection with several token
 *                            tiles and weights larger than L2 (the LM
 *                            head at batch 64): 1 token-tile major, the
 *                            grid cut to a multiple of the token tiles so
 *                            that the CTAs of every token tile take the
 *                            same k ranges of the same weight tiles at the
 *                            same time (each weight k-block from memory
 *                            once, then from L2); 0 weight-tile major (the
 *                            token tiles of a weight tile one after
 *                            another in one CTA's range, as the layer
 *                            projections always are: token-tile major
 *                            measured slower for them).  Default 1.
 * Returns PE_ERR_INVALID_ARGUMENT for an unknown key or a value out of
 * range.  PE_TUNE_GEMM_PRE_STAGES and PE_TUNE_ATTN_L2_AHEAD leave the
 * results bit-identical; the other keys move the points where a k range or
 * a key range is split, so fp32 partial sums may round differently (each
 * setting computes the same exact sums in another order). */
enum {
  PE_TUNE_GEMM_PRE_STAGES = 1,
  PE_TUNE_ATTN_L2_AHEAD = 2,
  PE_TUNE_GEMM_MAX_SPLIT = 3,
  PE_TUNE_ATTN_MIN_CHUNKS = 4,
  PE_TUNE_ATTN_MAX_CHUNKS = 5,
  PE_TUNE_GEMM_TILE_ORDER = 6
};
pe_status pe_set_tuning(pe_handle* h, int32_t key, int32_t value);

/* Tuning of the small-batch streaming kernel.  tiles: how many 16 KB
 * weight tiles each CTA brings into L2 ahead of its shared-memory ring
 * (default 0 = none; at most 4096).  boundary_tiles: how many weight tiles
 * a CTA may load into a phase whose inputs are not complete yet (default
 * -1 = no limit). */
pe_status pe_set_stream_prefetch(pe_handle* h, int32_t tiles, int32_t boundary_tiles);

/* Diagnostic timeline of the small-batch streaming kernel (no counterpart
 * on the pages).  stamps: caller-owned device buffer of sm_count * 64
 * uint64 (NULL turns it off); every segment launch overwrites it with
 * %globaltimer stamps in ns per CTA: [0] start, [1] tensor memory held,
 * [2] first weight load issued, then for phase p at 4 + 4p: [+0] previous
 * phase complete on every CTA, [+1] activation panel landed, [+2] last MMA
 * of the phase issued, [+3] the CTA's last tile of the phase done; [60] end.
 * Slots a launch does not reach keep their old contents. */
pe_status pe_set_stream_timeline(pe_handle* h, uint64_t* stamps);

/* Diagnostic timeline of the projection and attention kernels (no
 * counterpart on the pages).  stamps: caller-owned device buffer of
 * launches * 512 * 16 uint64 (NULL turns it off).  Launch k of a step's
 * projections and attentions (counted from the start of pe_draft_forward,
 * pe_lmhead_argmax continuing the count) writes per CTA c < 512 at
 * (k * 512 + c) * 16.  Projection: [0] start, [1] the wait for the
 * previous kernel returned, [2] first stage landed, [3] last MMA issued,
 * [4] the epilogue's main loop done, [5] every partial of a cluster split
 * ready, [8] the first reduction item summed, [7] the CTA's reduction
 * items applied, [6] exit.  Attention: [0] start, [1] set up, [2] the wait
 * returned, [3] Q staged, [4] first scores, [5] last P.V, [6] partial
 * written, [7] every split written, [8] merged, [9] exit.  (%globaltimer,
 * ns; slots not reached keep their old contents.) */
pe_status pe_set_gemm_timeline(pe_handle* h, uint64_t* stamps, int32_t launches);

/* y[M, N] = x[M, K] . w[N, K]^T with the library's GEMM for the model dtype
 * (tcgen05 tensor cores for bf16, FFMA for f32); y is fp32.  A diagnostic
 * entry point for checking the projection kernels in isolation; K % 64 == 0
 * for bf16. */
pe_status pe_linear(pe_handle* h, const void* x, const void* w, float* y,
                    int32_t M, int32_t N, int32_t K, void* stream);

/* y[M, N] = x[M, K] . w[N, K]^T in bf16 on the tensor cores (fp32 out),
 * without a handle and without allocating anything.  The P-EAGLE pages have
 * no counterpart: this is for callers that may not call cudaMalloc -- code
 * running inside an allocator or memory-pool callback, under a framework
 * that owns every byte of device memory, or on a path that must never enter
 * the driver's allocator.  x [M, K] and w [N, K] are 16-byte-aligned bf16,
 * y [M, N] fp32, all caller-owned device memory; K % 8 == 0.
 * The split-K scratch is one static device array of about 5.3 MB, reserved
 * on every GPU that loads the library until the process exits; it bounds
 * M <= 32 and N <= 4096 * 128, and larger sizes return PE_ERR_UNSUPPORTED
 * before launching anything.  It holds split-K partials for up to 160 SMs:
 * a GPU with more runs the projection on 160 of them.  The first call on a device looks up the
 * array's device address and prepares the kernels for that device; make
 * that first call before any stream capture.  All calls share the array,
 * so calls that overlap on the GPU race on it and must be serialised by the
 * caller.  Asynchronous on `stream`. */
pe_status pe_linear_static(const void* x, const void* w, float* y, int32_t M,
                           int32_t N, int32_t K, void* stream);

/* Read and clear the device error word that pe_linear_static's kernels
 * write into the same static array (0: nothing recorded since the last
 * read; PE_DEV_TIMEOUT: a bounded wait gave up and y may be incomplete).
 * The word persists across calls until this reads it.  Synchronises
 * `stream`; allocates nothing.  No counterpart on the P-EAGLE pages. */
pe_status pe_linear_static_error(int32_t* code, void* stream);

/* Number of kernels this handle has launched since pe_create (host-side
 * count, incremented per launch, including launches captured into a CUDA
 * graph).  A diagnostic for counting the kernels of one step. */
pe_status pe_get_launch_count(pe_handle* h, int64_t* count);

/* Static description of a status code. */
const char* pe_status_string(pe_status s);

#ifdef __cplusplus
}
#endif

#endif /* PEAGLE_H_ */
