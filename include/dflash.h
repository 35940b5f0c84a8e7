/*
 * dflash.h - C ABI of the DFlash KV-injection draft attention step on GB300 (sm_103a).
 *
 * The step (DFlash KV Injection Walkthrough, Steps 1-4 and 7; DFlash source
 * guide (II): Qwen3DFlashAttention, parts 1-5):
 *
 *   C      = RMSNorm_gh( concat[h^(l1) .. h^(lk)] W_fc^T )             dflash_ctx_project
 *   cache += RoPE(KNorm(C W_K^T)), C W_V^T  at the rows' positions     dflash_kv_inject
 *   Q, Kb, Vb = RoPE(QNorm(H W_Q^T)), RoPE(KNorm(H W_K^T)), H W_V^T
 *   out    = softmax(Q [cache K || Kb]^T d_h^-0.5) [cache V || Vb]      dflash_block_attn
 *   lens   = accepted prefix                                            dflash_cache_crop
 *
 * Conventions shared by every call:
 *  - Every pointer argument named "device" is CUDA device memory owned by the
 *    caller. The library never allocates or frees memory.
 *  - Every call enqueues kernels on the given stream and returns without
 *    synchronising, except dflash_status_get.
 *  - Matrices are row-major. Weights use the nn.Linear layout
 *    [out_features, in_features]; a projection is x W^T. (The walkthrough's
 *    "W_fc in R^{1536x512}" is the transpose of the fc array passed here.)
 *  - Element type of every activation, weight, gamma and cache buffer is
 *    dims->dtype (float32 or bfloat16). Arithmetic is fp32 throughout; bf16
 *    results are rounded once, when stored.
 *  - Errors the host can see (null pointers, unsupported dims, a workspace
 *    that is too small, a misaligned pointer) are returned at once and
 *    nothing is launched. Errors only the device can see (an append beyond
 *    the cache capacity or the RoPE table, a crop beyond the current length)
 *    set bits of a sticky per-device status word and skip the offending
 *    sequence, leaving its lengths unchanged; dflash_status_get reads them.
 *  - A launch failure returns DFLASH_ERR_CUDA.
 *  - Slot j of a sequence's cache holds the row at absolute position j.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, negative size, bad layer index */
  DFLASH_ERR_UNSUPPORTED = 2,  /* dims outside the supported set (see dflash_dims) */
  DFLASH_ERR_WORKSPACE = 3,    /* workspace smaller than dflash_workspace_bytes() asks */
  DFLASH_ERR_CUDA = 4,         /* a CUDA runtime error while launching */
  DFLASH_ERR_DEVICE = 5        /* dflash_status_get: the device status word is non-zero */
} dflash_status;

/* DFLASH_FP8_E4M3 is a cache element type only (dflash_kv_cache.kv_dtype). */
typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1, DFLASH_FP8_E4M3 = 2 } dflash_dtype;

/* Bits of the device status word (dflash_status_get). */
#define DFLASH_DEV_CAPACITY  1u  /* append beyond the cache capacity: sequence skipped */
#define DFLASH_DEV_ROPE      2u  /* a position beyond the RoPE table: sequence skipped */
#define DFLASH_DEV_CROP      4u  /* crop to a negative length or beyond the current one */
#define DFLASH_DEV_ROWS      8u  /* cu_rows not non-decreasing or beyond M */
#define DFLASH_DEV_TIMEOUT  16u  /* an internal pipeline wait gave up (kernel returned early) */

/*
 * Model dimensions.
 *   d          hidden size
 *   n_h, n_kv  query and key/value heads; G = n_h / n_kv query heads share a
 *              KV head, query head h reading KV head h / G (DFlash source
 *              guide (II), part 1: num_key_value_groups)
 *   d_h        head dimension
 *   k_layers   number of target layers whose hidden states are concatenated
 *   block_size block length bs (anchor + mask tokens)
 *   eps        RMSNorm epsilon (hidden_norm, q_norm, k_norm)
 *   dtype      dflash_dtype of all tensors
 * Supported: 1 <= k_layers <= 8; n_h % n_kv == 0; d % 8 == 0.
 *   bf16: d_h == 128, d % 64 == 0, G * block_size <= 128.
 *   Both: block_size <= 16.
 *   f32:  d_h even and <= 256.
 */
typedef struct {
  int d, n_h, n_kv, d_h, k_layers, block_size;
  float eps;
  int dtype;
} dflash_dims;

/*
 * Draft KV cache, all device memory owned by the caller.
 *   k, v      contiguous (block_table == NULL):
 *               [n_layers][batch][n_kv][capacity][d_h] elements of dims->dtype
 *             paged (block_table != NULL, bf16 only):
 *               [n_layers][n_pages][n_kv][page_size][d_h]; logical slot s of
 *               sequence b lives in page block_table[b][s / page_size] at row
 *               s % page_size of every layer's pool
 *             16-byte aligned
 *   lens      int32 [n_layers][batch]: rows held per layer and sequence
 *   capacity  logical rows per sequence (paged: a multiple of page_size)
 *   block_table  device int32 [batch][capacity / page_size] page ids in [0, n_pages),
 *             or NULL; page_size must be 128 (one page is one attention tile)
 *   kv_dtype  element type of k and v: 0 (the same as dims->dtype), or
 *             DFLASH_FP8_E4M3 (one byte per element; bf16 dims only, either layout):
 *             the code of x / scale, rounded to the nearest finite E4M3 value
 *             (ties to even, magnitudes beyond 448 saturate), which reads back as
 *             scale * value
 *   kv_scales fp8 only: HOST float [n_layers][2] = (k_scale, v_scale) per layer,
 *             each finite and > 0, read when a call is made (a captured graph keeps
 *             the values of its capture); NULL means 1 everywhere
 * (DFlash source guide (II), part 4: the DynamicCache that update() appends
 * to and crop(start) truncates. A paged cache holds the same logical rows; the
 * caller owns the page allocation, lengths and crops stay logical. KV Cache +
 * Speculative Decoding Interview Cheat Sheet, sections 2.1 and 4.5: an fp8 cache
 * element is one byte, half the bytes the attention streams.)
 */
typedef struct {
  void* k;
  void* v;
  int32_t* lens;
  int n_layers, batch, capacity;
  const int32_t* block_table;
  int page_size, n_pages;
  int kv_dtype;
  const float* kv_scales;
} dflash_kv_cache;

/*
 * Fills a RoPE table: table[p][i] = (cos(p w_i), sin(p w_i)) as float2,
 * w_i = theta^(-2 i / d_h), for p < max_pos and i < d_h / 2. Angles and
 * cosines are evaluated in double precision on the device.
 * (DFlash KV Injection Walkthrough, Step 4.3: cos/sin over the whole window;
 * Interview Cheat Sheet, section 6.3: the inverse-frequency formula.)
 *   table  device float [max_pos][d_h/2][2], 8-byte aligned
 */
dflash_status dflash_rope_table_build(double theta, int d_h, int max_pos, float* table,
                                      cudaStream_t stream);

/*
 * Bytes of scratch memory the calls below need for a cache of `batch`
 * sequences and `capacity` rows and for at most `max_rows` context rows per
 * ctx_project / kv_inject call. Pass at least this much as `workspace`.
 */
size_t dflash_workspace_bytes(const dflash_dims* dims, int batch, int capacity, int max_rows);

/*
 * Context signal C = RMSNorm_{gamma_h}(concat[hidden[0] .. hidden[k-1]] W_fc^T).
 * (DFlash KV Injection Walkthrough, Step 1: extract_context_feature, layers
 * concatenated on the feature axis in ascending order; Step 2: fc without
 * bias, then hidden_norm.) The concatenation is never formed: each hidden[j]
 * is read as the j-th K-segment of the projection. hidden_norm runs as a pass
 * over the projection's fp32 split partials (bf16 with DFLASH_FUSED_NORM=1 in
 * the environment: in the projection's epilogue instead, the tiles of a row
 * block exchanging their rows' sums of squares through the workspace, when all
 * the projection's CTAs fit on the GPU at once; slower at the measured shapes).
 *   hidden     host array of k_layers device pointers, each [M][d]
 *   M          rows (>= 0; 0 is a no-op)
 *   W_fc       device [d][k_layers * d]
 *   gamma_h    device [d]
 *   C_out      device [M][d]
 *   workspace  device scratch of ws_bytes bytes, 256-byte aligned
 */
dflash_status dflash_ctx_project(const dflash_dims* dims, const void* const* hidden, int M,
                                 const void* W_fc, const void* gamma_h, void* C_out,
                                 void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * dflash_ctx_project for callers that cannot allocate device memory: the
 * source pages have no counterpart to this call; it exists for code that runs
 * inside another runtime's launch path (a custom operator's enqueue in an
 * inference server, for example), where that runtime owns all device memory
 * and a cudaMalloc would break its accounting and stall the device. Same
 * arguments and results as dflash_ctx_project, minus the workspace: the
 * scratch is a fixed array of DFLASH_NOALLOC_SCRATCH_BYTES inside the library,
 * held on every GPU that loads it until the process exits.
 *  - No allocation of any kind happens in this call.
 *  - Size rule: the fc splits K over several CTAs, each split with its own
 *    M x d fp32 partial, as many as dflash_ctx_project uses (the array is sized
 *    so that at d = 4096 it always holds them, and the two calls give the same
 *    bits); where they would not fit, this call uses fewer splits, down to one.
 *    So a call fits exactly when its one-split scratch fits: M * d * 4 bytes of
 *    partial, M * (d / 256) * 4 bytes of per-tile row sums (bf16) and under 2 KB
 *    of counters, within 20 MiB: up to 1274 rows at d = 4096, and every smaller
 *    M. A larger call returns DFLASH_ERR_WORKSPACE and launches nothing.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps whatever the
 *    previous call left in it; the counters that must start at zero are
 *    cleared by each call on its own stream. Calls that can run at the same
 *    time on the GPU (other streams, other host threads) race on it:
 *    serialise them.
 */
#define DFLASH_NOALLOC_SCRATCH_BYTES ((size_t)20 << 20)
dflash_status dflash_ctx_project_noalloc(const dflash_dims* dims, const void* const* hidden, int M,
                                         const void* W_fc, const void* gamma_h, void* C_out,
                                         cudaStream_t stream);

/*
 * Injects context rows into one layer of the draft cache: for sequence b,
 * rows cu_rows[b] .. cu_rows[b+1]-1 of C give K = RoPE(KNorm(C W_K^T)) and
 * V = C W_V^T, written at slots lens[layer][b] .. lens[layer][b] + n_b - 1
 * (their absolute positions), then lens[layer][b] += n_b.
 * (DFlash KV Injection Walkthrough, Step 4.2: the same k_proj / v_proj serve
 * context and block, KNorm per head, V not normalised; Step 4.3: keys rotated
 * at their true positions; Step 7: accepted rows join the cache as new context.)
 *   C          device [M][d]
 *   cu_rows    device int32 [batch + 1], non-decreasing, cu_rows[0] = 0, cu_rows[batch] = M
 *   W_K, W_V   device [n_kv * d_h][d]
 *   gamma_k    device [d_h], shared by all heads
 *   rope_table device table of dflash_rope_table_build, table_len positions
 * Device errors: capacity or table overflow of a sequence -> status bit, that
 * sequence is skipped and its length unchanged.
 */
dflash_status dflash_kv_inject(const dflash_dims* dims, const dflash_kv_cache* cache, int layer,
                               const void* C, const int32_t* cu_rows, int M, const void* W_K,
                               const void* W_V, const void* gamma_k, const float* rope_table,
                               int table_len, void* workspace, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * Block attention of one draft layer. For every sequence b, with start =
 * lens[layer][b]: the block occupies positions start .. start + bs - 1;
 * Q = RoPE(QNorm(H_b W_Q^T)), Kb = RoPE(KNorm(H_b W_K^T)), Vb = H_b W_V^T at
 * those positions; Kb, Vb are appended to the cache (lens += bs, the
 * reference's update(); the caller crops them away after verification); then
 * out_b = softmax(Q K^T * scaling) V over every cached row 0 .. start + bs - 1,
 * non-causal, query head h reading KV head h / G.
 * (DFlash KV Injection Walkthrough, Steps 4.1-4.4; DFlash source guide (II),
 * non-causal design note: is_causal False, no mask; part 5: sliding window.)
 *   H              device [batch][bs][d]
 *   W_Q            device [n_h * d_h][d];  W_K, W_V device [n_kv * d_h][d]
 *   gamma_q, gamma_k device [d_h]
 *   sliding_window 0 = full attention; W > 0: key j is visible to the query
 *                  at position p iff p - j < W (requires W >= bs)
 *   scaling        <= 0 selects d_h^-0.5
 *   out            device [batch][bs][n_h * d_h] (heads concatenated, the
 *                  layout o_proj consumes, walkthrough Step 4.5)
 * Device errors: as dflash_kv_inject; a skipped sequence's out rows are zero.
 */
dflash_status dflash_block_attn(const dflash_dims* dims, const dflash_kv_cache* cache, int layer,
                                const void* H, const void* W_Q, const void* W_K, const void* W_V,
                                const void* gamma_q, const void* gamma_k, const float* rope_table,
                                int table_len, int sliding_window, float scaling, void* out,
                                void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * One draft layer in a single call: dflash_kv_inject of the context rows C
 * followed by dflash_block_attn of the block H, with the same arguments and the
 * same results, lengths and device errors as those two calls in that order (the
 * block of sequence b starts after the rows the inject appended for it). This is
 * the layer's single forward over concat[context; block] of the source guide
 * (part 2: K/V from the concatenation, Q from the block only; walkthrough Step
 * 4.2). With bf16 and shapes whose two projections fill the GPU without split-K,
 * both projections (context K/V and block Q/K/V, with their norm / RoPE / store
 * epilogues) and the attention work list run in one launch, followed by the
 * attention and its combine. With bf16, d_h = 128 and fewer rows (a few
 * sequences, M and batch * bs within one 128-row tile), both projections and the
 * work list run as one split-K launch, then one epilogue launch finishes both,
 * then the attention and its combine. Otherwise it issues the two calls.
 * DFLASH_FUSED_LAYER in the environment picks: 0 the two calls, 1 the first
 * form wherever the shapes allow it, 2 the split-K form wherever it applies.
 *   arguments      as dflash_kv_inject (C, cu_rows, M) and dflash_block_attn
 *   workspace      dflash_workspace_bytes(dims, batch, capacity, max(M, ...))
 */
dflash_status dflash_draft_layer(const dflash_dims* dims, const dflash_kv_cache* cache, int layer,
                                 const void* C, const int32_t* cu_rows, int M, const void* H,
                                 const void* W_Q, const void* W_K, const void* W_V,
                                 const void* gamma_q, const void* gamma_k, const float* rope_table,
                                 int table_len, int sliding_window, float scaling, void* out,
                                 void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * The rest of a draft decoder layer after its attention, for M rows (the blocks' rows):
 *   x1  = x + attn_out W_O^T                         (Walkthrough Step 4.5: the heads,
 *                                                     concatenated, times W_O)
 *   out = x1 + W_down( silu(n W_gate^T) * (n W_up^T) ),  n = RMSNorm_post(x1)
 * Step 5 of the walkthrough names the draft's decoder layers and the final norm but does
 * not print them; the residual blocks and the SwiGLU MLP follow the Qwen3 decoder layer
 * that the source guide's Qwen3DFlashAttention and Qwen3RMSNorm belong to.
 *   attn_out    device [M][n_h * d_h] (dflash_block_attn's out)
 *   x, x_out    device [M][d] residual stream in / out (x_out may be x)
 *   W_O         device [d][n_h * d_h];  gamma_post device [d]
 *   W_gate, W_up device [d_ff][d];      W_down     device [d][d_ff]
 *   d_ff        > 0, a multiple of 4 (bf16: of 64); d a multiple of 4, at most 8192
 *   workspace   dflash_layer_out_workspace_bytes(dims, M, d_ff) bytes, 256-byte aligned
 * All pointers 16-byte aligned. Host errors as the other calls.
 */
size_t dflash_layer_out_workspace_bytes(const dflash_dims* dims, int M, int d_ff);
dflash_status dflash_layer_out(const dflash_dims* dims, int M, const void* attn_out, const void* x,
                               const void* W_O, const void* gamma_post, int d_ff,
                               const void* W_gate, const void* W_up, const void* W_down,
                               void* x_out, void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * out = RMSNorm(x) * gamma over rows of width d (eps of dims): the layers' input norm and
 * the final norm after the last draft layer (Walkthrough Step 5).
 *   x, out  device [M][d], gamma device [d]; 16-byte aligned; d a multiple of 4, <= 8192
 */
dflash_status dflash_rms_norm(const dflash_dims* dims, int M, const void* x, const void* gamma,
                              void* out, cudaStream_t stream);

/*
 * crop(start) on every layer: lens[l][b] = new_lens[b] for all l. No cache
 * data moves. (DFlash source guide (II), part 4; DFlash KV Injection
 * Walkthrough, Step 7.) A target that is negative or above a layer's current
 * length sets DFLASH_DEV_CROP and leaves that layer's length unchanged.
 *   new_lens  device int32 [batch]
 */
dflash_status dflash_cache_crop(const dflash_kv_cache* cache, const int32_t* new_lens,
                                cudaStream_t stream);

/*
 * Acceptance bookkeeping of a verified round, on the device, for every sequence b
 * (DFlash KV Injection Walkthrough, Step 6: a = the number of leading i < bs - 1 with
 * block_ids[b][i + 1] == posterior[b][i], i.e. cumprod then sum of the matches; Step 7:
 * start += a + 1, the next round's context rows are the anchor's and the accepted
 * tokens', and the target's token after the accepted prefix is the next anchor):
 *   accept_len[b]   = a
 *   next_cu_rows    = [0, a_0 + 1, a_0 + a_1 + 2, ...]: cu_rows of the next round's inject
 *   ctx_next[b]     = ctx_len[b] + a + 1: the next block's first position, which is also
 *                     the next round's crop target (ctx_len[b] is this round's)
 *   next_anchor[b]  = posterior[b][a]
 * The draft cache itself is cropped with dflash_cache_crop(ctx_len). Nothing is read back
 * to the host.
 *   block_ids, posterior  device int32 [batch][bs], bs >= 1
 *   ctx_len               device int32 [batch]
 *   accept_len, ctx_next, next_anchor  device int32 [batch]; next_cu_rows [batch + 1]
 * Host errors: batch < 0, bs < 1, null or misaligned pointers (no launch).
 */
dflash_status dflash_accept(const int32_t* block_ids, const int32_t* posterior, int batch, int bs,
                            const int32_t* ctx_len, int32_t* accept_len, int32_t* next_cu_rows,
                            int32_t* ctx_next, int32_t* next_anchor, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's sticky
 * status word into *device_status (a mask of DFLASH_DEV_* bits). Returns
 * DFLASH_OK when the word was zero, DFLASH_ERR_DEVICE when not, and
 * DFLASH_ERR_CUDA if the synchronisation itself failed.
 */
dflash_status dflash_status_get(unsigned int* device_status, cudaStream_t stream);

/* Human-readable name of a dflash_status value (static string). */
const char* dflash_status_string(dflash_status s);

/*
 * Kernel tracing (no counterpart on the pages: a measurement aid).
 * Kernel kinds the library launches, as bit positions of a trace mask:
 */
#define DFLASH_KERNEL_GEMM          1  /* projection GEMM (fc, K/V, Q/K/V) */
#define DFLASH_KERNEL_RMSNORM       2  /* hidden_norm of the context signal */
#define DFLASH_KERNEL_HEAD_EPILOGUE 3  /* per-head norm, RoPE, cache scatter */
#define DFLASH_KERNEL_ATTENTION     4  /* block attention over the cache */
#define DFLASH_KERNEL_COMBINE       5  /* merge of the attention chunks */
#define DFLASH_KERNEL_LENS          6  /* cache length update */
#define DFLASH_KERNEL_CROP          7  /* crop */
#define DFLASH_KERNEL_ROPE_TABLE    8  /* RoPE table fill */
#define DFLASH_KERNEL_SCHEDULE      9  /* attention work list */
#define DFLASH_KERNEL_ACCEPT       10  /* acceptance bookkeeping */

/*
 * Starts recording a CUDA event pair around every launch whose kind bit
 * (1u << kind) is set in kernel_mask, on the launch's own stream, for at most
 * max_launches launches (later ones are not recorded). Inside a stream capture
 * the pairs become timestamped event nodes of the graph, read after a replay.
 * Each call creates fresh events (kept for the process, since a captured graph
 * may still refer to them). Recording adds a few microseconds per event to
 * the stream, so time a step without tracing when the total matters.
 */
dflash_status dflash_trace_start(unsigned int kernel_mask, int max_launches);

/*
 * Stops recording, waits for the recorded events and writes, for each recorded
 * launch i < *count, its kind into kinds[i] and its duration in milliseconds
 * into ms[i] (at most `capacity` entries; *count is the number recorded).
 */
dflash_status dflash_trace_stop(int* kinds, float* ms, int capacity, int* count);

/* Number of kernels the library has launched in this process so far. */
unsigned long long dflash_launch_count(void);

/*
 * Test aid (no counterpart in the source pages): sets the time limit, in ns, of the
 * pipeline waits of the tensor-core kernels (the waits of one role of a kernel for
 * another's data, and the context projection's waits for the other tiles of a row
 * block) in every launch made after the call, in this process; 0 restores the default
 * of 2 s. A wait that runs out sets DFLASH_DEV_TIMEOUT and makes its kernel stop: the
 * waits that let in-flight copies and MMAs finish before the kernel exits keep their
 * 2 s limit, so a kernel that gives up still frees its tensor memory and returns, and
 * later launches work. Not for production use: a short limit turns ordinary latency
 * into errors.
 */
void dflash_test_wait_limit(unsigned long long ns);

/*
 * Test aid (no counterpart in the source pages): builds on the device the work list the
 * tensor-core attention (bf16 dims) would use for layer `layer` of cache `c` — its current
 * lengths, plus the rows a KV inject of the same call appends (cu_rows [batch + 1] and M,
 * as for dflash_draft_layer; null and 0 for none), and a sliding window (0 = none) — in
 * `workspace` (dflash_workspace_bytes), then copies it to host memory `out` (int32):
 *   [0] n_ctas  [1] max_splits  [2] item_cost  [3] n_items  [4] n_merge
 *   first[n_ctas + 1]                 CTA i takes list items first[i] .. first[i + 1] - 1
 *   items[n_ctas + n_items][4]        {pair, k_begin, k_end, split (-1 = whole range)}: each
 *                                     CTA's first item, then the list
 *   splits[batch * n_kv]              items per pair (0: a refused sequence)
 *   merge_list[n_merge]               pair | items << 20, the pairs the combine writes
 * *n_out receives the number of ints written (or needed: DFLASH_ERR_INVALID_ARG when
 * out_ints is smaller; `out` may be null with out_ints 0 to ask for the size). Synchronises
 * `stream`; the cache is not modified.
 */
dflash_status dflash_test_attn_worklist(const dflash_dims* dims, const dflash_kv_cache* cache,
                                        int layer, const int32_t* cu_rows, int M, int window,
                                        void* workspace, size_t workspace_bytes, int32_t* out,
                                        size_t out_ints, size_t* n_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
