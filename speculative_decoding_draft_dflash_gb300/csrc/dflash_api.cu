// The C ABI: argument checks, scratch carving and kernel launches.
//
// Every entry point validates what the host can see, carves its scratch out
// of the caller's workspace and enqueues kernels on the caller's stream. No
// entry point allocates, frees or synchronises (dflash_status_get excepted).
#include <mutex>

#include "attn_sched.cuh"

#include <atomic>

namespace dflash {

__device__ unsigned int g_status_word;

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{0};  // 0: the default, 2 s
}  // namespace

unsigned long long wait_limit_ns() {
  const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : 2000000000ull;
}

unsigned* status_word() {
  static std::mutex mu;
  static unsigned* ptr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptr[dev] = (unsigned*)p;
  }
  return ptr[dev];
}

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

dflash_status check_dims(const dflash_dims* d) {
  if (!d) return DFLASH_ERR_INVALID_ARG;
  if (d->d <= 0 || d->n_h <= 0 || d->n_kv <= 0 || d->d_h <= 0 || d->k_layers <= 0 ||
      d->block_size <= 0 || !(d->eps >= 0.f))
    return DFLASH_ERR_INVALID_ARG;
  if (d->dtype != DFLASH_F32 && d->dtype != DFLASH_BF16) return DFLASH_ERR_UNSUPPORTED;
  if (d->k_layers > 8 || d->n_h % d->n_kv != 0 || d->d % 8 != 0 || d->d_h % 2 != 0)
    return DFLASH_ERR_UNSUPPORTED;
  if (d->block_size > 16) return DFLASH_ERR_UNSUPPORTED;
  if (d->dtype == DFLASH_F32) {
    if (d->d_h > 256) return DFLASH_ERR_UNSUPPORTED;
  } else {
    if (d->d_h != 128 || d->d % 64 != 0 || (d->n_h / d->n_kv) * d->block_size > 128)
      return DFLASH_ERR_UNSUPPORTED;
  }
  return DFLASH_OK;
}

dflash_status check_cache(const dflash_kv_cache* c, int layer) {
  if (!c || !c->k || !c->v || !c->lens) return DFLASH_ERR_INVALID_ARG;
  if (c->n_layers <= 0 || c->batch <= 0 || c->capacity <= 0) return DFLASH_ERR_INVALID_ARG;
  if (layer < 0 || layer >= c->n_layers) return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(c->k) || !aligned16(c->v) || ((uintptr_t)c->lens & 3)) return DFLASH_ERR_INVALID_ARG;
  if (c->block_table) {  // paged: 128-row pages (one attention tile each)
    if (c->page_size != 128 || c->capacity % 128 || c->n_pages <= 0 ||
        ((uintptr_t)c->block_table & 3))
      return DFLASH_ERR_INVALID_ARG;
  }
  if (c->kv_dtype == DFLASH_FP8_E4M3 && c->kv_scales) {
    for (int i = 0; i < 2 * c->n_layers; ++i)
      if (!(c->kv_scales[i] > 0.f) || !(c->kv_scales[i] < INFINITY)) return DFLASH_ERR_INVALID_ARG;
  }
  return DFLASH_OK;
}

bool kv_fp8(const dflash_kv_cache* c) { return c->kv_dtype == DFLASH_FP8_E4M3; }

// The paged layout and the fp8 cache are served by the bf16 tensor-core path only;
// the cache element type is the dims' one or E4M3.
dflash_status check_layout(const dflash_dims* d, const dflash_kv_cache* c) {
  if (c->kv_dtype != 0 && c->kv_dtype != d->dtype && c->kv_dtype != DFLASH_FP8_E4M3)
    return DFLASH_ERR_UNSUPPORTED;
  if ((c->block_table || kv_fp8(c)) && d->dtype != DFLASH_BF16) return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}

size_t esize(const dflash_dims* d) { return d->dtype == DFLASH_F32 ? 4 : 2; }

// bytes of one cache element
size_t kv_esize(const dflash_dims* d, const dflash_kv_cache* c) { return kv_fp8(c) ? 1 : esize(d); }

float kv_scale(const dflash_kv_cache* c, int layer, int which) {
  return kv_fp8(c) && c->kv_scales ? c->kv_scales[2 * layer + which] : 1.f;
}

// Fills the fp8 fields of a per-head epilogue: quantisation by the inverse scales, and
// Q as codes + remainder codes (the remainder array follows the codes in q_out).
void fp8_epilogue(HeadEpilogue& ep, const dflash_dims* d, const dflash_kv_cache* c, int layer) {
  ep.kv_fp8 = kv_fp8(c);
  if (!ep.kv_fp8) return;
  ep.k_inv = 1.f / kv_scale(c, layer, 0);
  ep.v_inv = 1.f / kv_scale(c, layer, 1);
  if (ep.q_out)
    ep.q_lo = (char*)ep.q_out + (size_t)c->batch * d->n_h * d->block_size * d->d_h;
}

dflash_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA; }

// Attention chunking for a cache of `capacity` rows and an optional window.
void attn_chunks(const dflash_dims* d, int capacity, int window, int* chunk, int* n_chunks) {
  int range = capacity;
  if (window > 0 && window + d->block_size - 1 < range) range = window + d->block_size - 1;
  *chunk = attn_chunk(d->dtype);
  *n_chunks = (range + *chunk - 1) / *chunk;
  if (*n_chunks < 1) *n_chunks = 1;
}

// Shapes of the stacked weights of each projection (pointers filled by the caller).
Weights ctx_weights(const dflash_dims* d, const void* W_fc) {
  Weights W;
  W.count = 1;
  W.p[0] = W_fc;
  W.n[0] = d->d;
  return W;
}
Weights kv_weights(const dflash_dims* d, const void* W_K, const void* W_V) {
  Weights W;
  W.count = 2;
  W.p[0] = W_K;
  W.p[1] = W_V;
  W.n[0] = W.n[1] = d->n_kv * d->d_h;
  return W;
}
Weights qkv_weights(const dflash_dims* d, const void* W_Q, const void* W_K, const void* W_V) {
  Weights W;
  W.count = 3;
  W.p[0] = W_Q;
  W.p[1] = W_K;
  W.p[2] = W_V;
  W.n[0] = d->n_h * d->d_h;
  W.n[1] = W.n[2] = d->n_kv * d->d_h;
  return W;
}

// Scratch of each call, carved in a fixed order (base == nullptr only sizes it).
struct CtxScratch { float* Y; int splits; float* rowpart; int* counters; };
struct InjectScratch { float* Y; int splits; };
struct BlockScratch { float* Y; int splits; void* q; float* part_acc; float2* part_ml; void* sched; };

CtxScratch carve_ctx(Carver& cv, const dflash_dims* d, int M, int split_cap = 0) {
  CtxScratch s;
  const Weights W = ctx_weights(d, nullptr);
  const int K = d->k_layers * d->d;
  s.splits = gemm_splits(d->dtype, M, W, K, split_cap);
  s.Y = cv.take<float>((size_t)s.splits * M * d->d);
  s.rowpart = nullptr;
  s.counters = nullptr;
  if (d->dtype == DFLASH_BF16) {  // the fused hidden_norm's per-tile row sums and counters
    s.rowpart = cv.take<float>((size_t)M * gemm_tc_norm_tiles_n(M, W, K));
    s.counters = cv.take<int>((size_t)gemm_tc_norm_counters(M, W, K, split_cap));
  }
  return s;
}

InjectScratch carve_inject(Carver& cv, const dflash_dims* d, int M) {
  InjectScratch s;
  const int N = 2 * d->n_kv * d->d_h;
  const Weights W = kv_weights(d, nullptr, nullptr);
  s.splits = gemm_splits(d->dtype, M, W, d->d);
  const bool fused = d->dtype == DFLASH_BF16 && gemm_tc_heads_ok(M, W, d->d);
  s.Y = fused ? nullptr : cv.take<float>((size_t)s.splits * M * N);
  return s;
}

BlockScratch carve_block(Carver& cv, const dflash_dims* d, int batch, int capacity, int window) {
  BlockScratch s;
  const int rows = batch * d->block_size;
  const int N = (d->n_h + 2 * d->n_kv) * d->d_h;
  int chunk, n_chunks;
  attn_chunks(d, capacity, window, &chunk, &n_chunks);
  const Weights W = qkv_weights(d, nullptr, nullptr, nullptr);
  s.splits = gemm_splits(d->dtype, rows, W, d->d);
  const bool fused = d->dtype == DFLASH_BF16 && gemm_tc_heads_ok(rows, W, d->d);
  s.Y = fused ? nullptr : cv.take<float>((size_t)s.splits * rows * N);
  s.q = cv.take<char>((size_t)batch * d->n_h * d->block_size * d->d_h * esize(d));
  const size_t part_rows = (size_t)batch * d->n_h * n_chunks * d->block_size;
  s.part_acc = cv.take<float>(part_rows * d->d_h);
  s.part_ml = cv.take<float2>(part_rows);
  // the attention's work list: items {pair, k_begin, k_end, split}, each CTA's range of
  // them, split count per pair, counters, per sequence the block start and the length
  // after the call, the pairs to combine
  s.sched = cv.take<char>(attn_sched_bytes(batch, d->n_kv));
  return s;
}

// A draft layer's two projections as one split-K launch (bf16, few sequences): the block's
// scratch, then fp32 partials of the context K/V (up to the launch's row tiles) and of the
// block Q/K/V (the block's own partials when they are large enough). splits = 0: the
// launch does not apply to this batch.
struct LayerSplitScratch { BlockScratch b; float* Y0; float* Y1; int splits; };

LayerSplitScratch carve_layer_split(Carver& cv, const dflash_dims* d, int batch, int capacity,
                                    int window, int M) {
  LayerSplitScratch s;
  s.b = carve_block(cv, d, batch, capacity, window);
  s.Y0 = s.Y1 = nullptr;
  s.splits = 0;
  if (d->dtype != DFLASH_BF16 || d->d_h != 128) return s;
  const int rows = batch * d->block_size;
  const Weights Wkv = kv_weights(d, nullptr, nullptr), Wqkv = qkv_weights(d, nullptr, nullptr, nullptr);
  s.splits = gemm_tc_layer_split_splits(rows, Wkv, Wqkv, d->d);
  if (s.splits == 0) return s;
  const int cap = gemm_tc_layer_split_rows(rows, Wkv, Wqkv, d->d);
  const int mc = M < cap ? M : cap;
  s.Y0 = cv.take<float>((size_t)s.splits * mc * Wkv.total());
  s.Y1 = s.b.Y && s.b.splits >= s.splits ? s.b.Y
                                         : cv.take<float>((size_t)s.splits * rows * Wqkv.total());
  return s;
}

// Projection + per-head epilogue: fused into the tcgen05 GEMM when no split-K
// is needed, else fp32 partials (ep.Y) and a separate epilogue kernel.
cudaError_t project_heads(const dflash_dims* d, const Segments& A, int M, const Weights& W,
                          const HeadEpilogue& ep, unsigned* status, cudaStream_t stream) {
  if (d->dtype == DFLASH_BF16 && gemm_tc_heads_ok(M, W, d->d))
    return gemm_tc_heads(A, M, W, ep, status, stream);
  cudaError_t e = gemm(d->dtype, A, M, W, const_cast<float*>(ep.Y), ep.ldY, status, stream);
  if (e != cudaSuccess) return e;
  return d->dtype == DFLASH_F32 ? head_epilogue(d->dtype, ep, stream) : head_epilogue_bf16(ep, stream);
}

}  // namespace
}  // namespace dflash

using namespace dflash;

DFLASH_API void dflash_test_wait_limit(unsigned long long ns) {
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
}

DFLASH_API const char* dflash_status_string(dflash_status s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported dimensions";
    case DFLASH_ERR_WORKSPACE: return "workspace too small";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_DEVICE: return "device status word set";
  }
  return "unknown status";
}

DFLASH_API size_t dflash_workspace_bytes(const dflash_dims* d, int batch, int capacity,
                                         int max_rows) {
  if (check_dims(d) != DFLASH_OK || batch < 0 || capacity < 0 || max_rows < 0) return 0;
  size_t need = 256;
  // every row count up to max_rows: the projections' K-split counts change with the
  // 128-row tiles M spans (fewer rows can mean more splits, each with its own partials),
  // and within one tile count the scratch grows with M, so the top of each tile count's
  // range bounds it; once both projections run unsplit, more rows only need more
  const Weights Wc = ctx_weights(d, nullptr), Wkv = kv_weights(d, nullptr, nullptr);
  for (long long m = 128; ; m += 128) {
    if (m < max_rows && gemm_splits(d->dtype, (int)m, Wc, d->k_layers * d->d) == 1 &&
        gemm_splits(d->dtype, (int)m, Wkv, d->d) == 1)
      m = max_rows;
    const int rows = m < max_rows ? (int)m : max_rows;
    {
      Carver cv(nullptr, ~size_t(0));
      carve_ctx(cv, d, rows);
      need = need > cv.off ? need : cv.off;
    }
    {
      Carver cv(nullptr, ~size_t(0));
      carve_inject(cv, d, rows);
      need = need > cv.off ? need : cv.off;
    }
    if (m >= max_rows) break;
  }
  {
    Carver cv(nullptr, ~size_t(0));
    carve_block(cv, d, batch, capacity, 0);
    need = need > cv.off ? need : cv.off;
  }
  {
    Carver cv(nullptr, ~size_t(0));
    carve_layer_split(cv, d, batch, capacity, 0, max_rows);
    need = need > cv.off ? need : cv.off;
  }
  return need;
}

DFLASH_API dflash_status dflash_rope_table_build(double theta, int d_h, int max_pos, float* table,
                                                 cudaStream_t stream) {
  if (!table || d_h <= 0 || d_h % 2 != 0 || max_pos < 0 || !(theta > 0.0) ||
      ((uintptr_t)table & 7))
    return DFLASH_ERR_INVALID_ARG;
  if (max_pos == 0) return DFLASH_OK;
  return cuda_status(rope_table(theta, d_h, max_pos, table, stream));
}

namespace dflash {

// The context projection with its scratch carved from `workspace`; split_cap > 0 bounds
// the fc's K-splits (so the scratch need shrinks with it).
dflash_status ctx_project_impl(const dflash_dims* d, const void* const* hidden, int M,
                               const void* W_fc, const void* gamma_h, void* C_out, void* workspace,
                               size_t ws_bytes, int split_cap, cudaStream_t stream) {
  dflash_status st = check_dims(d);
  if (st != DFLASH_OK) return st;
  if (M < 0) return DFLASH_ERR_INVALID_ARG;
  if (M == 0) return DFLASH_OK;
  if (!hidden || !W_fc || !gamma_h || !C_out || !workspace) return DFLASH_ERR_INVALID_ARG;
  Segments A;
  A.n = d->k_layers;
  A.kseg = d->d;
  for (int j = 0; j < d->k_layers; ++j) {
    if (!hidden[j] || !aligned16(hidden[j])) return DFLASH_ERR_INVALID_ARG;
    A.p[j] = hidden[j];
  }
  if (!aligned16(W_fc) || !aligned16(C_out) || ((uintptr_t)workspace & 255))
    return DFLASH_ERR_INVALID_ARG;
  Carver cv(workspace, ws_bytes);
  CtxScratch s = carve_ctx(cv, d, M, split_cap);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  const Weights W = ctx_weights(d, W_fc);
  const int K = d->k_layers * d->d;
  if (d->dtype == DFLASH_BF16 && gemm_tc_norm_ok(M, W, K, split_cap))
    return cuda_status(gemm_tc_norm(A, M, W, s.Y, s.rowpart, s.counters, gamma_h, d->eps, C_out,
                                    status, stream, split_cap));
  cudaError_t e = gemm(d->dtype, A, M, W, s.Y, d->d, status, stream, split_cap);
  if (e == cudaSuccess)
    e = rmsnorm_rows(d->dtype, s.Y, s.splits, M, d->d, gamma_h, d->eps, C_out, stream);
  return cuda_status(e);
}

// Scratch bytes of a context projection of M rows with at most split_cap K-splits (0: the
// planner's choice), or 0 for dims the library does not support.
size_t ctx_scratch_bytes(const dflash_dims* d, int M, int split_cap) {
  if (check_dims(d) != DFLASH_OK || M < 0) return 0;
  Carver cv(nullptr, ~size_t(0));
  carve_ctx(cv, d, M, split_cap);
  return cv.off;
}

// K-splits the planner gives a context projection of M rows (1 for the f32 path).
int ctx_splits(const dflash_dims* d, int M) {
  return gemm_splits(d->dtype, M, ctx_weights(d, nullptr), d->k_layers * d->d);
}

}  // namespace dflash

DFLASH_API dflash_status dflash_ctx_project(const dflash_dims* d, const void* const* hidden, int M,
                                            const void* W_fc, const void* gamma_h, void* C_out,
                                            void* workspace, size_t ws_bytes,
                                            cudaStream_t stream) {
  return ctx_project_impl(d, hidden, M, W_fc, gamma_h, C_out, workspace, ws_bytes, 0, stream);
}

namespace {

// elements of one layer's K (or V): [batch][n_kv][capacity][d_h], or a pool of
// [n_pages][n_kv][128][d_h] when paged
size_t layer_elems(const dflash_dims* d, const dflash_kv_cache* c) {
  if (c->block_table) return (size_t)c->n_pages * d->n_kv * 128 * d->d_h;
  return (size_t)c->batch * d->n_kv * c->capacity * d->d_h;
}

// Per-head epilogue of an inject: context rows (grouped by cu_rows) -> K-norm, RoPE at
// lens[b] + t, cache rows; V rows unchanged.
HeadEpilogue inject_epilogue(const dflash_dims* d, const dflash_kv_cache* c, int layer,
                             const int32_t* cu_rows, int M, const void* gamma_k, const float* rope,
                             int table_len, float* Y, int splits, unsigned* status) {
  HeadEpilogue ep;
  ep.Y = Y;
  ep.splits = splits;
  ep.rows = M;
  ep.ldY = 2 * d->n_kv * d->d_h;
  ep.n_q = 0;
  ep.n_kv = d->n_kv;
  ep.d_h = d->d_h;
  ep.eps = d->eps;
  ep.gamma_q = nullptr;
  ep.gamma_k = gamma_k;
  ep.rope = (const float2*)rope;
  ep.table_len = table_len;
  ep.cu_rows = cu_rows;
  ep.batch = c->batch;
  ep.bs = 0;
  ep.lens = c->lens + (size_t)layer * c->batch;
  ep.q_out = nullptr;
  ep.cache_k = (char*)c->k + (size_t)layer * layer_elems(d, c) * kv_esize(d, c);
  ep.cache_v = (char*)c->v + (size_t)layer * layer_elems(d, c) * kv_esize(d, c);
  ep.capacity = c->capacity;
  ep.status = status;
  ep.block_table = c->block_table;
  ep.pages_per_seq = c->block_table ? c->capacity / 128 : 0;
  fp8_epilogue(ep, d, c, layer);
  return ep;
}

// Per-head epilogue of a block: Q and K norms, RoPE at the block positions, Q to q_out,
// K/V to the block's cache rows.
HeadEpilogue block_epilogue(const dflash_dims* d, const dflash_kv_cache* c, int layer,
                            const void* gamma_q, const void* gamma_k, const float* rope,
                            int table_len, void* q_out, float* Y, int splits, unsigned* status) {
  HeadEpilogue ep;
  ep.Y = Y;
  ep.splits = splits;
  ep.rows = c->batch * d->block_size;
  ep.ldY = (d->n_h + 2 * d->n_kv) * d->d_h;
  ep.n_q = d->n_h;
  ep.n_kv = d->n_kv;
  ep.d_h = d->d_h;
  ep.eps = d->eps;
  ep.gamma_q = gamma_q;
  ep.gamma_k = gamma_k;
  ep.rope = (const float2*)rope;
  ep.table_len = table_len;
  ep.cu_rows = nullptr;
  ep.batch = c->batch;
  ep.bs = d->block_size;
  ep.lens = c->lens + (size_t)layer * c->batch;
  ep.q_out = q_out;
  ep.cache_k = (char*)c->k + (size_t)layer * layer_elems(d, c) * kv_esize(d, c);
  ep.cache_v = (char*)c->v + (size_t)layer * layer_elems(d, c) * kv_esize(d, c);
  ep.capacity = c->capacity;
  ep.status = status;
  ep.block_table = c->block_table;
  ep.pages_per_seq = c->block_table ? c->capacity / 128 : 0;
  fp8_epilogue(ep, d, c, layer);
  return ep;
}

AttnParams block_attention(const dflash_dims* d, const dflash_kv_cache* c, int layer,
                           const BlockScratch& s, int window, float scaling, int table_len,
                           void* out, unsigned* status) {
  AttnParams p;
  p.q = s.q;
  p.cache_k = (char*)c->k + (size_t)layer * layer_elems(d, c) * kv_esize(d, c);
  p.cache_v = (char*)c->v + (size_t)layer * layer_elems(d, c) * kv_esize(d, c);
  p.lens = c->lens + (size_t)layer * c->batch;
  p.out = out;
  p.part_acc = s.part_acc;
  p.part_ml = s.part_ml;
  p.sched = s.sched;
  p.status = status;
  p.batch = c->batch;
  p.n_h = d->n_h;
  p.n_kv = d->n_kv;
  p.d_h = d->d_h;
  p.bs = d->block_size;
  p.capacity = c->capacity;
  p.window = window;
  attn_chunks(d, c->capacity, window, &p.chunk, &p.n_chunks);
  p.table_len = table_len;
  p.scaling = scaling > 0.f ? scaling : 1.0f / sqrtf((float)d->d_h);
  p.pre_rows = nullptr;
  p.pre_M = 0;
  p.lens_out = nullptr;
  p.sched_ready = false;
  p.block_table = c->block_table;
  p.pages_per_seq = c->block_table ? c->capacity / 128 : 0;
  p.n_pages = c->n_pages;
  p.fp8 = kv_fp8(c);
  p.k_scale = kv_scale(c, layer, 0);
  p.v_scale = kv_scale(c, layer, 1);
  return p;
}

dflash_status check_inject(const dflash_dims* d, const dflash_kv_cache* c, int layer, const void* C,
                           const int32_t* cu_rows, int M, const void* W_K, const void* W_V,
                           const void* gamma_k, const float* rope, int table_len,
                           const void* workspace) {
  dflash_status st = check_dims(d);
  if (st != DFLASH_OK) return st;
  st = check_cache(c, layer);
  if (st != DFLASH_OK) return st;
  st = check_layout(d, c);
  if (st != DFLASH_OK) return st;
  if (M < 0 || table_len < 0) return DFLASH_ERR_INVALID_ARG;
  if (M == 0) return DFLASH_OK;
  if (!C || !cu_rows || !W_K || !W_V || !gamma_k || !rope || !workspace) return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(C) || !aligned16(W_K) || !aligned16(W_V) || ((uintptr_t)workspace & 255) ||
      ((uintptr_t)rope & 7))
    return DFLASH_ERR_INVALID_ARG;
  return DFLASH_OK;
}

dflash_status check_block(const dflash_dims* d, const dflash_kv_cache* c, int layer, const void* H,
                          const void* W_Q, const void* W_K, const void* W_V, const void* gamma_q,
                          const void* gamma_k, const float* rope, int table_len, int window,
                          const void* out, const void* workspace) {
  dflash_status st = check_dims(d);
  if (st != DFLASH_OK) return st;
  st = check_cache(c, layer);
  if (st != DFLASH_OK) return st;
  st = check_layout(d, c);
  if (st != DFLASH_OK) return st;
  if (table_len < 0 || window < 0) return DFLASH_ERR_INVALID_ARG;
  if (window > 0 && window < d->block_size) return DFLASH_ERR_INVALID_ARG;
  if (!H || !W_Q || !W_K || !W_V || !gamma_q || !gamma_k || !rope || !out || !workspace)
    return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(H) || !aligned16(W_Q) || !aligned16(W_K) || !aligned16(W_V) || !aligned16(out) ||
      ((uintptr_t)workspace & 255) || ((uintptr_t)rope & 7))
    return DFLASH_ERR_INVALID_ARG;
  return DFLASH_OK;
}

Segments one_segment(const dflash_dims* d, const void* X) {
  Segments A;
  A.n = 1;
  A.kseg = d->d;
  A.p[0] = X;
  return A;
}

}  // namespace

DFLASH_API dflash_status dflash_kv_inject(const dflash_dims* d, const dflash_kv_cache* c, int layer,
                                          const void* C, const int32_t* cu_rows, int M,
                                          const void* W_K, const void* W_V, const void* gamma_k,
                                          const float* rope, int table_len, void* workspace,
                                          size_t ws_bytes, cudaStream_t stream) {
  dflash_status st = check_inject(d, c, layer, C, cu_rows, M, W_K, W_V, gamma_k, rope, table_len,
                                  workspace);
  if (st != DFLASH_OK || M == 0) return st;
  Carver cv(workspace, ws_bytes);
  InjectScratch s = carve_inject(cv, d, M);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  const HeadEpilogue ep = inject_epilogue(d, c, layer, cu_rows, M, gamma_k, rope, table_len, s.Y,
                                          s.splits, status);
  cudaError_t e = project_heads(d, one_segment(d, C), M, kv_weights(d, W_K, W_V), ep, status, stream);
  if (e == cudaSuccess)
    e = lens_advance(c->lens + (size_t)layer * c->batch, cu_rows, c->batch, 0, M, c->capacity,
                     table_len, stream);
  return cuda_status(e);
}

DFLASH_API dflash_status dflash_block_attn(const dflash_dims* d, const dflash_kv_cache* c,
                                           int layer, const void* H, const void* W_Q,
                                           const void* W_K, const void* W_V, const void* gamma_q,
                                           const void* gamma_k, const float* rope, int table_len,
                                           int window, float scaling, void* out, void* workspace,
                                           size_t ws_bytes, cudaStream_t stream) {
  dflash_status st = check_block(d, c, layer, H, W_Q, W_K, W_V, gamma_q, gamma_k, rope, table_len,
                                 window, out, workspace);
  if (st != DFLASH_OK) return st;
  Carver cv(workspace, ws_bytes);
  BlockScratch s = carve_block(cv, d, c->batch, c->capacity, window);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  const int rows = c->batch * d->block_size;
  const HeadEpilogue ep = block_epilogue(d, c, layer, gamma_q, gamma_k, rope, table_len, s.q, s.Y,
                                         s.splits, status);
  cudaError_t e = project_heads(d, one_segment(d, H), rows, qkv_weights(d, W_Q, W_K, W_V), ep,
                                status, stream);
  AttnParams p = block_attention(d, c, layer, s, window, scaling, table_len, out, status);
  // the tensor-core attention's combine kernel publishes the new lengths itself
  const bool tc_attn = d->dtype != DFLASH_F32;
  p.lens_out = tc_attn ? c->lens + (size_t)layer * c->batch : nullptr;
  if (e == cudaSuccess)
    e = attention(d->dtype, p, stream);
  if (e == cudaSuccess && !tc_attn)
    e = lens_advance(c->lens + (size_t)layer * c->batch, nullptr, c->batch, d->block_size, rows,
                     c->capacity, table_len, stream);
  return cuda_status(e);
}

DFLASH_API dflash_status dflash_draft_layer(const dflash_dims* d, const dflash_kv_cache* c,
                                            int layer, const void* C, const int32_t* cu_rows, int M,
                                            const void* H, const void* W_Q, const void* W_K,
                                            const void* W_V, const void* gamma_q,
                                            const void* gamma_k, const float* rope, int table_len,
                                            int window, float scaling, void* out, void* workspace,
                                            size_t ws_bytes, cudaStream_t stream) {
  dflash_status st = check_inject(d, c, layer, C, cu_rows, M, W_K, W_V, gamma_k, rope, table_len,
                                  workspace);
  if (st != DFLASH_OK) return st;
  st = check_block(d, c, layer, H, W_Q, W_K, W_V, gamma_q, gamma_k, rope, table_len, window, out,
                   workspace);
  if (st != DFLASH_OK) return st;
  const int rows = c->batch * d->block_size;
  const Weights Wkv = kv_weights(d, W_K, W_V), Wqkv = qkv_weights(d, W_Q, W_K, W_V);
  const bool grouped = d->dtype == DFLASH_BF16 && M > 0 && gemm_tc_layer_ok(M, Wkv, rows, Wqkv, d->d);
  // few sequences: both projections as one split-K launch, both epilogues as one launch
  const bool split = d->dtype == DFLASH_BF16 && M > 0 && !grouped && d->d_h == 128 &&
                     gemm_tc_layer_split_splits(rows, Wkv, Wqkv, d->d) > 0 &&
                     M <= gemm_tc_layer_split_rows(rows, Wkv, Wqkv, d->d);
  if (split) {
    Carver cv(workspace, ws_bytes);
    LayerSplitScratch s = carve_layer_split(cv, d, c->batch, c->capacity, window, M);
    if (!cv.ok) return DFLASH_ERR_WORKSPACE;
    unsigned* status = status_word();
    if (!status) return DFLASH_ERR_CUDA;
    const HeadEpilogue ep_kv = inject_epilogue(d, c, layer, cu_rows, M, gamma_k, rope, table_len,
                                               s.Y0, s.splits, status);
    HeadEpilogue ep_qkv = block_epilogue(d, c, layer, gamma_q, gamma_k, rope, table_len, s.b.q,
                                         s.Y1, s.splits, status);
    ep_qkv.pre_rows = cu_rows;  // the block follows the rows injected here
    ep_qkv.pre_M = M;
    AttnParams p = block_attention(d, c, layer, s.b, window, scaling, table_len, out, status);
    p.pre_rows = cu_rows;
    p.pre_M = M;
    p.lens_out = c->lens + (size_t)layer * c->batch;
    p.sched_ready = true;
    const sched::Params sp = attn_sched_params(p);
    cudaError_t e = gemm_tc_layer_split(C, M, Wkv, s.Y0, H, rows, Wqkv, s.Y1, d->d, &sp, status,
                                        stream);
    if (e == cudaSuccess)
      e = head_epilogue_bf16_pair(ep_kv, ep_qkv, stream);
    if (e == cudaSuccess)
      e = attention(d->dtype, p, stream);
    return cuda_status(e);
  }
  if (!grouped) {
    // the same work as two calls
    st = dflash_kv_inject(d, c, layer, C, cu_rows, M, W_K, W_V, gamma_k, rope, table_len,
                          workspace, ws_bytes, stream);
    if (st != DFLASH_OK) return st;
    return dflash_block_attn(d, c, layer, H, W_Q, W_K, W_V, gamma_q, gamma_k, rope, table_len,
                             window, scaling, out, workspace, ws_bytes, stream);
  }
  Carver cv(workspace, ws_bytes);
  BlockScratch s = carve_block(cv, d, c->batch, c->capacity, window);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  const HeadEpilogue ep_kv = inject_epilogue(d, c, layer, cu_rows, M, gamma_k, rope, table_len,
                                             nullptr, 1, status);
  HeadEpilogue ep_qkv = block_epilogue(d, c, layer, gamma_q, gamma_k, rope, table_len, s.q,
                                       nullptr, 1, status);
  ep_qkv.pre_rows = cu_rows;  // the block follows the rows injected here
  ep_qkv.pre_M = M;
  AttnParams p = block_attention(d, c, layer, s, window, scaling, table_len, out, status);
  p.pre_rows = cu_rows;
  p.pre_M = M;
  p.lens_out = c->lens + (size_t)layer * c->batch;
  p.sched_ready = true;
  const sched::Params sp = attn_sched_params(p);
  cudaError_t e = gemm_tc_layer(C, M, Wkv, ep_kv, H, rows, Wqkv, ep_qkv, d->d, &sp, status, stream);
  if (e == cudaSuccess)
    e = attention(d->dtype, p, stream);
  return cuda_status(e);
}

namespace {
// shapes the layer-output kernels take: GEMM K and N in whole 64-wide blocks for the
// tensor-core path, rows of whole float4 / 4-element groups for the row kernels
dflash_status check_layer_out(const dflash_dims* d, int M, int d_ff) {
  dflash_status st = check_dims(d);
  if (st != DFLASH_OK) return st;
  if (M < 0 || d_ff <= 0 || d_ff % 4 || !rows_ok(d->d)) return DFLASH_ERR_INVALID_ARG;
  if (d->dtype == DFLASH_BF16 && (d_ff % 64 || (d->n_h * d->d_h) % 64))
    return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}
}  // namespace

DFLASH_API size_t dflash_layer_out_workspace_bytes(const dflash_dims* d, int M, int d_ff) {
  if (check_layer_out(d, M, d_ff) != DFLASH_OK) return 0;
  Carver cv(nullptr, ~size_t(0));
  carve_layer_out(cv, d->dtype, M, d->d, d->n_h * d->d_h, d_ff);
  return cv.off > 256 ? cv.off : 256;
}

DFLASH_API dflash_status dflash_layer_out(const dflash_dims* d, int M, const void* attn_out,
                                          const void* x, const void* W_O, const void* gamma_post,
                                          int d_ff, const void* W_gate, const void* W_up,
                                          const void* W_down, void* x_out, void* workspace,
                                          size_t ws_bytes, cudaStream_t stream) {
  dflash_status st = check_layer_out(d, M, d_ff);
  if (st != DFLASH_OK) return st;
  if (M == 0) return DFLASH_OK;
  const void* ptrs[] = {attn_out, x, W_O, gamma_post, W_gate, W_up, W_down, x_out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return DFLASH_ERR_INVALID_ARG;
  if (!workspace || ((uintptr_t)workspace & 255)) return DFLASH_ERR_INVALID_ARG;
  Carver cv(workspace, ws_bytes);
  const LayerOutScratch sc = carve_layer_out(cv, d->dtype, M, d->d, d->n_h * d->d_h, d_ff);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  return cuda_status(layer_out(d->dtype, M, d->d, d->n_h * d->d_h, d_ff, attn_out, x, W_O,
                               gamma_post, d->eps, W_gate, W_up, W_down, x_out, sc, status,
                               stream));
}

DFLASH_API dflash_status dflash_rms_norm(const dflash_dims* d, int M, const void* x,
                                         const void* gamma, void* out, cudaStream_t stream) {
  dflash_status st = check_dims(d);
  if (st != DFLASH_OK) return st;
  if (M < 0 || !rows_ok(d->d)) return DFLASH_ERR_INVALID_ARG;
  if (M == 0) return DFLASH_OK;
  if (!x || !gamma || !out || !aligned16(x) || !aligned16(gamma) || !aligned16(out))
    return DFLASH_ERR_INVALID_ARG;
  return cuda_status(norm_rows(d->dtype, M, d->d, x, gamma, d->eps, out, stream));
}

DFLASH_API dflash_status dflash_accept(const int32_t* block_ids, const int32_t* posterior,
                                       int batch, int bs, const int32_t* ctx_len,
                                       int32_t* accept_len, int32_t* next_cu_rows,
                                       int32_t* ctx_next, int32_t* next_anchor,
                                       cudaStream_t stream) {
  if (batch < 0 || bs < 1) return DFLASH_ERR_INVALID_ARG;
  if (!next_cu_rows || ((uintptr_t)next_cu_rows & 3)) return DFLASH_ERR_INVALID_ARG;
  if (batch > 0) {
    const void* ptrs[] = {block_ids, posterior, ctx_len, accept_len, ctx_next, next_anchor};
    for (const void* q : ptrs)
      if (!q || ((uintptr_t)q & 3)) return DFLASH_ERR_INVALID_ARG;
  }
  return cuda_status(accept_round(block_ids, posterior, batch, bs, ctx_len, accept_len,
                                  next_cu_rows, ctx_next, next_anchor, stream));
}

DFLASH_API dflash_status dflash_cache_crop(const dflash_kv_cache* c, const int32_t* new_lens,
                                           cudaStream_t stream) {
  dflash_status st = check_cache(c, 0);
  if (st != DFLASH_OK) return st;
  if (!new_lens || ((uintptr_t)new_lens & 3)) return DFLASH_ERR_INVALID_ARG;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  return cuda_status(crop_lens(c->lens, c->n_layers, c->batch, new_lens, status, stream));
}

DFLASH_API dflash_status dflash_test_attn_worklist(const dflash_dims* d, const dflash_kv_cache* c,
                                                   int layer, const int32_t* cu_rows, int M,
                                                   int window, void* workspace, size_t ws_bytes,
                                                   int32_t* out, size_t out_ints, size_t* n_out,
                                                   cudaStream_t stream) {
  dflash_status st = check_dims(d);
  if (st != DFLASH_OK) return st;
  st = check_cache(c, layer);
  if (st != DFLASH_OK) return st;
  if (d->dtype != DFLASH_BF16 || (!out && out_ints > 0) || !n_out || !workspace || window < 0 ||
      M < 0 || (M > 0 && !cu_rows))
    return DFLASH_ERR_INVALID_ARG;
  Carver cv(workspace, ws_bytes);
  BlockScratch s = carve_block(cv, d, c->batch, c->capacity, window);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  unsigned* status = status_word();
  if (!status) return DFLASH_ERR_CUDA;
  AttnParams p = block_attention(d, c, layer, s, window, 0.f, c->capacity, nullptr, status);
  p.pre_rows = M > 0 ? cu_rows : nullptr;
  p.pre_M = M;
  sched::Params sp;
  int cnt[2] = {0, 0};
  cudaError_t e = attn_worklist_build(p, stream, &sp);
  if (e == cudaSuccess) e = cudaMemcpyAsync(cnt, sp.n_items, sizeof(cnt), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return DFLASH_ERR_CUDA;
  const size_t n_ctas = (size_t)sp.n_sm, pairs = (size_t)c->batch * d->n_kv;
  const size_t need = 5 + (n_ctas + 1) + 4 * (n_ctas + (size_t)cnt[0]) + pairs + (size_t)cnt[1];
  *n_out = need;
  if (out_ints < need) return DFLASH_ERR_INVALID_ARG;
  out[0] = (int32_t)n_ctas;
  out[1] = sp.max_splits;
  out[2] = sp.item_cost;
  out[3] = cnt[0];
  out[4] = cnt[1];
  int32_t* o = out + 5;
  e = cudaMemcpyAsync(o, sp.first, (n_ctas + 1) * 4, cudaMemcpyDeviceToHost, stream);
  o += n_ctas + 1;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(o, sp.items, (n_ctas + cnt[0]) * 16, cudaMemcpyDeviceToHost, stream);
  o += 4 * (n_ctas + cnt[0]);
  if (e == cudaSuccess) e = cudaMemcpyAsync(o, sp.splits, pairs * 4, cudaMemcpyDeviceToHost, stream);
  o += pairs;
  if (e == cudaSuccess && cnt[1] > 0)
    e = cudaMemcpyAsync(o, sp.merge_list, (size_t)cnt[1] * 4, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return cuda_status(e);
}

DFLASH_API dflash_status dflash_status_get(unsigned int* out, cudaStream_t stream) {
  if (!out) return DFLASH_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DFLASH_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return DFLASH_ERR_CUDA;
  *out = v;
  return v ? DFLASH_ERR_DEVICE : DFLASH_OK;
}
