// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dflash.h"

#define DFLASH_API extern "C" __attribute__((visibility("default")))

namespace dflash {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// element conversions
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// scratch carving: every piece 256-byte aligned
// ---------------------------------------------------------------------------
struct Carver {
  char* base;
  size_t cap;
  size_t off = 0;
  bool ok = true;
  Carver(void* b, size_t c) : base((char*)b), cap(c) {}
  template <typename T> T* take(size_t count) {
    size_t bytes = (count * sizeof(T) + 255) & ~size_t(255);
    if (off + bytes > cap) { ok = false; return nullptr; }
    T* p = base ? (T*)(base + off) : nullptr;
    off += bytes;
    return p;
  }
};

// Limit of the pipeline waits of tensor-core kernels launched from now on (2 s unless a
// test lowered it with dflash_test_wait_limit; dflash_api.cu).
unsigned long long wait_limit_ns();

// per-device sticky status word (defined in dflash_api.cu)
unsigned* status_word();

// Brackets one kernel launch: counts it and, while tracing selects its kind,
// records CUDA events around it on its stream (trace.cu).
class LaunchScope {
 public:
  LaunchScope(int kind, cudaStream_t s);
  ~LaunchScope();
 private:
  int kind_;
  cudaStream_t stream_;
  int slot_;
};

// ---------------------------------------------------------------------------
// GEMM: Y[split][M][N] (fp32) = X[M][K] W[N][K]^T, X given as K-segments
// ---------------------------------------------------------------------------
struct Segments {
  const void* p[8];  // n device pointers, each [M][kseg]
  int n;
  int kseg;
};

// Weights stacked along N: columns [off_i, off_i + N_i) of Y come from Ws[i] ([N_i][K]).
struct Weights {
  const void* p[3];
  int n[3];
  int count;
  __host__ __device__ int total() const { int t = 0; for (int i = 0; i < count; ++i) t += n[i]; return t; }
};

// Number of K-splits the GEMM of this shape uses (partials summed by the epilogue).
// split_cap > 0 bounds the K-splits (a caller with a fixed scratch size).
int gemm_splits(int dtype, int M, const Weights& W, int K, int split_cap = 0);

// Y[split][M][ldY] (fp32) = X W^T. f32: SIMT FFMA; bf16: tcgen05 tensor cores.
cudaError_t gemm(int dtype, const Segments& A, int M, const Weights& W, float* Y, int ldY,
                 unsigned* status, cudaStream_t s, int split_cap = 0);

// tcgen05 / TMA GEMM (bf16 inputs, fp32 accumulation); gemm_tc.cu
int gemm_tc_splits(int M, const Weights& W, int K, int split_cap = 0);
cudaError_t gemm_tc(const Segments& A, int M, const Weights& W, float* Y, int ldY,
                    unsigned* status, cudaStream_t s, int split_cap = 0);

// The context projection with hidden_norm fused into its epilogue (bf16): C = RMSNorm of
// X W^T, from Y (split partials, [splits][M][N] fp32), rowpart ([M][N / BN] fp32) and
// gemm_tc_norm_counters() ints of scratch (cleared by the call on its stream). Only for
// shapes whose CTAs are all resident at once (gemm_tc_norm_ok); gemm_tc + rmsnorm_rows
// otherwise.
bool gemm_tc_norm_ok(int M, const Weights& W, int K, int split_cap = 0);
int gemm_tc_norm_counters(int M, const Weights& W, int K, int split_cap = 0);
int gemm_tc_norm_tiles_n(int M, const Weights& W, int K);  // N / BN: rowpart is [M][this]
cudaError_t gemm_tc_norm(const Segments& A, int M, const Weights& W, float* Y, float* rowpart,
                         int* counters, const void* gamma, float eps, void* C, unsigned* status,
                         cudaStream_t s, int split_cap = 0);

// The context projection on caller scratch (dflash_api.cu); split_cap > 0 bounds its
// K-splits, and ctx_scratch_bytes gives the scratch that needs.
dflash_status ctx_project_impl(const dflash_dims* d, const void* const* hidden, int M,
                               const void* W_fc, const void* gamma_h, void* C_out, void* workspace,
                               size_t ws_bytes, int split_cap, cudaStream_t stream);
size_t ctx_scratch_bytes(const dflash_dims* d, int M, int split_cap);
int ctx_splits(const dflash_dims* d, int M);

// SIMT fp32-accumulating GEMM for any M, N, K (the f32 path).
cudaError_t gemm_simt(int dtype, const Segments& A, int M, const Weights& W, float* Y, int ldY,
                      cudaStream_t s);

// ---------------------------------------------------------------------------
// epilogues
// ---------------------------------------------------------------------------
// C[row][:] = RMSNorm_gamma(sum_s Y[s][row][:])
cudaError_t rmsnorm_rows(int dtype, const float* Y, int splits, int M, int N, const void* gamma,
                         float eps, void* out, cudaStream_t s);

// Per-head epilogue of a projection whose N axis is [n_q Q heads | n_kv K heads | n_kv V heads].
struct HeadEpilogue {
  const float* Y;       // [splits][rows][ldY]
  int splits, rows, ldY;
  int n_q, n_kv, d_h;
  float eps;
  const void* gamma_q;  // [d_h] (Q heads)
  const void* gamma_k;  // [d_h] (K heads)
  const float2* rope;   // [table_len][d_h/2]
  int table_len;
  // rows -> sequences: cu_rows != nullptr: rows grouped by cu_rows[batch+1];
  // else row = b * bs + t
  const int32_t* cu_rows;
  int batch, bs;
  const int32_t* lens;  // [batch] for this layer
  void* q_out;          // [batch][n_q][bs][d_h]
  void* cache_k;        // layer base [batch][n_kv][capacity][d_h]
  void* cache_v;
  int capacity;
  unsigned* status;
  // block rows only: rows of an inject in the same call precede the block, so a
  // sequence's block starts after the rows that inject appended (cu_rows, row count)
  const int32_t* pre_rows = nullptr;
  int pre_M = 0;
  // paged cache: page ids [batch][pages_per_seq] of 128-row pages, or null (contiguous)
  const int32_t* block_table = nullptr;
  int pages_per_seq = 0;
  // fp8 (E4M3) cache: K / V rows are stored as codes of x * k_inv (x * v_inv), and Q as
  // two E4M3 arrays, q_out = codes of q and q_lo = codes of the remainder q - value(q_out)
  bool kv_fp8 = false;
  float k_inv = 1.f, v_inv = 1.f;
  void* q_lo = nullptr;
};
cudaError_t head_epilogue(int dtype, const HeadEpilogue& e, cudaStream_t s);

// Four E4M3 codes of (a, b, c, d) * inv (round to nearest even, saturating), packed with
// a in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}
// Values of the two E4M3 codes in the low (x) and high (y) byte of v.
__device__ __forceinline__ float2 e4m3x2_value(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  float2 f;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(f.x), "=f"(f.y)
      : "r"(h2));
  return f;
}
// E4M3 codes of four values and of their remainders: hi = codes(v), lo = codes(v - value(hi)).
__device__ __forceinline__ void e4m3x4_split(float a, float b, float c, float d, uint32_t& hi,
                                             uint32_t& lo) {
  hi = e4m3x4(a, b, c, d);
  const float2 v01 = e4m3x2_value((uint16_t)(hi & 0xFFFF));
  const float2 v23 = e4m3x2_value((uint16_t)(hi >> 16));
  lo = e4m3x4(a - v01.x, b - v01.y, c - v23.x, d - v23.y);
}

// Row index (in d_h-wide rows of one layer's K or V) of logical slot `pos` of sequence b,
// KV head kvh: [b][kvh][capacity] contiguous, or page table[b][pos / 128] of a pool of
// [n_pages][n_kv][128] rows.
__device__ __forceinline__ size_t cache_row(const int32_t* table, int pages_per_seq, int n_kv,
                                            int capacity, int b, int kvh, int pos) {
  if (table) {
    const int page = table[(size_t)b * pages_per_seq + (pos >> 7)];
    return ((size_t)page * n_kv + kvh) * 128 + (pos & 127);
  }
  return ((size_t)b * n_kv + kvh) * capacity + pos;
}

// tcgen05 GEMM with the per-head epilogue fused (bf16, d_h = 128), for shapes
// that fill the GPU without split-K (gemm_tc_heads_ok): the projection rows go
// through norm / RoPE straight into Q and the cache.
bool gemm_tc_heads_ok(int M, const Weights& W, int K);
cudaError_t gemm_tc_heads(const Segments& A, int M, const Weights& W, const HeadEpilogue& ep,
                          unsigned* status, cudaStream_t s);

// Both projections of one draft layer in a single tcgen05 launch (bf16, d_h = 128):
// the inject's context K/V and the block's Q/K/V, fused epilogues, plus optionally
// the attention work list (sched::Params, attn_sched.cuh) from one extra CTA.
namespace sched { struct Params; }
bool gemm_tc_layer_ok(int Mc, const Weights& Wkv, int Mb, const Weights& Wqkv, int K);
cudaError_t gemm_tc_layer(const void* C, int Mc, const Weights& Wkv, const HeadEpilogue& ep_kv,
                          const void* H, int Mb, const Weights& Wqkv, const HeadEpilogue& ep_qkv,
                          int K, const sched::Params* sp, unsigned* status, cudaStream_t s);

// The same two projections in one split-K launch (fp32 partials Y0: [splits][Mc][N0],
// Y1: [splits][Mb][N1]) for batches too small to fill the GPU without split-K, plus
// optionally the work-list CTA. The plan depends on Mb alone: _splits gives its K splits
// (0: not applicable) and _rows the most context rows it takes (Mc <= that).
int gemm_tc_layer_split_splits(int Mb, const Weights& Wkv, const Weights& Wqkv, int K);
int gemm_tc_layer_split_rows(int Mb, const Weights& Wkv, const Weights& Wqkv, int K);
cudaError_t gemm_tc_layer_split(const void* C, int Mc, const Weights& Wkv, float* Y0,
                                const void* H, int Mb, const Weights& Wqkv, float* Y1, int K,
                                const sched::Params* sp, unsigned* status, cudaStream_t s);

// Warp-per-(row, head) epilogue for bf16 with d_h = 128 (sums the split-K partials);
// _pair finishes two epilogues (an inject's and the block's) in one launch.
cudaError_t head_epilogue_bf16(const HeadEpilogue& e, cudaStream_t s);
cudaError_t head_epilogue_bf16_pair(const HeadEpilogue& e0, const HeadEpilogue& e1,
                                    cudaStream_t s);

// lens[b] += n_b where the append fitted (same checks as the epilogue)
cudaError_t lens_advance(int32_t* lens, const int32_t* cu_rows, int batch, int bs, int M,
                         int capacity, int table_len, cudaStream_t s);

// The rest of a draft decoder layer (layer_out.cu): o_proj + residual, post-attention
// RMSNorm, SwiGLU MLP + residual; and a plain row RMSNorm.
struct LayerOutScratch {
  float* Y;    // o_proj / down split-K partials
  float* Ygu;  // gate | up split-K partials
  void* x1;    // residual after o_proj
  void* n;     // RMSNorm_post(x1)
  void* h;     // silu(gate) * up
  int splits_o, splits_gu, splits_d;
};
bool rows_ok(int N);
LayerOutScratch carve_layer_out(Carver& cv, int dtype, int M, int d, int a_dim, int d_ff);
cudaError_t layer_out(int dtype, int M, int d, int a_dim, int d_ff, const void* attn_out,
                      const void* x, const void* W_O, const void* gamma_post, float eps,
                      const void* W_gate, const void* W_up, const void* W_down, void* x_out,
                      const LayerOutScratch& sc, unsigned* status, cudaStream_t s);
cudaError_t norm_rows(int dtype, int M, int N, const void* x, const void* gamma, float eps,
                      void* out, cudaStream_t s);

cudaError_t accept_round(const int32_t* block_ids, const int32_t* posterior, int batch, int bs,
                         const int32_t* ctx_len, int32_t* accept_len, int32_t* cu,
                         int32_t* ctx_next, int32_t* anchor, cudaStream_t s);
cudaError_t crop_lens(int32_t* lens, int n_layers, int batch, const int32_t* new_lens,
                      unsigned* status, cudaStream_t s);

cudaError_t rope_table(double theta, int d_h, int max_pos, float* table, cudaStream_t s);

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
struct AttnParams {
  const void* q;          // [batch][n_h][bs][d_h]
  const void* cache_k;    // layer base [batch][n_kv][capacity][d_h]
  const void* cache_v;
  const int32_t* lens;    // [batch], BEFORE the block's lens advance
  void* out;              // [batch][bs][n_h * d_h]
  float* part_acc;        // partial accumulators, per chunk
  float2* part_ml;        // partial (max, sum), per chunk
  void* sched;            // tensor-core path: work list, split counts, counters, lengths
  unsigned* status;       // device status word
  // tensor-core path only:
  const int32_t* pre_rows;  // cu_rows of rows injected in the same call (the block follows
  int pre_M;                // them), or null
  int32_t* lens_out;        // receives the lengths after the call (block appended), or null
  bool sched_ready;         // the work list was built by the projection launch
  const int32_t* block_table;  // paged cache (128-row pages), or null
  int pages_per_seq, n_pages;
  // fp8 (E4M3) cache: q holds the codes of Q then those of its remainder; scores are
  // scaled by k_scale and outputs by v_scale
  bool fp8;
  float k_scale, v_scale;
  int batch, n_h, n_kv, d_h, bs, capacity, window, chunk, n_chunks, table_len;
  float scaling;
};
int attn_simt_chunk();
cudaError_t attn_simt(int dtype, const AttnParams& p, cudaStream_t s);

// tcgen05 attention (bf16, d_h = 128); attn_tc.cu
int attn_tc_chunk();
// Bytes of the attention work-list area for `batch` sequences of n_kv KV heads.
size_t attn_sched_bytes(int batch, int n_kv);
cudaError_t attn_tc(const AttnParams& p, cudaStream_t s);

// Keys per attention chunk and the attention launch for a dtype.
int attn_chunk(int dtype);
cudaError_t attention(int dtype, const AttnParams& p, cudaStream_t s);

}  // namespace dflash
