// Tensor-core projection GEMMs for sm_103a: X W^T with bf16 inputs and an
// fp32 accumulator in tensor memory.
//
// One CTA computes a 128 x BN tile over its share of K (split-K across
// gridDim.z):
//   warp 0      TMA producer: 128 x 64 activation tile + BN x 64 weight tile
//               per stage, 128-byte swizzle, completion on a "full" mbarrier;
//   warp 1      allocates BN TMEM columns and issues tcgen05.mma (M=128,
//               N=BN, K=16, four per stage) from one thread; tcgen05.commit
//               frees each stage ("empty" mbarrier) and finally signals "done";
//   warps 2-5   epilogue, one thread per tile row (tcgen05.ld of its lanes).
// The activations arrive as up to eight K-segments (the k target layers'
// hidden states of the context projection), each with its own tensor map;
// the weights as up to three matrices stacked along N (W_Q | W_K | W_V).
//
// Two epilogues:
//   fp32 store   the tile (a split-K partial) goes to Y; the context
//                projection's RMSNorm kernel sums the splits;
//   heads        (no split-K) whole 128-dim heads per tile (BN = 128 or 256).
//                The thread owning a row applies the per-head RMSNorm (Q and K
//                heads), rotates the pair (i, i + 64) at the row's absolute
//                position and stores the bf16 row into the Q buffer or the
//                row's cache slot (DFlash KV Injection Walkthrough, Steps
//                4.1-4.3; DFlash source guide (II), parts 1-4). Shapes that need
//                split-K use the fp32 store and a separate epilogue kernel.
#include <cstdlib>
#include <mutex>

#include "attn_sched.cuh"
#include "sm100_ptx.cuh"

namespace dflash {
namespace {

constexpr int BM = 128, BK = 64, kThreads = 192;

struct TcGemmParams {
  CUtensorMap a[8];   // activation segments [M][kseg], box {64, 128}
  CUtensorMap b[3];   // weights [N_i][K], box {64, BN}
  int kseg_blocks;    // 64-wide K blocks per activation segment
  int w_count;
  int w_off[4];       // prefix offsets of the stacked weights along N
  int M, ldY;
  int kb_total, kb_per_split, splits;
  float* Y;           // fp32 store: [split][M][ldY]
  HeadEpilogue ep;    // heads: norm / RoPE / destination
  unsigned* status;
  // Grouped launch (heads epilogue, no split-K): grid columns [0, ny0) compute the
  // problem above, columns [ny0, ny0 + ny1) a second one with one activation segment
  // (same K), and with sched_cta one more column whose first CTA builds the
  // attention work list while the tiles run.
  int ny0, ny1, sched_cta;
  CUtensorMap a1;
  CUtensorMap b1[3];
  int w1_count;
  int w1_off[4];
  int M1;
  HeadEpilogue ep1;
  sched::Params sp;
};

template <int BN>
struct Cfg {
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + 256;
};

// Waits without honouring the abort flag (used to drain in-flight work before exit).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned* status) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
      atomicOr(status, DFLASH_DEV_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Per-head epilogue of one 128-wide row x[0..127] of the projection of tile
// row `row` (global), head `head` of the stacked [Q | K | V] layout.
__device__ __forceinline__ void head_row(const HeadEpilogue& e, int row, int head, float (&x)[128]) {
  int b, t, n_b;
  if (e.cu_rows) {
    int lo = 0, hi = e.batch - 1;
    while (lo < hi) {  // last b with cu_rows[b] <= row
      const int mid = (lo + hi + 1) >> 1;
      if (e.cu_rows[mid] <= row) lo = mid; else hi = mid - 1;
    }
    b = lo;
    t = row - e.cu_rows[b];
    n_b = e.cu_rows[b + 1] - e.cu_rows[b];
    if (n_b < 0 || e.cu_rows[b + 1] > e.rows || e.cu_rows[0] != 0 || t < 0 || t >= n_b) {
      atomicOr(e.status, DFLASH_DEV_ROWS);
      return;
    }
  } else {
    b = row / e.bs;
    t = row - b * e.bs;
    n_b = e.bs;
  }
  int start = e.lens[b];
  start += sched::injected_rows(e.pre_rows, e.pre_M, b, start, e.capacity, e.table_len);
  if (start < 0 || start + n_b > e.capacity || start + n_b > e.table_len) {
    if (t == 0 && head == 0)
      atomicOr(e.status, (start + n_b > e.capacity || start < 0) ? DFLASH_DEV_CAPACITY
                                                                 : DFLASH_DEV_ROPE);
    return;
  }
  const int pos = start + t;
  const int kind = head < e.n_q ? 0 : (head < e.n_q + e.n_kv ? 1 : 2);  // Q, K, V
  if (kind < 2) {
    float ss0 = 0.f, ss1 = 0.f, ss2 = 0.f, ss3 = 0.f;
#pragma unroll
    for (int i = 0; i < 128; i += 4) {
      ss0 = fmaf(x[i], x[i], ss0);
      ss1 = fmaf(x[i + 1], x[i + 1], ss1);
      ss2 = fmaf(x[i + 2], x[i + 2], ss2);
      ss3 = fmaf(x[i + 3], x[i + 3], ss3);
    }
    const float r = 1.0f / sqrtf(((ss0 + ss1) + (ss2 + ss3)) * (1.0f / 128.f) + e.eps);
    const bf16* g = (const bf16*)(kind == 0 ? e.gamma_q : e.gamma_k);
    const float2* cs = e.rope + (size_t)pos * 64;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float x0 = x[i] * r * __bfloat162float(g[i]);
      const float x1 = x[i + 64] * r * __bfloat162float(g[i + 64]);
      const float2 c = cs[i];
      x[i] = x0 * c.x - x1 * c.y;  // rotate_half: [-x1, x0]
      x[i + 64] = x1 * c.x + x0 * c.y;
    }
  }
  bf16* dst;
  if (kind == 0) {
    dst = (bf16*)e.q_out + (((size_t)b * e.n_q + head) * e.bs + t) * 128;
  } else {
    const int kvh = head - e.n_q - (kind == 2 ? e.n_kv : 0);
    bf16* base = (bf16*)(kind == 1 ? e.cache_k : e.cache_v);
    dst = base + (((size_t)b * e.n_kv + kvh) * e.capacity + pos) * 128;
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    uint4 w;
    w.x = pack_bf16(x[8 * k + 0], x[8 * k + 1]);
    w.y = pack_bf16(x[8 * k + 2], x[8 * k + 3]);
    w.z = pack_bf16(x[8 * k + 4], x[8 * k + 5]);
    w.w = pack_bf16(x[8 * k + 6], x[8 * k + 7]);
    d4[k] = w;
  }
}

template <int BN, bool HEADS>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcGemmParams p) {
  using C = Cfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + (size_t)STAGES * C::STAGE);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  // problem of this CTA (grouped launches); whole CTAs branch, before any barrier
  const int col = (int)blockIdx.y;
  if (p.sched_cta && col == p.ny0 + p.ny1) {
    if (blockIdx.x == 0 && blockIdx.z == 0) sched::build(p.sp);
    return;
  }
  const bool second = p.ny1 > 0 && col >= p.ny0;
  const CUtensorMap* amap = second ? &p.a1 : p.a;
  const CUtensorMap* bmap = second ? p.b1 : p.b;
  const int* w_off = second ? p.w1_off : p.w_off;
  const int w_count = second ? p.w1_count : p.w_count;
  const int M = second ? p.M1 : p.M;
  const int kseg_blocks = second ? p.kb_total : p.kseg_blocks;
  const HeadEpilogue& ep = second ? p.ep1 : p.ep;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM, n0 = (second ? col - p.ny0 : col) * BN;
  if (m0 >= M) return;  // grid.x covers the taller problem
  const int kb0 = blockIdx.z * p.kb_per_split;
  const int nkb = min(p.kb_total, kb0 + p.kb_per_split) - kb0;
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = ptx::smem_u32(bars + STAGES);
  const uint32_t done = ptx::smem_u32(bars + 2 * STAGES);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    ptx::mbar_init(done, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < (second ? 1 : 8); ++i) ptx::prefetch_tmap(&amap[i]);
    for (int i = 0; i < w_count; ++i) ptx::prefetch_tmap(&bmap[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), BN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  int wi = 0;
  while (wi + 1 < w_count && n0 >= w_off[wi + 1]) ++wi;
  const int nb = n0 - w_off[wi];

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (i >= STAGES && !ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, &abort_flag, p.status)) break;
        const int kb = kb0 + i;
        const int seg = kb / kseg_blocks;
        const int kx = (kb - seg * kseg_blocks) * BK;
        const uint32_t sa = ptx::smem_u32(smem + (size_t)s * C::STAGE);
        ptx::mbar_arrive_expect_tx(full0 + 8 * s, C::STAGE);
        ptx::tma_load_2d(sa, &amap[seg], full0 + 8 * s, kx, m0);
        ptx::tma_load_2d(sa + C::A_BYTES, &bmap[wi], full0 + 8 * s, kb * BK, nb);
        ++issued;
      }
      // no copy of ours may still be landing when the CTA exits
      for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
        drain_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!ptx::mbar_wait(full0 + 8 * s, ph, &abort_flag, p.status)) break;
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + (size_t)s * C::STAGE);
        const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          ptx::mma_bf16(tmem, ptx::smem_desc_sw128(sa + 32 * k), ptx::smem_desc_sw128(sb + 32 * k),
                        idesc, (i > 0 || k > 0) ? 1u : 0u);
        ptx::mma_commit(empty0 + 8 * s);
      }
      ptx::mma_commit(done);
      drain_wait(done, 0, p.status);  // every MMA has finished before TMEM can be freed
    }
  } else {
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 are this warp's
    const int row = q * 32 + lane;
    const bool in = (m0 + row) < M;
    // warp-uniform: tcgen05.ld below is a .sync.aligned instruction
    const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(done, 0, &abort_flag, p.status));
    ptx::tc_fence_after();
    if (ok && !HEADS) {
      float* y = p.Y + (size_t)blockIdx.z * M * p.ldY + (size_t)(m0 + row) * p.ldY + n0;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), r);
        ptx::tmem_ld_wait();
        if (in) {
          float4* dst = reinterpret_cast<float4*>(y + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
    }
    if (ok && HEADS) {
      // BN / 128 whole heads per tile, one after the other; each thread owns one row.
      // Every lane joins the tcgen05.ld (warp-collective); only rows < M are stored.
#pragma unroll 1
      for (int hd = 0; hd < BN / 128; ++hd) {
        float x[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hd * 128 + c * 32), r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c * 32 + j] = __uint_as_float(r[j]);
        }
        if (in) head_row(ep, m0 + row, n0 / 128 + hd, x);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, BN);
  }
}

// ---- host side ---------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

struct Plan {
  int bn, kb_total, kb_per_split, splits;
};

// The widest of 256/128/64 that divides every stacked weight (heads: 256 or
// 128, whole heads per tile). Split-K to about one wave on the GPU.
Plan plan(int M, const Weights& W, int K, bool heads) {
  Plan pl;
  pl.bn = 256;
  for (int i = 0; i < W.count; ++i)
    while (W.n[i] % pl.bn) pl.bn >>= 1;
  if (heads && pl.bn < 128) pl.bn = 0;  // heads need whole 128-dim heads per tile
  if (pl.bn == 0) return pl;
  pl.kb_total = K / BK;
  const int tiles = ((M + BM - 1) / BM) * (W.total() / pl.bn);
  int splits = 148 / (tiles > 0 ? tiles : 1);
  const int max_splits = pl.kb_total / 4 > 0 ? pl.kb_total / 4 : 1;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  pl.kb_per_split = (pl.kb_total + splits - 1) / splits;
  pl.splits = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  return pl;
}

template <int BN, bool HEADS>
cudaError_t launch(const TcGemmParams& p, dim3 grid, cudaStream_t s) {
  const size_t smem = Cfg<BN>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, HEADS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  LaunchScope ls_(DFLASH_KERNEL_GEMM, s);
  gemm_tc_kernel<BN, HEADS><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

// bf16 row-major [rows][cols] matrix, box {64 columns, box_rows rows}, 128-byte swizzle,
// zero fill outside the matrix.
bool encode_2d_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_tc_splits(int M, const Weights& W, int K) { return plan(M, W, K, false).splits; }

bool gemm_tc_heads_ok(int M, const Weights& W, int K) {
  const Plan pl = plan(M, W, K, true);
  return pl.bn >= 128 && pl.splits == 1;
}

namespace {

cudaError_t fill_common(TcGemmParams& p, const Segments& A, int M, const Weights& W, const Plan& pl,
                        int K) {
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < A.n; ++i)
    if (!encode_2d_bf16(&p.a[i], A.p[i], M, A.kseg, BM)) return cudaErrorInvalidValue;
  for (int i = A.n; i < 8; ++i) p.a[i] = p.a[0];
  int off = 0;
  for (int i = 0; i < W.count; ++i) {
    if (!encode_2d_bf16(&p.b[i], W.p[i], W.n[i], K, pl.bn)) return cudaErrorInvalidValue;
    p.w_off[i] = off;
    off += W.n[i];
  }
  p.w_off[W.count] = off;
  p.w_count = W.count;
  p.kseg_blocks = A.kseg / BK;
  p.M = M;
  p.kb_total = pl.kb_total;
  p.kb_per_split = pl.kb_per_split;
  p.splits = pl.splits;
  return cudaSuccess;
}

}  // namespace

cudaError_t gemm_tc(const Segments& A, int M, const Weights& W, float* Y, int ldY,
                    unsigned* status, cudaStream_t s) {
  const int N = W.total();
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int K = A.n * A.kseg;
  const Plan pl = plan(M, W, K, false);
  if (pl.bn < 64 || A.kseg % BK) return cudaErrorInvalidValue;
  TcGemmParams p;
  cudaError_t e = fill_common(p, A, M, W, pl, K);
  if (e != cudaSuccess) return e;
  p.ldY = ldY;
  p.Y = Y;
  p.status = status;
  dim3 grid((M + BM - 1) / BM, N / pl.bn, pl.splits);
  switch (pl.bn) {
    case 256: return launch<256, false>(p, grid, s);
    case 128: return launch<128, false>(p, grid, s);
    default: return launch<64, false>(p, grid, s);
  }
}

cudaError_t gemm_tc_heads(const Segments& A, int M, const Weights& W, const HeadEpilogue& ep,
                          unsigned* status, cudaStream_t s) {
  const int N = W.total();
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int K = A.n * A.kseg;
  const Plan pl = plan(M, W, K, true);
  if (pl.bn < 128 || pl.splits != 1 || ep.d_h != 128 || A.kseg % BK) return cudaErrorInvalidValue;
  TcGemmParams p;
  cudaError_t e = fill_common(p, A, M, W, pl, K);
  if (e != cudaSuccess) return e;
  p.ep = ep;
  p.status = status;
  dim3 grid((M + BM - 1) / BM, N / pl.bn, 1);
  return pl.bn == 256 ? launch<256, true>(p, grid, s) : launch<128, true>(p, grid, s);
}

// Both projections of a draft layer in one launch: the context rows' K/V (inject) and
// the block's Q/K/V, each with the fused per-head epilogue, plus (sp != null) the
// attention work list from an extra CTA. Worth it when the two tile sets together fill
// a good part of the GPU without split-K; gemm_tc_layer_ok decides.
namespace {
int layer_bn(int Mc, const Weights& Wkv, int Mb, const Weights& Wqkv, int K) {
  if (Mc <= 0 || Mb <= 0 || K % BK) return 0;
  const Plan a = plan(Mc, Wkv, K, true), b = plan(Mb, Wqkv, K, true);
  const int bn = a.bn < b.bn ? a.bn : b.bn;
  if (bn < 128) return 0;
  // DFLASH_FUSED_LAYER=0 never groups, =1 groups whenever the shapes allow (the two are
  // the same arithmetic); otherwise group when the tiles fill a good part of the GPU
  const char* env = getenv("DFLASH_FUSED_LAYER");
  if (env && env[0] == '0') return 0;
  if (env && env[0] == '1') return bn;
  const int tiles = ((Mc + BM - 1) / BM) * (Wkv.total() / bn) + ((Mb + BM - 1) / BM) * (Wqkv.total() / bn);
  return tiles >= 64 ? bn : 0;
}
}  // namespace

bool gemm_tc_layer_ok(int Mc, const Weights& Wkv, int Mb, const Weights& Wqkv, int K) {
  return layer_bn(Mc, Wkv, Mb, Wqkv, K) != 0;
}

cudaError_t gemm_tc_layer(const void* C, int Mc, const Weights& Wkv, const HeadEpilogue& ep_kv,
                          const void* H, int Mb, const Weights& Wqkv, const HeadEpilogue& ep_qkv,
                          int K, const sched::Params* sp, unsigned* status, cudaStream_t s) {
  const int bn = layer_bn(Mc, Wkv, Mb, Wqkv, K);
  if (!bn || ep_kv.d_h != 128 || ep_qkv.d_h != 128) return cudaErrorInvalidValue;
  Plan pl;
  pl.bn = bn;
  pl.kb_total = K / BK;
  pl.kb_per_split = pl.kb_total;
  pl.splits = 1;
  Segments A;
  A.n = 1;
  A.kseg = K;
  A.p[0] = C;
  TcGemmParams p;
  cudaError_t e = fill_common(p, A, Mc, Wkv, pl, K);
  if (e != cudaSuccess) return e;
  p.ep = ep_kv;
  p.status = status;
  if (!encode_2d_bf16(&p.a1, H, Mb, K, BM)) return cudaErrorInvalidValue;
  int off = 0;
  for (int i = 0; i < Wqkv.count; ++i) {
    if (!encode_2d_bf16(&p.b1[i], Wqkv.p[i], Wqkv.n[i], K, bn)) return cudaErrorInvalidValue;
    p.w1_off[i] = off;
    off += Wqkv.n[i];
  }
  p.w1_off[Wqkv.count] = off;
  p.w1_count = Wqkv.count;
  p.M1 = Mb;
  p.ep1 = ep_qkv;
  p.ny0 = Wkv.total() / bn;
  p.ny1 = Wqkv.total() / bn;
  p.sched_cta = sp != nullptr;
  if (sp) p.sp = *sp;
  const int mt0 = (Mc + BM - 1) / BM, mt1 = (Mb + BM - 1) / BM;
  dim3 grid(mt0 > mt1 ? mt0 : mt1, p.ny0 + p.ny1 + (sp ? 1 : 0), 1);
  return bn == 256 ? launch<256, true>(p, grid, s) : launch<128, true>(p, grid, s);
}

}  // namespace dflash
