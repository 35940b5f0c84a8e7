// Tensor-core projection GEMMs for sm_103a: X W^T with bf16 inputs and an
// fp32 accumulator in tensor memory.
//
// One CTA computes a 128 x BN tile over its share of K (split-K across
// gridDim.z). When M spans more than one 128-row tile, CTAs run in clusters of
// two (tcgen05.mma.cta_group::2): the even CTA issues M = 256 MMAs whose A rows
// come 128 from each CTA's shared memory and whose B rows come half from each,
// so every SM stages and reads half the weight bytes per MMA (the one-CTA tile
// is bound by shared-memory bandwidth near two thirds of the tensor rate). Both
// CTAs' copies complete on the even CTA's full barrier; its commits arrive on
// both CTAs' empty and done barriers; each CTA's epilogue reads its own 128 TMEM
// lanes. Roles per CTA:
//   warp 0      TMA producer: 128 x 64 activation tile + BN x 64 weight tile
//               per stage, 128-byte swizzle, completion on a "full" mbarrier;
//   warp 1      allocates BN TMEM columns and issues tcgen05.mma (M=128,
//               N=BN, K=16, four per stage) from one thread; tcgen05.commit
//               frees each stage ("empty" mbarrier) and finally signals "done";
//   warps 2-5   epilogue: one thread per tile row moves the accumulator from TMEM
//               (tcgen05.ld of its lanes) into a staging tile in shared memory; then
//               the CTA's threads copy the staged rows out. With the heads epilogue
//               these warps use the mainloop's time: each resolves its row's
//               destination and copies the row's RoPE cos/sin into spare TMEM
//               columns, so the epilogue itself issues no dependent global loads.
// The activations arrive as up to eight K-segments (the k target layers'
// hidden states of the context projection), each with its own tensor map;
// the weights as up to three matrices stacked along N (W_Q | W_K | W_V).
//
// Three epilogues, leaving the staged tile by bulk copies (cp.async.bulk, one per
// contiguous destination row), so the store phase costs a few instructions per row:
//   fp32 store   the tile (a split-K partial) goes to Y; the consumer sums the splits;
//   norm         the context projection with hidden_norm fused (DFlash KV Injection
//                Walkthrough, Step 2: C = RMSNorm(fc(raw))): the last split of a tile
//                adds the others' partials (published in Y), each tile reports its rows'
//                sums of squares over its columns, and once all tiles of a 128-row block
//                have reported (all CTAs resident; bounded waits) each scales its own
//                tile by 1 / rms(row) and gamma and stores C in bf16;
//   heads        (no split-K) whole 128-dim heads per tile (BN = 128 or 256).
//                The row's thread applies the per-head RMSNorm (Q and K heads),
//                rotates the pair (i, i + 64) at the row's absolute position and
//                stages the row in its stored form (bf16, or E4M3 codes); one copy
//                per (row, head) puts it into the Q buffer or the row's cache slot
//                (DFlash KV Injection Walkthrough, Steps 4.1-4.3; DFlash source
//                guide (II), parts 1-4). Shapes that need split-K use the fp32
//                store and a separate epilogue kernel.
#include <cstdlib>
#include <mutex>

#include "attn_sched.cuh"
#include "sm100_ptx.cuh"

namespace dflash {
namespace {

constexpr int BM = 128, BK = 64;
// warps 0-5: TMA, MMA, 4 x TMEM -> shared memory; all six store in the epilogue's second
// phase (more warps there measured no faster). Heads epilogue: warps 2-9, two per TMEM lane
// quarter, each computing one of the tile's two heads.
constexpr int gemm_threads(bool heads) { return heads ? 320 : 192; }

struct TcGemmParams {
  CUtensorMap a[8];   // activation segments [M][kseg], box {64, 128}
  CUtensorMap b[3];   // weights [N_i][K], box {64, BN}
  int kseg_blocks;    // 64-wide K blocks per activation segment
  int w_count;
  int w_off[4];       // prefix offsets of the stacked weights along N
  int M, ldY;
  int kb_total, kb_per_split, splits;
  unsigned long long wait_ns;  // limit of the pipeline waits (2 s unless a test lowers it)
  float* Y;           // fp32 store: [split][M][ldY]
  HeadEpilogue ep;    // heads: norm / RoPE / destination
  unsigned* status;
  // Grouped launch (heads epilogue without split-K, or fp32 split-K partials): grid
  // columns [0, ny0) compute the problem above, columns [ny0, ny0 + ny1) a second one
  // with one activation segment (same K and K split), and with sched_cta one more column
  // whose first CTA builds the attention work list while the tiles run.
  int ny0, ny1, sched_cta;
  // Fused hidden_norm (fp32-store launches of the context projection, norm != 0): the last
  // split of each tile to finish adds the other splits' partials (published in Y) to its
  // own, reports its rows' sums of squares over its BN columns, and once every tile of its
  // 128-row block has reported, scales its tile by 1 / rms(row) and gamma into C (bf16).
  // The counters start at zero (cleared before the launch); all CTAs are co-resident.
  int norm;
  void* C;              // bf16 [M][ldY]
  const void* gamma;    // bf16 [ldY]
  float eps;
  int* tickets;         // [gx * ny] splits of a tile that have finished
  int* ready;           // [gx * ny] partials of a tile published in Y
  int* rowcnt;          // [gx] tiles of a 128-row block whose sums of squares are in
  float* rowpart;       // [M][ny] per-tile sums of squares of each row
  CUtensorMap a1;
  CUtensorMap b1[3];
  int w1_count;
  int w1_off[4];
  int M1;
  HeadEpilogue ep1;
  // grouped split-K launch (fp32 store): the second problem's partials [split][M1][ldY1]
  float* Y1;
  int ldY1;
  sched::Params sp;
};

// PAIR: the tile is computed by a cluster of two CTAs (tcgen05.mma.cta_group::2, M = 256):
// each CTA holds its own 128 rows of A and half of B's BN rows per stage.
// AR < BM (single CTAs, M <= AR): a stage holds only AR rows of A, so more stages of B
// (the weights) fit; the MMA still reads 128 rows, and rows AR .. 127 of its A operand
// are whatever follows in the stage: they reach only accumulator rows >= M, which are
// never stored (each accumulator row depends on its own A row alone).
constexpr int kSmallRows = 32;
template <int BN, bool PAIR = false, int AR = BM>
struct Cfg {
  static_assert(AR % 8 == 0 && AR <= BM && (AR == BM || !PAIR), "A rows per stage");
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;
  static constexpr uint32_t A_BYTES = AR * BK * 2;
  static constexpr uint32_t B_BYTES = B_ROWS * BK * 2;
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = AR < BM ? ((BN == 256) ? 6 : 10)
                                        : PAIR ? ((BN == 256) ? 6 : 8) : ((BN == 256) ? 4 : 6);
  // pipeline stages, barriers (256 B), then gamma_q / gamma_k as fp32 (heads epilogue)
  static constexpr uint32_t OFF_GAMMA = STAGES * STAGE + 256;
  static constexpr size_t SMEM = 1024 + (size_t)OFF_GAMMA + 2 * 128 * 4;
  // epilogue staging tile over the stages: BM rows of BN fp32, padded, then row slots
  static constexpr int LD = BN + 4;
  static constexpr uint32_t STG_BYTES = BM * LD * 4;
  // heads: the finished rows in their stored form, 256 bytes per head (bf16, or E4M3 codes
  // with Q's remainder codes in the second half), rows 16 bytes apart from the bank pattern
  static constexpr uint32_t RSB = 2 * BN + 16;
  static_assert(BM * RSB <= STG_BYTES, "byte staging exceeds the fp32 staging area");
  static_assert(STG_BYTES + BM * 16 <= STAGES * STAGE, "staging tile exceeds the stages");
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

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits (bounded, like the pipeline waits) until *p >= target, where other CTAs of the same
// launch raise *p after publishing data (release); false when it gave up.
__device__ __forceinline__ bool spin_geq(const int* p, int target, unsigned* status,
                                         uint64_t limit_ns) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (ld_acquire(p) < target) {
    if (ptx::globaltimer() - t0 > limit_ns) {
      atomicOr(status, DFLASH_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// Sixteen finished values (dims d0 .. d0 + 15 of one head) into the head's 256-byte slot
// of the byte staging row: bf16 at 2 d0; E4M3 K / V codes of v * inv at d0; Q as codes at
// d0 and remainder codes at 128 + d0.
__device__ __forceinline__ void put16(uint8_t* slot, int d0, const float (&v)[16], bool fp8, bool q,
                                      float inv) {
  if (!fp8) {
    uint4 w0, w1;
    w0.x = pack_bf16(v[0], v[1]);
    w0.y = pack_bf16(v[2], v[3]);
    w0.z = pack_bf16(v[4], v[5]);
    w0.w = pack_bf16(v[6], v[7]);
    w1.x = pack_bf16(v[8], v[9]);
    w1.y = pack_bf16(v[10], v[11]);
    w1.z = pack_bf16(v[12], v[13]);
    w1.w = pack_bf16(v[14], v[15]);
    reinterpret_cast<uint4*>(slot + 2 * d0)[0] = w0;
    reinterpret_cast<uint4*>(slot + 2 * d0)[1] = w1;
  } else if (q) {
    uint4 hi, lo;
    e4m3x4_split(v[0], v[1], v[2], v[3], hi.x, lo.x);
    e4m3x4_split(v[4], v[5], v[6], v[7], hi.y, lo.y);
    e4m3x4_split(v[8], v[9], v[10], v[11], hi.z, lo.z);
    e4m3x4_split(v[12], v[13], v[14], v[15], hi.w, lo.w);
    *reinterpret_cast<uint4*>(slot + d0) = hi;
    *reinterpret_cast<uint4*>(slot + 128 + d0) = lo;
  } else {
    uint4 c;
    c.x = e4m3x4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
    c.y = e4m3x4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
    c.z = e4m3x4(v[8] * inv, v[9] * inv, v[10] * inv, v[11] * inv);
    c.w = e4m3x4(v[12] * inv, v[13] * inv, v[14] * inv, v[15] * inv);
    *reinterpret_cast<uint4*>(slot + d0) = c;
  }
}

// Sequence, index and position of projection row `row`, or pos = -1 when the row is
// not written (malformed cu_rows, or the sequence's rows do not fit the cache or the RoPE
// table). Status bits as the per-head epilogue kernels set them; `first_tile` marks the
// tile holding head 0, so each refused sequence is flagged once.
struct RowSlot {
  int b, t, pos, page;  // page: the slot's page of a paged cache, else -1
};
__device__ __forceinline__ RowSlot row_slot(const HeadEpilogue& e, int row, bool first_tile) {
  RowSlot rs{0, 0, -1, -1};
  int n_b;
  if (e.cu_rows) {
    int lo = 0, hi = e.batch - 1;
    while (lo < hi) {  // last b with cu_rows[b] <= row
      const int mid = (lo + hi + 1) >> 1;
      if (e.cu_rows[mid] <= row) lo = mid; else hi = mid - 1;
    }
    rs.b = lo;
    rs.t = row - e.cu_rows[lo];
    n_b = e.cu_rows[lo + 1] - e.cu_rows[lo];
    if (n_b < 0 || e.cu_rows[lo + 1] > e.rows || e.cu_rows[0] != 0 || rs.t < 0 || rs.t >= n_b) {
      atomicOr(e.status, DFLASH_DEV_ROWS);
      return rs;
    }
  } else {
    rs.b = row / e.bs;
    rs.t = row - rs.b * e.bs;
    n_b = e.bs;
  }
  int start = e.lens[rs.b];
  start += sched::injected_rows(e.pre_rows, e.pre_M, rs.b, start, e.capacity, e.table_len);
  if (start < 0 || start + n_b > e.capacity || start + n_b > e.table_len) {
    if (rs.t == 0 && first_tile)
      atomicOr(e.status, (start + n_b > e.capacity || start < 0) ? DFLASH_DEV_CAPACITY
                                                                 : DFLASH_DEV_ROPE);
    return rs;
  }
  rs.pos = start + rs.t;
  if (e.block_table) rs.page = e.block_table[(size_t)rs.b * e.pages_per_seq + (rs.pos >> 7)];
  return rs;
}

// The epilogue parameters of a CTA's problem, copied into registers field by field: each
// read stays a constant-bank access (a reference chosen at run time between the two
// parameter structs would turn every later field read into a generic memory load).
__device__ __forceinline__ HeadEpilogue pick_epilogue(const TcGemmParams& p, bool second) {
  HeadEpilogue e;
#define DFLASH_PICK(f) e.f = second ? p.ep1.f : p.ep.f
  DFLASH_PICK(Y);
  DFLASH_PICK(splits);
  DFLASH_PICK(rows);
  DFLASH_PICK(ldY);
  DFLASH_PICK(n_q);
  DFLASH_PICK(n_kv);
  DFLASH_PICK(d_h);
  DFLASH_PICK(eps);
  DFLASH_PICK(gamma_q);
  DFLASH_PICK(gamma_k);
  DFLASH_PICK(rope);
  DFLASH_PICK(table_len);
  DFLASH_PICK(cu_rows);
  DFLASH_PICK(batch);
  DFLASH_PICK(bs);
  DFLASH_PICK(lens);
  DFLASH_PICK(q_out);
  DFLASH_PICK(cache_k);
  DFLASH_PICK(cache_v);
  DFLASH_PICK(capacity);
  DFLASH_PICK(status);
  DFLASH_PICK(pre_rows);
  DFLASH_PICK(pre_M);
  DFLASH_PICK(block_table);
  DFLASH_PICK(pages_per_seq);
  DFLASH_PICK(kv_fp8);
  DFLASH_PICK(k_inv);
  DFLASH_PICK(v_inv);
  DFLASH_PICK(q_lo);
#undef DFLASH_PICK
  return e;
}

// Attention CTA c starts with the work list's item c (each CTA's first item has a slot of
// its own); this CTA (one of the grouped launch's GEMM CTAs) prefetches the first two K and
// V tiles of items L, L + nG, ... of those into L2, if the list is complete (its builder
// sets the flag with release order). Items are checked against the cache bounds first.
__device__ __noinline__ void prefetch_first_wave(const TcGemmParams& p) {
  const int* ready = p.sp.ready;
  if (!ready || ld_acquire(ready) != 1) return;
  const HeadEpilogue& e = p.ep;
  const int pairs = p.sp.batch * p.sp.n_kv;
  // the first item of each attention CTA (a workspace never written before may hold a stale
  // flag: each item is checked before use)
  const int wave = p.sp.n_sm;
  const int nG = (int)gridDim.x * (p.ny0 + p.ny1);
  const int rowbytes = e.kv_fp8 ? 128 : 256;
  for (int j = (int)blockIdx.y * (int)gridDim.x + (int)blockIdx.x; j < wave; j += nG) {
    const int4 it = p.sp.items[j];
    if (it.x < 0 || it.x >= pairs || it.y < 0 || it.z <= it.y || it.z > e.capacity) continue;
    const int b = it.x / p.sp.n_kv, kvh = it.x - b * p.sp.n_kv;
    int keys = min(it.z - it.y, 256);
    long long row;
    if (e.block_table) {
      const int page = e.block_table[(size_t)b * e.pages_per_seq + (it.y >> 7)];
      keys = min(keys, 128 - (it.y & 127));
      row = ((long long)page * e.n_kv + kvh) * 128 + (it.y & 127);
    } else {
      row = ((long long)b * e.n_kv + kvh) * e.capacity + it.y;
    }
    const uint32_t bytes = (uint32_t)keys * rowbytes;
    const char* k = (const char*)e.cache_k + row * rowbytes;
    const char* v = (const char*)e.cache_v + row * rowbytes;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(k), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(v), "r"(bytes) : "memory");
  }
}

// Phase 2 of a fused-norm launch, run by all threads of the CTA with the fp32 tile in the
// staging area (rows BN + 4 floats apart) and gamma of its columns in `gam`. Every thread
// reaches every barrier below whatever the outcome of a wait (decisions go through s_flag).
template <int BN, bool PAIR>
__device__ __forceinline__ void norm_epilogue(const TcGemmParams& p, float* stg, const float* gam,
                                              int m0, int n0, int M, volatile int* abort_flag,
                                              volatile int* s_role, volatile int* s_flag) {
  using C = Cfg<BN, PAIR>;
  constexpr int kT = gemm_threads(false);
  constexpr int Q4 = BN / 4;  // float4 groups of a row
  const int tid = threadIdx.x;
  const int ny = (int)gridDim.y, splits = (int)gridDim.z, z = (int)blockIdx.z;
  const int tile = (int)blockIdx.x * ny + (int)blockIdx.y;
  const int N = p.ldY;
  // 1) the last split of the tile to get here finishes it; the others publish their partial
  if (tid == 0) {
    int last = 1;
    if (*abort_flag) {
      last = -1;
    } else if (splits > 1) {
      const int t = atomicAdd(&p.tickets[tile], 1);
      last = t == splits - 1;
    }
    *s_role = last;
  }
  ptx::named_sync(1, kT);
  const int role = *s_role;
  if (role < 0) return;
  if (role == 0) {
    float* y = p.Y + (size_t)z * M * N + n0;
    for (int u = tid; u < BM * Q4; u += kT) {
      const int r = u / Q4, c = u - r * Q4;
      if (m0 + r < M)
        reinterpret_cast<float4*>(y + (size_t)(m0 + r) * N)[c] =
            *reinterpret_cast<const float4*>(stg + r * C::LD + 4 * c);
    }
    __threadfence();
    ptx::named_sync(1, kT);
    if (tid == 0) {  // after every thread's stores and fences
      __threadfence();
      atomicAdd(&p.ready[tile], 1);
    }
    return;
  }
  // 2) last split: add the other splits' partials (in L2) to the tile
  if (splits > 1) {
    if (tid == 0) *s_flag = spin_geq(&p.ready[tile], splits - 1, p.status, p.wait_ns) ? 1 : 0;
    ptx::named_sync(1, kT);
    if (!*s_flag) {
      if (tid == 0) *abort_flag = 1;
      return;
    }
    // the splits in index order, this CTA's own from shared memory: the sum does not
    // depend on which split finished last. Each thread keeps U float4 loads of a split in
    // flight (L2 latency, not bandwidth, bounds this step).
    constexpr int U = 16;
    for (int u0 = tid; u0 < BM * Q4; u0 += U * kT) {
      float4 v[U];
#pragma unroll
      for (int k = 0; k < U; ++k) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < splits; ++s) {
        float4 a[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int u = u0 + k * kT, r = u / Q4, c = u - r * Q4;
          a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (u < BM * Q4 && m0 + r < M)
            a[k] = s == z ? *reinterpret_cast<const float4*>(stg + r * C::LD + 4 * c)
                          : __ldcg(reinterpret_cast<const float4*>(
                                       p.Y + (size_t)s * M * N + n0 + (size_t)(m0 + r) * N) + c);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
          v[k].x += a[k].x;
          v[k].y += a[k].y;
          v[k].z += a[k].z;
          v[k].w += a[k].w;
        }
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int u = u0 + k * kT, r = u / Q4, c = u - r * Q4;
        if (u < BM * Q4 && m0 + r < M) *reinterpret_cast<float4*>(stg + r * C::LD + 4 * c) = v[k];
      }
    }
    ptx::named_sync(1, kT);
  }
  // 3) each row's sum of squares over this tile's columns, then wait for the row block
  if (tid < BM && m0 + tid < M) {
    const float4* r4 = reinterpret_cast<const float4*>(stg + tid * C::LD);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int c = 0; c < Q4; ++c) {
      const float4 v = r4[c];
      a0 = fmaf(v.x, v.x, a0);
      a1 = fmaf(v.y, v.y, a1);
      a2 = fmaf(v.z, v.z, a2);
      a3 = fmaf(v.w, v.w, a3);
    }
    p.rowpart[(size_t)(m0 + tid) * ny + blockIdx.y] = (a0 + a1) + (a2 + a3);
  }
  __threadfence();
  ptx::named_sync(1, kT);
  if (tid == 0) {
    __threadfence();
    atomicAdd(&p.rowcnt[blockIdx.x], 1);
    *s_flag = spin_geq(&p.rowcnt[blockIdx.x], ny, p.status, p.wait_ns) ? 1 : 0;
  }
  ptx::named_sync(1, kT);
  if (!*s_flag) {
    if (tid == 0) *abort_flag = 1;
    return;
  }
  // 4) C = x / sqrt(mean(x^2) + eps) * gamma, in bf16, written over the row's first half
  if (tid < BM && m0 + tid < M) {
    const float* pr = p.rowpart + (size_t)(m0 + tid) * ny;
    float ss = 0.f;
    for (int j0 = 0; j0 < ny; j0 += 16) {  // 16 loads in flight, summed in a fixed order
      float t[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) t[j] = j0 + j < ny ? __ldcg(pr + j0 + j) : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) ss += t[j];
    }
    const float rn = 1.0f / sqrtf(ss / (float)N + p.eps);
    float* row = stg + tid * C::LD;
    uint4* out = reinterpret_cast<uint4*>(row);
#pragma unroll 4
    for (int c = 0; c < BN / 8; ++c) {  // 8 values in, 16 bytes out, out never ahead of in
      const float4 v0 = reinterpret_cast<const float4*>(row)[2 * c];
      const float4 v1 = reinterpret_cast<const float4*>(row)[2 * c + 1];
      const float* g = gam + 8 * c;
      uint4 w;
      w.x = pack_bf16(v0.x * rn * g[0], v0.y * rn * g[1]);
      w.y = pack_bf16(v0.z * rn * g[2], v0.w * rn * g[3]);
      w.z = pack_bf16(v1.x * rn * g[4], v1.y * rn * g[5]);
      w.w = pack_bf16(v1.z * rn * g[6], v1.w * rn * g[7]);
      out[c] = w;
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::named_sync(1, kT);
  bf16* cb = reinterpret_cast<bf16*>(p.C) + n0;
  for (int r = tid; r < BM && m0 + r < M; r += kT)
    ptx::bulk_store(cb + (size_t)(m0 + r) * N, ptx::smem_u32(stg + r * C::LD), BN * 2);
  ptx::bulk_commit_wait_all();
}

template <int BN, bool HEADS, bool PAIR, int AR = BM>
__global__ void __launch_bounds__(gemm_threads(HEADS), 1) gemm_tc_kernel(const __grid_constant__ TcGemmParams p) {
  constexpr int kThreads = gemm_threads(HEADS);
  using C = Cfg<BN, PAIR, AR>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + (size_t)STAGES * C::STAGE);
  constexpr int NH = BN >= 128 ? BN / 128 : 1;                // heads per tile (heads epilogue)
  float* stg = reinterpret_cast<float*>(smem);                // epilogue only
  int4* slots = reinterpret_cast<int4*>(smem + C::STG_BYTES);  // epilogue only
  float* gam = reinterpret_cast<float*>(smem + C::OFF_GAMMA);   // heads: gamma_q, gamma_k
  // TMEM: the accumulator in columns [0, BN); heads: the row's RoPE (cos, sin) pairs in
  // [BN, BN + 128)
  constexpr uint32_t TMEM_COLS = HEADS ? 2 * BN : BN;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int s_role, s_flag;  // fused norm: decisions of thread 0 broadcast to the CTA

  // problem of this CTA (grouped launches); whole CTAs branch, before any barrier
  const int col = (int)blockIdx.y;
  if (p.sched_cta && col == p.ny0 + p.ny1) {
    if (blockIdx.x == 0 && blockIdx.z == 0) sched::build(p.sp);
    return;
  }
  const bool second = p.ny1 > 0 && col >= p.ny0;
  const CUtensorMap* amap = second ? &p.a1 : p.a;
  const CUtensorMap* bmap = second ? p.b1 : p.b;
  int w_off[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w_off[i] = second ? p.w1_off[i] : p.w_off[i];
  const int w_count = second ? p.w1_count : p.w_count;
  const int M = second ? p.M1 : p.M;
  const int kseg_blocks = second ? p.kb_total : p.kseg_blocks;
  const HeadEpilogue ep = pick_epilogue(p, second);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM, n0 = (second ? col - p.ny0 : col) * BN;
  // grid.x covers the taller problem. A pair leaves only as a whole (both CTAs take the
  // same branch), since each waits for the other below; a pair's odd CTA may hold no rows
  // of M (its A tile is zero fill, its epilogue stores nothing).
  if ((PAIR ? (int)(blockIdx.x & ~1u) * BM : m0) >= M) return;
  // PAIR: CTA 0 of the cluster issues the MMAs; CTA 1 loads its halves and runs its epilogue
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0;
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
  // PAIR: both CTAs' barriers are initialised before either CTA's copies or commits can
  // reach the other's: every thread arrives at the cluster barrier now and waits for it
  // after the TMEM allocation
  if (PAIR) {
    __syncwarp();  // the arrive is a warp-aligned instruction
    ptx::cluster_arrive();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < (second ? 1 : 8); ++i) ptx::prefetch_tmap(&amap[i]);
    for (int i = 0; i < w_count; ++i) ptx::prefetch_tmap(&bmap[i]);
  }
  if (warp == 1) {
    if (PAIR) {
      // collective with the peer CTA's warp 1: the same columns in both CTAs' TMEM
      ptx::tmem_alloc_pair(ptx::smem_u32(&tmem_slot), TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_wait();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  int wi = 0;
  while (wi + 1 < w_count && n0 >= w_off[wi + 1]) ++wi;
  const int nb = n0 - w_off[wi];

  if (warp == 0) {
    if (lane == 0) {
      // PAIR: both CTAs' copies complete on CTA 0's full barrier, which CTA 0 arms for the
      // bytes of both; CTA 1 loads the second half of the B tile
      const uint32_t brow = nb + rank * C::B_ROWS;
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (i >= STAGES && !ptx::mbar_wait(empty0 + 8 * s, ph ^ 1, &abort_flag, p.status, p.wait_ns)) break;
        const int kb = kb0 + i;
        const int seg = kb / kseg_blocks;
        const int kx = (kb - seg * kseg_blocks) * BK;
        const uint32_t sa = ptx::smem_u32(smem + (size_t)s * C::STAGE);
        if (!PAIR) {
          ptx::mbar_arrive_expect_tx(full0 + 8 * s, C::STAGE);
          ptx::tma_load_2d(sa, &amap[seg], full0 + 8 * s, kx, m0);
          ptx::tma_load_2d(sa + C::A_BYTES, &bmap[wi], full0 + 8 * s, kb * BK, nb);
        } else {
          if (rank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, 2 * C::STAGE);
          const uint32_t fb = ptx::mapa_shared(full0 + 8 * s, 0);
          ptx::tma_load_2d_pair(sa, &amap[seg], fb, kx, m0);
          ptx::tma_load_2d_pair(sa + C::A_BYTES, &bmap[wi], fb, kb * BK, brow);
        }
        ++issued;
      }
      // grouped launch: once its work-list CTA has finished, ask L2 for the first K and V
      // tiles of some of the attention's first-wave items (the attention's CTAs would
      // otherwise all request them from HBM at once); never waits for the list
      if (HEADS && p.sched_cta) prefetch_first_wave(p);
      // no copy of ours may still be landing when the CTA exits: CTA 0 (and a single CTA)
      // waits for its last stages to fill; CTA 1, whose copies count on CTA 0's barriers,
      // waits until the MMAs have released its last stages (they read them, so they landed)
      for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i) {
        if (rank == 0)
          drain_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1, p.status);
        else
          drain_wait(empty0 + 8 * (i % STAGES), (i / STAGES) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!ptx::mbar_wait(full0 + 8 * s, ph, &abort_flag, p.status, p.wait_ns)) break;
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + (size_t)s * C::STAGE);
        const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          if (PAIR)
            ptx::mma_bf16_pair(tmem, ptx::smem_desc_sw128(sa + 32 * k),
                               ptx::smem_desc_sw128(sb + 32 * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
          else
            ptx::mma_bf16(tmem, ptx::smem_desc_sw128(sa + 32 * k), ptx::smem_desc_sw128(sb + 32 * k),
                          idesc, (i > 0 || k > 0) ? 1u : 0u);
        }
        if (PAIR)
          ptx::mma_commit_pair(empty0 + 8 * s, 3);  // frees stage s in both CTAs
        else
          ptx::mma_commit(empty0 + 8 * s);
      }
      if (PAIR)
        ptx::mma_commit_pair(done, 3);
      else
        ptx::mma_commit(done);
      drain_wait(done, 0, p.status);  // every MMA has finished before TMEM can be freed
    }
  } else {
    // phase 1: TMEM -> a staging tile in the pipeline's shared memory (free once every
    // MMA is done), one row per thread. fp32 store: the accumulator row, rows padded by 4
    // floats so the float4 stores of a warp spread over all banks. heads: the finished
    // row in its stored form, in the byte tile (rows 2 BN + 16 bytes apart).
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 are this warp's
    const int eset = (warp - 2) >> 2;  // heads: warps 2-5 are set 0, warps 6-9 set 1
    const int row = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float* srow = stg + row * C::LD;
    RowSlot rs{0, 0, -1, -1};
    if (!HEADS && p.norm) {
      // while the MMAs run: gamma of the tile's columns, as fp32
      for (int c = threadIdx.x - 64; c < BN; c += 128)
        gam[c] = __bfloat162float(((const bf16*)p.gamma)[n0 + c]);
    }
    if (HEADS) {
      // while the MMAs run: the row's destination, gamma, and the row's RoPE pairs
      // (cos, sin of its position, 128 floats) into TMEM columns BN .. BN + 127
      // (set 0; set 1 only computes heads)
      if (eset == 0 && m0 + row < M) rs = row_slot(ep, m0 + row, n0 == 0);
      const int et = threadIdx.x - 64;  // 0 .. 127 in set 0
      if (eset == 0) {
        gam[et] = ep.gamma_q ? __bfloat162float(((const bf16*)ep.gamma_q)[et]) : 1.f;
        gam[128 + et] = ep.gamma_k ? __bfloat162float(((const bf16*)ep.gamma_k)[et]) : 1.f;
      }
      const bool ropes = n0 / 128 < ep.n_q + ep.n_kv;  // the tile's first head is a Q or K head
      __syncwarp();  // row_slot's search diverges; tcgen05.st is .sync.aligned
      if (ropes && eset == 0) {
        // the table is 8-byte aligned: float2 loads; rows that are not written (no
        // position, e.g. a table too short or empty) stage zeros and read nothing
        const bool has = rs.pos >= 0;
        const float2* cs = ep.rope + (size_t)(has ? rs.pos : 0) * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 f = has ? cs[c * 16 + j] : make_float2(0.f, 0.f);
            v[2 * j] = __float_as_uint(f.x);
            v[2 * j + 1] = __float_as_uint(f.y);
          }
          ptx::tmem_st_32x32b_x32(tmem + lane_base + (uint32_t)(BN + 32 * c), v);
        }
        ptx::tmem_st_wait();
      }
      ptx::named_sync(2, 256);  // gamma and RoPE pairs staged by set 0, for both sets
    }
    // warp-uniform: tcgen05.ld below is a .sync.aligned instruction
    // (the epilogue warps wait for the whole mainloop: suspended, off the issue slots of
    // the producer and the MMA issuer)
    const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_idle(done, 0, &abort_flag, p.status, p.wait_ns));
    ptx::tc_fence_after();
    if (ok && !HEADS) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(c * 32), r);
        ptx::tmem_ld_wait();
        float4* d = reinterpret_cast<float4*>(srow + c * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          d[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                             __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      }
    } else if (ok) {
      // the finished row: per-head RMSNorm (Q, K heads: sum of squares over the head's
      // 128 dims, then x / rms * gamma) and rotate_half RoPE on the pairs (i, i + 64);
      // V heads as they are; each head's 256-byte slot of the byte tile gets the values in
      // the form the destination stores (put16)
      if (eset == 0) slots[row] = make_int4(rs.b, rs.t, rs.pos, rs.page);
#pragma unroll 1
      for (int hd = eset; hd < NH; hd += 2) {
        const int head = n0 / 128 + hd;
        const int kind = head < ep.n_q ? 0 : (head < ep.n_q + ep.n_kv ? 1 : 2);  // Q, K, V
        const uint32_t hcol = (uint32_t)(hd * 128);
        uint8_t* hslot = smem + row * C::RSB + hd * 256;
        if (kind == 2) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + hcol + (uint32_t)(c * 32), r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float v[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[16 * hh + e]);
              put16(hslot, 32 * c + 16 * hh, v, ep.kv_fp8, false, ep.v_inv);
            }
          }
          continue;
        }
        float ssq = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_base + hcol + (uint32_t)(c * 32), r);
          ptx::tmem_ld_wait();
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            a0 = fmaf(__uint_as_float(r[j]), __uint_as_float(r[j]), a0);
            a1 = fmaf(__uint_as_float(r[j + 1]), __uint_as_float(r[j + 1]), a1);
            a2 = fmaf(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 2]), a2);
            a3 = fmaf(__uint_as_float(r[j + 3]), __uint_as_float(r[j + 3]), a3);
          }
          ssq += (a0 + a1) + (a2 + a3);
        }
        const float rn = 1.0f / sqrtf(ssq * (1.0f / 128.f) + ep.eps);
        const float* g = gam + (kind == 0 ? 0 : 128);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          // dims i = 32c + e and their partners i + 64, with the pairs' (cos, sin)
          uint32_t xa[32], xb[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_base + hcol + (uint32_t)(c * 32), xa);
          ptx::tmem_ld_32x32b_x32(tmem + lane_base + hcol + (uint32_t)(64 + c * 32), xb);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t cs[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(BN + 64 * c + 32 * hh), cs);
            ptx::tmem_ld_wait();
            float ya[16], yb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int i = 32 * c + 16 * hh + e;
              const float a = __uint_as_float(xa[16 * hh + e]) * rn * g[i];
              const float b = __uint_as_float(xb[16 * hh + e]) * rn * g[i + 64];
              const float co = __uint_as_float(cs[2 * e]), si = __uint_as_float(cs[2 * e + 1]);
              ya[e] = a * co - b * si;
              yb[e] = b * co + a * si;
            }
            put16(hslot, 32 * c + 16 * hh, ya, ep.kv_fp8, kind == 0, ep.k_inv);
            put16(hslot, 64 + 32 * c + 16 * hh, yb, ep.kv_fp8, kind == 0, ep.k_inv);
          }
        }
      }
    }
  }
  if (warp >= 2) ptx::fence_proxy_async_smem();  // staged rows leave by bulk copy
  // phase 2, all warps: bulk copies from the staging tile
  ptx::named_sync(1, kThreads);
  if (!HEADS && p.norm) {
    norm_epilogue<BN, PAIR>(p, stg, gam, m0, n0, M, &abort_flag, &s_role, &s_flag);
  } else if (!abort_flag) {
    if (!HEADS) {
      // fp32 partial rows, one contiguous copy each
      const int ldY = second ? p.ldY1 : p.ldY;
      float* ybase = (second ? p.Y1 : p.Y) + (size_t)blockIdx.z * M * ldY + n0;
      for (int r = threadIdx.x; r < BM && m0 + r < M; r += kThreads)
        ptx::bulk_store(ybase + (size_t)(m0 + r) * ldY, ptx::smem_u32(stg + r * C::LD), BN * 4);
    } else {
      // one copy per (row, head): the row's Q row, or its cache slot (bf16: 256 bytes;
      // E4M3: 128 bytes of codes, and for Q 128 bytes of remainder codes)
      for (int u = threadIdx.x; u < BM * NH; u += kThreads) {
        const int r = u / NH, hd = u - r * NH;
        const int4 rs = slots[r];
        if (rs.z < 0 || m0 + r >= M) continue;
        const int head = n0 / 128 + hd;
        const int kind = head < ep.n_q ? 0 : (head < ep.n_q + ep.n_kv ? 1 : 2);  // Q, K, V
        const bool qh = kind == 0;
        const int kvh = head - ep.n_q - (kind == 2 ? ep.n_kv : 0);
        // element offset of the destination row (Q, or the cache slot)
        const size_t eoff =
            qh ? (((size_t)rs.x * ep.n_q + head) * ep.bs + rs.y) * 128
               : (rs.w >= 0 ? ((size_t)rs.w * ep.n_kv + kvh) * 128 + (rs.z & 127)
                            : ((size_t)rs.x * ep.n_kv + kvh) * ep.capacity + rs.z) * 128;
        char* dbase = (char*)(qh ? ep.q_out : (kind == 1 ? ep.cache_k : ep.cache_v));
        const uint32_t src = ptx::smem_u32(smem + r * C::RSB + hd * 256);
        if (!ep.kv_fp8) {
          ptx::bulk_store(dbase + eoff * 2, src, 256);
        } else {
          ptx::bulk_store(dbase + eoff, src, 128);
          if (qh) ptx::bulk_store((char*)ep.q_lo + eoff, src + 128, 128);
        }
      }
    }
    ptx::bulk_commit_wait_read();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // PAIR: neither CTA leaves (or frees TMEM) while the other may still read its shared
  // memory through the MMAs or receive its commits; every path of both CTAs reaches this
  if (PAIR) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR)
      ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem, TMEM_COLS);
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
  bool pair;  // CTA pairs (M = 256 per MMA) instead of single CTAs
  int gx;     // grid.x: CTAs along M (even with pairs)
};

// CTA pairs halve the shared-memory operand bytes per SM (each CTA reads its own 128 rows
// of A and half of B) once M spans more than one 128-row tile; DFLASH_PAIR_GEMM=0 keeps
// single-CTA tiles everywhere (the same arithmetic).
bool pair_wanted(int M) {
  const char* env = getenv("DFLASH_PAIR_GEMM");
  if (env && env[0] == '0') return false;
  return M > BM;
}

int grid_x(int M, bool pair) {
  const int mt = (M + BM - 1) / BM;
  return pair ? (mt + 1) & ~1 : mt;
}

// The widest of 256/128/64 that divides every stacked weight (heads: 256 or
// 128, whole heads per tile). Split-K to about one wave on the GPU.
Plan plan(int M, const Weights& W, int K, bool heads, int split_cap = 0) {
  Plan pl;
  pl.bn = 256;
  for (int i = 0; i < W.count; ++i)
    while (W.n[i] % pl.bn) pl.bn >>= 1;
  if (heads && pl.bn < 128) pl.bn = 0;  // heads need whole 128-dim heads per tile
  if (pl.bn == 0) return pl;
  pl.pair = pl.bn >= 128 && pair_wanted(M);
  pl.gx = grid_x(M, pl.pair);
  pl.kb_total = K / BK;
  const int tiles = pl.gx * (W.total() / pl.bn);
  int splits = 148 / (tiles > 0 ? tiles : 1);
  const int max_splits = pl.kb_total / 4 > 0 ? pl.kb_total / 4 : 1;
  if (splits > max_splits) splits = max_splits;
  if (split_cap > 0 && splits > split_cap) splits = split_cap;
  if (splits < 1) splits = 1;
  pl.kb_per_split = (pl.kb_total + splits - 1) / splits;
  pl.splits = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  // heads: where 256-wide tiles need split-K (fp32 partials and a separate epilogue kernel)
  // but 128-wide ones fill most of the GPU in one pass, take the 128-wide ones, whose fused
  // heads epilogue writes the rows directly (the 1024-row K/V prefill: 33.6 -> 30.3 us for
  // GEMM + epilogue; DFLASH_HEADS_NARROW=0 keeps the split)
  const char* narrow = getenv("DFLASH_HEADS_NARROW");
  if (heads && pl.bn == 256 && pl.splits > 1 && split_cap == 0 && !(narrow && narrow[0] == '0')) {
    const int tiles128 = pl.gx * (W.total() / 128);
    if (tiles128 >= 96 && tiles128 <= 148) {
      pl.bn = 128;
      pl.kb_per_split = pl.kb_total;
      pl.splits = 1;
    }
  }
  return pl;
}

template <int BN, bool HEADS, bool PAIR, int AR = BM>
cudaError_t launch_one(const TcGemmParams& p, dim3 grid, cudaStream_t s) {
  const size_t smem = Cfg<BN, PAIR, AR>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, HEADS, PAIR, AR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  LaunchScope ls_(DFLASH_KERNEL_GEMM, s);
  if constexpr (!PAIR) {
    gemm_tc_kernel<BN, HEADS, false, AR><<<grid, gemm_threads(HEADS), smem, s>>>(p);
    return cudaGetLastError();
  } else {
    if (grid.x & 1) return cudaErrorInvalidValue;  // whole pairs only
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(gemm_threads(HEADS), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, HEADS, true>, p);
  }
}

// small: fp32-store launches whose rows fit kSmallRows (one row tile, single CTAs), with
// activation maps of kSmallRows-row boxes; anything else is refused, since the stage byte
// count the copies are awaited for follows the box
template <int BN, bool HEADS>
cudaError_t launch(const TcGemmParams& p, dim3 grid, bool pair, cudaStream_t s, bool small = false) {
  if (small) {
    if constexpr (!HEADS) {
      if (!pair && grid.x == 1) return launch_one<BN, false, false, kSmallRows>(p, grid, s);
    }
    return cudaErrorInvalidValue;
  }
  return pair ? launch_one<BN, HEADS, true>(p, grid, s) : launch_one<BN, HEADS, false>(p, grid, s);
}

// Whether an fp32-store launch of M rows (and M1 for a grouped one) takes the small-A
// stages; DFLASH_SMALL_A=0 keeps the 128-row stages (the same arithmetic).
bool small_rows(const Plan& pl, int M, int M1 = 0) {
  const char* env = getenv("DFLASH_SMALL_A");
  if (env && env[0] == '0') return false;
  return !pl.pair && pl.bn >= 128 && M <= kSmallRows && M1 <= kSmallRows;
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

// byte matrix [rows][128], box {128 bytes, box_rows rows}, 128-byte swizzle, zero fill.
bool encode_2d_u8(CUtensorMap* m, const void* base, long long rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_tc_splits(int M, const Weights& W, int K, int split_cap) {
  return plan(M, W, K, false, split_cap).splits;
}

bool gemm_tc_heads_ok(int M, const Weights& W, int K) {
  const Plan pl = plan(M, W, K, true);
  return pl.bn >= 128 && pl.splits == 1;
}

namespace {

cudaError_t fill_common(TcGemmParams& p, const Segments& A, int M, const Weights& W, const Plan& pl,
                        int K, int a_rows = BM) {
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < A.n; ++i)
    if (!encode_2d_bf16(&p.a[i], A.p[i], M, A.kseg, a_rows)) return cudaErrorInvalidValue;
  for (int i = A.n; i < 8; ++i) p.a[i] = p.a[0];
  int off = 0;
  for (int i = 0; i < W.count; ++i) {
    if (!encode_2d_bf16(&p.b[i], W.p[i], W.n[i], K, pl.pair ? pl.bn / 2 : pl.bn))
      return cudaErrorInvalidValue;
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
  p.wait_ns = wait_limit_ns();
  return cudaSuccess;
}

}  // namespace

cudaError_t gemm_tc(const Segments& A, int M, const Weights& W, float* Y, int ldY,
                    unsigned* status, cudaStream_t s, int split_cap) {
  const int N = W.total();
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int K = A.n * A.kseg;
  const Plan pl = plan(M, W, K, false, split_cap);
  if (pl.bn < 64 || A.kseg % BK) return cudaErrorInvalidValue;
  const bool small = small_rows(pl, M);
  TcGemmParams p;
  cudaError_t e = fill_common(p, A, M, W, pl, K, small ? kSmallRows : BM);
  if (e != cudaSuccess) return e;
  p.ldY = ldY;
  p.Y = Y;
  p.status = status;
  dim3 grid(pl.gx, N / pl.bn, pl.splits);
  switch (pl.bn) {
    case 256: return launch<256, false>(p, grid, pl.pair, s, small);
    case 128: return launch<128, false>(p, grid, pl.pair, s, small);
    default: return launch_one<64, false, false>(p, grid, s);
  }
}

// Can every CTA of a launch of `pl` over N columns be resident at once (so CTAs may wait
// for one another)? One CTA per SM (the shared memory of a stage ring); pairs also need two
// SMs of one cluster slot.
namespace {
template <int BN, bool PAIR>
int max_resident_ctas() {
  const size_t smem = Cfg<BN, PAIR>::SMEM;
  if (cudaFuncSetAttribute(gemm_tc_kernel<BN, false, PAIR>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(gemm_threads(false), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_kernel<BN, false, true>, &cfg) !=
        cudaSuccess)
      return 0;
    return 2 * clusters;
  } else {
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_tc_kernel<BN, false, false>,
                                                      gemm_threads(false), smem) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    return per_sm * sms;
  }
}

int resident_ctas(const Plan& pl) {
  static std::mutex mu;
  static int cache[128][2][2];  // [device][bn == 256][pair], 0 = not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& v = cache[dev][pl.bn == 256][pl.pair];
  if (!v) {
    if (pl.bn == 256)
      v = pl.pair ? max_resident_ctas<256, true>() : max_resident_ctas<256, false>();
    else
      v = pl.pair ? max_resident_ctas<128, true>() : max_resident_ctas<128, false>();
    if (!v) v = -1;
  }
  return v;
}
}  // namespace

// The fused norm measured slower than the separate pass at every shape tried (the wait for
// the last tile of a row block puts the slowest CTA's reduction on the critical path), so it
// runs only when DFLASH_FUSED_NORM=1 asks for it.
bool gemm_tc_norm_ok(int M, const Weights& W, int K, int split_cap) {
  const Plan pl = plan(M, W, K, false, split_cap);
  if (pl.bn < 128 || W.count != 1 || K % BK) return false;
  const char* env = getenv("DFLASH_FUSED_NORM");
  if (!(env && env[0] == '1')) return false;
  const long long ctas = (long long)pl.gx * (W.total() / pl.bn) * pl.splits;
  return ctas <= resident_ctas(pl);
}

int gemm_tc_norm_counters(int M, const Weights& W, int K, int split_cap) {
  const Plan pl = plan(M, W, K, false, split_cap);
  const int ny = pl.bn > 0 ? W.total() / pl.bn : 0;
  return 2 * pl.gx * ny + pl.gx;
}

int gemm_tc_norm_tiles_n(int M, const Weights& W, int K) {
  const Plan pl = plan(M, W, K, false);
  return pl.bn > 0 ? W.total() / pl.bn : 0;
}

cudaError_t gemm_tc_norm(const Segments& A, int M, const Weights& W, float* Y, float* rowpart,
                         int* counters, const void* gamma, float eps, void* C, unsigned* status,
                         cudaStream_t s, int split_cap) {
  const int N = W.total();
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int K = A.n * A.kseg;
  const Plan pl = plan(M, W, K, false, split_cap);
  if (pl.bn < 128 || A.kseg % BK) return cudaErrorInvalidValue;
  TcGemmParams p;
  cudaError_t e = fill_common(p, A, M, W, pl, K);
  if (e != cudaSuccess) return e;
  const int ny = N / pl.bn;
  p.ldY = N;
  p.Y = Y;
  p.status = status;
  p.norm = 1;
  p.C = C;
  p.gamma = gamma;
  p.eps = eps;
  p.tickets = counters;
  p.ready = counters + pl.gx * ny;
  p.rowcnt = counters + 2 * pl.gx * ny;
  p.rowpart = rowpart;
  e = cudaMemsetAsync(counters, 0, sizeof(int) * (size_t)(2 * pl.gx * ny + pl.gx), s);
  if (e != cudaSuccess) return e;
  dim3 grid(pl.gx, ny, pl.splits);
  return pl.bn == 256 ? launch<256, false>(p, grid, pl.pair, s) : launch<128, false>(p, grid, pl.pair, s);
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
  dim3 grid(pl.gx, N / pl.bn, 1);
  return pl.bn == 256 ? launch<256, true>(p, grid, pl.pair, s)
                      : launch<128, true>(p, grid, pl.pair, s);
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
  // DFLASH_FUSED_LAYER=0 never groups, =1 groups whenever the shapes allow, =2 takes the
  // split-K grouping wherever it applies (all the same arithmetic); otherwise group when
  // the tiles fill a good part of the GPU
  const char* env = getenv("DFLASH_FUSED_LAYER");
  if (env && (env[0] == '0' || env[0] == '2')) return 0;
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
  // one instantiation serves both problems: pairs when both span more than one M tile and
  // the launch fits one wave of resident pairs (with two waves, as for 64 sequences, the
  // pairs measured slower here: 97.6 against 92.5 us per grouped launch)
  pl.pair = pair_wanted(Mc) && pair_wanted(Mb);
  if (pl.pair) {
    Plan pp = pl;
    const long long ctas = (long long)(grid_x(Mc, true) > grid_x(Mb, true) ? grid_x(Mc, true)
                                                                          : grid_x(Mb, true)) *
                           (Wkv.total() / bn + Wqkv.total() / bn);
    if (ctas > resident_ctas(pp)) pl.pair = false;
  }
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
    if (!encode_2d_bf16(&p.b1[i], Wqkv.p[i], Wqkv.n[i], K, pl.pair ? bn / 2 : bn))
      return cudaErrorInvalidValue;
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
  const int mt0 = grid_x(Mc, pl.pair), mt1 = grid_x(Mb, pl.pair);
  dim3 grid(mt0 > mt1 ? mt0 : mt1, p.ny0 + p.ny1 + (sp ? 1 : 0), 1);
  return bn == 256 ? launch<256, true>(p, grid, pl.pair, s) : launch<128, true>(p, grid, pl.pair, s);
}

// Both projections of a draft layer in one split-K launch, for batches whose tiles fill
// too little of the GPU to run without split-K (a few sequences): the two problems share
// one K split, each writes fp32 partials [split][M][N] that one per-head epilogue launch
// finishes, and (sp != null) one extra CTA builds the attention work list. The plan
// depends on the block rows alone; the context rows must fit the block's row tiles.
namespace {
bool layer_split_plan(int Mb, const Weights& Wkv, const Weights& Wqkv, int K, Plan* out) {
  if (Mb <= 0 || K % BK) return false;
  const char* env = getenv("DFLASH_FUSED_LAYER");
  if (env && env[0] == '0') return false;
  Plan pl;
  pl.bn = 256;
  for (int i = 0; i < Wkv.count; ++i)
    while (Wkv.n[i] % pl.bn) pl.bn >>= 1;
  for (int i = 0; i < Wqkv.count; ++i)
    while (Wqkv.n[i] % pl.bn) pl.bn >>= 1;
  if (pl.bn < 128) return false;
  pl.pair = pair_wanted(Mb);
  pl.gx = grid_x(Mb, pl.pair);
  pl.kb_total = K / BK;
  const int tiles = pl.gx * (Wkv.total() / pl.bn + Wqkv.total() / pl.bn);
  int splits = 148 / tiles;
  const int max_splits = pl.kb_total / 4 > 0 ? pl.kb_total / 4 : 1;
  if (splits > max_splits) splits = max_splits;
  if (splits < 2) return false;  // one pass fills the GPU: the fused-epilogue launches
  pl.kb_per_split = (pl.kb_total + splits - 1) / splits;
  pl.splits = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  *out = pl;
  return true;
}
}  // namespace

int gemm_tc_layer_split_splits(int Mb, const Weights& Wkv, const Weights& Wqkv, int K) {
  Plan pl;
  return layer_split_plan(Mb, Wkv, Wqkv, K, &pl) ? pl.splits : 0;
}

int gemm_tc_layer_split_rows(int Mb, const Weights& Wkv, const Weights& Wqkv, int K) {
  Plan pl;
  return layer_split_plan(Mb, Wkv, Wqkv, K, &pl) ? pl.gx * BM : 0;
}

cudaError_t gemm_tc_layer_split(const void* C, int Mc, const Weights& Wkv, float* Y0,
                                const void* H, int Mb, const Weights& Wqkv, float* Y1, int K,
                                const sched::Params* sp, unsigned* status, cudaStream_t s) {
  Plan pl;
  if (Mc <= 0 || !layer_split_plan(Mb, Wkv, Wqkv, K, &pl) || grid_x(Mc, pl.pair) > pl.gx)
    return cudaErrorInvalidValue;
  Segments A;
  A.n = 1;
  A.kseg = K;
  A.p[0] = C;
  const bool small = small_rows(pl, Mc, Mb);
  const int a_rows = small ? kSmallRows : BM;
  TcGemmParams p;
  cudaError_t e = fill_common(p, A, Mc, Wkv, pl, K, a_rows);
  if (e != cudaSuccess) return e;
  p.Y = Y0;
  p.ldY = Wkv.total();
  p.status = status;
  if (!encode_2d_bf16(&p.a1, H, Mb, K, a_rows)) return cudaErrorInvalidValue;
  int off = 0;
  for (int i = 0; i < Wqkv.count; ++i) {
    if (!encode_2d_bf16(&p.b1[i], Wqkv.p[i], Wqkv.n[i], K, pl.pair ? pl.bn / 2 : pl.bn))
      return cudaErrorInvalidValue;
    p.w1_off[i] = off;
    off += Wqkv.n[i];
  }
  p.w1_off[Wqkv.count] = off;
  p.w1_count = Wqkv.count;
  p.M1 = Mb;
  p.Y1 = Y1;
  p.ldY1 = Wqkv.total();
  p.ny0 = Wkv.total() / pl.bn;
  p.ny1 = Wqkv.total() / pl.bn;
  p.sched_cta = sp != nullptr;
  if (sp) p.sp = *sp;
  dim3 grid(pl.gx, p.ny0 + p.ny1 + (sp ? 1 : 0), pl.splits);
  return pl.bn == 256 ? launch<256, false>(p, grid, pl.pair, s, small)
                      : launch<128, false>(p, grid, pl.pair, s, small);
}

}  // namespace dflash
